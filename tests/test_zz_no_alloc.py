"""The no-allocation entry point, attn_bwd_noalloc, on the GPU.

Some callers cannot call cudaMalloc: code inside a framework hook that must
not re-enter the framework's allocator, deployments whose device memory is
fixed at start-up, or paths that must not stall other streams. For them the
library keeps its workspace in a fixed device array. This test calls that
entry point through the C ABI twice in a row (the second call runs on the
array's stale contents from the first) and checks each result against the
regular attn_bwd_preprocess + attn_bwd path, and against the float64 oracle,
with the parity tolerance of the other tests. It lives in its own file,
collected last.
"""

import numpy as np
import pytest

import harness as H
from workloads import make_dense

pytestmark = pytest.mark.gpu


def _noalloc_run(ab, torch, plan):
    """Same problem as `plan`, through attn_bwd_noalloc into fresh outputs."""
    dq = torch.full_like(plan.dq, float("nan"))
    dk = torch.full_like(plan.dk, float("nan"))
    dv = torch.full_like(plan.dv, float("nan"))
    delta = torch.full_like(plan.delta, float("nan"))
    dbias = None if plan.dbias is None else torch.full_like(plan.dbias, float("nan"))
    code, detail = ab.attn_bwd_noalloc(plan.prob, plan.mask, None, plan.q, plan.k, plan.v, plan.o,
                                       plan.do, plan.lse, plan.bias, delta, dq, dk, dv, dbias,
                                       read_status=True)
    assert code == 0, (code, detail)
    return dict(dq=dq, dk=dk, dv=dv, delta=delta, dbias=dbias)


CASES = [
    # GQA 4:1 causal at D = 128 (tensor-core path)
    lambda: make_dense("na1", 51, B=1, Hq=8, Hk=2, Sq=512, Sk=512, D=128, window_left=-1,
                       window_right=0),
    # ALiBi bias + dbias at D = 64 (tensor-core path, different workspace layout)
    lambda: make_dense("na2", 52, B=2, Hq=2, Hk=2, Sq=256, Sk=256, D=64, alibi=True,
                       want_dbias=True),
]


@pytest.mark.parametrize("first,second", [(0, 1), (1, 0), (0, 0)])
def test_noalloc_matches_regular_path_twice(first, second):
    import torch
    import attention_backward_attn_gb300 as ab
    for idx in (first, second):
        w = CASES[idx]()
        O_b, L_f, _, _ = H.dense_forward_inputs(w)
        plan = H.gpu_dense_plan(w, O_b, L_f)
        plan.run()
        got = _noalloc_run(ab, torch, plan)
        torch.cuda.synchronize()
        assert plan.device_status()[0] == 0
        names = ("dq", "dk", "dv", "delta") + (("dbias",) if w.want_dbias else ())
        for name in names:
            ref = getattr(plan, name).cpu().numpy()
            H.check_close(name, got[name].cpu().numpy(), ref)
        oracle_ref = H.dense_reference(w, O_b, L_f)
        for name in names:
            H.check_close(name, got[name].cpu().numpy(), oracle_ref[name])


def test_noalloc_rejects_problems_beyond_its_workspace():
    import ctypes
    import torch
    import attention_backward_attn_gb300 as ab
    # D = 128, B*Hq*Sq = 2^17 rows: the fp16 staging alone is 64 MiB > 32 MiB
    B, S, Hq, Hk, D = 1, 8192, 16, 4, 128
    q = torch.empty((B, S, Hq, D), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((B, S, Hk, D), dtype=torch.bfloat16, device="cuda")
    prob = ab.problem_from(q, k, k, q, q, D ** -0.5)
    assert ab.attn_bwd_workspace_size(prob) > (32 << 20)
    code = ab.lib.attn_bwd_noalloc(ctypes.byref(prob), None, None, q.data_ptr(), k.data_ptr(),
                                   k.data_ptr(), q.data_ptr(), q.data_ptr(), 1 << 20, None,
                                   1 << 20, 1 << 20, 1 << 20, 1 << 20, None, None, None)
    assert code == 7  # ATTN_ERR_WORKSPACE, nothing enqueued
