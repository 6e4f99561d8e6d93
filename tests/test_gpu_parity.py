"""GPU parity: the CUDA backward (through the C ABI) against the float64 oracle.

Small cases compare every element; they span several 128-row tiles and a
ragged tail. Full-size cases run the exact launch the benchmark times and
compare complete head groups (dense) or every output (sparse).
"""

import numpy as np
import pytest

import harness as H
import oracle
from workloads import make_workload, make_dense, make_sparse, make_varlen

pytestmark = pytest.mark.gpu


def _torch():
    import torch
    return torch


def _run_dense(w, expect_path=None):
    # path 2 (the SIMT kernels) runs only when the problem asks for it
    torch = _torch()
    O_b, L_f, _, _ = H.dense_forward_inputs(w)
    plan = H.gpu_dense_plan(w, O_b, L_f, cuda_cores=expect_path == 2)
    if expect_path is not None:
        assert plan.path == expect_path
    plan.run()
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    assert code == 0, (code, detail)
    return plan, O_b, L_f


def _compare_dense(w, plan, O_b, L_f, batches=None, kv_heads=None):
    ref = H.dense_reference(w, O_b, L_f, batches, kv_heads)
    r = w.Hq // w.Hk
    bs = batches if batches is not None else slice(0, w.B)
    ks = kv_heads if kv_heads is not None else slice(0, w.Hk)
    qs = slice(ks.start * r, ks.stop * r)
    H.check_close("dq", plan.dq.cpu().numpy()[bs][:, :, qs], ref["dq"])
    H.check_close("dk", plan.dk.cpu().numpy()[bs][:, :, ks], ref["dk"])
    H.check_close("dv", plan.dv.cpu().numpy()[bs][:, :, ks], ref["dv"])
    delta = plan.delta.cpu().numpy()[bs][:, qs]
    np.testing.assert_allclose(delta, ref["delta"], rtol=1e-5, atol=1e-5 * np.abs(ref["delta"]).max())
    if w.want_dbias:
        assert batches is None
        H.check_close("dbias", plan.dbias.cpu().numpy()[qs], ref["dbias"])


SMALL_DENSE = {
    # the exact 64-token MHA workload
    "mha_s64_d64": lambda: make_workload("mha_s64_d64"),
    # GQA 4:1 causal, 3 query tiles
    "gqa4_causal_s384_d128": lambda: make_workload("gqa4_causal_s1024_d128", Hq=8, Hk=2,
                                                   Sq=384, Sk=384),
    # ALiBi bias + dbias, D = 64
    "alibi_dbias_s256_d64": lambda: make_workload("mha_alibi_dbias_s2048_d64", B=3, Hq=4,
                                                  Hk=4, Sq=256, Sk=256),
    # window 128 + 4 sinks, GQA 4:1
    "window128_sink4_s640_d128": lambda: make_workload("gqa4_window1024_sink4_s8192_d128",
                                                       Hq=8, Hk=2, Sq=640, Sk=640,
                                                       window_left=127),
    # ragged lengths (not a multiple of the tile), causal + sinks, D = 64
    "ragged_causal_sink_s200_d64": lambda: make_dense("r", 21, B=2, Hq=4, Hk=2, Sq=200,
                                                      Sk=200, D=64, window_left=-1,
                                                      window_right=0, num_sink=3),
    # Sq != Sk, GQA 8:1, no mask
    "gqa8_sq128_sk320_d128": lambda: make_dense("x", 22, B=1, Hq=8, Hk=1, Sq=128, Sk=320,
                                                D=128),
    # dbias in the batch-inner query-major CTAs with a mask that leaves whole
    # tiles dead (zeroed first) and cuts others (per-element mask), GQA 2:1,
    # four batches (the most those CTAs take)
    "window_sinks_alibi_dbias_s512_d64": lambda: make_dense("qb", 29, B=4, Hq=4, Hk=2, Sq=512,
                                                            Sk=512, D=64, window_left=150,
                                                            window_right=0, num_sink=3,
                                                            alibi=True, want_dbias=True),
    # Sq > Sk, two-sided window, bias without dbias request
    "window_lr_sq320_sk192_d64": lambda: make_dense("y", 23, B=2, Hq=2, Hk=1, Sq=320, Sk=192,
                                                    D=64, window_left=40, window_right=25,
                                                    alibi=True),
    # bottom-right causal, Sq < Sk (tensor-core path), GQA 4:1
    "br_causal_sq128_sk384_d128": lambda: make_dense("br1", 27, B=1, Hq=8, Hk=2, Sq=128,
                                                     Sk=384, D=128, window_left=-1,
                                                     window_right=0, bottom_right=True),
    # bottom-right causal, Sq > Sk: the first 256 queries have no key
    "br_causal_sq384_sk128_d64": lambda: make_dense("br2", 28, B=2, Hq=4, Hk=4, Sq=384,
                                                    Sk=128, D=64, window_left=-1,
                                                    window_right=0, bottom_right=True),
    # bottom-right window + sinks, ragged lengths, bias
    "br_window_sink_sq150_sk230_d64": lambda: make_dense("br3", 29, B=1, Hq=4, Hk=2, Sq=150,
                                                         Sk=230, D=64, window_left=31,
                                                         window_right=0, num_sink=3,
                                                         alibi=True, bottom_right=True),
    # MHA D = 512 through the dense path
    "mha_s128_d512": lambda: make_dense("z", 24, B=1, Hq=2, Hk=2, Sq=128, Sk=128, D=512,
                                        window_left=-1, window_right=0),
    # bias at D = 128: window + sinks on ragged lengths (bias rows clamped past
    # Sk, partial tiles), and whole tiles without a mask (16-byte bias loads)
    "bias_window_sinks_s300_d128": lambda: make_dense("fb1", 47, B=2, Hq=4, Hk=2, Sq=300,
                                                      Sk=300, D=128, window_left=90,
                                                      window_right=0, num_sink=2,
                                                      alibi=True),
    "bias_gqa2_s256_d128": lambda: make_dense("fb2", 48, B=1, Hq=4, Hk=2, Sq=256, Sk=256,
                                              D=128, alibi=True),
}


def _dense_path(w):
    """The tcgen05 kernel takes every dense problem with D in {64, 128}, of any
    lengths (a ragged last tile is masked per element); the SIMT kernels the
    rest, when the problem asks for them (ATTN_FLAG_CUDA_CORES)."""
    return 1 if w.D in (64, 128) else 2


@pytest.mark.parametrize("name", list(SMALL_DENSE))
def test_dense_small(name):
    w = SMALL_DENSE[name]()
    plan, O_b, L_f = _run_dense(w, expect_path=_dense_path(w))
    _compare_dense(w, plan, O_b, L_f)


@pytest.mark.parametrize("name", list(SMALL_DENSE))
def test_dense_small_cuda_cores(name):
    # the same cases through the SIMT kernels (ATTN_FLAG_CUDA_CORES)
    torch = _torch()
    w = SMALL_DENSE[name]()
    O_b, L_f, _, _ = H.dense_forward_inputs(w)
    plan = H.gpu_dense_plan(w, O_b, L_f, cuda_cores=True)
    assert plan.path == 2
    plan.run()
    torch.cuda.synchronize()
    assert plan.device_status()[0] == 0
    _compare_dense(w, plan, O_b, L_f)


# Lengths that are not whole 128-row tiles on the tensor-core path: the staged
# fp16 copies are zero past each length and the last query / key tile takes
# the per-element mask.
RAGGED_TC = {
    # GQA 4:1 causal, both lengths ragged, D = 128
    "gqa4_causal_sq200_sk200_d128": lambda: make_dense("rg1", 60, B=2, Hq=8, Hk=2, Sq=200,
                                                       Sk=200, D=128, window_left=-1,
                                                       window_right=0),
    # bias + dbias with a key length that is not a multiple of 4 (scalar bias
    # reads), Sq < Sk
    "alibi_dbias_sq130_sk250_d64": lambda: make_dense("rg2", 61, B=2, Hq=2, Hk=2, Sq=130,
                                                      Sk=250, D=64, alibi=True,
                                                      want_dbias=True),
    # bias with Sk a multiple of 4 (vector bias reads on whole key tiles), a
    # two-sided window and sinks, Sq > Sk
    "window_sinks_bias_sq300_sk260_d64": lambda: make_dense("rg3", 62, B=1, Hq=2, Hk=1,
                                                            Sq=300, Sk=260, D=64,
                                                            window_left=70, window_right=9,
                                                            num_sink=2, alibi=True),
    # one query against 5 keys (a single key would make dS = P (dP - D)
    # vanish identically: exact zeros the fp16 operands do not reproduce)
    "single_query_sk5_d128": lambda: make_dense("rg4", 63, B=1, Hq=2, Hk=1, Sq=1, Sk=5, D=128),
    # 5 queries at the end of 700 keys: bottom-right causal with sinks
    "br_sink_sq5_sk700_d64": lambda: make_dense("rg5", 64, B=1, Hq=4, Hk=2, Sq=5, Sk=700,
                                                D=64, window_left=-1, window_right=0,
                                                num_sink=4, bottom_right=True),
    # GQA 8:1 on one ragged key tile: the query heads are split over CTAs whose
    # partial dK / dV rows are added (rows past Sk are not)
    "gqa8_split_sq96_sk100_d128": lambda: make_dense("rg6", 65, B=1, Hq=8, Hk=1, Sq=96,
                                                     Sk=100, D=128, want_dbias=True),
}


@pytest.mark.parametrize("name", list(RAGGED_TC))
def test_ragged_tensor_core(name):
    w = RAGGED_TC[name]()
    plan, O_b, L_f = _run_dense(w, expect_path=1)
    _compare_dense(w, plan, O_b, L_f)


TC_EXTRA = {
    # one tile, no mask: the plain five-GEMM pipeline
    "mha_s128_d128": lambda: make_dense("a", 40, B=1, Hq=1, Hk=1, Sq=128, Sk=128, D=128),
    "mha_s128_d64": lambda: make_dense("b", 41, B=1, Hq=1, Hk=1, Sq=128, Sk=128, D=64),
    # Sq != Sk and GQA 8:1 (several query tiles per key tile, group sum on chip)
    "gqa8_sq256_sk512_d128": lambda: make_dense("c", 42, B=2, Hq=8, Hk=1, Sq=256, Sk=512,
                                                D=128),
    # causal + 3 sinks + two-sided window at D = 64, with bias but no dbias
    "window_sinks_bias_s512_d64": lambda: make_dense("d", 43, B=1, Hq=2, Hk=2, Sq=512, Sk=512,
                                                     D=64, window_left=150, window_right=20,
                                                     num_sink=3, alibi=True),
    # dbias without bias (gradient of a zero bias), GQA 2:1
    "dbias_only_gqa2_s256_d128": lambda: make_dense("e", 44, B=2, Hq=4, Hk=2, Sq=256, Sk=256,
                                                    D=128, want_dbias=True),
    # rows with no live key inside a partial tile, and a fully empty query tile
    # (Sq > Sk, window of 11 keys: rows i >= 138 see nothing)
    "empty_rows_sq384_sk128_d64": lambda: make_dense("f", 45, B=1, Hq=2, Hk=1, Sq=384, Sk=128,
                                                     D=64, window_left=10, window_right=0),
}


@pytest.mark.parametrize("name", list(TC_EXTRA))
def test_tensor_core_cases(name):
    w = TC_EXTRA[name]()
    plan, O_b, L_f = _run_dense(w, expect_path=1)
    _compare_dense(w, plan, O_b, L_f)


# Variable-length batches (packed token-major rows, cu_seqlens): every
# sequence is its own problem, masks align per sequence.
VARLEN = {
    # GQA 4:1 causal, D = 128: an empty query sequence, ragged and aligned lengths
    "gqa4_causal_mixed_d128": lambda: make_varlen("vl1", 70, [100, 0, 300, 257],
                                                  [100, 64, 300, 257], Hq=8, Hk=2, D=128,
                                                  window_left=-1, window_right=0),
    # bottom-right causal per sequence with ALiBi bias and dbias, D = 64; Sq < Sk,
    # Sq = Sk, a single query against 129 keys
    "br_alibi_dbias_d64": lambda: make_varlen("vl2", 71, [130, 64, 1], [200, 64, 129], Hq=2,
                                              Hk=2, D=64, window_left=-1, window_right=0,
                                              bottom_right=True, alibi=True, want_dbias=True),
    # GQA 8:1 window + sinks, a sequence without keys, max lengths above every length
    "window_sinks_gqa8_d128": lambda: make_varlen("vl3", 72, [384, 5, 200, 30], [384, 700, 90, 0],
                                                  Hq=8, Hk=1, D=128, window_left=60,
                                                  window_right=3, num_sink=2, max_q=400,
                                                  max_k=720),
}


@pytest.mark.parametrize("name", list(VARLEN))
def test_varlen(name):
    torch = _torch()
    w = VARLEN[name]()
    O_b, L_f = H.varlen_forward_inputs(w)
    plan = H.gpu_varlen_plan(w, O_b, L_f)
    assert plan.path == 1
    plan.run()
    torch.cuda.synchronize()
    assert plan.device_status()[0] == 0
    ref = H.varlen_reference(w, O_b, L_f)
    H.check_close("dq", plan.dq.cpu().numpy(), ref["dq"])
    H.check_close("dk", plan.dk.cpu().numpy(), ref["dk"])
    H.check_close("dv", plan.dv.cpu().numpy(), ref["dv"])
    if w.want_dbias:
        H.check_close("dbias", plan.dbias.cpu().numpy(), ref["dbias"])
    delta = plan.delta.cpu().numpy()
    for b in range(w.B):
        n = int(w.cu_q[b + 1] - w.cu_q[b])
        rows = slice(int(w.cu_q[b]), int(w.cu_q[b + 1]))
        want = (O_b[rows].astype(np.float64) * w.do[rows].astype(np.float64)).sum(-1).T
        np.testing.assert_allclose(delta[b, :, :n], want, rtol=1e-5,
                                   atol=1e-5 * max(1.0, np.abs(want).max(initial=0.0)))


def test_varlen_deterministic_dbias():
    # per-sequence dbias slices summed in sequence order: bitwise repeatable
    torch = _torch()
    w = VARLEN["br_alibi_dbias_d64"]()
    O_b, L_f = H.varlen_forward_inputs(w)
    plan = H.gpu_varlen_plan(w, O_b, L_f, deterministic=True)
    outs = []
    for _ in range(2):
        plan.run()
        torch.cuda.synchronize()
        assert plan.device_status()[0] == 0
        outs.append(plan.dbias.clone())
    assert torch.equal(outs[0], outs[1])
    ref = H.varlen_reference(w, O_b, L_f)
    H.check_close("dbias", plan.dbias.cpu().numpy(), ref["dbias"])
    H.check_close("dq", plan.dq.cpu().numpy(), ref["dq"])


def test_varlen_equal_lengths_match_the_fixed_length_run():
    # the same three sequences as a padded batch and as a packed one: the
    # same tiles in the same order, so bitwise-equal gradients (deterministic
    # mode, so that no partial sums are added in arrival order)
    torch = _torch()
    w = make_dense("ve", 73, B=3, Hq=4, Hk=1, Sq=200, Sk=200, D=128, window_left=-1,
                   window_right=0)
    O_b, L_f, _, _ = H.dense_forward_inputs(w)
    dense = H.gpu_dense_plan(w, O_b, L_f, deterministic=True)
    dense.run()
    pack = lambda x: np.ascontiguousarray(x.reshape(-1, *x.shape[2:]))
    v = make_varlen("ve", 73, [200] * 3, [200] * 3, Hq=4, Hk=1, D=128, window_left=-1,
                    window_right=0)
    v.q, v.k, v.v, v.do = pack(w.q), pack(w.k), pack(w.v), pack(w.do)
    var = H.gpu_varlen_plan(v, pack(O_b), L_f, deterministic=True)
    var.run()
    torch.cuda.synchronize()
    assert dense.device_status()[0] == 0 and var.device_status()[0] == 0
    for a, b in ((dense.dq, var.dq), (dense.dk, var.dk), (dense.dv, var.dv)):
        assert torch.equal(a.reshape(b.shape), b)


def test_varlen_bad_bounds_are_reported():
    # decreasing bounds for sequence 1 (the others stay valid): it is skipped
    # and recorded (detail 1)
    torch = _torch()
    w = VARLEN["gqa4_causal_mixed_d128"]()
    O_b, L_f = H.varlen_forward_inputs(w)
    plan = H.gpu_varlen_plan(w, O_b, L_f)
    plan._keep[0].copy_(torch.tensor([0, 100, 90, 390, 647], dtype=torch.int32))
    plan.run()
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    assert code == 1 and detail == 1


# Deterministic mode (ATTN_FLAG_DETERMINISTIC): bitwise-identical outputs over
# repeated runs, and the usual oracle parity.
DETERMINISTIC = {
    # dbias over 3 batches on the tensor-core path: per-batch slices summed in order
    "alibi_dbias_s256_d64": (lambda: SMALL_DENSE["alibi_dbias_s256_d64"](), 1),
    # GQA 8:1 on two key tiles: by default each query head of a key tile gets its
    # own CTA and the 8 partial dK / dV sums are added in arrival order
    "gqa8_s256_d128": (lambda: make_dense("det", 25, B=1, Hq=8, Hk=1, Sq=256, Sk=256, D=128,
                                          window_left=-1, window_right=0), 1),
    # ragged lengths (staged copies padded to whole tiles), dbias over 3 batches
    "ragged_alibi_dbias_s200_d64": (lambda: make_dense("detr", 26, B=3, Hq=2, Hk=2, Sq=200,
                                                       Sk=200, D=64, alibi=True,
                                                       want_dbias=True), 1),
    # the same on the SIMT kernels (ATTN_FLAG_CUDA_CORES): per-batch dbias slices too
    "simt_alibi_dbias_s200_d64": (lambda: make_dense("dets", 27, B=3, Hq=2, Hk=2, Sq=200,
                                                     Sk=200, D=64, alibi=True,
                                                     want_dbias=True), 2),
}


@pytest.mark.parametrize("name", list(DETERMINISTIC))
def test_deterministic_mode(name):
    torch = _torch()
    make, path = DETERMINISTIC[name]
    w = make()
    O_b, L_f, _, _ = H.dense_forward_inputs(w)
    plan = H.gpu_dense_plan(w, O_b, L_f, deterministic=True, cuda_cores=(path == 2))
    assert plan.path == path
    runs = []
    for _ in range(3):
        plan.run()
        torch.cuda.synchronize()
        code, detail = plan.device_status()
        assert code == 0, (code, detail)
        outs = [plan.dq, plan.dk, plan.dv] + ([plan.dbias] if w.want_dbias else [])
        runs.append([t.cpu().numpy().copy() for t in outs])
    for later in runs[1:]:
        for a, b in zip(runs[0], later):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    _compare_dense(w, plan, O_b, L_f)


def test_deterministic_dbias_graph_replay_full_size():
    # per-batch dbias slices summed in batch order, captured in a CUDA graph
    # and replayed as the benchmark does: every replay gives the same bits
    torch = _torch()
    w = make_workload("mha_alibi_dbias_s2048_d64")
    up = lambda x: torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda().to(torch.bfloat16)
    import attention_backward_attn_gb300 as ab
    q, k, v, do = (up(x) for x in (w.q, w.k, w.v, w.do))
    bias = torch.from_numpy(w.bias).cuda()
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device="cuda")
    ab.attn_fwd_lse(ab.problem_from(q, k, v, o, do, w.scale), None, None, q, k, v, bias, o, lse)
    plan = ab.BackwardPlan(q, k, v, o, do, lse, w.scale, bias=bias, want_dbias=True,
                           deterministic=True)
    assert plan.path == 1
    plan.run()
    torch.cuda.synchronize()
    assert plan.device_status()[0] == 0
    ref = [t.clone() for t in (plan.dq, plan.dk, plan.dbias)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        plan.run()
    for _ in range(5):
        g.replay()
        torch.cuda.synchronize()
        assert plan.device_status()[0] == 0
        for a, b in zip(ref, (plan.dq, plan.dk, plan.dbias)):
            assert torch.equal(a, b)
    # and the replayed result is the oracle's, on heads 0 and 15 (all batches)
    O_b = o.float().cpu().numpy()
    L_f = lse.cpu().numpy()
    heads = [0, w.Hq - 1]
    bh = lambda x: H.bhsd(x[:, :, heads])
    dQ, dK, dV, dB = oracle.backward(bh(w.q), bh(w.k), bh(w.v), bh(O_b), bh(w.do),
                                     L_f[:, heads].astype(np.float64), w.scale, None,
                                     w.bias[heads].astype(np.float64))
    t = lambda x: x.transpose(0, 2, 1, 3)
    H.check_close("dq", plan.dq.cpu().numpy()[:, :, heads], t(dQ))
    H.check_close("dk", plan.dk.cpu().numpy()[:, :, heads], t(dK))
    H.check_close("dv", plan.dv.cpu().numpy()[:, :, heads], t(dV))
    H.check_close("dbias", plan.dbias.cpu().numpy()[heads], dB)


def test_batch_inner_outputs_only_16_byte_aligned():
    # The API asks dq and dbias to be 16-byte aligned only; the batch-inner
    # dbias CTAs store 32 bytes at a time where the address allows it and
    # 16 bytes where it does not. Buffers that start 16 bytes past a 32-byte
    # boundary must give the same bits as the regular ones.
    torch = _torch()
    import attention_backward_attn_gb300 as ab
    w = SMALL_DENSE["alibi_dbias_s256_d64"]()
    O_b, L_f, _, _ = H.dense_forward_inputs(w)
    plan = H.gpu_dense_plan(w, O_b, L_f)
    assert plan.path == 1
    plan.run()
    torch.cuda.synchronize()
    assert plan.device_status()[0] == 0

    def shifted_like(t):
        big = torch.full((t.numel() + 8,), float("nan"), dtype=t.dtype, device=t.device)
        assert big.data_ptr() % 32 == 0
        v = big[4:4 + t.numel()].view(t.shape)
        assert v.data_ptr() % 32 == 16
        return v

    dq16, db16 = shifted_like(plan.dq), shifted_like(plan.dbias)
    ab.attn_bwd_preprocess(plan.prob, plan.sparse, plan.q, plan.k, plan.v, plan.o, plan.do,
                           plan.delta, db16, plan.dk, plan.dv, plan.workspace, plan.ws_bytes)
    ab.attn_bwd(plan.prob, plan.mask, plan.sparse, plan.q, plan.k, plan.v, plan.do, plan.lse,
                plan.delta, plan.bias, dq16, plan.dk, plan.dv, db16, plan.workspace,
                plan.ws_bytes)
    torch.cuda.synchronize()
    assert plan.device_status()[0] == 0
    assert torch.equal(dq16, plan.dq)
    assert torch.equal(db16, plan.dbias)


def test_head_split_needs_the_prepared_dk_dv():
    # GQA 8:1 on a small problem splits each key tile's query heads over
    # several CTAs that add partial sums into dk / dv; the pre-pass zeroes the
    # buffers it was given, so attn_bwd with other buffers must refuse them
    torch = _torch()
    import attention_backward_attn_gb300 as ab
    w = TC_EXTRA["gqa8_sq256_sk512_d128"]()
    O_b, L_f, _, _ = H.dense_forward_inputs(w)
    plan = H.gpu_dense_plan(w, O_b, L_f)
    assert plan.path == 1
    other_dk = torch.full_like(plan.dk, float("nan"))
    ab.attn_bwd_preprocess(plan.prob, plan.sparse, plan.q, plan.k, plan.v, plan.o, plan.do,
                           plan.delta, plan.dbias, plan.dk, plan.dv, plan.workspace,
                           plan.ws_bytes)
    ab.attn_bwd(plan.prob, plan.mask, plan.sparse, plan.q, plan.k, plan.v, plan.do, plan.lse,
                plan.delta, plan.bias, plan.dq, other_dk, plan.dv, plan.dbias, plan.workspace,
                plan.ws_bytes)
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    assert code == 1 and detail == 3
    assert torch.isnan(other_dk).all()  # left unwritten
    # the regular pairing still works afterwards
    plan.run()
    torch.cuda.synchronize()
    assert plan.device_status()[0] == 0
    _compare_dense(w, plan, O_b, L_f)


def test_fully_masked_rows_and_empty_query():
    # keys live only for rows 0..7 (window_right = -1 .. left 3 at Sk = 8): rows
    # beyond see nothing -> LSE = -inf, zero gradients.
    w = make_dense("m", 25, B=1, Hq=2, Hk=1, Sq=136, Sk=8, D=64, window_left=3,
                   window_right=0)
    plan, O_b, L_f = _run_dense(w)
    assert np.all(np.isneginf(L_f[:, :, 12:]))
    _compare_dense(w, plan, O_b, L_f)
    # Sq = 0: nothing to differentiate; dK, dV must come back as exact zeros.
    torch = _torch()
    import attention_backward_attn_gb300 as ab
    B, Sk, Hq, Hk, D = 1, 64, 2, 1, 64
    q = torch.empty((B, 0, Hq, D), dtype=torch.bfloat16, device="cuda")
    k = torch.randn((B, Sk, Hk, D), device="cuda").to(torch.bfloat16)
    lse = torch.empty((B, Hq, 0), dtype=torch.float32, device="cuda")
    plan = ab.BackwardPlan(q, k, k.clone(), q, q, lse, D ** -0.5)
    plan.dk.fill_(1.0)
    plan.dv.fill_(1.0)
    plan.run()
    torch.cuda.synchronize()
    assert float(plan.dk.abs().max()) == 0.0 and float(plan.dv.abs().max()) == 0.0


FORWARD_CASES = ["window128_sink4_s640_d128", "alibi_dbias_s256_d64", "mha_s64_d64",
                 "ragged_causal_sink_s200_d64", "gqa8_sq128_sk320_d128",
                 "window_lr_sq320_sk192_d64", "br_causal_sq384_sk128_d64",
                 "br_window_sink_sq150_sk230_d64", "gqa4_causal_s384_d128",
                 "bias_window_sinks_s300_d128", "bias_gqa2_s256_d128"]


@pytest.mark.parametrize("cuda_cores", [False, True])
@pytest.mark.parametrize("name", FORWARD_CASES)
def test_forward_matches_oracle(name, cuda_cores):
    # the tensor-core forward (bf16 operands, P rounded to bf16) and the SIMT
    # forward (fp32 throughout) against the float64 oracle forward
    torch = _torch()
    import attention_backward_attn_gb300 as ab
    w = SMALL_DENSE[name]()
    O_b, L_f, O, L = H.dense_forward_inputs(w)
    q, k, v = (H.to_dev_bf16(x, "cuda") for x in (w.q, w.k, w.v))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device="cuda")
    bias = None if w.bias is None else H.to_dev_f32(w.bias, "cuda")
    prob = ab.problem_from(q, k, v, o, o, w.scale, cuda_cores=cuda_cores)
    mask = ab.mask_from(w.window_left, w.window_right, w.num_sink, w.bottom_right)
    ab.attn_fwd_lse(prob, mask, None, q, k, v, bias, o, lse)
    torch.cuda.synchronize()
    got_l = lse.cpu().numpy()
    dead = np.isneginf(L)
    assert np.array_equal(np.isneginf(got_l), dead)
    np.testing.assert_allclose(got_l[~dead], L[~dead], rtol=0,
                               atol=2e-5 * max(1, np.abs(L[~dead]).max(initial=0)))
    got = o.float().cpu().numpy()
    ref = O.transpose(0, 2, 1, 3)
    if cuda_cores:
        assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
    else:
        # bf16 output plus bf16 P: a few 2^-9 roundings per element
        H.check_close("o", got, ref, max_rel=1e-2, mean_rel=3e-3)


SMALL_SPARSE = {
    "scfa_s256_h16_d512": lambda: make_sparse("s", 31, Sq=256, Hq=16, Hk=1, D=512, n_ori=256,
                                              n_cmp=64, topk=32, cmp_ratio=4, ori_win_left=31),
    "swa_s192_h8_d512": lambda: make_sparse("w", 32, Sq=192, Hq=8, Hk=1, D=512, n_ori=192,
                                            n_cmp=0, topk=0, cmp_ratio=1, ori_win_left=63,
                                            with_cmp=False),
    "cfa_hk2_d512": lambda: make_sparse("c", 34, Sq=96, Hq=8, Hk=2, D=512, n_ori=160,
                                        n_cmp=40, topk=1, cmp_ratio=4, ori_win_left=20,
                                        cfa=True),
    "scfa_delta_hk2_d512": lambda: make_sparse("d", 33, Sq=96, Hq=8, Hk=2, D=512, n_ori=160,
                                               n_cmp=40, topk=16, cmp_ratio=4, ori_win_left=20,
                                               ori_win_right=3),
}


# Shapes of the tensor-core sparse path (64 query heads per KV head, D = 512).
TC_SPARSE = {
    # at most one ragged 128-row tile per token: window then compressed rows
    "tc_scfa_s200_h64": lambda: make_sparse("t1", 41, Sq=200, Hq=64, Hk=1, D=512, n_ori=200,
                                            n_cmp=50, topk=40, cmp_ratio=4, ori_win_left=127),
    # two KV heads, a right window, queries offset by delta_s = 28
    "tc_scfa_hk2_delta": lambda: make_sparse("t2", 42, Sq=72, Hq=128, Hk=2, D=512, n_ori=100,
                                             n_cmp=30, topk=24, cmp_ratio=4, ori_win_left=20,
                                             ori_win_right=3),
    # window only, no compressed KV
    "tc_swa_s160_h64": lambda: make_sparse("t3", 43, Sq=160, Hq=64, Hk=1, D=512, n_ori=160,
                                           n_cmp=0, topk=0, cmp_ratio=1, ori_win_left=63,
                                           with_cmp=False),
    # 500 selected rows per token: four tiles, the last one ragged
    "tc_scfa_rows500": lambda: make_sparse("t4", 44, Sq=96, Hq=64, Hk=1, D=512, n_ori=1000,
                                           n_cmp=250, topk=200, cmp_ratio=4, ori_win_left=299),
    # CFA: compressed KV without an index list (every block that ended by the query)
    "tc_cfa_s200_h64": lambda: make_sparse("t7", 47, Sq=200, Hq=64, Hk=1, D=512, n_ori=200,
                                           n_cmp=50, topk=1, cmp_ratio=4, ori_win_left=127,
                                           cfa=True),
    # CFA, two KV heads, queries offset by delta_s = 60, two 128-row tiles per token
    "tc_cfa_hk2_delta": lambda: make_sparse("t8", 48, Sq=100, Hq=128, Hk=2, D=512, n_ori=160,
                                            n_cmp=40, topk=1, cmp_ratio=4, ori_win_left=99,
                                            cfa=True),
    # about eight work items per persistent CTA: row counts from 0 to two tiles
    # vary between a CTA's items, and each CTA ends on items with no row
    "tc_scfa_persistent_mix": lambda: make_sparse("t6", 46, Sq=600, Hq=128, Hk=2, D=512,
                                                  n_ori=360, n_cmp=90, topk=40, cmp_ratio=4,
                                                  ori_win_left=200),
    # n_ori < Sq: the first 36 tokens select no row at all (dQ = 0, LSE = -inf)
    "tc_scfa_empty_rows": lambda: make_sparse("t5", 45, Sq=100, Hq=64, Hk=1, D=512, n_ori=64,
                                              n_cmp=16, topk=8, cmp_ratio=4, ori_win_left=15),
}


def _run_sparse(w, expect_path=None):
    # path 2 (the SIMT kernels) runs only when the problem asks for it
    torch = _torch()
    O_b, L_f, _, _ = H.sparse_forward_inputs(w)
    plan = H.gpu_sparse_plan(w, O_b, L_f, cuda_cores=expect_path == 2)
    if expect_path is not None:
        assert plan.path == expect_path
    plan.run()
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    assert code == 0, (code, detail)
    return plan, O_b, L_f


@pytest.mark.parametrize("name", list(SMALL_SPARSE))
def test_sparse_small(name):
    w = SMALL_SPARSE[name]()
    plan, O_b, L_f = _run_sparse(w, expect_path=2)
    _compare_sparse(w, plan, O_b, L_f)


def _compare_sparse(w, plan, O_b, L_f):
    ref = H.sparse_reference(w, O_b, L_f)
    H.check_close("dq", plan.dq.cpu().numpy()[0], ref["dq"])
    H.check_close("d_ori", plan.d_ori.cpu().numpy(), ref["d_ori"])
    if w.cmp_kv is not None:
        H.check_close("d_cmp", plan.d_cmp.cpu().numpy(), ref["d_cmp"])


@pytest.mark.parametrize("name", list(TC_SPARSE))
def test_sparse_tensor_core(name):
    w = TC_SPARSE[name]()
    plan, O_b, L_f = _run_sparse(w, expect_path=1)
    _compare_sparse(w, plan, O_b, L_f)
    if name == "tc_scfa_empty_rows":
        assert np.all(plan.dq.cpu().numpy()[0, :36] == 0)


def _with_repeats(w):
    """Top-k lists in which some indices repeat (each repeat counts once more)."""
    idx = w.cmp_idx.copy()
    idx[1::3, :, 1] = idx[1::3, :, 0]
    idx[2::5, :, 2:4] = idx[2::5, :, 0:1]
    w.cmp_idx = idx
    return w


# Deterministic sparse dKV: per-slot rows added in token order afterwards.
DET_SPARSE = {
    "tc_scfa_s200_h64": lambda: TC_SPARSE["tc_scfa_s200_h64"](),
    "tc_scfa_hk2_delta": lambda: TC_SPARSE["tc_scfa_hk2_delta"](),
    "tc_swa_s160_h64": lambda: TC_SPARSE["tc_swa_s160_h64"](),
    "tc_cfa_hk2_delta": lambda: TC_SPARSE["tc_cfa_hk2_delta"](),
    "tc_scfa_rows500": lambda: TC_SPARSE["tc_scfa_rows500"](),
    "tc_scfa_repeats": lambda: _with_repeats(TC_SPARSE["tc_scfa_persistent_mix"]()),
}


@pytest.mark.parametrize("name", list(DET_SPARSE))
def test_sparse_deterministic_mode(name):
    torch = _torch()
    w = DET_SPARSE[name]()
    O_b, L_f, _, _ = H.sparse_forward_inputs(w)
    plan = H.gpu_sparse_plan(w, O_b, L_f, deterministic=True)
    assert plan.path == 1
    runs = []
    for _ in range(3):
        plan.d_ori.fill_(float("nan"))  # every row is written, not added
        if plan.d_cmp is not None:
            plan.d_cmp.fill_(float("nan"))
        plan.run()
        torch.cuda.synchronize()
        code, detail = plan.device_status()
        assert code == 0, (code, detail)
        outs = [plan.dq, plan.d_ori] + ([plan.d_cmp] if plan.d_cmp is not None else [])
        runs.append([t.cpu().numpy().copy() for t in outs])
    for later in runs[1:]:
        for a, b in zip(runs[0], later):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    _compare_sparse(w, plan, O_b, L_f)


def test_sparse_tensor_core_bad_index_is_reported():
    torch = _torch()
    w = TC_SPARSE["tc_scfa_s200_h64"]()
    O_b, L_f, _, _ = H.sparse_forward_inputs(w)
    w.cmp_idx = w.cmp_idx.copy()
    w.cmp_idx[150, 0, 1] = -7  # neither a row nor the empty marker: skipped and reported
    plan = H.gpu_sparse_plan(w, O_b, L_f)
    assert plan.path == 1
    plan.run()
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    assert code == 5 and detail == 150


@pytest.mark.parametrize("where", ["ori_kv", "q"])
def test_sparse_tensor_core_fp16_range_is_reported(where):
    torch = _torch()
    w = TC_SPARSE["tc_swa_s160_h64"]()
    O_b, L_f, _, _ = H.sparse_forward_inputs(w)
    if where == "ori_kv":
        w.ori_kv = w.ori_kv.copy()
        w.ori_kv[7, 0, 100] = 1.0e5  # representable in bf16, not in fp16
    else:
        w.q = w.q.copy()
        w.q[9, 3, 200] = -1.0e5
    plan = H.gpu_sparse_plan(w, O_b, L_f)
    assert plan.path == 1
    plan.run()
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    assert code == 6 and detail & (2 if where == "ori_kv" else 16)


def test_sparse_bad_index_is_reported_not_trapped():
    torch = _torch()
    w = SMALL_SPARSE["scfa_s256_h16_d512"]()
    O_b, L_f, _, _ = H.sparse_forward_inputs(w)
    w.cmp_idx = w.cmp_idx.copy()
    w.cmp_idx[200, 0, 0] = w.n_cmp + 5  # out of range: must be skipped and reported
    plan = H.gpu_sparse_plan(w, O_b, L_f, cuda_cores=True)
    assert plan.path == 2
    plan.run()
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    assert code == 5 and detail == 200


def test_fp16_range_overflow_is_reported():
    # The tensor-core path works on exact fp16 copies of the bf16 inputs; a
    # value beyond the fp16 range must surface as ATTN_ERR_RANGE, not as a trap.
    torch = _torch()
    w = TC_EXTRA["mha_s128_d64"]()
    O_b, L_f, _, _ = H.dense_forward_inputs(w)
    w.k = w.k.copy()
    w.k[0, 5, 0, 3] = 1.0e5  # representable in bf16, not in fp16
    plan = H.gpu_dense_plan(w, O_b, L_f)
    assert plan.path == 1
    plan.run()
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    assert code == 6 and detail & 2  # ATTN_ERR_RANGE, flag of k
    # the next clean call clears the condition
    w2 = TC_EXTRA["mha_s128_d64"]()
    plan2 = H.gpu_dense_plan(w2, O_b, L_f)
    plan2.workspace = plan.workspace
    plan2.run()
    torch.cuda.synchronize()
    assert plan2.device_status()[0] == 0


# ------------------------------------------------------------- full size ----

def test_full_gqa4_causal_s1024_d128():
    w = make_workload("gqa4_causal_s1024_d128")
    plan, O_b, L_f = _run_dense(w, expect_path=1)
    _compare_dense(w, plan, O_b, L_f)


def test_full_mha_alibi_dbias_s2048_d64():
    w = make_workload("mha_alibi_dbias_s2048_d64")
    plan, O_b, L_f = _run_dense(w, expect_path=1)
    for h in (0, 15):
        ref = H.dense_reference(w, O_b, L_f, kv_heads=slice(h, h + 1))
        H.check_close("dq", plan.dq.cpu().numpy()[:, :, h:h + 1], ref["dq"])
        H.check_close("dk", plan.dk.cpu().numpy()[:, :, h:h + 1], ref["dk"])
        H.check_close("dv", plan.dv.cpu().numpy()[:, :, h:h + 1], ref["dv"])
        H.check_close("dbias", plan.dbias.cpu().numpy()[h:h + 1], ref["dbias"])


def test_full_gqa4_window1024_sink4_s8192_d128():
    w = make_workload("gqa4_window1024_sink4_s8192_d128")
    plan, O_b, L_f = _run_dense(w, expect_path=1)
    for g in (0, 7):
        _compare_dense(w, plan, O_b, L_f, kv_heads=slice(g, g + 1))


def test_full_sparse_scfa_s4096_h64_d512():
    torch = _torch()
    w = make_workload("sparse_scfa_s4096_h64_d512")
    plan, O_b, L_f = _run_sparse(w, expect_path=1)
    _compare_sparse(w, plan, O_b, L_f)
    # the deterministic mode at full size: twice bitwise the same, and parity
    del plan
    det = H.gpu_sparse_plan(w, O_b, L_f, deterministic=True)
    outs = []
    for _ in range(2):
        det.run()
        torch.cuda.synchronize()
        assert det.device_status()[0] == 0
        outs.append((det.d_ori.clone(), det.d_cmp.clone()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    _compare_sparse(w, det, O_b, L_f)


SINK_CASES = {
    # dense, tensor-core path, GQA 4:1 causal
    "dense_tc": lambda: make_workload("gqa4_causal_s1024_d128", Hq=8, Hk=2, Sq=256, Sk=256),
    # dense, ragged lengths, window + sinks tokens
    "dense_simt": lambda: SMALL_DENSE["ragged_causal_sink_s200_d64"](),
    # sparse, tensor-core path
    "sparse_tc": lambda: TC_SPARSE["tc_scfa_hk2_delta"](),
}


@pytest.mark.parametrize("name", list(SINK_CASES))
def test_sink_logits(name):
    # Learnable sink logits: the forward's LSE contains them, attn_bwd is
    # unchanged, and attn_bwd_dsinks gives their gradient.
    torch = _torch()
    import attention_backward_attn_gb300 as ab
    w = SINK_CASES[name]()
    rng = np.random.default_rng(90)
    sinks = rng.standard_normal(w.Hq).astype(np.float32)
    sparse = w.__class__.__name__ == "SparseWorkload"
    if sparse:
        q = np.asarray(w.q, np.float64)
        okv = np.asarray(w.ori_kv, np.float64)
        ckv = None if w.cmp_kv is None else np.asarray(w.cmp_kv, np.float64)
        O, L = oracle.sparse_forward(q, okv, ckv, w.cmp_idx, w.scale, w.ori_win_left,
                                     w.ori_win_right, H.cfa_ratio(w), sinks=sinks)
        O_b = np.ascontiguousarray(H.bf16_round(O.astype(np.float32)))
        L_f = L.astype(np.float32)
        plan = H.gpu_sparse_plan(w, O_b, L_f)
    else:
        O, L = oracle.forward(H.bhsd(w.q), H.bhsd(w.k), H.bhsd(w.v), w.scale, H.mask_of(w),
                              None if w.bias is None else w.bias.astype(np.float64), sinks)
        O_b = np.ascontiguousarray(H.bf16_round(O.transpose(0, 2, 1, 3).astype(np.float32)))
        L_f = L.astype(np.float32)
        plan = H.gpu_dense_plan(w, O_b, L_f)
    plan.run()
    torch.cuda.synchronize()
    code, detail = plan.device_status()
    assert code == 0, (code, detail)
    if sparse:
        _compare_sparse(w, plan, O_b, L_f)
        lse3 = L_f[None].astype(np.float64)
        dlt = (np.asarray(w.do, np.float64) * O_b.astype(np.float64)).sum(-1).T[None]
    else:
        _compare_dense(w, plan, O_b, L_f)
        lse3 = L_f.astype(np.float64)
        dlt = oracle.preprocess(H.bhsd(O_b), H.bhsd(w.do))
    ref = oracle.dsinks(lse3, dlt, sinks.astype(np.float64))
    sk = torch.from_numpy(sinks).cuda()
    got = torch.empty(w.Hq, dtype=torch.float32, device="cuda")
    ab.attn_bwd_dsinks(plan.prob, sk, plan.lse, plan.delta, got)
    got2 = torch.empty_like(got)
    ab.attn_bwd_dsinks(plan.prob, sk, plan.lse, plan.delta, got2)
    torch.cuda.synchronize()
    H.check_close("dsinks", got.cpu().numpy(), ref)
    assert torch.equal(got, got2)  # fixed-order reduction
