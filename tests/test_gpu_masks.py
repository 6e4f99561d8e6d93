"""GPU: the device-side mask and gather-index logic against the oracle, bit for bit.

The backward kernels decide per element which (query, key) pairs are live:
a tile walk over closed-form live-tile ranges, then a per-row predicate on the
tiles the mask cuts ("22_sink_tokens_fmha.py" mask builders). The sparse
kernel builds each token's selected-row list on the device (Ascend
"sparse_flash_mla_grad" formula, phase 1). A slip there of one key at a window
edge could hide inside the gradient tolerance, so these tests read the
decisions back exactly:

* attn_debug_mask_live runs the kernel's own walk and predicates for both
  kinds of CTA and must reproduce oracle.live_mask as 0 / 1 bytes, with no
  live entry outside the lengths and no tile visited twice;
* the backward itself, with dbias requested and B = 1, must leave dbias
  exactly zero off the mask and nonzero on every live entry of a row with
  at least two live keys (on a row with a single live key P = 1 and O is
  that key's value row, so dS = P (dP - D) is zero up to rounding: those
  entries may hold rounding noise either way);
* attn_debug_sparse_rows runs the kernel's row-list builder and must return
  oracle.selected_rows for every (token, KV head), in order.
"""

import numpy as np
import pytest

import harness as H
import oracle
from workloads import make_dense, make_sparse, make_workload

pytestmark = pytest.mark.gpu


def _probe(Sq, Sk, wl, wr, ns, br, variant):
    import torch
    import attention_backward_attn_gb300 as ab
    kv = torch.zeros((Sq, Sk), dtype=torch.uint8, device="cuda")
    q = torch.zeros((Sq, Sk), dtype=torch.uint8, device="cuda")
    out = torch.zeros(1, dtype=torch.int32, device="cuda")
    ab.attn_debug_mask_live(ab.mask_from(wl, wr, ns, br), Sq, Sk, variant, kv, q, out)
    torch.cuda.synchronize()
    return kv.cpu().numpy(), q.cpu().numpy(), int(out.item())


def _check_probe(Sq, Sk, wl, wr, ns, br):
    ref = oracle.live_mask(Sq, Sk, wl, wr, ns, br).astype(np.uint8)
    variants = [0] + ([1] if Sq % 128 == 0 and Sk % 128 == 0 else [])
    for variant in variants:
        kv, q, outside = _probe(Sq, Sk, wl, wr, ns, br, variant)
        where = (Sq, Sk, wl, wr, ns, br, variant)
        assert outside == 0, where
        if not np.array_equal(kv, ref):
            bad = np.argwhere(kv != ref)[:5]
            raise AssertionError(f"key-major view differs at {bad.tolist()} for {where}")
        if not np.array_equal(q, ref):
            bad = np.argwhere(q != ref)[:5]
            raise AssertionError(f"query-major view differs at {bad.tolist()} for {where}")


# (Sq, Sk, window_left, window_right, num_sink, bottom_right)
WORKLOAD_MASKS = {
    "mha_s64_d64": (64, 64, -1, -1, 0, False),
    "gqa4_causal_s1024_d128": (1024, 1024, -1, 0, 0, False),
    "mha_alibi_dbias_s2048_d64": (2048, 2048, -1, -1, 0, False),
    "gqa4_window1024_sink4_s8192_d128": (8192, 8192, 1023, 0, 4, False),
}

RAGGED_MASKS = [
    (1000, 1000, -1, 0, 0, False),     # causal, ragged last tile
    (1, 1, -1, 0, 0, False),
    (200, 330, -1, 0, 0, True),        # bottom-right causal, Sk > Sq
    (330, 200, -1, 0, 0, True),        # bottom-right causal, Sk < Sq: empty rows
    (330, 200, 50, 7, 0, True),        # bottom-right two-sided window
    (129, 127, 30, 0, 5, False),       # window + sinks across a tile edge
    (300, 5, -1, 0, 2, False),         # few keys, sinks
    (5, 300, -1, -1, 200, False),      # sinks spanning two key tiles
    (640, 640, 0, 0, 0, False),        # the diagonal only
    (384, 512, 127, 128, 1, False),    # window edges on tile edges
    (256, 256, 10, 0, 130, False),     # sinks longer than a tile
    (700, 450, 1023, 0, 4, True),      # the workload-4 mask, bottom-right, ragged
]


@pytest.mark.parametrize("name", list(WORKLOAD_MASKS))
def test_mask_probe_workload_shapes(name):
    _check_probe(*WORKLOAD_MASKS[name])


@pytest.mark.parametrize("case", RAGGED_MASKS, ids=lambda c: "_".join(map(str, c)))
def test_mask_probe_ragged_shapes(case):
    _check_probe(*case)


def test_mask_probe_random_masks():
    rng = np.random.default_rng(2024)
    for t in range(300):
        if t % 3 == 0:  # whole tiles, so the aligned instantiation is probed too
            Sq, Sk = 128 * int(rng.integers(1, 6)), 128 * int(rng.integers(1, 6))
        else:
            Sq, Sk = int(rng.integers(1, 600)), int(rng.integers(1, 600))
        wl = int(rng.choice([-1, int(rng.integers(0, 400))]))
        wr = int(rng.choice([-1, 0, int(rng.integers(0, 200))]))
        ns = int(rng.choice([0, 0, int(rng.integers(1, 150))]))
        br = bool(rng.integers(0, 2))
        _check_probe(Sq, Sk, wl, wr, ns, br)


# dbias of the backward itself: zero off the mask, nonzero on it (B = 1)
DBIAS_MASKS = {
    "window_sinks_s384": dict(Sq=384, Sk=384, window_left=100, window_right=0, num_sink=3),
    "br_causal_sq200_sk330": dict(Sq=200, Sk=330, window_left=-1, window_right=0,
                                  bottom_right=True),
    "br_window_sq330_sk200": dict(Sq=330, Sk=200, window_left=50, window_right=7,
                                  bottom_right=True),
    "two_sided_s256": dict(Sq=256, Sk=256, window_left=20, window_right=33),
    "ragged_causal_sinks_s300": dict(Sq=300, Sk=300, window_left=-1, window_right=0,
                                     num_sink=5),
}


@pytest.mark.parametrize("name", list(DBIAS_MASKS))
@pytest.mark.parametrize("D", [64, 128])
def test_dbias_support_is_the_mask(name, D):
    import torch
    spec = DBIAS_MASKS[name]
    w = make_dense(name, 61, B=1, Hq=2, Hk=1, D=D, want_dbias=True, **spec)
    O_b, L_f, _, _ = H.dense_forward_inputs(w)
    plan = H.gpu_dense_plan(w, O_b, L_f)
    assert plan.path == 1
    # every entry must be written by the call (zeroed, or computed), whatever
    # the buffer held before
    plan.dbias.fill_(float("nan"))
    plan.run()
    torch.cuda.synchronize()
    assert plan.device_status() == (0, 0)
    assert torch.isfinite(plan.dbias).all()
    live = oracle.live_mask(w.Sq, w.Sk, w.window_left, w.window_right, w.num_sink,
                            w.bottom_right)
    multi = live & (live.sum(axis=1) >= 2)[:, None]
    assert multi.any()
    db = plan.dbias.cpu().numpy()
    for h in range(w.Hq):
        off = (db[h] != 0) & ~live
        if off.any():
            raise AssertionError(f"head {h}: dbias nonzero off the mask at "
                                 f"{np.argwhere(off)[:5].tolist()}")
        missing = (db[h] == 0) & multi
        if missing.any():
            raise AssertionError(f"head {h}: dbias zero on live entries at "
                                 f"{np.argwhere(missing)[:5].tolist()}")


# ------------------------------------------------------------- sparse rows ----

def _rows_probe(w, idx_override=None):
    import torch
    import attention_backward_attn_gb300 as ab
    idx_np = w.cmp_idx if idx_override is None else idx_override
    q = H.to_dev_bf16(w.q[None], "cuda")
    okv = H.to_dev_bf16(w.ori_kv, "cuda")
    ckv = None if w.cmp_kv is None else H.to_dev_bf16(w.cmp_kv, "cuda")
    idx = None if idx_np is None else torch.from_numpy(np.ascontiguousarray(idx_np)).to("cuda")
    cfa = H.cfa_ratio(w) or 0
    sp = ab.sparse_from(okv, ckv, idx, w.ori_win_left, w.ori_win_right, None, None, cfa)
    prob = ab.problem_from(q, None, None, q, q, w.scale, Sk=0, Hk=w.Hk)
    win = (w.ori_win_left + w.ori_win_right + 1 if w.ori_win_left >= 0 and w.ori_win_right >= 0
           else w.n_ori)
    bound = min(win, w.n_ori) + (0 if w.cmp_kv is None else (w.n_cmp if cfa else w.topk))
    items = w.Sq * w.Hk
    rows = torch.full((items, bound), -7, dtype=torch.int32, device="cuda")
    counts = torch.full((items,), -7, dtype=torch.int32, device="cuda")
    ab.attn_debug_sparse_rows(prob, sp, rows, counts, bound)
    torch.cuda.synchronize()
    return rows.cpu().numpy(), counts.cpu().numpy(), idx_np


def _expected_rows(w, i, g, idx_np):
    cfa = H.cfa_ratio(w)
    row = None if idx_np is None else idx_np[i, g]
    if row is not None:
        row = row[(row >= 0) & (row < w.n_cmp)]  # out-of-range entries are skipped
    ori, cmp = oracle.selected_rows(i, w.Sq, w.n_ori, w.ori_win_left, w.ori_win_right, row,
                                    w.n_cmp, cfa)
    return np.concatenate([ori * w.Hk + g, (w.n_ori + cmp) * w.Hk + g]).astype(np.int64)


def _check_rows(w, idx_override=None):
    rows, counts, idx_np = _rows_probe(w, idx_override)
    for i in range(w.Sq):
        for g in range(w.Hk):
            item = i * w.Hk + g
            exp = _expected_rows(w, i, g, idx_np)
            n = int(counts[item])
            assert n == exp.size, (i, g, n, exp.size)
            if not np.array_equal(rows[item, :n].astype(np.int64), exp):
                raise AssertionError(f"token {i}, KV head {g}: row list differs")
            assert (rows[item, n:] == -7).all(), (i, g)  # nothing written past the list


SPARSE_ROW_CASES = {
    "scfa_s4096_full": lambda: make_workload("sparse_scfa_s4096_h64_d512"),
    "scfa_hk2_delta": lambda: make_sparse("t2", 42, Sq=72, Hq=128, Hk=2, D=512, n_ori=100,
                                          n_cmp=30, topk=24, cmp_ratio=4, ori_win_left=20,
                                          ori_win_right=3),
    "swa_s160": lambda: make_sparse("t3", 43, Sq=160, Hq=64, Hk=1, D=512, n_ori=160, n_cmp=0,
                                    topk=0, cmp_ratio=1, ori_win_left=63, with_cmp=False),
    "cfa_s200": lambda: make_sparse("t7", 47, Sq=200, Hq=64, Hk=1, D=512, n_ori=200, n_cmp=50,
                                    topk=1, cmp_ratio=4, ori_win_left=127, cfa=True),
    "cfa_hk2_delta": lambda: make_sparse("t8", 48, Sq=100, Hq=128, Hk=2, D=512, n_ori=160,
                                         n_cmp=40, topk=1, cmp_ratio=4, ori_win_left=99,
                                         cfa=True),
    "scfa_rows500": lambda: make_sparse("t4", 44, Sq=96, Hq=64, Hk=1, D=512, n_ori=1000,
                                        n_cmp=250, topk=200, cmp_ratio=4, ori_win_left=299),
    "scfa_empty_rows": lambda: make_sparse("t5", 45, Sq=100, Hq=64, Hk=1, D=512, n_ori=64,
                                           n_cmp=16, topk=8, cmp_ratio=4, ori_win_left=15),
}


@pytest.mark.parametrize("name", list(SPARSE_ROW_CASES))
def test_sparse_row_lists_match_oracle(name):
    _check_rows(SPARSE_ROW_CASES[name]())


def test_sparse_row_lists_skip_unused_and_bad_slots():
    # -1 slots between valid ones, repeated indices and out-of-range indices:
    # the list keeps the valid entries in slot order (repeats included) and
    # drops the rest
    w = make_sparse("t9", 49, Sq=64, Hq=64, Hk=2, D=512, n_ori=64, n_cmp=40, topk=24,
                    cmp_ratio=1, ori_win_left=9)
    rng = np.random.default_rng(5)
    idx = rng.integers(-1, 40, size=w.cmp_idx.shape).astype(np.int32)
    idx[::7, :, 3] = 40           # one past the end
    idx[::5, :, 5] = -9           # below -1
    idx[::3, :, 8] = idx[::3, :, 9]  # a repeat
    _check_rows(w, idx)
