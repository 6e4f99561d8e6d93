"""Pins for the sparse (selected, shared-latent-KV) float64 oracle (CPU only)."""

import json
import math
import os

import numpy as np
import pytest

import oracle
import brute
from workloads import make_sparse, topk_compressed_indices

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _small(seed=3, Sq=12, Hq=4, Hk=1, D=3, n_ori=12, n_cmp=4, topk=3, ratio=3,
           left=3, right=0, with_cmp=True):
    return make_sparse("s", seed=seed, Sq=Sq, Hq=Hq, Hk=Hk, D=D, n_ori=n_ori, n_cmp=n_cmp,
                       topk=topk, cmp_ratio=ratio, ori_win_left=left, ori_win_right=right,
                       with_cmp=with_cmp)


def _f64(x):
    return None if x is None else np.asarray(x, np.float64)


def test_index_generator_rule_and_counts():
    # Ascend example: query i may pick compressed row c iff c < (delta_s + i + 1) // ratio;
    # min(eligible, K) distinct picks, rest -1.
    rng = np.random.default_rng(0)
    Sq, n_ori, n_cmp, ratio, K = 64, 80, 20, 4, 8
    idx = topk_compressed_indices(rng, Sq, n_ori, n_cmp, ratio, K, 2)
    delta = n_ori - Sq
    for i in range(Sq):
        elig = min((delta + i + 1) // ratio, n_cmp)
        row = idx[i, 0]
        valid = row[row >= 0]
        assert np.array_equal(idx[i, 0], idx[i, 1])
        assert valid.size == min(elig, K)
        assert np.all(row[valid.size:] == -1)
        assert len(set(valid.tolist())) == valid.size
        assert np.all(valid < elig)


def test_benchmark_live_counts_closed_form():
    # Window of 128 original rows: sum_i min(i + 1, 128) = 128*129/2 + (4096 - 128) * 128.
    ori = sum(min(i + 1, 128) for i in range(4096))
    assert ori == 128 * 129 // 2 + (4096 - 128) * 128 == 516160
    # Top-512 of floor((i + 1) / 4) eligible rows: 4 * sum_{m<512} m + 2049 * 512.
    cmp = sum(min((i + 1) // 4, 512) for i in range(4096))
    assert cmp == 4 * (511 * 512 // 2) + 2049 * 512 == 1572352


def test_selected_rows_window():
    ori, cmp = oracle.selected_rows(5, 10, 10, 2, 0, np.array([3, -1, 1]))
    assert ori.tolist() == [3, 4, 5] and cmp.tolist() == [3, 1]
    ori, _ = oracle.selected_rows(0, 4, 8, 1, 1, None)  # bottom-right: position 4
    assert ori.tolist() == [3, 4, 5]
    ori, _ = oracle.selected_rows(0, 4, 4, 5, 0, None)
    assert ori.tolist() == [0]


@pytest.mark.parametrize("with_cmp", [False, True])
def test_sparse_matches_brute_force(with_cmp):
    w = _small(with_cmp=with_cmp, Hk=2, Hq=4)
    q, okv, ckv, do = _f64(w.q), _f64(w.ori_kv), _f64(w.cmp_kv), _f64(w.do)
    O, L = oracle.sparse_forward(q, okv, ckv, w.cmp_idx, w.scale, w.ori_win_left, w.ori_win_right)
    got = oracle.sparse_backward(q, okv, ckv, w.cmp_idx, O, do, L, w.scale,
                                 w.ori_win_left, w.ori_win_right)
    ref = brute.sparse_backward(q.tolist(), okv.tolist(), None if ckv is None else ckv.tolist(),
                                None if w.cmp_idx is None else w.cmp_idx.tolist(),
                                O.tolist(), do.tolist(), L.tolist(), w.scale,
                                w.ori_win_left, w.ori_win_right)
    for g, r in zip(got, ref):
        if g is None:
            assert r is None
            continue
        np.testing.assert_allclose(g, np.array(r), rtol=0, atol=1e-12)


def test_window_only_reduces_to_dense_window_mask():
    # No compressed KV (the page's SWA case): K = V = ori_kv with the window mask,
    # and dKV must equal dK + dV of the dense oracle.
    w = _small(with_cmp=False, Sq=10, n_ori=10, left=3)
    q, okv, do = _f64(w.q), _f64(w.ori_kv), _f64(w.do)
    O, L = oracle.sparse_forward(q, okv, None, None, w.scale, 3, 0)
    dq, dkv, _ = oracle.sparse_backward(q, okv, None, None, O, do, L, w.scale, 3, 0)
    Q = q.transpose(1, 0, 2)[None]
    KV = okv.transpose(1, 0, 2)[None]
    dO = do.transpose(1, 0, 2)[None]
    m = oracle.window_sink_mask(10, 10, 4, 0)
    Od, Ld = oracle.forward(Q, KV, KV, w.scale, m)
    np.testing.assert_allclose(Od[0].transpose(1, 0, 2), O, atol=1e-13)
    np.testing.assert_allclose(Ld[0], L, atol=1e-13)
    dQd, dKd, dVd, _ = oracle.backward(Q, KV, KV, Od, dO, Ld, w.scale, m)
    np.testing.assert_allclose(dQd[0].transpose(1, 0, 2), dq, atol=1e-12)
    np.testing.assert_allclose((dKd + dVd)[0].transpose(1, 0, 2), dkv, atol=1e-12)


def test_gathered_rows_reduce_to_dense_mask_over_concatenated_kv():
    # Selecting compressed rows by index == a dense mask over [ori_kv ; cmp_kv].
    w = _small(Sq=12, n_ori=12, n_cmp=4, topk=3, ratio=3, left=2, Hq=2, Hk=1)
    q, okv, ckv, do = _f64(w.q), _f64(w.ori_kv), _f64(w.cmp_kv), _f64(w.do)
    O, L = oracle.sparse_forward(q, okv, ckv, w.cmp_idx, w.scale, 2, 0)
    dq, dori, dcmp = oracle.sparse_backward(q, okv, ckv, w.cmp_idx, O, do, L, w.scale, 2, 0)
    kv = np.concatenate([okv, ckv], axis=0)
    m = np.zeros((12, 16), dtype=bool)
    for i in range(12):
        m[i, max(0, i - 2):i + 1] = True
        for c in w.cmp_idx[i, 0]:
            if c >= 0:
                m[i, 12 + c] = True
    Q, KV, dO = q.transpose(1, 0, 2)[None], kv.transpose(1, 0, 2)[None], do.transpose(1, 0, 2)[None]
    Od, Ld = oracle.forward(Q, KV, KV, w.scale, m)
    np.testing.assert_allclose(Od[0].transpose(1, 0, 2), O, atol=1e-13)
    dQd, dKd, dVd, _ = oracle.backward(Q, KV, KV, Od, dO, Ld, w.scale, m)
    dkv = (dKd + dVd)[0].transpose(1, 0, 2)
    np.testing.assert_allclose(dQd[0].transpose(1, 0, 2), dq, atol=1e-12)
    np.testing.assert_allclose(dkv[:12], dori, atol=1e-12)
    np.testing.assert_allclose(dkv[12:], dcmp, atol=1e-12)


def test_sparse_finite_differences():
    # L = sum(O * dO); perturbing a shared KV row checks dKV = dK + dV in one shot.
    w = _small(Sq=8, n_ori=8, n_cmp=3, topk=2, ratio=2, left=2, Hq=2, Hk=1, D=2)
    q, okv, ckv, do = _f64(w.q), _f64(w.ori_kv), _f64(w.cmp_kv), _f64(w.do)
    O, L = oracle.sparse_forward(q, okv, ckv, w.cmp_idx, w.scale, 2, 0)
    dq, dori, dcmp = oracle.sparse_backward(q, okv, ckv, w.cmp_idx, O, do, L, w.scale, 2, 0)

    def loss(qq, oo, cc):
        Ox, _ = oracle.sparse_forward(qq, oo, cc, w.cmp_idx, w.scale, 2, 0)
        return float((Ox * do).sum())

    eps = 1e-6
    rng = np.random.default_rng(1)
    for name, G in (("q", dq), ("ori", dori), ("cmp", dcmp)):
        for _ in range(6):
            X = {"q": q, "ori": okv, "cmp": ckv}[name]
            idx = tuple(int(rng.integers(0, s)) for s in X.shape)
            vals = []
            for sgn in (1, -1):
                Xs = X.copy()
                Xs[idx] += sgn * eps
                args = {"q": q, "ori": okv, "cmp": ckv}
                args[name] = Xs
                vals.append(loss(args["q"], args["ori"], args["cmp"]))
            num = (vals[0] - vals[1]) / (2 * eps)
            assert abs(num - G[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx, num, G[idx])


def test_sparse_ds_rows_sum_to_zero():
    # sum over selected rows of dS = 0 for each (token, head) (exact O), which
    # makes sum_d dQ_d-weighted terms consistent; checked through dQ with kv = const:
    # if every selected row is the same vector, dS = 0 and dQ = 0.
    w = _small(Sq=6, n_ori=6, n_cmp=2, topk=1, ratio=2, left=2, Hq=2, Hk=1, D=3)
    okv = np.broadcast_to(_f64(w.ori_kv)[:1], w.ori_kv.shape).copy()
    ckv = np.broadcast_to(_f64(w.ori_kv)[:1], w.cmp_kv.shape).copy()
    q, do = _f64(w.q), _f64(w.do)
    O, L = oracle.sparse_forward(q, okv, ckv, w.cmp_idx, w.scale, 2, 0)
    dq, _, _ = oracle.sparse_backward(q, okv, ckv, w.cmp_idx, O, do, L, w.scale, 2, 0)
    assert np.abs(dq).max() < 1e-13


def _ev(x):
    if isinstance(x, list):
        return [_ev(y) for y in x]
    if isinstance(x, str):
        return eval(x, {"__builtins__": {}}, {"ln3": math.log(3.0), "ln4": math.log(4.0)})
    return float(x)


def test_hand_derived_sparse_example():
    ex = json.load(open(GOLDEN))["sparse_shared_kv_two_rows"]
    q, okv, do = (np.array(_ev(ex[k])) for k in ("q", "ori_kv", "do"))
    O, L = oracle.sparse_forward(q, okv, None, None, ex["scale"], ex["win_left"], ex["win_right"])
    dq, dori, _ = oracle.sparse_backward(q, okv, None, None, O, do, L, ex["scale"],
                                         ex["win_left"], ex["win_right"])
    got = dict(O=O, LSE=L, dQ=dq, d_ori_kv=dori)
    for key, val in ex["expect"].items():
        np.testing.assert_allclose(got[key], np.array(_ev(val)), rtol=0, atol=1e-14, err_msg=key)


def _small_cfa(Sq, n_ori, n_cmp, ratio, left, Hq, Hk, D=4, seed=7):
    return make_sparse("cfa", seed, Sq=Sq, Hq=Hq, Hk=Hk, D=D, n_ori=n_ori, n_cmp=n_cmp, topk=1,
                       cmp_ratio=ratio, ori_win_left=left, cfa=True)


def test_cfa_selects_every_block_that_ends_by_the_query():
    # Compressed row c covers positions [c * ratio, (c + 1) * ratio): it is live
    # for position p once that block has ended, c < (p + 1) // ratio.
    _, cmp = oracle.selected_rows(0, 12, 12, 2, 0, None, n_cmp=4, cmp_ratio=3)
    assert cmp.size == 0                                  # p = 0: block 0 not complete
    _, cmp = oracle.selected_rows(2, 12, 12, 2, 0, None, n_cmp=4, cmp_ratio=3)
    assert list(cmp) == [0]                               # p = 2 ends block 0
    _, cmp = oracle.selected_rows(11, 12, 12, 2, 0, None, n_cmp=3, cmp_ratio=3)
    assert list(cmp) == [0, 1, 2]                         # clipped to n_cmp
    _, cmp = oracle.selected_rows(1, 4, 8, 2, 0, None, n_cmp=4, cmp_ratio=2)
    assert list(cmp) == [0, 1, 2]                         # bottom-right: p = 5 ends block 2


def test_cfa_reduces_to_dense_mask_over_concatenated_kv():
    # CFA == a dense mask over [ori_kv ; cmp_kv] with the window plus every
    # compressed block that ended by the query.
    w = _small_cfa(Sq=12, n_ori=12, n_cmp=4, ratio=3, left=2, Hq=2, Hk=1)
    assert w.cmp_idx is None and w.cmp_kv is not None
    q, okv, ckv, do = _f64(w.q), _f64(w.ori_kv), _f64(w.cmp_kv), _f64(w.do)
    O, L = oracle.sparse_forward(q, okv, ckv, None, w.scale, 2, 0, cmp_ratio=3)
    dq, dori, dcmp = oracle.sparse_backward(q, okv, ckv, None, O, do, L, w.scale, 2, 0,
                                            cmp_ratio=3)
    kv = np.concatenate([okv, ckv], axis=0)
    m = np.zeros((12, 16), dtype=bool)
    for i in range(12):
        m[i, max(0, i - 2):i + 1] = True
        for c in range(4):
            if (c + 1) * 3 <= i + 1:
                m[i, 12 + c] = True
    Q, KV, dO = q.transpose(1, 0, 2)[None], kv.transpose(1, 0, 2)[None], do.transpose(1, 0, 2)[None]
    Od, Ld = oracle.forward(Q, KV, KV, w.scale, m)
    np.testing.assert_allclose(Od[0].transpose(1, 0, 2), O, atol=1e-13)
    dQd, dKd, dVd, _ = oracle.backward(Q, KV, KV, Od, dO, Ld, w.scale, m)
    dkv = (dKd + dVd)[0].transpose(1, 0, 2)
    np.testing.assert_allclose(dQd[0].transpose(1, 0, 2), dq, atol=1e-12)
    np.testing.assert_allclose(dkv[:12], dori, atol=1e-12)
    np.testing.assert_allclose(dkv[12:], dcmp, atol=1e-12)


def test_cfa_matches_brute_force_with_the_explicit_row_list():
    # The pure-Python brute force takes index lists: give it the eligible rows.
    w = _small_cfa(Sq=6, n_ori=8, n_cmp=3, ratio=2, left=1, Hq=2, Hk=1, D=3)
    q, okv, ckv, do = _f64(w.q), _f64(w.ori_kv), _f64(w.cmp_kv), _f64(w.do)
    O, L = oracle.sparse_forward(q, okv, ckv, None, w.scale, 1, 0, cmp_ratio=2)
    got = oracle.sparse_backward(q, okv, ckv, None, O, do, L, w.scale, 1, 0, cmp_ratio=2)
    idx = np.full((6, 1, 3), -1, dtype=np.int32)
    for i in range(6):
        p = (8 - 6) + i
        n = min(3, (p + 1) // 2)
        idx[i, 0, :n] = np.arange(n)
    ref = brute.sparse_backward(q.tolist(), okv.tolist(), ckv.tolist(), idx.tolist(), O.tolist(),
                                do.tolist(), L.tolist(), w.scale, 1, 0)
    for g_, r_ in zip(got, ref):
        np.testing.assert_allclose(g_, np.asarray(r_), atol=1e-12)


def test_cfa_without_a_ratio_is_rejected():
    w = _small_cfa(Sq=4, n_ori=4, n_cmp=2, ratio=2, left=1, Hq=1, Hk=1)
    with pytest.raises(ValueError):
        oracle.sparse_forward(_f64(w.q), _f64(w.ori_kv), _f64(w.cmp_kv), None, w.scale, 1, 0)


def test_sparse_sinks_match_the_dense_extra_key():
    # With sinks the sparse forward equals the dense one over the concatenated
    # selected rows plus a zero key carrying the sink as its bias.
    w = _small(Sq=8, n_ori=8, n_cmp=3, topk=2, ratio=2, left=2, Hq=2, Hk=1, D=3)
    q, okv, ckv = _f64(w.q), _f64(w.ori_kv), _f64(w.cmp_kv)
    sinks = np.array([0.3, -1.2])
    O, L = oracle.sparse_forward(q, okv, ckv, w.cmp_idx, w.scale, 2, 0, sinks=sinks)
    kv = np.concatenate([okv, ckv, np.zeros((1, 1, 3))], axis=0)
    m = np.zeros((8, 12), dtype=bool)
    for i in range(8):
        m[i, max(0, i - 2):i + 1] = True
        for c in w.cmp_idx[i, 0]:
            if c >= 0:
                m[i, 8 + c] = True
    m[:, 11] = True
    bias = np.zeros((2, 8, 12))
    bias[:, :, 11] = sinks[:, None]
    KV = kv.transpose(1, 0, 2)[None]
    Od, Ld = oracle.forward(q.transpose(1, 0, 2)[None], KV, KV, w.scale, m, bias)
    np.testing.assert_allclose(Od[0].transpose(1, 0, 2), O, atol=1e-13)
    np.testing.assert_allclose(Ld[0], L, atol=1e-13)
