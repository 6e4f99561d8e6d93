"""Pins for the oracle's variable-length (packed, token-major) batches (CPU only).

varlen_forward / varlen_backward split a packed batch into its sequences and
run the dense oracle on each. The pins: equal lengths reproduce the batched
problem; sequences do not see each other (and empty ones contribute
nothing); and a bottom-right mask aligns on each sequence's own lengths,
checked against the scalar-loop attention of tests/brute.py.
"""

import numpy as np

import brute
import oracle
from workloads import make_dense, make_varlen


def _pack(x):
    """[B, S, H, D] -> packed [B * S, H, D]."""
    B, S, H, D = x.shape
    return np.ascontiguousarray(x.reshape(B * S, H, D))


def test_equal_lengths_reproduce_the_batched_problem():
    w = make_dense("v", 3, B=3, Hq=4, Hk=2, Sq=37, Sk=29, D=16, window_left=9, window_right=2,
                   num_sink=2, alibi=True)
    bh = lambda x: np.asarray(x, np.float64).transpose(0, 2, 1, 3)
    m = oracle.live_mask(37, 29, 9, 2, 2)
    bias = w.bias.astype(np.float64)
    O, L = oracle.forward(bh(w.q), bh(w.k), bh(w.v), w.scale, m, bias)
    dO = bh(w.do)
    ref = oracle.backward(bh(w.q), bh(w.k), bh(w.v), O, dO, L, w.scale, m, bias)
    cu_q = np.arange(4, dtype=np.int32) * 37
    cu_k = np.arange(4, dtype=np.int32) * 29
    Ov, Lv = oracle.varlen_forward(_pack(w.q), _pack(w.k), _pack(w.v), cu_q, cu_k, w.scale, 37,
                                   9, 2, 2, bias=bias)
    np.testing.assert_allclose(Ov, _pack(O.transpose(0, 2, 1, 3)), rtol=0, atol=1e-13)
    np.testing.assert_allclose(Lv, L, rtol=0, atol=1e-13)
    got = oracle.varlen_backward(_pack(w.q), _pack(w.k), _pack(w.v), Ov, _pack(w.do), Lv, cu_q,
                                 cu_k, w.scale, 37, 29, 9, 2, 2, bias=bias)
    for g, r in zip(got[:3], ref[:3]):
        np.testing.assert_allclose(g, _pack(r.transpose(0, 2, 1, 3)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(got[3], ref[3], rtol=0, atol=1e-12)  # dbias summed over sequences


def test_sequences_are_independent_and_empty_ones_add_nothing():
    lq, lk = [6, 0, 9, 4], [7, 5, 0, 8]
    w = make_varlen("i", 5, lq, lk, Hq=2, Hk=1, D=8, window_left=-1, window_right=0,
                    num_sink=1, alibi=True)
    args = dict(window_left=-1, window_right=0, num_sink=1, bias=w.bias.astype(np.float64))
    O, L = oracle.varlen_forward(w.q, w.k, w.v, w.cu_q, w.cu_k, w.scale, w.max_q, **args)
    g1 = oracle.varlen_backward(w.q, w.k, w.v, O, w.do, L, w.cu_q, w.cu_k, w.scale, w.max_q,
                                w.max_k, **args)
    # the sequence with queries but no keys: LSE = -inf, O = 0, no gradient
    a, e = w.cu_q[2], w.cu_q[3]
    assert np.all(np.isneginf(L[2, :, :9])) and not O[a:e].any() and not g1[0][a:e].any()
    # keys of the sequence without queries get no gradient
    ka, ke = w.cu_k[1], w.cu_k[2]
    assert not g1[1][ka:ke].any() and not g1[2][ka:ke].any()
    # change the last sequence: the others are bitwise unchanged
    k2, q2 = w.k.copy(), w.q.copy()
    k2[w.cu_k[3]:] *= -0.5
    q2[w.cu_q[3]:] += 1.0
    O2, L2 = oracle.varlen_forward(q2, k2, w.v, w.cu_q, w.cu_k, w.scale, w.max_q, **args)
    g2 = oracle.varlen_backward(q2, k2, w.v, O2, w.do, L2, w.cu_q, w.cu_k, w.scale, w.max_q,
                                w.max_k, **args)
    qa, ka = w.cu_q[3], w.cu_k[3]
    assert np.array_equal(O[:qa], O2[:qa]) and np.array_equal(L[:3], L2[:3])
    assert np.array_equal(g1[0][:qa], g2[0][:qa])
    assert np.array_equal(g1[1][:ka], g2[1][:ka]) and np.array_equal(g1[2][:ka], g2[2][:ka])
    assert not np.array_equal(g1[0][qa:], g2[0][qa:])


def test_bottom_right_aligns_on_each_sequence():
    # two sequences with different Sk - Sq: brute-force scalar attention per
    # sequence with the offset of that sequence
    lq, lk = [3, 5], [6, 4]
    w = make_varlen("br", 6, lq, lk, Hq=2, Hk=2, D=4, window_left=1, window_right=0,
                    bottom_right=True)
    args = dict(window_left=1, window_right=0, bottom_right=True)
    O, L = oracle.varlen_forward(w.q, w.k, w.v, w.cu_q, w.cu_k, w.scale, w.max_q, **args)
    g = oracle.varlen_backward(w.q, w.k, w.v, O, w.do, L, w.cu_q, w.cu_k, w.scale, w.max_q,
                               w.max_k, **args)
    for b in range(2):
        qa, qe, ka, ke = w.cu_q[b], w.cu_q[b + 1], w.cu_k[b], w.cu_k[b + 1]
        off = (ke - ka) - (qe - qa)

        def live(i, j, off=off):
            return j >= i + off - 1 and j <= i + off

        seq = lambda x, a, e: np.asarray(x[a:e], np.float64).transpose(1, 0, 2)[None].tolist()
        Ob, Lb = brute.dense_forward(seq(w.q, qa, qe), seq(w.k, ka, ke), seq(w.v, ka, ke), w.scale,
                                     live)
        np.testing.assert_allclose(O[qa:qe], np.array(Ob)[0].transpose(1, 0, 2), atol=1e-12)
        np.testing.assert_allclose(L[b, :, :qe - qa], np.array(Lb)[0], atol=1e-12)
        dq, dk, dv, _ = brute.dense_backward(seq(w.q, qa, qe), seq(w.k, ka, ke), seq(w.v, ka, ke),
                                             seq(O, qa, qe), seq(w.do, qa, qe),
                                             L[b:b + 1, :, :qe - qa].tolist(), w.scale, live)
        np.testing.assert_allclose(g[0][qa:qe], np.array(dq)[0].transpose(1, 0, 2), atol=1e-12)
        np.testing.assert_allclose(g[1][ka:ke], np.array(dk)[0].transpose(1, 0, 2), atol=1e-12)
        np.testing.assert_allclose(g[2][ka:ke], np.array(dv)[0].transpose(1, 0, 2), atol=1e-12)
    # the first sequence's own offset (Sk - Sq = 3) is what decides: the
    # offset of the max lengths (6 - 5 = 1) gives another LSE
    seq = lambda x, a, e: np.asarray(x[a:e], np.float64).transpose(1, 0, 2)[None].tolist()
    _, L1 = brute.dense_forward(seq(w.q, 0, 3), seq(w.k, 0, 6), seq(w.v, 0, 6), w.scale,
                                lambda i, j: i <= j <= i + 1)
    assert not np.allclose(np.array(L1)[0], L[0, :, :3])
