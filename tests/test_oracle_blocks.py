"""Pins for the row-block path of the dense float64 oracle (CPU only).

oracle.forward / oracle.backward walk the query rows in blocks of
oracle.dense._ROW_BLOCK rows and, inside a block, visit only the key columns
that are live for some row of the block (dbias strips are scattered back by
column position). Every full-size GPU parity comparison goes through that
path with many blocks, so it is checked here against two things that have
no blocking at all:

* the scalar-loop attention of tests/brute.py, with the block size shrunk to
  a few rows so that tiny problems span many blocks;
* a whole-matrix restatement of the page formulas (composable_kernel
  "34_bwd_gqa_fmha.py" cpu_fwd_with_intermediates / cpu_bwd_gqa,
  "28_backward_dbias_fmha.py" cpu_attention_bwd_dbias), on problems longer
  than the real block size with uneven block edges (Sq = 300, 520).

The masks are chosen so that a later block's live columns start past key 0
and are not contiguous (sinks plus a window), which is where a wrong row
slice, column selection or strip offset would move values.
"""

import numpy as np
import pytest

import brute
import oracle
import oracle.dense as odense


def _problem(seed, B, Hq, Hk, Sq, Sk, D, with_bias):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, Hq, Sq, D))
    K = rng.standard_normal((B, Hk, Sk, D))
    V = rng.standard_normal((B, Hk, Sk, D))
    dO = rng.standard_normal((B, Hq, Sq, D))
    bias = rng.standard_normal((Hq, Sq, Sk)) if with_bias else None
    return Q, K, V, dO, bias


def _whole_matrix(Q, K, V, dO, scale, live, bias):
    """Forward and backward of every (b, h) on the full [Sq, Sk] matrices."""
    B, Hq, Sq, D = Q.shape
    Hk, Sk = K.shape[1], K.shape[2]
    r = Hq // Hk
    O = np.zeros_like(Q)
    L = np.full((B, Hq, Sq), -np.inf)
    dQ = np.zeros_like(Q)
    dK = np.zeros_like(K)
    dV = np.zeros_like(V)
    dB = np.zeros((Hq, Sq, Sk))
    for b in range(B):
        for h in range(Hq):
            g = h // r
            S = scale * Q[b, h] @ K[b, g].T
            if bias is not None:
                S = S + bias[h]
            S = np.where(live, S, -np.inf)
            mx = S.max(axis=1, keepdims=True)
            mx = np.where(np.isfinite(mx), mx, 0.0)
            tot = np.exp(S - mx).sum(axis=1, keepdims=True)
            with np.errstate(divide="ignore", invalid="ignore"):
                lse = (mx + np.log(tot))[:, 0]
                P = np.where(live, np.exp(S - lse[:, None]), 0.0)
            O[b, h] = P @ V[b, g]
            L[b, h] = lse
    for b in range(B):
        for h in range(Hq):
            g = h // r
            S = scale * Q[b, h] @ K[b, g].T
            if bias is not None:
                S = S + bias[h]
            ok = live & np.isfinite(L[b, h])[:, None]
            P = np.where(ok, np.exp(np.where(ok, S, 0.0) - np.where(ok, L[b, h][:, None], 0.0)),
                         0.0)
            Dl = (dO[b, h] * O[b, h]).sum(axis=1)
            dS = P * (dO[b, h] @ V[b, g].T - Dl[:, None])
            dQ[b, h] = scale * dS @ K[b, g]
            dK[b, g] += scale * dS.T @ Q[b, h]
            dV[b, g] += P.T @ dO[b, h]
            dB[h] += dS
    return O, L, dQ, dK, dV, dB


# (Sq, Sk, window_left, window_right, num_sink, bottom_right, Hq, Hk, bias)
TINY = [
    (11, 11, -1, 0, 0, False, 4, 1, False),   # causal, GQA 4:1
    (13, 13, 3, 0, 2, False, 2, 1, True),     # window 4 + 2 sinks, bias (cols not contiguous)
    (9, 14, -1, 0, 0, True, 2, 2, True),      # bottom-right causal, Sk > Sq
    (14, 9, 2, 1, 1, True, 2, 1, False),      # bottom-right two-sided window, Sk < Sq (empty rows)
    (10, 12, -1, -1, 0, False, 1, 1, True),   # no mask, bias
]


@pytest.mark.parametrize("block", [1, 3, 4])
@pytest.mark.parametrize("case", TINY, ids=lambda c: f"sq{c[0]}_sk{c[1]}_w{c[2]}_{c[3]}_s{c[4]}"
                         f"{'_br' if c[5] else ''}_h{c[6]}x{c[7]}{'_bias' if c[8] else ''}")
def test_blocked_oracle_matches_scalar_loops(monkeypatch, block, case):
    Sq, Sk, wl, wr, ns, br, Hq, Hk, with_bias = case
    monkeypatch.setattr(odense, "_ROW_BLOCK", block)
    Q, K, V, dO, bias = _problem(7 + block, 1, Hq, Hk, Sq, Sk, 3, with_bias)
    scale = 0.6
    m = oracle.live_mask(Sq, Sk, wl, wr, ns, br)
    live = lambda i, j: bool(m[i, j])
    O, L = oracle.forward(Q, K, V, scale, m, bias)
    Ob, Lb = brute.dense_forward(Q, K, V, scale, live, bias)
    np.testing.assert_allclose(O, np.array(Ob), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(L), np.isinf(np.array(Lb)))
    fin = np.isfinite(L)
    np.testing.assert_allclose(L[fin], np.array(Lb)[fin], rtol=0, atol=1e-12)
    dQ, dK, dV, dB = oracle.backward(Q, K, V, O, dO, L, scale, m, bias)
    gQ, gK, gV, gB = brute.dense_backward(Q, K, V, O, dO, L, scale, live, bias)
    for got, ref in ((dQ, gQ), (dK, gK), (dV, gV), (dB, gB)):
        np.testing.assert_allclose(got, np.array(ref), rtol=0, atol=1e-12)


# Longer than the real block (256 rows): 2 and 3 blocks, ragged last block.
LONG = [
    (300, 300, -1, 0, 0, False, 4, 1, False),   # causal GQA 4:1
    (300, 310, 40, 0, 3, False, 2, 2, True),    # window 41 + 3 sinks, bias + dbias
    (520, 260, -1, 0, 0, True, 2, 1, True),     # bottom-right causal, Sk < Sq
    (290, 300, 100, 7, 0, True, 1, 1, False),   # bottom-right two-sided window
]


@pytest.mark.parametrize("case", LONG, ids=lambda c: f"sq{c[0]}_sk{c[1]}_w{c[2]}_{c[3]}_s{c[4]}"
                         f"{'_br' if c[5] else ''}_h{c[6]}x{c[7]}{'_bias' if c[8] else ''}")
def test_blocked_oracle_matches_whole_matrix(case):
    Sq, Sk, wl, wr, ns, br, Hq, Hk, with_bias = case
    assert Sq > odense._ROW_BLOCK and Sq % odense._ROW_BLOCK != 0
    Q, K, V, dO, bias = _problem(Sq + Sk, 1, Hq, Hk, Sq, Sk, 4, with_bias)
    scale = 0.5
    m = oracle.live_mask(Sq, Sk, wl, wr, ns, br)
    O, L = oracle.forward(Q, K, V, scale, m, bias)
    Ow, Lw, dQw, dKw, dVw, dBw = _whole_matrix(Q, K, V, dO, scale, m, bias)
    np.testing.assert_allclose(O, Ow, rtol=0, atol=1e-11)
    np.testing.assert_array_equal(np.isinf(L), np.isinf(Lw))
    fin = np.isfinite(L)
    np.testing.assert_allclose(L[fin], Lw[fin], rtol=0, atol=1e-11)
    dQ, dK, dV, dB = oracle.backward(Q, K, V, O, dO, L, scale, m, bias)
    for got, ref in ((dQ, dQw), (dK, dKw), (dV, dVw), (dB, dBw)):
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-10)
    # entries outside the mask carry no bias gradient at all
    assert not dB[:, ~m].any()


def test_block_columns_are_not_contiguous_in_the_long_window_case():
    # The sink + window case above must really exercise a non-contiguous,
    # non-zero-based column set in a later block (otherwise it would not pin
    # the strip offset of the dbias scatter).
    m = oracle.live_mask(300, 310, 40, 0, 3)
    cols, _ = odense._block_cols(m, 256, 300, 310)
    assert cols[0] == 0 and cols[3] > 3  # sinks, then a gap, then the window
    assert (np.diff(cols) > 1).any()
