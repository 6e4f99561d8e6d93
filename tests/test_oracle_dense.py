"""Pins for the dense float64 oracle (CPU only).

Each test checks the oracle against something other than itself: page
definitions written as loops, closed-form counts, brute-force scalar loops,
central finite differences of L = sum(O * dO), invariants and closed-form
special cases, and hand-derived values in tests/golden/.
"""

import json
import math
import os

import numpy as np
import pytest

import oracle
import brute
from workloads import make_dense, alibi_bias

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")


def _bhsd(x):
    """BSHD -> BHSD (the oracle's layout)."""
    return np.ascontiguousarray(np.asarray(x, np.float64).transpose(0, 2, 1, 3))


def _mask_of(w):
    if not w.masked and w.num_sink == 0:
        return None
    return oracle.live_mask(w.Sq, w.Sk, w.window_left, w.window_right, w.num_sink)


# ---------------------------------------------------------------- masks ----

def _loop_mask(sq, sk, pred):
    m = np.zeros((sq, sk), dtype=bool)
    for i in range(sq):
        for j in range(sk):
            m[i, j] = pred(i, j)
    return m


@pytest.mark.parametrize("sq,sk", [(1, 1), (7, 7), (16, 16), (5, 9), (9, 5)])
@pytest.mark.parametrize("sink", [0, 1, 4])
@pytest.mark.parametrize("window", [1, 3, 8])
def test_masks_equal_page_definitions(sq, sk, sink, window):
    # "22_sink_tokens_fmha.py": the three mask builders, as scalar loops.
    causal = _loop_mask(sq, sk, lambda i, j: j <= i)
    csink = _loop_mask(sq, sk, lambda i, j: j < sink or j <= i)
    wsink = _loop_mask(sq, sk, lambda i, j: j < sink or (i - window + 1 <= j <= i))
    assert np.array_equal(oracle.causal_mask(sq, sk), causal)
    assert np.array_equal(oracle.causal_sink_mask(sq, sk, sink), csink)
    assert np.array_equal(oracle.window_sink_mask(sq, sk, window, sink), wsink)
    # The library parametrisation (left, right, sink) maps onto them.
    assert np.array_equal(oracle.live_mask(sq, sk, -1, 0, 0), causal)
    assert np.array_equal(oracle.live_mask(sq, sk, -1, 0, sink), csink)
    assert np.array_equal(oracle.live_mask(sq, sk, window - 1, 0, sink), wsink)
    assert oracle.live_mask(sq, sk, -1, -1, 0).all()


@pytest.mark.parametrize("sq,sk", [(5, 5), (5, 9), (9, 5), (1, 6), (6, 1)])
@pytest.mark.parametrize("left,right,sink", [(-1, 0, 0), (-1, 0, 2), (2, 0, 1), (1, 2, 0)])
def test_bottom_right_alignment(sq, sk, left, right, sink):
    # Bottom-right: the diagonal ends in the last query / key corner, i.e. the
    # window test uses i + (sk - sq); checked as a scalar loop.
    off = sk - sq

    def live(i, j):
        if j < sink:
            return True
        ii = i + off
        return (left < 0 or j >= ii - left) and (right < 0 or j <= ii + right)

    got = oracle.live_mask(sq, sk, left, right, sink, bottom_right=True)
    assert np.array_equal(got, _loop_mask(sq, sk, live))
    if sq == sk:  # the two alignments coincide
        assert np.array_equal(got, oracle.live_mask(sq, sk, left, right, sink))
    if left < 0 and right == 0 and sink == 0:
        # causal: sk >= sq is top-left causal widened by sk - sq; sk < sq leaves
        # the first sq - sk queries without a key
        if sk >= sq:
            assert np.array_equal(got, oracle.live_mask(sq, sk, -1, sk - sq, 0))
        else:
            assert not got[:sq - sk].any() and got[sq - sk:].any(axis=1).all()


def test_live_entry_counts_closed_form():
    # Causal S=1024: sum_{i} (i + 1) = S (S + 1) / 2.
    assert oracle.live_mask(1024, 1024, -1, 0, 0).sum() == 1024 * 1025 // 2
    # Window 1024 + 4 sinks, S = 8192 (derived by hand, row by row):
    #   rows 0..3 see the 4 sinks (which cover j <= i): 4 each;
    #   rows 4..1023 see j <= i: i + 1 each;
    #   rows 1024, 1025, 1026 see the window plus 1, 2, 3 sinks outside it;
    #   rows >= 1027 see 1024 window keys + 4 sinks.
    s, w, n = 8192, 1024, 4
    expect = 4 * 4 + sum(i + 1 for i in range(4, 1024)) + (1025 + 1026 + 1027) + (s - 1027) * (w + n)
    assert expect == 7893504
    assert oracle.live_mask(s, s, w - 1, 0, n).sum() == expect


# ---------------------------------------------------------- brute force ----

def _tiny_cases():
    return [
        dict(B=1, Hq=1, Hk=1, Sq=3, Sk=4, D=2),
        dict(B=2, Hq=4, Hk=2, Sq=5, Sk=5, D=3, window_left=-1, window_right=0),
        dict(B=1, Hq=4, Hk=1, Sq=6, Sk=6, D=2, window_left=1, window_right=0, num_sink=2),
        dict(B=2, Hq=2, Hk=2, Sq=4, Sk=3, D=2, alibi=True),
        dict(B=1, Hq=2, Hk=1, Sq=4, Sk=6, D=2, window_left=2, window_right=1),
    ]


@pytest.mark.parametrize("case", _tiny_cases())
def test_oracle_matches_brute_force(case):
    w = make_dense("tiny", seed=11, **case)
    m = _mask_of(w)
    Q, K, V, dO = _bhsd(w.q), _bhsd(w.k), _bhsd(w.v), _bhsd(w.do)
    live = (lambda i, j: True) if m is None else (lambda i, j: bool(m[i, j]))
    O_b, L_b = brute.dense_forward(Q.tolist(), K.tolist(), V.tolist(), w.scale, live, w.bias)
    O, L = oracle.forward(Q, K, V, w.scale, m, w.bias)
    np.testing.assert_allclose(O, np.array(O_b), rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, np.array(L_b), rtol=0, atol=1e-12)
    got = oracle.backward(Q, K, V, O, dO, L, w.scale, m, w.bias)
    ref = brute.dense_backward(Q.tolist(), K.tolist(), V.tolist(), O.tolist(), dO.tolist(),
                               L.tolist(), w.scale, live, w.bias)
    for g, r in zip(got, ref):
        np.testing.assert_allclose(g, np.array(r), rtol=0, atol=1e-12)


# ---------------------------------------------------- finite differences ----

def _loss(Q, K, V, dO, scale, m, bias):
    O, _ = oracle.forward(Q, K, V, scale, m, bias)
    return float((O * dO).sum())


FD_CASES = [
    dict(B=1, Hq=2, Hk=2, Sq=5, Sk=6, D=4),
    dict(B=2, Hq=4, Hk=2, Sq=6, Sk=6, D=3, window_left=-1, window_right=0),
    dict(B=1, Hq=4, Hk=1, Sq=7, Sk=7, D=3, window_left=2, window_right=0, num_sink=2),
    dict(B=2, Hq=2, Hk=2, Sq=4, Sk=5, D=3, alibi=True),
]


@pytest.mark.parametrize("case", FD_CASES)
def test_finite_differences(case):
    w = make_dense("fd", seed=5, **case)
    m = _mask_of(w)
    Q, K, V, dO = _bhsd(w.q), _bhsd(w.k), _bhsd(w.v), _bhsd(w.do)
    bias = None if w.bias is None else w.bias.astype(np.float64)
    O, L = oracle.forward(Q, K, V, w.scale, m, bias)  # exact mode: unrounded O, LSE
    dQ, dK, dV, dB = oracle.backward(Q, K, V, O, dO, L, w.scale, m, bias)
    rng = np.random.default_rng(3)
    eps = 1e-6
    targets = [("Q", Q, dQ), ("K", K, dK), ("V", V, dV)]
    if bias is not None:
        targets.append(("bias", bias, dB))
    for name, X, G in targets:
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in X.shape)
            Xp, Xm = X.copy(), X.copy()
            Xp[idx] += eps
            Xm[idx] -= eps
            args_p = dict(Q=Q, K=K, V=V, bias=bias)
            args_m = dict(Q=Q, K=K, V=V, bias=bias)
            args_p[name] = Xp
            args_m[name] = Xm
            num = (_loss(args_p["Q"], args_p["K"], args_p["V"], dO, w.scale, m, args_p["bias"])
                   - _loss(args_m["Q"], args_m["K"], args_m["V"], dO, w.scale, m, args_m["bias"])) / (2 * eps)
            assert abs(num - G[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx, num, G[idx])


# ------------------------------------------------------------ invariants ----

@pytest.mark.parametrize("case", FD_CASES)
def test_ds_rows_sum_to_zero_and_vanish_on_masked(case):
    # sum_j dS_ij = sum_j P_ij dP_ij - D_i = dO_i . O_i - D_i = 0 (exact O).
    # dbias sums dS over the batch, so its rows sum to zero as well.
    w = make_dense("inv", seed=7, **case)
    m = _mask_of(w)
    Q, K, V, dO = _bhsd(w.q), _bhsd(w.k), _bhsd(w.v), _bhsd(w.do)
    O, L = oracle.forward(Q, K, V, w.scale, m, w.bias)
    _, _, _, dB = oracle.backward(Q, K, V, O, dO, L, w.scale, m, w.bias)
    np.testing.assert_allclose(dB.sum(axis=-1), 0.0, atol=1e-12)
    if m is not None:
        assert np.all(dB[:, ~m] == 0.0)


@pytest.mark.parametrize("ratio", [1, 2, 4])
def test_gqa_equals_expanded_mha_then_group_sum(ratio):
    # "34_bwd_gqa_fmha.py": GQA backward == MHA backward on np.repeat-expanded
    # K / V followed by summing dK / dV over each query-head group.
    Hq = 8
    w = make_dense("gqa", seed=9, B=2, Hq=Hq, Hk=Hq // ratio, Sq=12, Sk=10, D=4,
                   window_left=-1, window_right=0)
    m = _mask_of(w)
    Q, K, V, dO = _bhsd(w.q), _bhsd(w.k), _bhsd(w.v), _bhsd(w.do)
    O, L = oracle.forward(Q, K, V, w.scale, m)
    dQ, dK, dV, _ = oracle.backward(Q, K, V, O, dO, L, w.scale, m)
    Ke, Ve = np.repeat(K, ratio, axis=1), np.repeat(V, ratio, axis=1)
    Oe, Le = oracle.forward(Q, Ke, Ve, w.scale, m)
    np.testing.assert_allclose(Oe, O, atol=1e-12)
    dQe, dKe, dVe, _ = oracle.backward(Q, Ke, Ve, Oe, dO, Le, w.scale, m)
    B, Hk, Sk, D = K.shape
    np.testing.assert_allclose(dQe, dQ, atol=1e-12)
    np.testing.assert_allclose(dKe.reshape(B, Hk, ratio, Sk, D).sum(axis=2), dK, atol=1e-12)
    np.testing.assert_allclose(dVe.reshape(B, Hk, ratio, Sk, D).sum(axis=2), dV, atol=1e-12)


# ---------------------------------------------------------- closed forms ----

def test_single_key_closed_form():
    # Sk = 1: P = 1, dS = 0, so dQ = dK = 0 and dV = sum over rows and heads of dO.
    w = make_dense("sk1", seed=1, B=2, Hq=4, Hk=2, Sq=5, Sk=1, D=3)
    Q, K, V, dO = _bhsd(w.q), _bhsd(w.k), _bhsd(w.v), _bhsd(w.do)
    O, L = oracle.forward(Q, K, V, w.scale)
    np.testing.assert_allclose(O, np.repeat(V, 2, axis=1).repeat(5, axis=2), atol=1e-15)
    dQ, dK, dV, _ = oracle.backward(Q, K, V, O, dO, L, w.scale)
    assert np.abs(dQ).max() < 1e-14 and np.abs(dK).max() < 1e-14
    expect = dO.reshape(2, 2, 2, 5, 3).sum(axis=(2, 3))[:, :, None, :]
    np.testing.assert_allclose(dV, expect, atol=1e-13)


def test_constant_value_rows_give_zero_dq_dk():
    # All V rows equal: O_i = v, dP_ij = dO_i . v = D_i, so dS = 0.
    w = make_dense("cv", seed=2, B=1, Hq=2, Hk=1, Sq=6, Sk=7, D=4,
                   window_left=2, window_right=1, num_sink=1)
    m = _mask_of(w)
    Q, K, dO = _bhsd(w.q), _bhsd(w.k), _bhsd(w.do)
    V = np.broadcast_to(_bhsd(w.v)[:, :, :1, :], K.shape).copy()
    O, L = oracle.forward(Q, K, V, w.scale, m)
    dQ, dK, dV, dB = oracle.backward(Q, K, V, O, dO, L, w.scale, m)
    assert np.abs(dQ).max() < 1e-13 and np.abs(dK).max() < 1e-13 and np.abs(dB).max() < 1e-13


def test_bias_constant_along_keys_is_invisible():
    # bias[h, i, j] = c[h, i] shifts every logit of a row equally: O and dQ/dK/dV
    # are unchanged, LSE moves by c, and dbias rows sum to zero.
    w = make_dense("bc", seed=4, B=2, Hq=2, Hk=2, Sq=5, Sk=6, D=3)
    Q, K, V, dO = _bhsd(w.q), _bhsd(w.k), _bhsd(w.v), _bhsd(w.do)
    c = np.random.default_rng(0).standard_normal((2, 5))
    bias = np.repeat(c[:, :, None], 6, axis=2)
    O0, L0 = oracle.forward(Q, K, V, w.scale)
    O1, L1 = oracle.forward(Q, K, V, w.scale, None, bias)
    np.testing.assert_allclose(O1, O0, atol=1e-13)
    np.testing.assert_allclose(L1 - L0, np.broadcast_to(c, L0.shape), atol=1e-13)
    g0 = oracle.backward(Q, K, V, O0, dO, L0, w.scale)
    g1 = oracle.backward(Q, K, V, O1, dO, L1, w.scale, None, bias)
    for a, b in zip(g0[:3], g1[:3]):
        np.testing.assert_allclose(a, b, atol=1e-12)
    np.testing.assert_allclose(g1[3].sum(axis=-1), 0.0, atol=1e-12)


def test_fully_masked_row_is_zero():
    # A key window that excludes every key of a row: LSE = -inf, O = 0, no gradient.
    w = make_dense("empty", seed=6, B=1, Hq=1, Hk=1, Sq=4, Sk=4, D=2)
    Q, K, V, dO = _bhsd(w.q), _bhsd(w.k), _bhsd(w.v), _bhsd(w.do)
    m = np.ones((4, 4), dtype=bool)
    m[2] = False
    O, L = oracle.forward(Q, K, V, w.scale, m)
    assert L[0, 0, 2] == -np.inf and np.all(O[0, 0, 2] == 0)
    dQ, dK, dV, dB = oracle.backward(Q, K, V, O, dO, L, w.scale, m)
    assert np.all(dQ[0, 0, 2] == 0) and np.all(dB[0, 2] == 0)


# -------------------------------------------------------- hand examples ----

def _ev(x):
    if isinstance(x, list):
        return [_ev(y) for y in x]
    if isinstance(x, str):
        return eval(x, {"__builtins__": {}}, {"ln3": math.log(3.0), "ln4": math.log(4.0)})
    return float(x)


@pytest.mark.parametrize("name", ["dense_two_keys", "causal_two_rows", "bias_two_keys_two_batches"])
def test_hand_derived_examples(name):
    ex = json.load(open(GOLDEN))[name]
    Q, K, V, dO = (np.array(_ev(ex[k])) for k in ("q", "k", "v", "do"))
    bias = np.array(_ev(ex["bias"])) if "bias" in ex else None
    m = oracle.causal_mask(Q.shape[2], K.shape[2]) if ex.get("mask") == "causal" else None
    O, L = oracle.forward(Q, K, V, ex["scale"], m, bias)
    dQ, dK, dV, dB = oracle.backward(Q, K, V, O, dO, L, ex["scale"], m, bias)
    got = dict(O=O, LSE=L, dQ=dQ, dK=dK, dV=dV, dbias=dB)
    for key, val in ex["expect"].items():
        np.testing.assert_allclose(got[key], np.array(_ev(val)), rtol=0, atol=1e-14, err_msg=key)


def test_alibi_generator_matches_formula():
    # "28_backward_dbias_fmha.py" make_alibi_bias, spot values by hand:
    # H = 4: slope_0 = 2^-2, slope_3 = 2^-8.
    b = alibi_bias(4, 5, 6)
    assert b.shape == (4, 5, 6) and b.dtype == np.float32
    assert b[0, 0, 0] == 0.0 and b[0, 0, 4] == np.float32(-0.25 * 4)
    assert b[3, 4, 1] == np.float32(-(2.0 ** -8) * 3)
    sq = alibi_bias(3, 7, 7)
    assert np.array_equal(sq, sq.transpose(0, 2, 1))  # |i - j| is symmetric


def _sink_case(seed=11, B=2, Hq=4, Hk=2, Sq=6, Sk=7, D=3):
    rng = np.random.default_rng(seed)
    Q = rng.standard_normal((B, Hq, Sq, D))
    K = rng.standard_normal((B, Hk, Sk, D))
    V = rng.standard_normal((B, Hk, Sk, D))
    dO = rng.standard_normal((B, Hq, Sq, D))
    sinks = rng.standard_normal(Hq)
    return Q, K, V, dO, sinks


def test_sink_logit_equals_an_extra_key_with_zero_value():
    # A sink logit s_h behaves as one more key, live for every query, with a
    # zero key and value vector and bias s_h: the same O and LSE, and dsink_h
    # is that column's bias gradient summed over the queries.
    Q, K, V, dO, sinks = _sink_case()
    B, Hq, Sq, D = Q.shape
    Hk, Sk = K.shape[1], K.shape[2]
    m = oracle.live_mask(Sq, Sk, 1, 0, 1)
    O, L = oracle.forward(Q, K, V, 0.7, m, None, sinks)
    Kx = np.concatenate([K, np.zeros((B, Hk, 1, D))], axis=2)
    Vx = np.concatenate([V, np.zeros((B, Hk, 1, D))], axis=2)
    mx = np.concatenate([m, np.ones((Sq, 1), dtype=bool)], axis=1)
    bx = np.zeros((Hq, Sq, Sk + 1))
    bx[:, :, Sk] = sinks[:, None]
    Ox, Lx = oracle.forward(Q, Kx, Vx, 0.7, mx, bx)
    np.testing.assert_allclose(O, Ox, atol=1e-13)
    np.testing.assert_allclose(L, Lx, atol=1e-13)
    dQ, dK, dV, _ = oracle.backward(Q, K, V, O, dO, L, 0.7, m)
    dQx, dKx, dVx, dbx = oracle.backward(Q, Kx, Vx, Ox, dO, Lx, 0.7, mx, bx)
    np.testing.assert_allclose(dQ, dQx, atol=1e-12)
    np.testing.assert_allclose(dK, dKx[:, :, :Sk], atol=1e-12)
    np.testing.assert_allclose(dV, dVx[:, :, :Sk], atol=1e-12)
    ds = oracle.dsinks(L, oracle.preprocess(O, dO), sinks)
    np.testing.assert_allclose(ds, dbx[:, :, Sk].sum(axis=1), atol=1e-12)


def test_dsinks_finite_differences():
    Q, K, V, dO, sinks = _sink_case(seed=12)
    m = oracle.live_mask(Q.shape[2], K.shape[2], -1, 0, 0)
    O, L = oracle.forward(Q, K, V, 0.5, m, None, sinks)
    ds = oracle.dsinks(L, oracle.preprocess(O, dO), sinks)
    eps = 1e-6
    for h in range(len(sinks)):
        vals = []
        for sgn in (1, -1):
            s2 = sinks.copy()
            s2[h] += sgn * eps
            O2, _ = oracle.forward(Q, K, V, 0.5, m, None, s2)
            vals.append(float((O2 * dO).sum()))
        num = (vals[0] - vals[1]) / (2 * eps)
        assert abs(num - ds[h]) <= 1e-6 * max(1.0, abs(num)), (h, num, ds[h])


def test_sinks_at_minus_infinity_change_nothing():
    Q, K, V, dO, _ = _sink_case(seed=13)
    m = oracle.live_mask(Q.shape[2], K.shape[2], -1, 0, 0)
    off = np.full(Q.shape[1], -np.inf)
    O, L = oracle.forward(Q, K, V, 0.5, m)
    O2, L2 = oracle.forward(Q, K, V, 0.5, m, None, off)
    np.testing.assert_array_equal(O, O2)
    np.testing.assert_array_equal(L, L2)
    assert np.all(oracle.dsinks(L2, oracle.preprocess(O2, dO), off) == 0)
