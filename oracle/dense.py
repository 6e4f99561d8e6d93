"""Dense / masked / biased / GQA attention forward and backward in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring). Layout follows the
source pages: Q [B, Hq, Sq, D], K [B, Hk, Sk, D], V [B, Hk, Sk, Dv],
O and dO [B, Hq, Sq, Dv], LSE [B, Hq, Sq], bias [Hq, Sq, Sk] broadcast over
the batch. Query head h reads KV head h // (Hq // Hk) (np.repeat along the
head axis in "34_bwd_gqa_fmha.py", cpu_fwd_with_intermediates).

Masked entries are excluded from the softmax (P = 0, dS = 0 exactly). The
page's masked forward writes float32-min into the logits instead; the two
agree whenever a row has at least one live entry. A row with no live entry
gets LSE = -inf, O = 0 and zero gradients.

Rows are processed in blocks and, inside a block, only the key columns that
are live for at least one row of the block are visited; columns dead for the
whole block contribute exactly zero, so this is the same sum.
"""

from __future__ import annotations

from typing import Optional, Tuple

import numpy as np

_ROW_BLOCK = 256


# --------------------------------------------------------------------------
# Masks ("22_sink_tokens_fmha.py": make_causal_mask, make_causal_sink_mask,
# make_sliding_window_sink_mask). True = attend.
# --------------------------------------------------------------------------

def _grid(seqlen_q: int, seqlen_k: int):
    i = np.arange(seqlen_q)[:, None]
    j = np.arange(seqlen_k)[None, :]
    return i, j


def causal_mask(seqlen_q: int, seqlen_k: int) -> np.ndarray:
    """Top-left causal: query i attends key j iff j <= i."""
    i, j = _grid(seqlen_q, seqlen_k)
    return j <= i


def causal_sink_mask(seqlen_q: int, seqlen_k: int, num_sink: int) -> np.ndarray:
    """Causal plus sinks: j < num_sink or j <= i (sinks override causality)."""
    i, j = _grid(seqlen_q, seqlen_k)
    return (j < num_sink) | (j <= i)


def window_sink_mask(seqlen_q: int, seqlen_k: int, window: int, num_sink: int) -> np.ndarray:
    """Sliding window plus sinks: j < num_sink or i - window + 1 <= j <= i."""
    i, j = _grid(seqlen_q, seqlen_k)
    return (j < num_sink) | ((i - window + 1 <= j) & (j <= i))


def live_mask(seqlen_q: int, seqlen_k: int, window_left: int = -1,
              window_right: int = -1, num_sink: int = 0,
              bottom_right: bool = False) -> np.ndarray:
    """The library's mask parametrisation.

    live(i, j) = (j < num_sink) or (i' - window_left <= j <= i' + window_right),
    where a negative window bound means that side is unbounded. So causal is
    (-1, 0, 0), causal + n sinks is (-1, 0, n) and a window of w keys plus n
    sinks is (w - 1, 0, n). Positions are aligned top-left (i' = i) or, with
    bottom_right, so that the diagonal ends in the last query / key corner
    (i' = i + seqlen_k - seqlen_q: the "22_sink_tokens_fmha.py" mask format
    names both alignments for the causal mask).
    """
    i, j = _grid(seqlen_q, seqlen_k)
    if bottom_right:
        i = i + (seqlen_k - seqlen_q)
    inside = np.ones((seqlen_q, seqlen_k), dtype=bool)
    if window_left >= 0:
        inside &= j >= i - window_left
    if window_right >= 0:
        inside &= j <= i + window_right
    return inside | (j < num_sink)


# --------------------------------------------------------------------------
# Forward with LSE ("34_bwd_gqa_fmha.py" cpu_fwd_with_intermediates,
# "28_backward_dbias_fmha.py" cpu_attention_fwd_bias,
# "22_sink_tokens_fmha.py" cpu_attention_fwd_masked)
# --------------------------------------------------------------------------

def _blocks(n: int):
    for r0 in range(0, n, _ROW_BLOCK):
        yield r0, min(n, r0 + _ROW_BLOCK)


def _block_cols(mask: Optional[np.ndarray], r0: int, r1: int, seqlen_k: int):
    if mask is None:
        return np.arange(seqlen_k), None
    m = mask[r0:r1]
    cols = np.nonzero(m.any(axis=0))[0]
    return cols, m[:, cols]


def forward(Q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
            mask: Optional[np.ndarray] = None,
            bias: Optional[np.ndarray] = None,
            sinks: Optional[np.ndarray] = None) -> Tuple[np.ndarray, np.ndarray]:
    """O = softmax(scale Q K^T + bias, masked) V and LSE = natural log-sum-exp.

    sinks (float [Hq], optional): a learnable logit per query head that joins
    every row's softmax denominator without a value vector (the Ascend
    "sparse_flash_mla_grad" sinks input): LSE = log(sum_j exp(S_ij) +
    exp(sink_h)), O = sum_j exp(S_ij - LSE) V_j.

    Returns (O [B, Hq, Sq, Dv] float64, LSE [B, Hq, Sq] float64).
    """
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    B, Hq, Sq, _ = Q.shape
    Hk, Sk, Dv = K.shape[1], K.shape[2], V.shape[3]
    ratio = Hq // Hk
    O = np.zeros((B, Hq, Sq, Dv))
    LSE = np.full((B, Hq, Sq), -np.inf)
    sk = None if sinks is None else np.asarray(sinks, np.float64)
    for b in range(B):
        for h in range(Hq):
            g = h // ratio
            sink = -np.inf if sk is None else sk[h]
            for r0, r1 in _blocks(Sq):
                cols, m = _block_cols(mask, r0, r1, Sk)
                if cols.size == 0:
                    LSE[b, h, r0:r1] = sink  # only the sink (or nothing) in the row
                    continue
                S = scale * (Q[b, h, r0:r1] @ K[b, g, cols].T)
                if bias is not None:
                    S = S + np.asarray(bias[h, r0:r1][:, cols], np.float64)
                if m is not None:
                    S = np.where(m, S, -np.inf)
                row_max = np.maximum(S.max(axis=1), sink)
                shift = np.where(np.isfinite(row_max), row_max, 0.0)
                E = np.exp(S - shift[:, None])
                denom = E.sum(axis=1) + np.exp(sink - shift)
                live = denom > 0
                P = np.zeros_like(E)
                P[live] = E[live] / denom[live, None]
                O[b, h, r0:r1] = P @ V[b, g, cols]
                with np.errstate(divide="ignore"):
                    LSE[b, h, r0:r1] = np.where(live, shift + np.log(denom), -np.inf)
    return O, LSE


# --------------------------------------------------------------------------
# Backward ("34_bwd_gqa_fmha.py" cpu_bwd_gqa; "28_backward_dbias_fmha.py"
# cpu_attention_bwd_dbias)
# --------------------------------------------------------------------------

def preprocess(O: np.ndarray, dO: np.ndarray) -> np.ndarray:
    """D = rowsum(dO * O) over the value dimension, [B, Hq, Sq]."""
    return (np.asarray(dO, np.float64) * np.asarray(O, np.float64)).sum(axis=-1)


def dsinks(LSE: np.ndarray, Dlt: np.ndarray, sinks: np.ndarray) -> np.ndarray:
    """Gradient of the sink logits, float [Hq] (Ascend "sparse_flash_mla_grad"
    formula, phase 3: dSinks = ReduceSum(-P x dP x SimpleSoftmax(sinks, lse))).

    The sink's probability in row (b, h, i) is p = exp(sink_h - LSE[b, h, i]);
    sum_j P_ij dP_ij = D[b, h, i]; so dsink_h = -sum_{b, i} p D[b, h, i]. A row
    with LSE = -inf (no live key and no sink) contributes nothing.
    """
    LSE = np.asarray(LSE, np.float64)
    Dlt = np.asarray(Dlt, np.float64)
    s = np.asarray(sinks, np.float64)[None, :, None]
    with np.errstate(invalid="ignore", over="ignore"):
        p = np.where(np.isfinite(LSE), np.exp(s - LSE), 0.0)
    return -(p * Dlt).sum(axis=(0, 2))


def backward(Q: np.ndarray, K: np.ndarray, V: np.ndarray, O: np.ndarray,
             dO: np.ndarray, LSE: np.ndarray, scale: float,
             mask: Optional[np.ndarray] = None,
             bias: Optional[np.ndarray] = None):
    """Gradients of the attention output with respect to Q, K, V and the bias.

    P is rebuilt from the given LSE: P = exp(scale Q K^T + bias - LSE) on live
    entries, 0 elsewhere. Then D = rowsum(dO * O), dP = dO V^T,
    dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO, with
    dK / dV summed over the Hq / Hk query heads that share a KV head, and
    dbias = sum over the batch of dS (no scale).

    Returns (dQ, dK, dV, dbias) in float64; dbias has shape [Hq, Sq, Sk].
    """
    Q = np.asarray(Q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    O = np.asarray(O, np.float64)
    dO = np.asarray(dO, np.float64)
    LSE = np.asarray(LSE, np.float64)
    B, Hq, Sq, D = Q.shape
    Hk, Sk, Dv = K.shape[1], K.shape[2], V.shape[3]
    ratio = Hq // Hk
    Dlt = preprocess(O, dO)
    dQ = np.zeros((B, Hq, Sq, D))
    dK = np.zeros((B, Hk, Sk, D))
    dV = np.zeros((B, Hk, Sk, Dv))
    dbias = np.zeros((Hq, Sq, Sk))
    for b in range(B):
        for h in range(Hq):
            g = h // ratio
            for r0, r1 in _blocks(Sq):
                cols, m = _block_cols(mask, r0, r1, Sk)
                if cols.size == 0:
                    continue
                S = scale * (Q[b, h, r0:r1] @ K[b, g, cols].T)
                if bias is not None:
                    S = S + np.asarray(bias[h, r0:r1][:, cols], np.float64)
                arg = S - LSE[b, h, r0:r1, None]
                live = np.isfinite(LSE[b, h, r0:r1])[:, None]
                if m is not None:
                    live = live & m
                arg = np.where(live, arg, -np.inf)
                P = np.exp(arg)
                dP = dO[b, h, r0:r1] @ V[b, g, cols].T
                dS = P * (dP - Dlt[b, h, r0:r1, None])
                dQ[b, h, r0:r1] = scale * (dS @ K[b, g, cols])
                dK[b, g, cols] += scale * (dS.T @ Q[b, h, r0:r1])
                dV[b, g, cols] += P.T @ dO[b, h, r0:r1]
                dbias[h, r0:r1, cols[0]:cols[-1] + 1] += _scatter_cols(dS, cols)
    return dQ, dK, dV, dbias


def _scatter_cols(block: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """Place the columns of `block` at positions cols - cols[0] of a dense strip."""
    out = np.zeros((block.shape[0], int(cols[-1] - cols[0] + 1)))
    out[:, cols - cols[0]] = block
    return out


# --------------------------------------------------------------------------
# Variable-length batches: packed sequences in token-major rows [T, H, D]
# (the TND layout of the Ascend "sparse_flash_mla_grad" page), each sequence
# its own attention problem.
# --------------------------------------------------------------------------

def _sequence(X: np.ndarray, a: int, e: int) -> np.ndarray:
    """Rows [a, e) of a packed [T, H, D] tensor as a [1, H, e - a, D] batch."""
    return np.asarray(X[a:e], np.float64).transpose(1, 0, 2)[None]


def varlen_forward(Q, K, V, cu_q, cu_k, scale: float, max_q: int, window_left: int = -1,
                   window_right: int = -1, num_sink: int = 0, bottom_right: bool = False,
                   bias: Optional[np.ndarray] = None):
    """forward() on every sequence of a packed batch.

    Sequence b holds query rows cu_q[b] .. cu_q[b+1]-1 and key rows
    cu_k[b] .. cu_k[b+1]-1; its mask is live_mask over its own lengths (so a
    bottom-right alignment uses its own Sk - Sq) and its bias is the
    top-left [Sq_b, Sk_b] corner of bias [Hq, max_q, max_k].
    Returns O [Tq, Hq, Dv] and LSE [B, Hq, max_q] (-inf past each length).
    """
    B = len(cu_q) - 1
    Hq, Dv = Q.shape[1], V.shape[2]
    O = np.zeros((Q.shape[0], Hq, Dv))
    LSE = np.full((B, Hq, max_q), -np.inf)
    for b in range(B):
        qa, qe, ka, ke = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        if qe == qa:
            continue
        m = live_mask(qe - qa, ke - ka, window_left, window_right, num_sink, bottom_right)
        bb = None if bias is None else bias[:, :qe - qa, :ke - ka]
        Ob, Lb = forward(_sequence(Q, qa, qe), _sequence(K, ka, ke), _sequence(V, ka, ke), scale,
                         m, bb)
        O[qa:qe] = Ob[0].transpose(1, 0, 2)
        LSE[b, :, :qe - qa] = Lb[0]
    return O, LSE


def varlen_backward(Q, K, V, O, dO, LSE, cu_q, cu_k, scale: float, max_q: int, max_k: int,
                    window_left: int = -1, window_right: int = -1, num_sink: int = 0,
                    bottom_right: bool = False, bias: Optional[np.ndarray] = None):
    """backward() on every sequence of a packed batch (layouts as in
    varlen_forward; LSE [B, Hq, max_q]).

    Returns dQ [Tq, Hq, D], dK [Tk, Hk, D], dV [Tk, Hk, Dv], and dbias
    [Hq, max_q, max_k]: the sum over sequences of each sequence's dS placed
    at its positions.
    """
    B = len(cu_q) - 1
    Hq = Q.shape[1]
    dQ = np.zeros(Q.shape)
    dK = np.zeros(K.shape)
    dV = np.zeros(V.shape)
    dbias = np.zeros((Hq, max_q, max_k))
    for b in range(B):
        qa, qe, ka, ke = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        if qe == qa or ke == ka:
            continue
        m = live_mask(qe - qa, ke - ka, window_left, window_right, num_sink, bottom_right)
        bb = None if bias is None else bias[:, :qe - qa, :ke - ka]
        gq, gk, gv, gb = backward(_sequence(Q, qa, qe), _sequence(K, ka, ke), _sequence(V, ka, ke),
                                  _sequence(O, qa, qe), _sequence(dO, qa, qe),
                                  np.asarray(LSE, np.float64)[b:b + 1, :, :qe - qa], scale, m, bb)
        dQ[qa:qe] = gq[0].transpose(1, 0, 2)
        dK[ka:ke] = gk[0].transpose(1, 0, 2)
        dV[ka:ke] = gv[0].transpose(1, 0, 2)
        dbias[:, :qe - qa, :ke - ka] += gb
    return dQ, dK, dV, dbias
