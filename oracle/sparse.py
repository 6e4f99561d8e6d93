"""Selected-KV sparse attention backward with shared latent KV, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring). Follows the Ascend
"sparse_flash_mla_grad" formula section:
  phase 1: selectedKv(i) = concat(oriKv rows in the window of query i,
           Gather(cmpKv, topkIndices[i])) in the SCFA case, concat(oriKv
           window, cmpKv) in the CFA case (no index list), the window alone in
           the SWA case;  K = V = selectedKv;
  phase 2: P = SimpleSoftmax(Mask(Q selectedKv^T scale), lse), i.e. P is
           rebuilt from the given LSE; dP = dO selectedKv^T;
           dS = P (dP - SoftmaxGrad(dO, O)) with SoftmaxGrad = rowsum(dO * O);
  phase 3: dQ = dS selectedKv scale;  dKV = dS^T Q scale + P^T dO, added back
           into the original and compressed KV rows it came from.

Layout (one sequence, "TND"): q, O, dO [Sq, Hq, D]; ori_kv [n_ori, Hk, D];
cmp_kv [n_cmp, Hk, D]; cmp_idx int [Sq, Hk, topk] with -1 = unused slot;
LSE [Hq, Sq]. Query head h reads KV head h // (Hq // Hk).

Query i sits at position p = (n_ori - Sq) + i of the original sequence (the
page's delta_s offset). Its original-KV window is [p - win_left,
p + win_right] clipped to [0, n_ori); a negative bound means unbounded.

CFA reading (the page's mask-mode table did not survive): compressed row c
summarises original positions [c * cmp_ratio, (c + 1) * cmp_ratio), and the
phase-2 Mask keeps it for query i when that block ends at or before p, i.e.
c < (p + 1) // cmp_ratio, clipped to n_cmp. This is the eligibility rule the
page's own example uses when it draws SCFA indices.
"""

from __future__ import annotations

from typing import Optional, Tuple

import numpy as np


def selected_rows(i: int, seqlen_q: int, n_ori: int, win_left: int, win_right: int,
                  idx_row: Optional[np.ndarray], n_cmp: int = 0,
                  cmp_ratio: Optional[int] = None) -> Tuple[np.ndarray, np.ndarray]:
    """(original rows, compressed rows) selected by query i for one KV head.

    idx_row given: SCFA (the listed rows, -1 = unused). idx_row None and
    cmp_ratio given: CFA (every eligible compressed row). Neither: SWA.
    """
    p = (n_ori - seqlen_q) + i
    lo = p - win_left if win_left >= 0 else 0
    hi = p + win_right if win_right >= 0 else n_ori - 1
    lo, hi = max(lo, 0), min(hi, n_ori - 1)
    ori = np.arange(lo, hi + 1) if hi >= lo else np.zeros(0, dtype=np.int64)
    if idx_row is None and cmp_ratio is not None:
        cmp = np.arange(min(n_cmp, max(p + 1, 0) // cmp_ratio), dtype=np.int64)
    elif idx_row is None:
        cmp = np.zeros(0, dtype=np.int64)
    else:
        idx_row = np.asarray(idx_row)
        cmp = idx_row[idx_row >= 0].astype(np.int64)
    return ori, cmp


def _gather(i, g, ori_kv, cmp_kv, cmp_idx, seqlen_q, win_left, win_right, cmp_ratio):
    n_ori = ori_kv.shape[0]
    idx_row = None if cmp_idx is None else cmp_idx[i, g]
    cfa_ratio = cmp_ratio if (cmp_kv is not None and cmp_idx is None) else None
    ori, cmp = selected_rows(i, seqlen_q, n_ori, win_left, win_right, idx_row,
                             0 if cmp_kv is None else cmp_kv.shape[0], cfa_ratio)
    parts = [ori_kv[ori, g]]
    if cmp.size:
        parts.append(cmp_kv[cmp, g])
    return ori, cmp, np.concatenate(parts, axis=0)


def _check_case(cmp_kv, cmp_idx, cmp_ratio):
    if cmp_kv is not None and cmp_idx is None and not (cmp_ratio and cmp_ratio >= 1):
        raise ValueError("CFA (compressed KV without an index list) needs cmp_ratio >= 1")


def sparse_forward(q: np.ndarray, ori_kv: np.ndarray, cmp_kv: Optional[np.ndarray],
                   cmp_idx: Optional[np.ndarray], scale: float, win_left: int,
                   win_right: int, cmp_ratio: Optional[int] = None,
                   sinks: Optional[np.ndarray] = None):
    """O [Sq, Hq, D] and LSE [Hq, Sq] (natural log) over the selected rows.

    sinks (float [Hq], optional): per-head logits that join the softmax
    denominator without a value vector (the page's sinks input)."""
    _check_case(cmp_kv, cmp_idx, cmp_ratio)
    q = np.asarray(q, np.float64)
    ori_kv = np.asarray(ori_kv, np.float64)
    cmp_kv = None if cmp_kv is None else np.asarray(cmp_kv, np.float64)
    Sq, Hq, D = q.shape
    Hk = ori_kv.shape[1]
    ratio = Hq // Hk
    O = np.zeros((Sq, Hq, D))
    LSE = np.full((Hq, Sq), -np.inf)
    sk = np.full(Hq, -np.inf) if sinks is None else np.asarray(sinks, np.float64)
    for i in range(Sq):
        for g in range(Hk):
            _, _, sel = _gather(i, g, ori_kv, cmp_kv, cmp_idx, Sq, win_left, win_right,
                                cmp_ratio)
            hs = slice(g * ratio, (g + 1) * ratio)
            if sel.shape[0] == 0:
                LSE[hs, i] = sk[hs]  # only the sink (or nothing)
                continue
            S = scale * (q[i, hs] @ sel.T)
            row_max = np.maximum(S.max(axis=1), sk[hs])
            E = np.exp(S - row_max[:, None])
            denom = E.sum(axis=1) + np.exp(sk[hs] - row_max)
            O[i, hs] = (E / denom[:, None]) @ sel
            LSE[hs, i] = row_max + np.log(denom)
    return O, LSE


def sparse_backward(q: np.ndarray, ori_kv: np.ndarray, cmp_kv: Optional[np.ndarray],
                    cmp_idx: Optional[np.ndarray], O: np.ndarray, dO: np.ndarray,
                    LSE: np.ndarray, scale: float, win_left: int, win_right: int,
                    cmp_ratio: Optional[int] = None):
    """Returns (dQ [Sq, Hq, D], d_ori_kv [n_ori, Hk, D], d_cmp_kv [n_cmp, Hk, D] or None)."""
    _check_case(cmp_kv, cmp_idx, cmp_ratio)
    q = np.asarray(q, np.float64)
    ori_kv = np.asarray(ori_kv, np.float64)
    cmp_kv = None if cmp_kv is None else np.asarray(cmp_kv, np.float64)
    O = np.asarray(O, np.float64)
    dO = np.asarray(dO, np.float64)
    LSE = np.asarray(LSE, np.float64)
    Sq, Hq, D = q.shape
    Hk = ori_kv.shape[1]
    ratio = Hq // Hk
    Dlt = (dO * O).sum(axis=-1)  # SoftmaxGrad(dO, O), [Sq, Hq]
    dQ = np.zeros((Sq, Hq, D))
    d_ori = np.zeros(ori_kv.shape)
    d_cmp = None if cmp_kv is None else np.zeros(cmp_kv.shape)
    for i in range(Sq):
        for g in range(Hk):
            ori, cmp, sel = _gather(i, g, ori_kv, cmp_kv, cmp_idx, Sq, win_left, win_right,
                                    cmp_ratio)
            if sel.shape[0] == 0:
                continue
            hs = slice(g * ratio, (g + 1) * ratio)
            lse = LSE[hs, i]
            S = scale * (q[i, hs] @ sel.T)
            arg = np.where(np.isfinite(lse)[:, None], S - lse[:, None], -np.inf)
            P = np.exp(arg)
            dP = dO[i, hs] @ sel.T
            dS = P * (dP - Dlt[i, hs][:, None])
            dQ[i, hs] = scale * (dS @ sel)
            dsel = scale * (dS.T @ q[i, hs]) + P.T @ dO[i, hs]
            n_o = ori.size
            np.add.at(d_ori[:, g], ori, dsel[:n_o])
            if cmp.size:
                np.add.at(d_cmp[:, g], cmp, dsel[n_o:])
    return dQ, d_ori, d_cmp
