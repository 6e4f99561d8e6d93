"""Shared test plumbing: oracle expectations for a workload and GPU runs of it.

The oracle side receives exactly the values the GPU receives: bf16 inputs,
O rounded to bf16 and LSE rounded to fp32 (both produced by the oracle
forward). Tolerances follow the parity bar of the backward: per output
tensor, max|g - r| <= 1e-2 max|r| and sum|g - r| / sum|r| <= 1e-3.
"""

from __future__ import annotations

import numpy as np

import oracle
from workloads import bf16_round

MAX_REL = 1e-2
MEAN_REL = 1e-3


def bhsd(x):
    return np.ascontiguousarray(np.asarray(x, np.float64).transpose(0, 2, 1, 3))


def mask_of(w):
    if w.window_left < 0 and w.window_right < 0 and w.num_sink == 0:
        return None
    return oracle.live_mask(w.Sq, w.Sk, w.window_left, w.window_right, w.num_sink,
                            getattr(w, "bottom_right", False))


def dense_forward_inputs(w):
    """Oracle forward -> (O bf16-exact float32 BSHD, LSE float32 [B, Hq, Sq])."""
    m = mask_of(w)
    bias = None if w.bias is None else w.bias.astype(np.float64)
    O, L = oracle.forward(bhsd(w.q), bhsd(w.k), bhsd(w.v), w.scale, m, bias)
    O_b = bf16_round(O.transpose(0, 2, 1, 3).astype(np.float32))
    return np.ascontiguousarray(O_b), L.astype(np.float32), O, L


def dense_reference(w, O_b, L_f, batches=None, kv_heads=None):
    """Oracle backward on the rounded O / LSE, optionally on a subset.

    batches: slice of the batch; kv_heads: slice of KV heads (with their query
    heads). Returns dict dq [B', Sq, Hq', D], dk, dv [B', Sk, Hk', D], dbias
    [Hq', Sq, Sk] (summed over the selected batches only) in BSHD float64.
    """
    r = w.Hq // w.Hk
    bs = batches if batches is not None else slice(0, w.B)
    ks = kv_heads if kv_heads is not None else slice(0, w.Hk)
    qs = slice(ks.start * r, ks.stop * r)
    m = mask_of(w)
    bias = None if w.bias is None else w.bias[qs].astype(np.float64)
    Q = bhsd(w.q[bs][:, :, qs])
    K = bhsd(w.k[bs][:, :, ks])
    V = bhsd(w.v[bs][:, :, ks])
    dO = bhsd(w.do[bs][:, :, qs])
    O = bhsd(O_b[bs][:, :, qs])
    L = np.asarray(L_f[bs][:, qs], np.float64)
    dQ, dK, dV, dB = oracle.backward(Q, K, V, O, dO, L, w.scale, m, bias)
    t = lambda x: x.transpose(0, 2, 1, 3)
    return dict(dq=t(dQ), dk=t(dK), dv=t(dV), dbias=dB, delta=oracle.preprocess(O, dO))


def cfa_ratio(w):
    """cmp_ratio for the CFA case (compressed KV without an index list), else None."""
    return w.cmp_ratio if (w.cmp_kv is not None and w.cmp_idx is None) else None


def sparse_forward_inputs(w):
    q = np.asarray(w.q, np.float64)
    okv = np.asarray(w.ori_kv, np.float64)
    ckv = None if w.cmp_kv is None else np.asarray(w.cmp_kv, np.float64)
    O, L = oracle.sparse_forward(q, okv, ckv, w.cmp_idx, w.scale, w.ori_win_left, w.ori_win_right,
                                 cfa_ratio(w))
    return np.ascontiguousarray(bf16_round(O.astype(np.float32))), L.astype(np.float32), O, L


def sparse_reference(w, O_b, L_f):
    q = np.asarray(w.q, np.float64)
    okv = np.asarray(w.ori_kv, np.float64)
    ckv = None if w.cmp_kv is None else np.asarray(w.cmp_kv, np.float64)
    dq, dori, dcmp = oracle.sparse_backward(q, okv, ckv, w.cmp_idx, np.asarray(O_b, np.float64),
                                            np.asarray(w.do, np.float64),
                                            np.asarray(L_f, np.float64), w.scale,
                                            w.ori_win_left, w.ori_win_right, cfa_ratio(w))
    return dict(dq=dq, d_ori=dori, d_cmp=dcmp)


def check_close(name, got, ref, max_rel=MAX_REL, mean_rel=MEAN_REL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    scale = np.abs(ref).max()
    tot = np.abs(ref).sum()
    if scale == 0:
        assert err.max() == 0, f"{name}: expected zeros, max err {err.max()}"
        return 0.0, 0.0
    mx = err.max() / scale
    mr = err.sum() / tot
    assert mx <= max_rel, f"{name}: max|err|/max|ref| = {mx:.3e} > {max_rel}"
    assert mr <= mean_rel, f"{name}: sum|err|/sum|ref| = {mr:.3e} > {mean_rel}"
    return mx, mr


# ------------------------------------------------------------------ GPU ----

def to_dev_bf16(x, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev).to(torch.bfloat16)


def to_dev_f32(x, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev)


def gpu_dense_plan(w, O_b, L_f, dev="cuda", deterministic=False, cuda_cores=False):
    import attention_backward_attn_gb300 as ab
    q, k, v, o, do = (to_dev_bf16(x, dev) for x in (w.q, w.k, w.v, O_b, w.do))
    lse = to_dev_f32(L_f, dev)
    bias = None if w.bias is None else to_dev_f32(w.bias, dev)
    mask = ab.mask_from(w.window_left, w.window_right, w.num_sink,
                        getattr(w, "bottom_right", False))
    return ab.BackwardPlan(q, k, v, o, do, lse, w.scale, mask=mask, bias=bias,
                           want_dbias=w.want_dbias, deterministic=deterministic,
                           cuda_cores=cuda_cores)


def gpu_sparse_plan(w, O_b, L_f, dev="cuda", cuda_cores=False, deterministic=False):
    import torch
    import attention_backward_attn_gb300 as ab
    q = to_dev_bf16(w.q[None], dev)
    do = to_dev_bf16(w.do[None], dev)
    o = to_dev_bf16(O_b[None], dev)
    lse = to_dev_f32(L_f[None], dev)
    okv = to_dev_bf16(w.ori_kv, dev)
    ckv = None if w.cmp_kv is None else to_dev_bf16(w.cmp_kv, dev)
    idx = None if w.cmp_idx is None else torch.from_numpy(w.cmp_idx).to(dev)
    return ab.BackwardPlan(q, None, None, o, do, lse, w.scale, ori_kv=okv, cmp_kv=ckv,
                           cmp_idx=idx, ori_win_left=w.ori_win_left,
                           ori_win_right=w.ori_win_right, cmp_ratio=cfa_ratio(w) or 0,
                           cuda_cores=cuda_cores, deterministic=deterministic)


def varlen_forward_inputs(w):
    """Oracle forward of a packed batch -> (O bf16-exact float32 [Tq, Hq, D],
    LSE float32 [B, Hq, max_q])."""
    bias = None if w.bias is None else w.bias.astype(np.float64)
    O, L = oracle.varlen_forward(w.q, w.k, w.v, w.cu_q, w.cu_k, w.scale, w.max_q,
                                 w.window_left, w.window_right, w.num_sink, w.bottom_right, bias)
    return np.ascontiguousarray(bf16_round(O.astype(np.float32))), L.astype(np.float32)


def varlen_reference(w, O_b, L_f):
    bias = None if w.bias is None else w.bias.astype(np.float64)
    dq, dk, dv, db = oracle.varlen_backward(w.q, w.k, w.v, O_b, w.do, L_f, w.cu_q, w.cu_k,
                                            w.scale, w.max_q, w.max_k, w.window_left,
                                            w.window_right, w.num_sink, w.bottom_right, bias)
    return dict(dq=dq, dk=dk, dv=dv, dbias=db)


def gpu_varlen_plan(w, O_b, L_f, dev="cuda", deterministic=False):
    import torch
    import attention_backward_attn_gb300 as ab
    q, k, v, o, do = (to_dev_bf16(x, dev) for x in (w.q, w.k, w.v, O_b, w.do))
    lse = to_dev_f32(L_f, dev)
    bias = None if w.bias is None else to_dev_f32(w.bias, dev)
    mask = ab.mask_from(w.window_left, w.window_right, w.num_sink, w.bottom_right)
    cu_q = torch.from_numpy(np.asarray(w.cu_q, np.int32)).to(dev)
    cu_k = torch.from_numpy(np.asarray(w.cu_k, np.int32)).to(dev)
    return ab.BackwardPlan(q, k, v, o, do, lse, w.scale, mask=mask, bias=bias,
                           want_dbias=w.want_dbias, deterministic=deterministic,
                           cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=w.max_q,
                           max_seqlen_k=w.max_k)
