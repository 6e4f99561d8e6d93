"""Seeded synthetic inputs for the attention backward pass.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark. It only draws and rounds input values and builds the input
structures (bias tables, top-k index lists). It contains none of the backward
pass arithmetic, and neither the oracle nor the CUDA library imports it.

Sources of the input recipes:
  * bf16 N(0, 1) tensors, seed per workload: the five workload descriptions
    of the attention backward benchmark (B, H, S, D, mask, bias, sparsity).
  * ALiBi bias, bias[h, i, j] = -2^(-8 (h + 1) / H) * |i - j|:
    composable_kernel example "28_backward_dbias_fmha.py", make_alibi_bias.
  * Top-k compressed-KV indices drawn uniformly without replacement from the
    eligible compressed rows, padded with -1: Ascend "sparse_flash_mla_grad",
    single-operator example (cmp_sparse_indices construction).
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "bf16_round",
    "bf16_bits",
    "alibi_bias",
    "topk_compressed_indices",
    "DenseWorkload",
    "SparseWorkload",
    "WORKLOADS",
    "make_dense",
    "make_sparse",
    "make_workload",
]


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bfloat16 (ties to even).

    Returns float32 values that are exactly representable in bfloat16.
    Inputs must be finite (the generators only produce finite values).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # For finite x the sum stays below 2^32 (largest finite pattern 0xFF7FFFFF).
    r = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    r &= np.uint32(0xFFFF0000)
    return r.view(np.float32).reshape(x.shape)


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """The upper 16 bits of float32 values that are already bf16-exact."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def alibi_bias(nhead: int, seqlen_q: int, seqlen_k: int) -> np.ndarray:
    """ALiBi distance penalty, float32 [H, Sq, Sk].

    slope_h = 2^(-8 (h + 1) / H); bias[h, i, j] = -slope_h * |i - j|
    (the slope is formed in double precision, the product stored as float32).
    """
    slopes = np.array([2.0 ** (-(8.0 * (h + 1) / nhead)) for h in range(nhead)])
    dist = np.abs(np.arange(seqlen_q)[:, None] - np.arange(seqlen_k)[None, :])
    out = np.empty((nhead, seqlen_q, seqlen_k), dtype=np.float32)
    for h in range(nhead):
        out[h] = (-slopes[h] * dist).astype(np.float32)
    return out


def topk_compressed_indices(
    rng: np.random.Generator,
    seqlen_q: int,
    n_ori: int,
    n_cmp: int,
    cmp_ratio: int,
    topk: int,
    n_kv_heads: int = 1,
) -> np.ndarray:
    """Top-k compressed-row indices, int32 [Sq, Hk, topk], -1 = unused slot.

    Query i sits at position delta_s + i of the original KV sequence
    (delta_s = n_ori - Sq). Compressed row c summarises original rows
    [c * cmp_ratio, (c + 1) * cmp_ratio); it is eligible for query i when
    c < (delta_s + i + 1) // cmp_ratio (clamped at 0), i.e. the compressed
    block ends at or before the query. min(eligible, topk) distinct rows are
    drawn uniformly without replacement into the leading slots; the rest stay
    -1. All KV heads share the draw of their token.
    """
    out = np.full((seqlen_q, n_kv_heads, topk), -1, dtype=np.int32)
    delta_s = n_ori - seqlen_q
    for i in range(seqlen_q):
        threshold = max(delta_s + i + 1, 0)
        eligible = min(threshold // cmp_ratio, n_cmp)
        if eligible == 0:
            continue
        count = min(eligible, topk)
        pick = rng.choice(eligible, size=count, replace=False).astype(np.int32)
        out[i, :, :count] = pick[None, :]
    return out


@dataclasses.dataclass
class DenseWorkload:
    """A dense (or masked / biased / GQA) backward problem.

    Tensors are float32 holding bf16-exact values, in the library's BSHD
    layout: q, do [B, Sq, Hq, D]; k, v [B, Sk, Hk, D]. bias is float32
    [Hq, Sq, Sk] or None. The mask is (window_left, window_right, num_sink)
    with -1 meaning unbounded, positions aligned top-left (bottom_right=True:
    the window is taken around j = i + Sk - Sq).
    """

    name: str
    B: int
    Hq: int
    Hk: int
    Sq: int
    Sk: int
    D: int
    scale: float
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray
    bias: Optional[np.ndarray] = None
    window_left: int = -1
    window_right: int = -1
    num_sink: int = 0
    want_dbias: bool = False
    bottom_right: bool = False

    @property
    def masked(self) -> bool:
        return self.window_left >= 0 or self.window_right >= 0


@dataclasses.dataclass
class SparseWorkload:
    """A shared-latent-KV sparse backward problem (one sequence, TND layout).

    q, do [Sq, Hq, D]; ori_kv [n_ori, Hk, D]; cmp_kv [n_cmp, Hk, D] or None;
    cmp_idx int32 [Sq, Hk, topk] or None. Original-KV window around the
    query's aligned position: [p - ori_win_left, p + ori_win_right] with
    p = (n_ori - Sq) + i.
    """

    name: str
    Sq: int
    Hq: int
    Hk: int
    D: int
    n_ori: int
    n_cmp: int
    topk: int
    cmp_ratio: int
    ori_win_left: int
    ori_win_right: int
    scale: float
    q: np.ndarray
    do: np.ndarray
    ori_kv: np.ndarray
    cmp_kv: Optional[np.ndarray]
    cmp_idx: Optional[np.ndarray]


def _normal_bf16(rng: np.random.Generator, shape, mult: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(shape, dtype=np.float32)
    if mult != 1.0:
        x *= np.float32(mult)
    return bf16_round(x)


def make_dense(
    name: str,
    seed: int,
    B: int,
    Hq: int,
    Hk: int,
    Sq: int,
    Sk: int,
    D: int,
    window_left: int = -1,
    window_right: int = -1,
    num_sink: int = 0,
    alibi: bool = False,
    want_dbias: bool = False,
    scale: Optional[float] = None,
    mult: float = 1.0,
    bottom_right: bool = False,
) -> DenseWorkload:
    """Draw q, k, v, dO (in that order) from default_rng(seed), N(0,1)*mult, bf16."""
    rng = np.random.default_rng(seed)
    q = _normal_bf16(rng, (B, Sq, Hq, D), mult)
    k = _normal_bf16(rng, (B, Sk, Hk, D), mult)
    v = _normal_bf16(rng, (B, Sk, Hk, D), mult)
    do = _normal_bf16(rng, (B, Sq, Hq, D), mult)
    bias = alibi_bias(Hq, Sq, Sk) if alibi else None
    return DenseWorkload(
        name=name, B=B, Hq=Hq, Hk=Hk, Sq=Sq, Sk=Sk, D=D,
        scale=float(1.0 / np.sqrt(D)) if scale is None else float(scale),
        q=q, k=k, v=v, do=do, bias=bias,
        window_left=window_left, window_right=window_right, num_sink=num_sink,
        want_dbias=want_dbias, bottom_right=bottom_right,
    )


@dataclasses.dataclass
class VarlenWorkload:
    """Variable-length batch in packed token-major ("TND") layout:
    q, do [Tq, Hq, D]; k, v [Tk, Hk, D]; sequence b holds query rows
    cu_q[b] .. cu_q[b + 1] - 1 and key rows cu_k[b] .. cu_k[b + 1] - 1.
    max_q / max_k bound the lengths; bias is float32 [Hq, max_q, max_k]
    indexed by positions within a sequence."""
    name: str
    Hq: int
    Hk: int
    D: int
    cu_q: np.ndarray
    cu_k: np.ndarray
    max_q: int
    max_k: int
    scale: float
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    do: np.ndarray
    bias: Optional[np.ndarray] = None
    window_left: int = -1
    window_right: int = -1
    num_sink: int = 0
    want_dbias: bool = False
    bottom_right: bool = False

    @property
    def B(self) -> int:
        return len(self.cu_q) - 1


def make_varlen(
    name: str,
    seed: int,
    lens_q,
    lens_k,
    Hq: int,
    Hk: int,
    D: int,
    window_left: int = -1,
    window_right: int = -1,
    num_sink: int = 0,
    alibi: bool = False,
    want_dbias: bool = False,
    bottom_right: bool = False,
    max_q: Optional[int] = None,
    max_k: Optional[int] = None,
) -> VarlenWorkload:
    """Draw packed q, k, v, dO (in that order) from default_rng(seed), N(0,1), bf16."""
    lens_q = np.asarray(lens_q, np.int64)
    lens_k = np.asarray(lens_k, np.int64)
    cu_q = np.concatenate([[0], np.cumsum(lens_q)]).astype(np.int32)
    cu_k = np.concatenate([[0], np.cumsum(lens_k)]).astype(np.int32)
    max_q = int(lens_q.max()) if max_q is None else int(max_q)
    max_k = int(lens_k.max()) if max_k is None else int(max_k)
    rng = np.random.default_rng(seed)
    q = _normal_bf16(rng, (int(cu_q[-1]), Hq, D))
    k = _normal_bf16(rng, (int(cu_k[-1]), Hk, D))
    v = _normal_bf16(rng, (int(cu_k[-1]), Hk, D))
    do = _normal_bf16(rng, (int(cu_q[-1]), Hq, D))
    bias = alibi_bias(Hq, max_q, max_k) if alibi else None
    return VarlenWorkload(
        name=name, Hq=Hq, Hk=Hk, D=D, cu_q=cu_q, cu_k=cu_k, max_q=max_q, max_k=max_k,
        scale=float(1.0 / np.sqrt(D)), q=q, k=k, v=v, do=do, bias=bias,
        window_left=window_left, window_right=window_right, num_sink=num_sink,
        want_dbias=want_dbias, bottom_right=bottom_right,
    )


def make_sparse(
    name: str,
    seed: int,
    Sq: int,
    Hq: int,
    Hk: int,
    D: int,
    n_ori: int,
    n_cmp: int,
    topk: int,
    cmp_ratio: int,
    ori_win_left: int,
    ori_win_right: int = 0,
    mult: float = 0.5,
    with_cmp: bool = True,
    cfa: bool = False,
) -> SparseWorkload:
    """Draw q, ori_kv, cmp_kv, dO (in that order), then the top-k indices.

    cfa=True keeps cmp_kv but draws no index list: every compressed row whose
    block of cmp_ratio positions ends at or before the query is selected.
    """
    rng = np.random.default_rng(seed)
    q = _normal_bf16(rng, (Sq, Hq, D), mult)
    ori_kv = _normal_bf16(rng, (n_ori, Hk, D), mult)
    cmp_kv = _normal_bf16(rng, (n_cmp, Hk, D), mult) if with_cmp else None
    do = _normal_bf16(rng, (Sq, Hq, D), mult)
    idx = (topk_compressed_indices(rng, Sq, n_ori, n_cmp, cmp_ratio, topk, Hk)
           if with_cmp and not cfa else None)
    return SparseWorkload(
        name=name, Sq=Sq, Hq=Hq, Hk=Hk, D=D, n_ori=n_ori,
        n_cmp=n_cmp if with_cmp else 0, topk=topk if with_cmp else 0,
        cmp_ratio=cmp_ratio, ori_win_left=ori_win_left, ori_win_right=ori_win_right,
        scale=float(1.0 / np.sqrt(D)), q=q, do=do, ori_kv=ori_kv,
        cmp_kv=cmp_kv, cmp_idx=idx,
    )


# The five benchmark workloads. Seed = workload number - 1.
WORKLOADS = {
    "mha_s64_d64": dict(kind="dense", seed=0, B=1, Hq=2, Hk=2, Sq=64, Sk=64, D=64),
    "gqa4_causal_s1024_d128": dict(kind="dense", seed=1, B=2, Hq=16, Hk=4, Sq=1024,
                                   Sk=1024, D=128, window_left=-1, window_right=0),
    "mha_alibi_dbias_s2048_d64": dict(kind="dense", seed=2, B=4, Hq=16, Hk=16, Sq=2048,
                                      Sk=2048, D=64, alibi=True, want_dbias=True),
    "gqa4_window1024_sink4_s8192_d128": dict(kind="dense", seed=3, B=1, Hq=32, Hk=8,
                                             Sq=8192, Sk=8192, D=128, window_left=1023,
                                             window_right=0, num_sink=4),
    "sparse_scfa_s4096_h64_d512": dict(kind="sparse", seed=4, Sq=4096, Hq=64, Hk=1, D=512,
                                       n_ori=4096, n_cmp=1024, topk=512, cmp_ratio=4,
                                       ori_win_left=127, ori_win_right=0),
}


def make_workload(name: str, **overrides):
    """Build one of the named workloads; keyword overrides shrink shapes for tests."""
    spec = dict(WORKLOADS[name])
    spec.update(overrides)
    kind = spec.pop("kind")
    if kind == "dense":
        return make_dense(name, **spec)
    return make_sparse(name, **spec)
