"""Python binding of the GB300 fused attention backward C ABI (include/attn_bwd.h).

Argument marshalling only: every function here builds the C descriptors from
torch tensors (shapes, element strides, device pointers, the current CUDA
stream) and calls the same-named entry point of libattn_bwd.so. All
arithmetic runs in the library's CUDA kernels. Importing this package fails
loudly if the library has not been built (see `_build.build`).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

from . import _build

__all__ = [
    "AttnError", "Problem", "Mask", "Sparse", "lib", "status_string",
    "problem_from", "varlen_problem", "mask_from", "sparse_from", "ATTN_FLAG_DETERMINISTIC",
    "ATTN_FLAG_CUDA_CORES",
    "attn_fwd_lse", "attn_bwd_preprocess", "attn_bwd", "attn_bwd_workspace_size",
    "attn_read_device_status", "attn_bwd_path", "attn_bwd_noalloc", "BackwardPlan",
    "attn_bwd_dsinks", "attn_mask_tile_classes", "attn_debug_mask_live",
    "attn_debug_sparse_rows",
]

ATTN_OK = 0
STATUS_NAMES = {
    0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED", 3: "ATTN_ERR_CUDA",
    4: "ATTN_ERR_DEVICE_TIMEOUT", 5: "ATTN_ERR_INDEX_OOB", 6: "ATTN_ERR_RANGE",
    7: "ATTN_ERR_WORKSPACE",
}


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


class Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("Hq", ctypes.c_int32), ("Hk", ctypes.c_int32),
        ("Sq", ctypes.c_int32), ("Sk", ctypes.c_int32), ("D", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3),
        ("do_stride", ctypes.c_int64 * 3),
        ("flags", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("total_q", ctypes.c_int32), ("total_k", ctypes.c_int32),
    ]


class Mask(ctypes.Structure):
    _fields_ = [("window_left", ctypes.c_int32), ("window_right", ctypes.c_int32),
                ("num_sink", ctypes.c_int32), ("bottom_right", ctypes.c_int32)]


class Sparse(ctypes.Structure):
    _fields_ = [
        ("ori_kv", ctypes.c_void_p), ("cmp_kv", ctypes.c_void_p), ("cmp_idx", ctypes.c_void_p),
        ("n_ori", ctypes.c_int32), ("n_cmp", ctypes.c_int32), ("topk", ctypes.c_int32),
        ("ori_win_left", ctypes.c_int32), ("ori_win_right", ctypes.c_int32),
        ("d_ori_kv", ctypes.c_void_p), ("d_cmp_kv", ctypes.c_void_p),
        ("cmp_ratio", ctypes.c_int32),
    ]


def _load():
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(path)
    P = ctypes.POINTER
    vp, sz, st = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    L.attn_fwd_lse.argtypes = [P(Problem), P(Mask), P(Sparse), vp, vp, vp, vp, vp, vp, vp]
    L.attn_fwd_lse.restype = st
    L.attn_bwd_workspace_size.argtypes = [P(Problem), P(Mask), P(Sparse)]
    L.attn_bwd_workspace_size.restype = sz
    L.attn_bwd_preprocess.argtypes = [P(Problem), P(Sparse), vp, vp, vp, vp, vp, vp, vp, vp,
                                      vp, vp, sz, vp]
    L.attn_bwd_preprocess.restype = st
    L.attn_bwd.argtypes = [P(Problem), P(Mask), P(Sparse), vp, vp, vp, vp, vp, vp, vp,
                           vp, vp, vp, vp, vp, sz, vp]
    L.attn_bwd.restype = st
    L.attn_bwd_dsinks.argtypes = [P(Problem), vp, vp, vp, vp, vp]
    L.attn_bwd_dsinks.restype = st
    L.attn_read_device_status.argtypes = [vp, vp, P(ctypes.c_int32)]
    L.attn_read_device_status.restype = st
    L.attn_status_string.argtypes = [st]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_bwd_path.argtypes = [P(Problem), P(Mask), P(Sparse)]
    L.attn_bwd_path.restype = ctypes.c_int32
    L.attn_bwd_noalloc.argtypes = [P(Problem), P(Mask), P(Sparse), vp, vp, vp, vp, vp, vp, vp,
                                   vp, vp, vp, vp, vp, vp, P(ctypes.c_int32)]
    L.attn_bwd_noalloc.restype = st
    L.attn_mask_tile_classes.argtypes = [P(Mask), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_int32, vp]
    L.attn_mask_tile_classes.restype = st
    L.attn_debug_mask_live.argtypes = [P(Mask), ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       vp, vp, vp, vp]
    L.attn_debug_mask_live.restype = st
    L.attn_debug_sparse_rows.argtypes = [P(Problem), P(Sparse), vp, vp, ctypes.c_int32, vp]
    L.attn_debug_sparse_rows.restype = st
    return L


lib = _load()


def status_string(code: int) -> str:
    return lib.attn_status_string(code).decode()


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _ref(x):
    return None if x is None else ctypes.byref(x)


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code: int, where: str):
    if code != ATTN_OK:
        raise AttnError(code, where)


def _strides(t):
    s = t.stride()
    return (ctypes.c_int64 * 3)(s[0], s[1], s[2])


ATTN_FLAG_DETERMINISTIC = 1
ATTN_FLAG_CUDA_CORES = 2


def problem_from(q, k=None, v=None, o=None, do=None, scale: Optional[float] = None,
                 Sk: Optional[int] = None, Hk: Optional[int] = None,
                 deterministic: bool = False, cuda_cores: bool = False) -> Problem:
    """Problem descriptor from BSHD tensors (q [B, Sq, Hq, D], k / v [B, Sk, Hk, D])."""
    B, Sq, Hq, D = q.shape
    p = Problem()
    p.B, p.Sq, p.Hq, p.D = B, Sq, Hq, D
    p.Sk = k.shape[1] if k is not None else (Sk or 0)
    p.Hk = k.shape[2] if k is not None else (Hk or Hq)
    p.scale = float(scale if scale is not None else D ** -0.5)
    p.q_stride = _strides(q)
    p.k_stride = _strides(k if k is not None else q)
    p.v_stride = _strides(v if v is not None else (k if k is not None else q))
    p.o_stride = _strides(o if o is not None else q)
    p.do_stride = _strides(do if do is not None else (o if o is not None else q))
    p.flags = ((ATTN_FLAG_DETERMINISTIC if deterministic else 0) |
               (ATTN_FLAG_CUDA_CORES if cuda_cores else 0))
    return p


def varlen_problem(q, k, v, o, do, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                   max_seqlen_k: int, scale: Optional[float] = None,
                   deterministic: bool = False) -> Problem:
    """Problem descriptor of a variable-length batch: packed q / o / do
    [total_q, Hq, D] and k / v [total_k, Hk, D]; cu_seqlens_* int32 device
    tensors of B + 1 cumulative lengths; the max lengths bound every sequence."""
    Tq, Hq, D = q.shape
    Tk, Hk = k.shape[0], k.shape[1]

    def st(t):  # (batch: unused, token, head) strides
        return (ctypes.c_int64 * 3)(0, t.stride(0), t.stride(1))

    p = Problem()
    p.B = cu_seqlens_q.numel() - 1
    p.Hq, p.Hk, p.D = Hq, Hk, D
    p.Sq, p.Sk = int(max_seqlen_q), int(max_seqlen_k)
    p.scale = float(scale if scale is not None else D ** -0.5)
    p.q_stride, p.k_stride, p.v_stride = st(q), st(k), st(v)
    p.o_stride, p.do_stride = st(o), st(do)
    p.flags = ATTN_FLAG_DETERMINISTIC if deterministic else 0
    p.cu_seqlens_q = cu_seqlens_q.data_ptr()
    p.cu_seqlens_k = cu_seqlens_k.data_ptr()
    p.total_q, p.total_k = Tq, Tk
    return p


def mask_from(window_left: int = -1, window_right: int = -1, num_sink: int = 0,
              bottom_right: bool = False) -> Optional[Mask]:
    """(window_left, window_right) around the diagonal j = i (top-left) or
    j = i + Sk - Sq (bottom_right); negative = unbounded; plus num_sink keys."""
    if window_left < 0 and window_right < 0 and num_sink == 0:
        return None
    return Mask(window_left, window_right, num_sink, 1 if bottom_right else 0)


def sparse_from(ori_kv, cmp_kv=None, cmp_idx=None, ori_win_left=-1, ori_win_right=-1,
                d_ori_kv=None, d_cmp_kv=None, cmp_ratio=0) -> Sparse:
    """cmp_kv with cmp_idx: SCFA (listed rows); cmp_kv without cmp_idx: CFA
    (every compressed row whose block of cmp_ratio positions ends by the query);
    neither: SWA."""
    s = Sparse()
    s.ori_kv = _ptr(ori_kv)
    s.cmp_kv = _ptr(cmp_kv)
    s.cmp_idx = _ptr(cmp_idx)
    s.n_ori = ori_kv.shape[0]
    s.n_cmp = cmp_kv.shape[0] if cmp_kv is not None else 0
    s.topk = cmp_idx.shape[-1] if cmp_idx is not None else 0
    s.ori_win_left, s.ori_win_right = ori_win_left, ori_win_right
    s.d_ori_kv = _ptr(d_ori_kv)
    s.d_cmp_kv = _ptr(d_cmp_kv)
    s.cmp_ratio = cmp_ratio
    return s


def attn_bwd_workspace_size(prob: Problem, mask: Optional[Mask] = None,
                            sparse: Optional[Sparse] = None) -> int:
    return int(lib.attn_bwd_workspace_size(ctypes.byref(prob), _ref(mask), _ref(sparse)))


def attn_bwd_path(prob: Problem, mask: Optional[Mask] = None,
                  sparse: Optional[Sparse] = None) -> int:
    return int(lib.attn_bwd_path(ctypes.byref(prob), _ref(mask), _ref(sparse)))


def attn_fwd_lse(prob, mask, sparse, q, k, v, bias, o, lse, stream=None):
    _check(lib.attn_fwd_lse(ctypes.byref(prob), _ref(mask), _ref(sparse), _ptr(q), _ptr(k),
                            _ptr(v), _ptr(bias), _ptr(o), _ptr(lse), _stream(stream)),
           "attn_fwd_lse")


def attn_bwd_preprocess(prob, sparse, q, k, v, o, do, delta, dbias, dk, dv, workspace,
                        workspace_bytes, stream=None):
    _check(lib.attn_bwd_preprocess(ctypes.byref(prob), _ref(sparse), _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(o), _ptr(do), _ptr(delta), _ptr(dbias), _ptr(dk),
                                   _ptr(dv), _ptr(workspace), workspace_bytes, _stream(stream)),
           "attn_bwd_preprocess")


def attn_bwd(prob, mask, sparse, q, k, v, do, lse, delta, bias, dq, dk, dv, dbias,
             workspace, workspace_bytes, stream=None):
    _check(lib.attn_bwd(ctypes.byref(prob), _ref(mask), _ref(sparse), _ptr(q), _ptr(k), _ptr(v),
                        _ptr(do), _ptr(lse), _ptr(delta), _ptr(bias), _ptr(dq), _ptr(dk),
                        _ptr(dv), _ptr(dbias), _ptr(workspace), workspace_bytes,
                        _stream(stream)),
           "attn_bwd")


def attn_bwd_dsinks(prob, sinks, lse, delta, dsinks, stream=None):
    """dsinks [Hq] = -sum_{b,i} exp(sinks - lse) * delta (see include/attn_bwd.h)."""
    _check(lib.attn_bwd_dsinks(ctypes.byref(prob), _ptr(sinks), _ptr(lse), _ptr(delta),
                               _ptr(dsinks), _stream(stream)),
           "attn_bwd_dsinks")


def attn_bwd_noalloc(prob, mask, sparse, q, k, v, o, do, lse, bias, delta, dq, dk, dv, dbias,
                     stream=None, read_status=False):
    """Pre-pass + backward with the library's fixed device workspace (no allocation).

    For callers that cannot allocate device memory; see include/attn_bwd.h.
    With read_status=True the call synchronises the stream and returns the
    device status (code, detail); otherwise it returns None.
    """
    status = (ctypes.c_int32 * 2)() if read_status else None
    _check(lib.attn_bwd_noalloc(ctypes.byref(prob), _ref(mask), _ref(sparse), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(bias), _ptr(delta),
                                _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias), _stream(stream),
                                status),
           "attn_bwd_noalloc")
    return (int(status[0]), int(status[1])) if read_status else None


def attn_mask_tile_classes(mask: Optional[Mask], Sq: int, Sk: int, tile_q: int = 128,
                           tile_k: int = 128):
    """Host-side tile classes (0 empty, 1 partial, 2 full) as a nested list."""
    nmt, nnt = -(-Sq // tile_q), -(-Sk // tile_k)
    buf = (ctypes.c_int8 * (nmt * nnt))()
    _check(lib.attn_mask_tile_classes(_ref(mask), Sq, Sk, tile_q, tile_k, buf),
           "attn_mask_tile_classes")
    return [[buf[m * nnt + n] for n in range(nnt)] for m in range(nmt)]


def attn_debug_mask_live(mask: Optional[Mask], Sq: int, Sk: int, aligned_variant: int,
                         kv_live, q_live, outside, stream=None):
    """Per-element live sets of the dense tensor-core backward's two kinds of
    CTA (see include/attn_bwd.h): kv_live / q_live uint8 [Sq, Sk] and outside
    int32 [1], zeroed device tensors."""
    _check(lib.attn_debug_mask_live(_ref(mask), Sq, Sk, aligned_variant, _ptr(kv_live),
                                    _ptr(q_live), _ptr(outside), _stream(stream)),
           "attn_debug_mask_live")


def attn_debug_sparse_rows(prob: Problem, sparse: Sparse, rows, counts, max_rows: int,
                           stream=None):
    """Selected-row lists of the sparse tensor-core backward: rows int32
    [Sq * Hk, max_rows] and counts int32 [Sq * Hk] device tensors."""
    _check(lib.attn_debug_sparse_rows(ctypes.byref(prob), ctypes.byref(sparse), _ptr(rows),
                                      _ptr(counts), max_rows, _stream(stream)),
           "attn_debug_sparse_rows")


def attn_read_device_status(workspace, stream=None):
    detail = ctypes.c_int32(0)
    code = lib.attn_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(detail))
    return int(code), int(detail.value)


class BackwardPlan:
    """Preallocated outputs + workspace for repeated backward calls.

    Dense: q, k, v, o, do bf16 BSHD; lse fp32 [B, Hq, Sq]; bias fp32 [Hq, Sq, Sk]
    or None. Sparse (pass ori_kv etc. and k = v = None): q, o, do [1, Sq, Hq, D].
    Variable-length (pass cu_seqlens_q / cu_seqlens_k, int32 device tensors of
    B + 1 cumulative lengths, and the max lengths): q, o, do packed
    [total_q, Hq, D], k, v [total_k, Hk, D]; lse fp32 [B, Hq, max_seqlen_q].
    run() enqueues attn_bwd_preprocess then attn_bwd on the current stream.
    """

    def __init__(self, q, k, v, o, do, lse, scale, mask: Optional[Mask] = None, bias=None,
                 want_dbias=False, ori_kv=None, cmp_kv=None, cmp_idx=None,
                 ori_win_left=-1, ori_win_right=-1, cmp_ratio=0, deterministic=False,
                 cuda_cores=False, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None,
                 max_seqlen_k=None):
        import torch
        dev = q.device
        self.q, self.k, self.v, self.o, self.do, self.lse, self.bias = q, k, v, o, do, lse, bias
        self.sparse = None
        if cu_seqlens_q is not None:
            B, Sq, Hq = cu_seqlens_q.numel() - 1, int(max_seqlen_q), q.shape[1]
            Sk = int(max_seqlen_k)
        else:
            B, Sq, Hq, _ = q.shape
            Sk = k.shape[1] if k is not None else 0
        if cu_seqlens_q is not None:
            self._keep = (cu_seqlens_q, cu_seqlens_k)
            self.prob = varlen_problem(q, k, v, o, do, cu_seqlens_q, cu_seqlens_k, Sq, Sk,
                                       scale, deterministic=deterministic)
            self.dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
            self.dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
        elif ori_kv is not None:
            Hk = ori_kv.shape[1]
            self.d_ori = torch.empty(ori_kv.shape, dtype=torch.float32, device=dev)
            self.d_cmp = (torch.empty(cmp_kv.shape, dtype=torch.float32, device=dev)
                          if cmp_kv is not None else None)
            self.sparse = sparse_from(ori_kv, cmp_kv, cmp_idx, ori_win_left, ori_win_right,
                                      self.d_ori, self.d_cmp, cmp_ratio)
            self._keep = (ori_kv, cmp_kv, cmp_idx)
            self.prob = problem_from(q, None, None, o, do, scale, Sk=0, Hk=Hk,
                                     deterministic=deterministic, cuda_cores=cuda_cores)
            self.dk = self.dv = None
        else:
            self.prob = problem_from(q, k, v, o, do, scale, deterministic=deterministic,
                                     cuda_cores=cuda_cores)
            self.dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
            self.dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
        self.mask = mask
        self.dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
        self.delta = torch.empty((B, Hq, Sq), dtype=torch.float32, device=dev)
        self.dbias = None
        if want_dbias:
            self.dbias = torch.empty((Hq, Sq, Sk), dtype=torch.float32, device=dev)
        self.ws_bytes = attn_bwd_workspace_size(self.prob, mask, self.sparse)
        if self.ws_bytes == 0:
            raise AttnError(1, "attn_bwd_workspace_size")
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.path = attn_bwd_path(self.prob, mask, self.sparse)

    def run(self, stream=None):
        attn_bwd_preprocess(self.prob, self.sparse, self.q, self.k, self.v, self.o, self.do,
                            self.delta, self.dbias, self.dk, self.dv, self.workspace,
                            self.ws_bytes, stream)
        attn_bwd(self.prob, self.mask, self.sparse, self.q, self.k, self.v, self.do, self.lse,
                 self.delta, self.bias, self.dq, self.dk, self.dv, self.dbias, self.workspace,
                 self.ws_bytes, stream)

    def device_status(self, stream=None):
        return attn_read_device_status(self.workspace, stream)
