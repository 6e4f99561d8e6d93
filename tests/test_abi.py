"""Host-side checks of the C ABI (no GPU needed).

The library must load, export every function include/attn_bwd.h declares,
and reject bad arguments with an error code before enqueuing any work (these
calls never reach a kernel launch, so they run without a device).
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def ab():
    import __graft_entry__
    __graft_entry__.build()
    import attention_backward_attn_gb300 as mod
    return mod


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            names += re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(attn_[a-z_0-9]+)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("attn_fwd_lse", "attn_bwd_preprocess", "attn_bwd", "attn_bwd_workspace_size",
              "attn_read_device_status", "attn_status_string", "attn_bwd_path"):
        assert n in names


def test_library_exports_every_declared_symbol(ab):
    lib = ctypes.CDLL(ab._build.LIB_PATH)
    for n in _declared_functions():
        assert hasattr(lib, n), n


def test_status_strings(ab):
    assert ab.status_string(0) == "ATTN_OK"
    assert ab.status_string(5) == "ATTN_ERR_INDEX_OOB"
    assert ab.status_string(99) == "ATTN_ERR_UNKNOWN"


def _prob(ab, B=2, Hq=8, Hk=2, Sq=256, Sk=256, D=128, scale=None):
    p = ab.Problem()
    p.B, p.Hq, p.Hk, p.Sq, p.Sk, p.D = B, Hq, Hk, Sq, Sk, D
    p.scale = scale if scale is not None else D ** -0.5
    qs = (Sq * Hq * D, Hq * D, D)
    ks = (Sk * Hk * D, Hk * D, D)
    p.q_stride = (ctypes.c_int64 * 3)(*qs)
    p.o_stride = (ctypes.c_int64 * 3)(*qs)
    p.do_stride = (ctypes.c_int64 * 3)(*qs)
    p.k_stride = (ctypes.c_int64 * 3)(*ks)
    p.v_stride = (ctypes.c_int64 * 3)(*ks)
    return p


def test_workspace_size_and_validation(ab):
    p = _prob(ab)
    assert ab.attn_bwd_workspace_size(p) >= 256
    bad = _prob(ab, Hq=6, Hk=4)
    assert ab.attn_bwd_workspace_size(bad) == 0
    assert ab.attn_bwd_path(bad) == 0
    assert ab.attn_bwd_path(_prob(ab, D=96)) == 0  # unsupported head dim
    assert ab.attn_bwd_workspace_size(_prob(ab, scale=0.0)) == 0
    assert ab.attn_bwd_workspace_size(_prob(ab, scale=float("nan"))) == 0
    odd = _prob(ab)
    odd.q_stride = (ctypes.c_int64 * 3)(256 * 8 * 128, 8 * 128 + 4, 128)
    assert ab.attn_bwd_workspace_size(odd) == 0
    assert ab.attn_bwd_path(p) in (1, 2)


def _call_bwd(ab, p, mask=None, sparse=None, ptrs=None, ws_bytes=1 << 20):
    fake = 1 << 20  # never dereferenced: every case below fails host validation
    args = dict(q=fake, k=fake, v=fake, do=fake, lse=fake, delta=fake, bias=None, dq=fake,
                dk=fake, dv=fake, dbias=None, ws=fake)
    args.update(ptrs or {})
    return ab.lib.attn_bwd(ctypes.byref(p), None if mask is None else ctypes.byref(mask),
                           None if sparse is None else ctypes.byref(sparse), args["q"],
                           args["k"], args["v"], args["do"], args["lse"], args["delta"],
                           args["bias"], args["dq"], args["dk"], args["dv"], args["dbias"],
                           args["ws"], ws_bytes, None)


def test_bwd_rejects_bad_arguments_on_the_host(ab):
    p = _prob(ab)
    assert _call_bwd(ab, p, ptrs=dict(q=None)) == 1
    assert _call_bwd(ab, p, ptrs=dict(dk=None)) == 1
    assert _call_bwd(ab, p, ptrs=dict(q=(1 << 20) + 8)) == 1  # misaligned
    assert _call_bwd(ab, p, ptrs=dict(ws=None)) == 7
    assert _call_bwd(ab, p, ws_bytes=16) == 7
    assert _call_bwd(ab, _prob(ab, D=80)) == 2
    m = ab.Mask(-1, 0, -3)
    assert _call_bwd(ab, p, mask=m) == 1


def _call_pre(ab, p, sparse=None, ptrs=None, ws_bytes=1 << 20):
    fake = 1 << 20  # never dereferenced: every case below fails host validation
    args = dict(q=fake, k=fake, v=fake, o=fake, do=fake, delta=fake, dbias=None, dk=fake,
                dv=fake, ws=fake)
    args.update(ptrs or {})
    return ab.lib.attn_bwd_preprocess(ctypes.byref(p),
                                      None if sparse is None else ctypes.byref(sparse),
                                      args["q"], args["k"], args["v"], args["o"], args["do"],
                                      args["delta"], args["dbias"], args["dk"], args["dv"],
                                      args["ws"], ws_bytes, None)


def test_preprocess_validates_dk_dv(ab):
    # dense problems hand dk / dv to the pre-pass (it zeroes them when the
    # head-split kernel adds partial sums into them); the sparse variant has none
    p = _prob(ab)
    assert _call_pre(ab, p, ptrs=dict(dk=None)) == 1
    assert _call_pre(ab, p, ptrs=dict(dv=None)) == 1
    assert _call_pre(ab, p, ptrs=dict(dv=(1 << 20) + 4)) == 1  # misaligned
    assert _call_pre(ab, p, ptrs=dict(ws=None)) == 7
    fake = 1 << 20
    sp = _prob(ab, B=1, Hq=16, Hk=1, Sq=128, Sk=0, D=512)
    s = ab.Sparse()
    s.ori_kv, s.n_ori, s.ori_win_left, s.ori_win_right = fake, 128, 31, 0
    s.d_ori_kv = fake
    assert _call_pre(ab, sp, sparse=s, ptrs=dict(k=None, v=None)) == 1
    # 16 query heads per KV head: CUDA-core kernels only, and only when asked for
    assert _call_pre(ab, sp, sparse=s,
                     ptrs=dict(k=None, v=None, dk=None, dv=None, ws=None)) == 2  # ATTN_ERR_UNSUPPORTED
    sp.flags = ab.ATTN_FLAG_CUDA_CORES
    assert _call_pre(ab, sp, sparse=s, ptrs=dict(k=None, v=None, dk=None, dv=None, ws=None)) == 7


def test_sparse_descriptor_validation(ab):
    fake = 1 << 20
    p = _prob(ab, B=1, Hq=16, Hk=1, Sq=128, Sk=0, D=512)
    s = ab.Sparse()
    s.ori_kv, s.n_ori, s.ori_win_left, s.ori_win_right = fake, 128, 31, 0
    s.d_ori_kv = fake
    # 16 query heads per KV head: the SIMT kernels, only when asked for
    assert ab.attn_bwd_path(p, None, s) == 0
    assert ab.attn_bwd_workspace_size(p, None, s) == 0
    p.flags = ab.ATTN_FLAG_CUDA_CORES
    assert ab.attn_bwd_path(p, None, s) == 2
    # k / v must be NULL for the shared-KV variant
    assert _call_bwd(ab, p, sparse=s) == 1
    # compressed KV without an index list is the CFA case: it needs cmp_ratio >= 1
    s.cmp_kv, s.n_cmp, s.topk, s.d_cmp_kv = fake, 32, 8, fake
    s.cmp_ratio = 0
    assert ab.attn_bwd_path(p, None, s) == 0
    assert _call_bwd(ab, p, sparse=s, ptrs=dict(k=None, v=None, dk=None, dv=None)) == 1
    s.cmp_ratio = 4
    assert ab.attn_bwd_path(p, None, s) == 2  # 16 query heads per KV head: SIMT kernels (asked for)
    s.n_cmp = 0
    assert ab.attn_bwd_path(p, None, s) == 0  # compressed KV needs rows
    s.n_cmp = 32
    # batch must be 1
    p2 = _prob(ab, B=2, Hq=16, Hk=1, Sq=128, Sk=0, D=512)
    s.cmp_idx = fake
    assert ab.attn_bwd_path(p2, None, s) == 0
    # a mask descriptor is not allowed with the sparse window
    assert ab.attn_bwd_path(p, ab.Mask(-1, 0, 0), s) == 0
    # the deterministic mode covers the dense path only (sparse dKV is a
    # reduction over tokens in arrival order)
    p.flags = ab.ATTN_FLAG_DETERMINISTIC
    assert ab.attn_bwd_path(p, None, s) == 0
    assert _call_bwd(ab, p, sparse=s, ptrs=dict(k=None, v=None, dk=None, dv=None)) == 2
    p.flags = 0


def test_problem_flags(ab):
    p = _prob(ab)
    assert ab.attn_bwd_path(p, None, None) in (1, 2)
    p.flags = ab.ATTN_FLAG_DETERMINISTIC
    assert ab.attn_bwd_path(p, None, None) in (1, 2)
    p.flags = ab.ATTN_FLAG_CUDA_CORES  # the SIMT kernels, whatever the shape
    assert ab.attn_bwd_path(p, None, None) == 2
    p.flags = ab.ATTN_FLAG_CUDA_CORES | ab.ATTN_FLAG_DETERMINISTIC
    assert ab.attn_bwd_path(p, None, None) == 2
    p.flags = 4  # unknown bit
    assert ab.attn_bwd_path(p, None, None) == 0


def test_deterministic_workspace_holds_the_dbias_slices(ab):
    # deterministic mode with B > 1 reserves one dbias slice per batch
    # (B * Hq * Sq * Sk floats) on top of the default workspace
    p = _prob(ab, B=3, Hq=4, Hk=2, Sq=200, Sk=136, D=64)
    base = ab.attn_bwd_workspace_size(p)
    p.flags = ab.ATTN_FLAG_DETERMINISTIC
    det = ab.attn_bwd_workspace_size(p)
    assert det >= base + 3 * 4 * 200 * 136 * 4
    # a single batch needs no slices
    p1 = _prob(ab, B=1, Hq=4, Hk=2, Sq=200, Sk=136, D=64)
    base1 = ab.attn_bwd_workspace_size(p1)
    p1.flags = ab.ATTN_FLAG_DETERMINISTIC
    assert ab.attn_bwd_workspace_size(p1) == base1


def test_varlen_descriptor_validation(ab):
    fake = 1 << 20  # never dereferenced: host validation only
    p = _prob(ab, B=3, Sq=300, Sk=300)
    p.cu_seqlens_q = fake  # without cu_seqlens_k
    p.total_q, p.total_k = 500, 500
    assert ab.attn_bwd_path(p, None, None) == 0
    assert _call_bwd(ab, p) == 1
    p.cu_seqlens_k = fake
    p.total_q = -1
    assert _call_bwd(ab, p) == 1
    p.total_q = 500
    # the variable-length layout runs on the dense tensor-core kernel only
    p.flags = ab.ATTN_FLAG_CUDA_CORES
    assert ab.attn_bwd_path(p, None, None) == 0
    p.flags = 0
    assert ab.attn_bwd_path(_varlen(ab, D=512), None, None) == 0
    sp = _varlen(ab, B=1, Hq=16, Hk=1, Sk=0, D=512)
    s = ab.Sparse()
    s.ori_kv, s.n_ori, s.ori_win_left, s.ori_win_right, s.d_ori_kv = fake, 128, 31, 0, fake
    assert ab.attn_bwd_path(sp, None, s) == 0
    # lse / delta of a packed batch hold unused entries: no dsinks
    assert ab.lib.attn_bwd_dsinks(ctypes.byref(p), fake, fake, fake, fake, None) == 2


def _varlen(ab, **kw):
    p = _prob(ab, **kw)
    p.cu_seqlens_q = p.cu_seqlens_k = 1 << 20
    p.total_q = p.total_k = 64
    return p


def test_read_status_rejects_null(ab):
    code = ab.lib.attn_read_device_status(None, None, None)
    assert code == 1


@pytest.mark.parametrize("spec", [
    # (Sq, Sk, window_left, window_right, num_sink, tile_q, tile_k)
    (1024, 1024, -1, 0, 0, 128, 128),       # the causal benchmark workload
    (8192, 8192, 1023, 0, 4, 128, 128),     # window 1024 + 4 sinks workload
    (2048, 2048, -1, -1, 0, 128, 128),      # no mask
    (640, 640, 127, 0, 4, 128, 128),
    (200, 328, 40, 25, 3, 64, 32),          # ragged tails, two-sided window
    (384, 128, 10, 0, 0, 128, 128),         # rows without live keys
    (97, 61, -1, 0, 70, 16, 8),             # sinks beyond the diagonal
    # bottom-right alignment (last column: 1)
    (128, 384, -1, 0, 0, 128, 128, 1),      # causal, Sq < Sk
    (384, 128, -1, 0, 0, 128, 128, 1),      # causal, Sq > Sk: rows without keys
    (200, 328, 40, 25, 3, 64, 32, 1),       # ragged, two-sided window + sinks
    (97, 61, 5, 0, 2, 16, 8, 1),
])
def test_tile_classes_match_oracle_mask(ab, spec):
    # The kernels skip tiles classed 0 and mask tiles classed 1 per element;
    # the classes must agree bit-exactly with the oracle's element mask.
    import numpy as np
    import oracle
    Sq, Sk, wl, wr, ns, tq, tk = spec[:7]
    br = spec[7] if len(spec) > 7 else 0
    m = oracle.live_mask(Sq, Sk, wl, wr, ns, bottom_right=bool(br))
    got = ab.attn_mask_tile_classes(ab.Mask(wl, wr, ns, br), Sq, Sk, tq, tk)
    for mt, row in enumerate(got):
        for nt, cls in enumerate(row):
            tile = m[mt * tq:(mt + 1) * tq, nt * tk:(nt + 1) * tk]
            expect = 0 if not tile.any() else (2 if tile.all() else 1)
            assert cls == expect, (mt, nt, cls, expect)


def test_tile_classes_random_masks(ab):
    # 300 random (lengths, window, sinks, alignment, tile) draws against the
    # oracle's element mask, vectorised per draw
    import numpy as np
    import oracle
    rng = np.random.default_rng(123)
    for _ in range(300):
        Sq, Sk = (int(x) for x in rng.integers(1, 300, size=2))
        wl = int(rng.choice([-1, int(rng.integers(0, 200))]))
        wr = int(rng.choice([-1, int(rng.integers(0, 200))]))
        ns = int(rng.choice([0, int(rng.integers(0, 40))]))
        br = int(rng.integers(0, 2))
        tq, tk = (int(rng.choice([8, 16, 32, 64, 128])) for _ in range(2))
        m = oracle.live_mask(Sq, Sk, wl, wr, ns, bottom_right=bool(br))
        got = np.asarray(ab.attn_mask_tile_classes(ab.Mask(wl, wr, ns, br), Sq, Sk, tq, tk))
        nmt, nnt = -(-Sq // tq), -(-Sk // tk)
        pad = np.zeros((nmt * tq, nnt * tk), dtype=np.int8)
        pad[:Sq, :Sk] = m
        cnt = pad.reshape(nmt, tq, nnt, tk).sum(axis=(1, 3))
        rows = np.minimum(tq, Sq - np.arange(nmt) * tq)[:, None]
        cols = np.minimum(tk, Sk - np.arange(nnt) * tk)[None, :]
        expect = np.where(cnt == 0, 0, np.where(cnt == rows * cols, 2, 1))
        assert np.array_equal(got, expect), (Sq, Sk, wl, wr, ns, br, tq, tk)
