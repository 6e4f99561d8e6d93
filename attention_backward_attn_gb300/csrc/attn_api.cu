// C ABI entry points: argument validation, workspace layout, kernel dispatch.
// See include/attn_bwd.h for the contract of each function.

#include "internal.h"

#include <math.h>

namespace attn {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool strides_ok(const int64_t* s) {
  for (int t = 0; t < 3; ++t)
    if (s[t] < 0 || (s[t] % 8) != 0) return false;
  return true;
}

// The mask descriptor as window bounds around the diagonal (MaskSpec): a
// negative window bound means unbounded; bounds beyond any sequence are
// unbounded too; bottom-right alignment shifts both bounds by Sk - Sq.
attn_status_t mask_spec_of(const attn_mask_t* mask, int Sq, int Sk, MaskSpec* out) {
  MaskSpec m{kMaskUnbounded, kMaskUnbounded, 0};
  if (mask != nullptr) {
    if (mask->num_sink < 0 || (mask->bottom_right != 0 && mask->bottom_right != 1))
      return ATTN_ERR_INVALID_ARG;
    const bool open_l = mask->window_left < 0 || mask->window_left >= kMaskMaxBound;
    const bool open_r = mask->window_right < 0 || mask->window_right >= kMaskMaxBound;
    m.wl = open_l ? kMaskUnbounded : mask->window_left;
    m.wr = open_r ? kMaskUnbounded : mask->window_right;
    m.sink = mask->num_sink;
    m = mask_aligned(m, mask->bottom_right ? Sk - Sq : 0);
  }
  *out = m;
  return ATTN_OK;
}

// Validates the shared problem / mask / sparse descriptors and fills `out`.
attn_status_t make_problem(const attn_problem_t* prob, const attn_mask_t* mask,
                           const attn_sparse_t* sp, Problem* out) {
  if (prob == nullptr) return ATTN_ERR_INVALID_ARG;
  const attn_problem_t& a = *prob;
  if (a.B < 0 || a.Hq < 1 || a.Hk < 1 || a.Sq < 0 || a.D < 1) return ATTN_ERR_INVALID_ARG;
  if (a.Hq % a.Hk != 0) return ATTN_ERR_INVALID_ARG;
  if (!(a.scale > 0.f) || !isfinite(a.scale)) return ATTN_ERR_INVALID_ARG;
  if (!strides_ok(a.q_stride) || !strides_ok(a.o_stride) || !strides_ok(a.do_stride))
    return ATTN_ERR_INVALID_ARG;
  if (a.D != 64 && a.D != 128 && a.D != 512) return ATTN_ERR_UNSUPPORTED;
  // row counts of the [B, S, H] index spaces, staged rows included (a length
  // rounded up to whole tiles), must fit 31 bits (32-bit index math)
  const int64_t rows_q = (int64_t)a.B * (a.Sq + 128) * a.Hq;
  const int64_t rows_k = (int64_t)a.B * ((a.Sk > 0 ? a.Sk : 0) + 128) * a.Hk * 2;
  if (rows_q >= (int64_t(1) << 31) || rows_k >= (int64_t(1) << 31)) return ATTN_ERR_UNSUPPORTED;
  Problem p{};
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hk = a.Hk;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.D = a.D;
  p.scale = a.scale;
  for (int t = 0; t < 3; ++t) {
    p.qs[t] = a.q_stride[t];
    p.ks[t] = a.k_stride[t];
    p.vs[t] = a.v_stride[t];
    p.os[t] = a.o_stride[t];
    p.dos[t] = a.do_stride[t];
  }
  if (a.flags & ~(ATTN_FLAG_DETERMINISTIC | ATTN_FLAG_CUDA_CORES)) return ATTN_ERR_INVALID_ARG;
  p.deterministic = (a.flags & ATTN_FLAG_DETERMINISTIC) != 0;
  p.cuda_cores = (a.flags & ATTN_FLAG_CUDA_CORES) != 0;
  if (a.Sq > kMaxMaskedLen || a.Sk > kMaxMaskedLen) return ATTN_ERR_UNSUPPORTED;
  p.varlen = a.cu_seqlens_q != nullptr || a.cu_seqlens_k != nullptr;
  if (p.varlen) {
    // per-sequence lengths live on the device: the mask stays top-left here
    // and the kernels align it per sequence
    if (a.cu_seqlens_q == nullptr || a.cu_seqlens_k == nullptr) return ATTN_ERR_INVALID_ARG;
    if (a.total_q < 0 || a.total_k < 0 || a.Sk < 0) return ATTN_ERR_INVALID_ARG;
    if (sp != nullptr || p.cuda_cores || (a.D != 64 && a.D != 128)) return ATTN_ERR_UNSUPPORTED;
    if ((int64_t)a.total_q * a.Hq >= (int64_t(1) << 31) ||
        (int64_t)a.total_k * a.Hk >= (int64_t(1) << 31))
      return ATTN_ERR_UNSUPPORTED;
    p.cu_q = a.cu_seqlens_q;
    p.cu_k = a.cu_seqlens_k;
    p.total_q = a.total_q;
    p.total_k = a.total_k;
    p.br = mask != nullptr && mask->bottom_right == 1;
  }
  const attn_status_t ms =
      p.varlen ? mask_spec_of(mask, 0, 0, &p.mask) : mask_spec_of(mask, a.Sq, a.Sk, &p.mask);
  if (ms != ATTN_OK) return ms;
  p.sparse = sp != nullptr;
  if (p.sparse) {
    if (mask != nullptr) return ATTN_ERR_INVALID_ARG;  // the sparse window replaces it
    if (a.B != 1) return ATTN_ERR_INVALID_ARG;
    if (sp->n_ori < 0) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(sp->ori_kv) || !aligned16(sp->cmp_kv)) return ATTN_ERR_INVALID_ARG;
    const bool cfa = sp->cmp_kv != nullptr && sp->cmp_idx == nullptr;
    if (sp->cmp_kv != nullptr) {
      if (sp->n_cmp < 1) return ATTN_ERR_INVALID_ARG;
      if (cfa ? sp->cmp_ratio < 1 : sp->topk < 1) return ATTN_ERR_INVALID_ARG;
    } else if (sp->cmp_idx != nullptr) {
      return ATTN_ERR_INVALID_ARG;
    }
    p.n_ori = sp->n_ori;
    p.n_cmp = sp->cmp_kv ? sp->n_cmp : 0;
    p.topk = sp->cmp_kv && !cfa ? sp->topk : 0;
    p.cmp_ratio = cfa ? sp->cmp_ratio : 0;
    p.ori_wl = sp->ori_win_left < 0 ? -1 : sp->ori_win_left;
    p.ori_wr = sp->ori_win_right < 0 ? -1 : sp->ori_win_right;
    p.Sk = 0;
  } else {
    if (a.Sk < 0) return ATTN_ERR_INVALID_ARG;
    if (!strides_ok(a.k_stride) || !strides_ok(a.v_stride)) return ATTN_ERR_INVALID_ARG;
  }
  // variable-length batches run on the dense tensor-core kernel only
  if (p.varlen && !tc_supported(p)) return ATTN_ERR_UNSUPPORTED;
  // the ordered sparse dKV reduction follows the tensor-core kernel's slots
  if (p.sparse && p.deterministic && (p.cuda_cores || !tc_sparse_supported(p)))
    return ATTN_ERR_UNSUPPORTED;
  *out = p;
  return ATTN_OK;
}

// Element counts of the tensors of a problem. A pointer may be NULL only for
// a tensor with no elements.
struct Sizes {
  int64_t q, k, rows, ori;
};

Sizes sizes_of(const Problem& p) {
  Sizes n;
  n.q = (int64_t)(p.varlen ? p.total_q : (int64_t)p.B * p.Sq) * p.Hq * p.D;
  n.k = (int64_t)(p.varlen ? p.total_k : (int64_t)p.B * p.Sk) * p.Hk * p.D;
  n.rows = (int64_t)p.B * p.Hq * p.Sq;
  n.ori = (int64_t)p.n_ori * p.Hk * p.D;
  return n;
}

bool need(const void* ptr, int64_t count) { return count == 0 || ptr != nullptr; }

bool use_tensor_cores(const Problem& p) {
  if (p.cuda_cores) return false;
  return p.sparse ? tc_sparse_supported(p) : tc_supported(p);
}

// One backward per problem: the tensor-core kernels, or the CUDA-core kernels
// when the caller asks for them (ATTN_FLAG_CUDA_CORES). A problem outside the
// tensor-core kernels' shapes is not sent to the CUDA-core kernels unasked.
bool backward_available(const Problem& p) { return p.cuda_cores || use_tensor_cores(p); }

// dbias computed by the tensor-core kernel's batch-inner query-major CTAs:
// stored once per element, neither zeroed first nor split by batch.
bool dbias_in_q(const Problem& p, const float* dbias) {
  return dbias != nullptr && !p.sparse && use_tensor_cores(p) && tc_dbias_in_q(p);
}

// Deterministic dense mode with dbias over several batches (other than the
// batch-inner case): per-batch slices of dbias in the workspace, summed in
// batch order afterwards.
bool dbias_split(const Problem& p, const float* dbias) {
  return !p.sparse && p.deterministic && p.B > 1 && dbias != nullptr && !dbias_in_q(p, dbias);
}

attn_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace

WorkspaceLayout workspace_layout(const Problem& p, bool tensor_core_path) {
  WorkspaceLayout w;
  size_t off = kStatusBytes;
  if (tensor_core_path && p.sparse) {
    const size_t kvbytes = (size_t)(p.n_ori + p.n_cmp) * p.Hk * p.D * sizeof(__half);
    off = align_up(off, 1024);
    w.kv16 = off;
    off = align_up(off + kvbytes, 1024);
    w.staged = true;
    if (p.deterministic) {
      // per item (token, KV head): dKV rows at their slots, the row list,
      // {count, window rows, first window row}; per item and compressed row:
      // first slot and multiplicity
      const size_t items = (size_t)p.Sq * p.Hk;
      const size_t slots = items * (size_t)sparse_det_stride(p);
      w.det_part = off;
      off = align_up(off + slots * p.D * sizeof(float), 1024);
      w.det_rows = off;
      off = align_up(off + slots * sizeof(int32_t), 1024);
      w.det_meta = off;
      off = align_up(off + items * 3 * sizeof(int32_t), 1024);
      w.det_slot = off;
      off = align_up(off + items * p.n_cmp * sizeof(int32_t), 1024);
      w.det_mult = off;
      off = align_up(off + items * p.n_cmp * sizeof(int32_t), 1024);
    }
  } else if (tensor_core_path) {
    const size_t qbytes = (size_t)p.B * p.Hq * tc_rows(p.Sq) * p.D * sizeof(__half);
    const size_t kbytes = (size_t)p.B * p.Hk * tc_rows(p.Sk) * p.D * sizeof(__half);
    off = align_up(off, 1024);
    w.q16 = off;
    off = align_up(off + qbytes, 1024);
    w.do16 = off;
    off = align_up(off + qbytes, 1024);
    w.k16 = off;
    off = align_up(off + kbytes, 1024);
    w.v16 = off;
    off = align_up(off + kbytes, 1024);
    w.staged = true;
  }
  if (!p.sparse && p.deterministic && p.B > 1 && !(tensor_core_path && tc_dbias_in_q(p))) {
    // per-batch dbias slices (used when dbias is requested and the
    // batch-inner kernel does not apply)
    off = align_up(off, 1024);
    w.det_dbias = off;
    off = align_up(off + (size_t)p.B * p.Hq * p.Sq * p.Sk * sizeof(float), 1024);
  }
  w.total = off;
  return w;
}

}  // namespace attn

using namespace attn;

extern "C" {

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
    case ATTN_ERR_INDEX_OOB: return "ATTN_ERR_INDEX_OOB";
    case ATTN_ERR_RANGE: return "ATTN_ERR_RANGE";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
  }
  return "ATTN_ERR_UNKNOWN";
}

attn_status_t attn_mask_tile_classes(const attn_mask_t* mask, int32_t Sq, int32_t Sk,
                                     int32_t tile_q, int32_t tile_k, int8_t* out) {
  if (Sq <= 0 || Sk <= 0 || tile_q <= 0 || tile_k <= 0 || out == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (Sq > kMaxMaskedLen || Sk > kMaxMaskedLen) return ATTN_ERR_UNSUPPORTED;
  MaskSpec m;
  const attn_status_t ms = mask_spec_of(mask, Sq, Sk, &m);
  if (ms != ATTN_OK) return ms;
  const int nmt = (Sq + tile_q - 1) / tile_q, nnt = (Sk + tile_k - 1) / tile_k;
  for (int mt = 0; mt < nmt; ++mt) {
    const int m0 = mt * tile_q, m1 = m0 + tile_q < Sq ? m0 + tile_q : Sq;
    for (int nt = 0; nt < nnt; ++nt) {
      const int n0 = nt * tile_k, n1 = n0 + tile_k < Sk ? n0 + tile_k : Sk;
      out[(int64_t)mt * nnt + nt] =
          !tile_any(m, m0, m1, n0, n1) ? 0 : (tile_full(m, m0, m1, n0, n1) ? 2 : 1);
    }
  }
  return ATTN_OK;
}

attn_status_t attn_debug_mask_live(const attn_mask_t* mask, int32_t Sq, int32_t Sk,
                                   int32_t aligned_variant, uint8_t* kv_live, uint8_t* q_live,
                                   int32_t* outside, cudaStream_t stream) {
  if (Sq <= 0 || Sk <= 0 || kv_live == nullptr || q_live == nullptr || outside == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (aligned_variant != 0 && aligned_variant != 1) return ATTN_ERR_INVALID_ARG;
  if (aligned_variant == 1 && (Sq % 128 != 0 || Sk % 128 != 0)) return ATTN_ERR_INVALID_ARG;
  if (Sq > kMaxMaskedLen || Sk > kMaxMaskedLen) return ATTN_ERR_UNSUPPORTED;
  MaskSpec m;
  const attn_status_t ms = mask_spec_of(mask, Sq, Sk, &m);
  if (ms != ATTN_OK) return ms;
  return cuda_status(
      launch_mask_probe(m, Sq, Sk, aligned_variant == 1, kv_live, q_live, outside, stream));
}

attn_status_t attn_debug_sparse_rows(const attn_problem_t* prob, const attn_sparse_t* sparse,
                                     int32_t* rows, int32_t* counts, int32_t max_rows,
                                     cudaStream_t stream) {
  if (sparse == nullptr || rows == nullptr || counts == nullptr) return ATTN_ERR_INVALID_ARG;
  Problem p;
  attn_status_t s = make_problem(prob, nullptr, sparse, &p);
  if (s != ATTN_OK) return s;
  const int64_t bound = sparse_row_bound(p);
  if (bound > 1024) return ATTN_ERR_UNSUPPORTED;
  if (max_rows < bound) return ATTN_ERR_INVALID_ARG;
  if (p.topk > 0 && sparse->cmp_idx == nullptr) return ATTN_ERR_INVALID_ARG;
  return cuda_status(launch_rows_probe(p, sparse->cmp_idx, rows, counts, max_rows, stream));
}

int32_t attn_bwd_path(const attn_problem_t* prob, const attn_mask_t* mask,
                      const attn_sparse_t* sparse) {
  Problem p;
  if (make_problem(prob, mask, sparse, &p) != ATTN_OK) return 0;
  if (!backward_available(p)) return 0;
  return use_tensor_cores(p) ? 1 : 2;
}

size_t attn_bwd_workspace_size(const attn_problem_t* prob, const attn_mask_t* mask,
                               const attn_sparse_t* sparse) {
  Problem p;
  if (make_problem(prob, mask, sparse, &p) != ATTN_OK || !backward_available(p)) return 0;
  return workspace_layout(p, use_tensor_cores(p)).total;
}

attn_status_t attn_fwd_lse(const attn_problem_t* prob, const attn_mask_t* mask,
                           const attn_sparse_t* sparse, const void* q, const void* k,
                           const void* v, const float* bias, void* o, float* lse,
                           cudaStream_t stream) {
  Problem p;
  attn_status_t s = make_problem(prob, mask, sparse, &p);
  if (s != ATTN_OK) return s;
  if (p.varlen) return ATTN_ERR_UNSUPPORTED;  // the forward has no varlen variant
  const Sizes n = sizes_of(p);
  if (!need(q, n.q) || !need(o, n.q) || !need(lse, n.rows)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse) || !aligned16(bias))
    return ATTN_ERR_INVALID_ARG;
  if (p.sparse) {
    if (k != nullptr || v != nullptr || bias != nullptr) return ATTN_ERR_INVALID_ARG;
    if (!need(sparse->ori_kv, n.ori)) return ATTN_ERR_INVALID_ARG;
  } else {
    if (!need(k, n.k) || !need(v, n.k) || !aligned16(k) || !aligned16(v))
      return ATTN_ERR_INVALID_ARG;
  }
  if (fwd_tc_supported(p)) return cuda_status(launch_fwd_tc(p, q, k, v, bias, o, lse, stream));
  // Device conditions of the forward (bad sparse indices) are skipped but not
  // recorded: the forward has no workspace.
  return cuda_status(launch_fwd_simt(p, q, k, v, bias, sparse ? sparse->ori_kv : nullptr,
                                     sparse ? sparse->cmp_kv : nullptr,
                                     sparse ? sparse->cmp_idx : nullptr, o, lse, nullptr,
                                     stream));
}

attn_status_t attn_bwd_preprocess(const attn_problem_t* prob, const attn_sparse_t* sparse,
                                  const void* q, const void* k, const void* v,
                                  const void* o, const void* dO, float* delta,
                                  float* dbias, float* dk, float* dv, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream) {
  Problem p;
  attn_status_t s = make_problem(prob, nullptr, sparse, &p);
  if (s != ATTN_OK) return s;
  const Sizes n = sizes_of(p);
  if (!need(o, n.q) || !need(dO, n.q) || !need(delta, n.rows)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dO) || !aligned16(dbias)) return ATTN_ERR_INVALID_ARG;
  float* d_ori = nullptr;
  float* d_cmp = nullptr;
  if (p.sparse) {
    if (dbias != nullptr || dk != nullptr || dv != nullptr) return ATTN_ERR_INVALID_ARG;
    d_ori = sparse->d_ori_kv;
    d_cmp = sparse->cmp_kv ? sparse->d_cmp_kv : nullptr;
    if (!need(d_ori, n.ori) || (sparse->cmp_kv && d_cmp == nullptr)) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(d_ori) || !aligned16(d_cmp)) return ATTN_ERR_INVALID_ARG;
  } else if (!need(dk, n.k) || !need(dv, n.k) || !aligned16(dk) || !aligned16(dv)) {
    return ATTN_ERR_INVALID_ARG;
  }
  if (!backward_available(p)) return ATTN_ERR_UNSUPPORTED;
  const bool tc = use_tensor_cores(p);
  // the head-split tensor-core kernel adds partial dK / dV sums into zeroed buffers
  const bool zero_kv = tc && !p.sparse && tc_head_split(p) > 1;
  if (tc && !p.sparse &&
      (!need(q, n.q) || !need(k, n.k) || !need(v, n.k) || !aligned16(q) || !aligned16(k) ||
       !aligned16(v)))
    return ATTN_ERR_INVALID_ARG;
  if (tc && p.sparse && !need(sparse->ori_kv, n.ori)) return ATTN_ERR_INVALID_ARG;
  const WorkspaceLayout w = workspace_layout(p, tc);
  if (workspace == nullptr || workspace_bytes < w.total || !aligned16(workspace))
    return ATTN_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  DevStatus* st = reinterpret_cast<DevStatus*>(ws + w.status);
  auto staged = [&](size_t off) {
    return w.staged ? reinterpret_cast<__half*>(ws + off) : nullptr;
  };
  const bool dense_staged = w.staged && !p.sparse;
  // deterministic dbias over several batches: zero the per-batch slices
  const bool split = dbias_split(p, dbias);
  Problem pk = p;
  pk.dbias_bstride = split ? (int64_t)p.Hq * p.Sq * p.Sk : 0;
  // (the batch-inner kernel stores every dbias entry itself)
  float* dbias_zero = split ? reinterpret_cast<float*>(ws + w.det_dbias)
                            : (dbias_in_q(p, dbias) ? nullptr : dbias);
  return cuda_status(launch_preprocess(
      pk, q, k, v, o, dO, delta, dbias_zero, d_ori, d_cmp, dense_staged ? staged(w.q16) : nullptr,
      dense_staged ? staged(w.k16) : nullptr, dense_staged ? staged(w.v16) : nullptr,
      dense_staged ? staged(w.do16) : nullptr, p.sparse ? sparse->ori_kv : nullptr,
      p.sparse ? sparse->cmp_kv : nullptr, (w.staged && p.sparse) ? staged(w.kv16) : nullptr,
      // dk / dv are recorded (for attn_bwd's check) only when zeroed here:
      // only then may the head-split kernel add partial sums into them
      zero_kv ? dk : nullptr, zero_kv ? dv : nullptr, zero_kv ? dk : nullptr,
      zero_kv ? dv : nullptr, st, stream));
}

attn_status_t attn_bwd(const attn_problem_t* prob, const attn_mask_t* mask,
                       const attn_sparse_t* sparse, const void* q, const void* k,
                       const void* v, const void* dO, const float* lse, const float* delta,
                       const float* bias, float* dq, float* dk, float* dv, float* dbias,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  Problem p;
  attn_status_t s = make_problem(prob, mask, sparse, &p);
  if (s != ATTN_OK) return s;
  const Sizes n = sizes_of(p);
  if (!need(q, n.q) || !need(dO, n.q) || !need(lse, n.rows) || !need(delta, n.rows) ||
      !need(dq, n.q))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(dO) || !aligned16(dq)) return ATTN_ERR_INVALID_ARG;
  if (p.sparse) {
    if (k || v || bias || dk || dv || dbias) return ATTN_ERR_INVALID_ARG;
    if (!need(sparse->d_ori_kv, n.ori) || !need(sparse->ori_kv, n.ori) ||
        (sparse->cmp_kv && sparse->d_cmp_kv == nullptr))
      return ATTN_ERR_INVALID_ARG;
    if (!aligned16(sparse->d_ori_kv) || !aligned16(sparse->d_cmp_kv)) return ATTN_ERR_INVALID_ARG;
  } else {
    if (!need(k, n.k) || !need(v, n.k) || !need(dk, n.k) || !need(dv, n.k))
      return ATTN_ERR_INVALID_ARG;
    if (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv) || !aligned16(bias) ||
        !aligned16(dbias))
      return ATTN_ERR_INVALID_ARG;
  }
  if (!backward_available(p)) return ATTN_ERR_UNSUPPORTED;
  const bool tc = use_tensor_cores(p);
  if (tc && (!aligned16(lse) || !aligned16(delta))) return ATTN_ERR_INVALID_ARG;
  const WorkspaceLayout w = workspace_layout(p, tc);
  if (workspace == nullptr || workspace_bytes < w.total || !aligned16(workspace))
    return ATTN_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  DevStatus* st = reinterpret_cast<DevStatus*>(ws + w.status);
  if (tc && p.sparse) {
    const __half* kv16 = reinterpret_cast<const __half*>(ws + w.kv16);
    SparseDet det;
    if (p.deterministic) {
      det.part = reinterpret_cast<float*>(ws + w.det_part);
      det.rows = reinterpret_cast<int32_t*>(ws + w.det_rows);
      det.meta = reinterpret_cast<int32_t*>(ws + w.det_meta);
      det.slot = reinterpret_cast<int32_t*>(ws + w.det_slot);
      det.mult = reinterpret_cast<int32_t*>(ws + w.det_mult);
      det.stride = (int)sparse_det_stride(p);
    }
    cudaError_t e = launch_bwd_sparse_tc(p, q, dO, kv16, sparse->cmp_idx, lse, delta, dq,
                                         sparse->d_ori_kv, sparse->d_cmp_kv, det, st, stream);
    if (e == cudaSuccess && p.deterministic)
      e = launch_sparse_det_reduce(p, det, sparse->d_ori_kv, sparse->d_cmp_kv, stream);
    return cuda_status(e);
  }
  if (p.sparse) {
    return cuda_status(launch_bwd_simt(p, q, k, v, dO, lse, delta, bias, dq, dk, dv, dbias,
                                       sparse->ori_kv, sparse->cmp_kv, sparse->cmp_idx,
                                       sparse->d_ori_kv, sparse->d_cmp_kv, st, stream));
  }
  // Deterministic dbias over several batches: every batch adds its terms
  // into its own zeroed slice of the workspace (one writer per element, so
  // each slice holds exact values), and a second pass sums the slices in
  // batch order into dbias.
  const bool split = dbias_split(p, dbias);
  float* dbias_acc = split ? reinterpret_cast<float*>(ws + w.det_dbias) : dbias;
  Problem pk = p;
  pk.dbias_bstride = split ? (int64_t)p.Hq * p.Sq * p.Sk : 0;
  cudaError_t e;
  if (tc) {
    e = launch_bwd_tc(pk, reinterpret_cast<const __half*>(ws + w.q16),
                      reinterpret_cast<const __half*>(ws + w.k16),
                      reinterpret_cast<const __half*>(ws + w.v16),
                      reinterpret_cast<const __half*>(ws + w.do16), lse, delta, bias, dq, dk, dv,
                      dbias_acc, st, stream);
  } else {
    e = launch_bwd_simt(pk, q, k, v, dO, lse, delta, bias, dq, dk, dv, dbias_acc, nullptr,
                        nullptr, nullptr, nullptr, nullptr, st, stream);
  }
  if (e == cudaSuccess && split)
    e = launch_sum_slices(dbias_acc, p.B, pk.dbias_bstride, dbias, stream);
  if (e != cudaSuccess) return cuda_status(e);
  return ATTN_OK;
}

attn_status_t attn_bwd_dsinks(const attn_problem_t* prob, const float* sinks,
                              const float* lse, const float* delta, float* dsinks,
                              cudaStream_t stream) {
  if (prob == nullptr || sinks == nullptr || lse == nullptr || delta == nullptr ||
      dsinks == nullptr)
    return ATTN_ERR_INVALID_ARG;
  if (prob->B <= 0 || prob->Hq <= 0 || prob->Sq <= 0) return ATTN_ERR_INVALID_ARG;
  // lse / delta of a variable-length batch hold unused entries past each length
  if (prob->cu_seqlens_q != nullptr || prob->cu_seqlens_k != nullptr)
    return ATTN_ERR_UNSUPPORTED;
  const uintptr_t mis = reinterpret_cast<uintptr_t>(sinks) | reinterpret_cast<uintptr_t>(lse) |
                        reinterpret_cast<uintptr_t>(delta) | reinterpret_cast<uintptr_t>(dsinks);
  if (mis & 3u) return ATTN_ERR_INVALID_ARG;
  return cuda_status(launch_dsinks(prob->B, prob->Hq, prob->Sq, sinks, lse, delta, dsinks,
                                   stream));
}

attn_status_t attn_read_device_status(const void* workspace, cudaStream_t stream,
                                      int32_t* detail) {
  if (workspace == nullptr) return ATTN_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int32_t host[2] = {0, 0};
  if (cudaMemcpy(host, workspace, sizeof(host), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (detail != nullptr) *detail = host[1];
  return static_cast<attn_status_t>(host[0]);
}

}  // extern "C"
