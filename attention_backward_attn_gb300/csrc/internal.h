// Host-side launchers shared between the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace attn {

// Rows of one head in the dense tensor-core path's fp16 copies: the length
// rounded up to whole 128-row tiles. The rows past the length are zero, so a
// tile that crosses the end of a sequence loads finite values; the kernel's
// per-element mask keeps them out of every sum.
inline int tc_rows(int s) { return (s + 127) / 128 * 128; }

// Workspace layout: [DevStatus (256 B)] then, for the tensor-core path, fp16
// copies of Q, dO [B, Hq, tc_rows(Sq), D] and K, V [B, Hk, tc_rows(Sk), D]
// (head-major rows, zero past the length), each region aligned to 1 KiB.
// The sparse tensor-core path stages one fp16 copy of the shared KV rows
// [ori rows ; cmp rows] ([(n_ori + n_cmp) * Hk][D]) instead.
struct WorkspaceLayout {
  size_t status = 0;
  size_t q16 = 0, k16 = 0, v16 = 0, do16 = 0, kv16 = 0;
  // deterministic sparse dKV (SparseDet below)
  size_t det_part = 0, det_rows = 0, det_meta = 0, det_slot = 0, det_mult = 0;
  // deterministic dense dbias over several batches: B per-batch slices
  size_t det_dbias = 0;
  size_t total = 0;
  bool staged = false;
};

WorkspaceLayout workspace_layout(const Problem& p, bool tensor_core_path);

// ---- simt_kernels.cu ----
cudaError_t launch_fwd_simt(const Problem& p, const void* q, const void* k, const void* v,
                            const float* bias, const void* ori_kv, const void* cmp_kv,
                            const int32_t* cmp_idx, void* o, float* lse, DevStatus* st,
                            cudaStream_t stream);

cudaError_t launch_bwd_simt(const Problem& p, const void* q, const void* k, const void* v,
                            const void* dO, const float* lse, const float* delta,
                            const float* bias, float* dq, float* dk, float* dv, float* dbias,
                            const void* ori_kv, const void* cmp_kv, const int32_t* cmp_idx,
                            float* d_ori, float* d_cmp, DevStatus* st, cudaStream_t stream);

// ---- preprocess.cu ----
// One fused kernel: clears the status record, zeroes dbias / the sparse dKV
// buffers, computes delta, and (if do16 != nullptr) writes fp16
// head-major copies of q, k, v and dO with tc_rows(S) rows per head (zero
// past the length), and (if kv16 != nullptr) the fp16
// copy of the sparse shared KV rows. dk_zero / dv_zero (may be nullptr) are
// zeroed; dk / dv are recorded in the status record (reserved[2..5]) so the
// backward can check it received the buffers this pass prepared. An fp16
// overflow sets bits (1 q, 2 k or shared KV, 4 v, 8 dO) in the block's flag
// slot after the status record; the tensor-core backward ORs the slots and
// reports ATTN_ERR_RANGE.
cudaError_t launch_preprocess(const Problem& p, const void* q, const void* k, const void* v,
                              const void* o, const void* dO, float* delta,
                              float* dbias, float* d_ori, float* d_cmp, __half* q16, __half* k16,
                              __half* v16, __half* do16, const void* ori_kv, const void* cmp_kv,
                              __half* kv16, float* dk_zero, float* dv_zero, float* dk,
                              float* dv, DevStatus* st, cudaStream_t stream);

// out[e] = slices[0][e] + slices[1][e] + ... + slices[n - 1][e] (in that
// order), slices `stride` floats apart, e < stride.
cudaError_t launch_sum_slices(const float* slices, int n, int64_t stride, float* out,
                              cudaStream_t stream);

// dsinks[h] = -sum_{b, i} exp(sinks[h] - lse[b, h, i]) delta[b, h, i], one
// CTA per head, fixed-order reduction.
cudaError_t launch_dsinks(int B, int Hq, int Sq, const float* sinks, const float* lse,
                          const float* delta, float* dsinks, cudaStream_t stream);

// ---- tc_bwd.cu ----
bool tc_supported(const Problem& p);
// Whether the dense tensor-core kernel computes a requested dbias in its
// batch-inner query-major CTAs (D = 64, B <= 4, whole tiles, fixed lengths):
// every element of a live tile is stored once (no atomics, no zero-filled
// buffer, fixed summation order), so the pre-pass does not zero dbias and
// deterministic mode needs no per-batch slices.
bool tc_dbias_in_q(const Problem& p);
// Key-major CTAs per (key tile, KV head) of the dense tensor-core kernel; when
// above 1 they add partial dK / dV sums into buffers the pre-pass zeroed.
int tc_head_split(const Problem& p);
// Diagnostic: the per-element live sets of the dense tensor-core kernel's
// key-major and query-major CTAs for one sequence of lengths Sq x Sk
// (mask_probe_kernel in tc_bwd.cu). aligned_variant selects the
// instantiation that assumes whole tiles (Sq, Sk multiples of 128).
cudaError_t launch_mask_probe(const MaskSpec& m, int Sq, int Sk, bool aligned_variant,
                              uint8_t* kv_live, uint8_t* q_live, int32_t* outside,
                              cudaStream_t stream);
cudaError_t launch_bwd_tc(const Problem& p, const __half* q16, const __half* k16,
                          const __half* v16, const __half* do16, const float* lse,
                          const float* delta, const float* bias, float* dq, float* dk,
                          float* dv, float* dbias, DevStatus* st, cudaStream_t stream);

// ---- fwd_tc.cu ----
// Dense forward on the tensor cores (D in {64, 128}, q / k / v rows evenly
// spaced over batch and position); attn_fwd_lse falls back to the SIMT
// forward otherwise.
bool fwd_tc_supported(const Problem& p);
cudaError_t launch_fwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          const float* bias, void* o, float* lse, cudaStream_t stream);

// ---- tc_sparse.cu ----
// Deterministic sparse dKV: the tensor-core kernel stores every item's
// (item = token Hk + KV head) dKV rows at their slots in `part`
// ([items * stride][512] fp32) with the item's row list in `rows` and
// {row count, window rows, first window row} in `meta`; sparse_det.cu then
// finds, per item and compressed row, the first slot holding it (`slot`,
// [items * n_cmp]) and how many slots do (`mult`), and adds each dKV row's
// contributions in token order.
struct SparseDet {
  float* part = nullptr;
  int32_t* rows = nullptr;
  int32_t* meta = nullptr;
  int32_t* slot = nullptr;
  int32_t* mult = nullptr;
  int stride = 0;
};
int64_t sparse_det_stride(const Problem& p);  // slots per item: the row bound rounded to 128

bool tc_sparse_supported(const Problem& p);
cudaError_t launch_bwd_sparse_tc(const Problem& p, const void* q, const void* dO,
                                 const __half* kv16, const int32_t* idx, const float* lse,
                                 const float* delta, float* dq, float* d_ori, float* d_cmp,
                                 const SparseDet& det, DevStatus* st, cudaStream_t stream);

// Selected rows per (token, KV head) of a sparse problem: the window plus the
// compressed rows (before padding to whole tiles).
int64_t sparse_row_bound(const Problem& p);
// Diagnostic: the selected-row lists of the sparse tensor-core kernel
// (build_rows), one per item = token Hk + KV head, into rows[item][stride]
// with their lengths in counts[item]; stride >= sparse_row_bound(p) and the
// bound must be at most 1024.
cudaError_t launch_rows_probe(const Problem& p, const int32_t* idx, int32_t* rows,
                              int32_t* counts, int stride, cudaStream_t stream);

// ---- sparse_det.cu ----
// After launch_bwd_sparse_tc in deterministic mode: writes d_ori / d_cmp
// (every row, zero where no token selected it) from det.part.
cudaError_t launch_sparse_det_reduce(const Problem& p, const SparseDet& det, float* d_ori,
                                     float* d_cmp, cudaStream_t stream);

}  // namespace attn
