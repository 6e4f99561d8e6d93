/*
 * attn_bwd.h -- C ABI of the GB300 (sm_103a) fused attention backward library.
 *
 * The library computes, for softmax attention with an optional mask, an
 * optional elementwise bias and grouped-query heads,
 *
 *   S  = scale * Q K^T + bias            (masked entries excluded)
 *   P  = exp(S - LSE)                    (LSE given by the forward)
 *   D  = rowsum(dO * O)
 *   dP = dO V^T,   dS = P * (dP - D)
 *   dQ = scale * dS K,   dK = scale * dS^T Q,   dV = P^T dO,
 *   dbias = sum over the batch of dS,
 *
 * following composable_kernel "34_bwd_gqa_fmha.py" (docstring "CPU backward
 * reference" and cpu_bwd_gqa), "28_backward_dbias_fmha.py"
 * (cpu_attention_bwd_dbias) and "22_sink_tokens_fmha.py" (mask builders), and
 * a selected-KV sparse variant with shared latent KV (K = V) following the
 * Ascend "sparse_flash_mla_grad" formula (phases 1-3).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller. The library
 *    allocates no device memory and keeps no state between calls; all work is
 *    enqueued on `stream` and nothing blocks except attn_read_device_status.
 *  - Host-side argument checks return an error code synchronously and enqueue
 *    nothing. Conditions found on the device (an out-of-range sparse index, an
 *    fp16 range overflow of the staged operands, a bounded wait that ran out)
 *    never trap: the kernel records the first such condition in the status
 *    record at the start of the workspace and skips the offending work;
 *    attn_read_device_status returns it.
 *  - Layouts: q, o, dO are [B, Sq, Hq, D] and k, v are [B, Sk, Hk, D]
 *    ("BSHD", the flash-attn layout of the ring-attention page), addressed
 *    through the element strides in attn_problem_t; the last (D) dimension
 *    must be contiguous. bf16 inputs. lse and delta are fp32 [B, Hq, Sq],
 *    contiguous, natural log. bias and dbias are fp32 [Hq, Sq, Sk],
 *    contiguous, broadcast / summed over the batch. dq is fp32 contiguous
 *    [B, Sq, Hq, D]; dk, dv are fp32 contiguous [B, Sk, Hk, D].
 *  - Query head h reads KV head h / (Hq / Hk) (consecutive grouping, np.repeat
 *    in "34_bwd_gqa_fmha.py"); dk / dv are summed over each group.
 */
#ifndef ATTN_BWD_H
#define ATTN_BWD_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,    /* null pointer, bad shape, bad stride, bad scale */
  ATTN_ERR_UNSUPPORTED = 2,    /* valid request this build does not implement */
  ATTN_ERR_CUDA = 3,           /* a CUDA runtime call failed (launch, attribute) */
  ATTN_ERR_DEVICE_TIMEOUT = 4, /* device: a bounded wait ran out; outputs invalid */
  ATTN_ERR_INDEX_OOB = 5,      /* device: a sparse index >= n_cmp or < -1; entry skipped */
  ATTN_ERR_RANGE = 6,          /* device: an input is outside the fp16 range of the
                                  tensor-core path (|x| > 65504); outputs invalid */
  ATTN_ERR_WORKSPACE = 7       /* workspace null or smaller than attn_bwd_workspace_size */
} attn_status_t;

/* Problem shape and input layout (the FmhaProblem pattern of
 * "34_bwd_gqa_fmha.py": batch, nhead_q, nhead_k, seqlen_q, seqlen_k, hdim).
 * Head dims of q/k and v/o are equal (D). Strides are in ELEMENTS for the
 * (batch, sequence, head) dimensions; each must be a multiple of 8 (16-byte
 * rows) and the base pointers 16-byte aligned. Hq % Hk == 0. */
typedef struct attn_problem {
  int32_t B, Hq, Hk, Sq, Sk, D;
  float scale;            /* softmax scale, finite and > 0 (usually 1/sqrt(D)) */
  int64_t q_stride[3];
  int64_t k_stride[3];
  int64_t v_stride[3];
  int64_t o_stride[3];    /* o (written by attn_fwd_lse, read by preprocess) */
  int64_t do_stride[3];
  int32_t flags;          /* ATTN_FLAG_* bits; 0 = defaults. Pass the same value to
                             attn_bwd_preprocess and attn_bwd. */
  /* Variable-length batch, packed token-major ("TND") rows. With
   * cu_seqlens_q == NULL (zero-initialised struct) the fixed-length layout
   * above applies. Otherwise sequence b holds the query rows
   * [cu_seqlens_q[b], cu_seqlens_q[b + 1]) and the key rows
   * [cu_seqlens_k[b], cu_seqlens_k[b + 1]) (device arrays of B + 1 int32:
   * first entry 0, nondecreasing, last at most total_q / total_k), and Sq, Sk
   * are upper bounds of the per-sequence lengths. Then:
   *  - q, o, dO, dq are [total_q, Hq, D] (stride[1] between tokens,
   *    stride[2] between heads, stride[0] unused; dq contiguous), k, v, dk,
   *    dv are [total_k, Hk, D];
   *  - lse and delta keep the padded [B, Hq, Sq] layout (entries past a
   *    sequence's length are neither read nor written);
   *  - bias / dbias [Hq, Sq, Sk] are indexed by positions within the sequence;
   *  - a mask aligns per sequence (bottom-right uses that sequence's lengths).
   * The dense tensor-core path only: the sparse variant, D = 512,
   * ATTN_FLAG_CUDA_CORES, attn_fwd_lse and attn_bwd_dsinks return
   * ATTN_ERR_UNSUPPORTED. cu_seqlens are
   * checked on the device: a sequence whose bounds are out of order or out
   * of range is skipped and ATTN_ERR_INVALID_ARG recorded in the status
   * record with detail = its index. (Ascend "sparse_flash_mla_grad" takes
   * the TND layout with per-sequence lengths; the CK sink-token page names
   * both causal alignments.) */
  const int32_t* cu_seqlens_q;
  const int32_t* cu_seqlens_k;
  int32_t total_q, total_k;
} attn_problem_t;

/* Deterministic dense backward: dq, dk, dv and dbias are bitwise the same on
 * every run. dk / dv are then written by one CTA per key tile (no split of a
 * key tile's query heads over CTAs, whose partial sums would be added in
 * arrival order). dbias on the tensor-core path at D = 64 with B <= 4 and
 * fixed lengths in whole 128-row tiles is deterministic in either mode (one
 * CTA sums dS over the batches in a fixed order and stores each element
 * once). Other dbias problems with B > 1: the backward kernel (still one
 * launch) adds each batch's terms into that batch's own slice of the
 * workspace (one writer per element, so every slice holds exact values), and
 * a second kernel sums the slices into dbias in batch order; the workspace
 * then holds B * Hq * Sq * Sk more fp32 values. Slower than the default.
 * Sparse variant: the tensor-core kernel stores
 * every (token, KV head)'s dKV rows in the workspace instead of adding them
 * into d_ori_kv / d_cmp_kv, and a second pass adds each row's terms in token
 * order and writes the rows (the workspace then holds Sq * Hk * (selected-row
 * bound rounded up to 128) * D fp32 values, 5.4 GB at 4096 tokens x 640
 * rows); sparse shapes outside the tensor-core kernel return
 * ATTN_ERR_UNSUPPORTED. (Composable_kernel "34_bwd_gqa_fmha.py" names
 * atomics vs a deterministic reduction for dK / dV; the Ascend
 * "sparse_flash_mla_grad" page notes its operator is not deterministic by
 * default.) */
#define ATTN_FLAG_DETERMINISTIC 1

/* Run the CUDA-core kernels (no tensor cores, bf16 operands read directly):
 * a second, independent implementation of the same backward, for
 * cross-checks and for the shapes the tensor-core kernels do not take
 * (dense D = 512, sparse variants other than 64 query heads per KV head at
 * D = 512). The backward runs on them only when this flag asks for it:
 * without it such a problem returns ATTN_ERR_UNSUPPORTED (and
 * attn_bwd_workspace_size / attn_bwd_path return 0). attn_bwd_path returns
 * 2 with the flag. Much slower. */
#define ATTN_FLAG_CUDA_CORES 2

/* Key mask, positions aligned top-left ("22_sink_tokens_fmha.py"):
 *   live(i, j) = (j < num_sink) || (i - window_left <= j && j <= i + window_right)
 * with a negative window bound meaning that side is unbounded. Causal is
 * (-1, 0, 0); causal + n sinks is (-1, 0, n); sliding window of w keys plus n
 * sinks is (w - 1, 0, n). A NULL mask pointer means every entry is live.
 * A row with no live key gets LSE = -inf, O = 0 and no gradient. */
typedef struct attn_mask {
  int32_t window_left;
  int32_t window_right;
  int32_t num_sink;
  int32_t bottom_right; /* 0: top-left as above; 1: bottom-right, i.e. i is
                           replaced by i + (Sk - Sq) in the window test (the
                           diagonal ends in the last query / key corner; with
                           Sk < Sq the first Sq - Sk queries of a causal mask
                           then have no live key). Equal to top-left when
                           Sq == Sk. Sinks are unaffected. */
} attn_mask_t;

/* Selected-KV sparse attention with shared latent KV (Ascend
 * "sparse_flash_mla_grad" formula, phase 1: selectedKv = concat(oriKv
 * window, Gather(cmpKv, topkIndices[i])) in the SCFA case, concat(oriKv
 * window, cmpKv) in the CFA case, oriKv window alone in the SWA case;
 * K = V = selectedKv).
 * One sequence: the problem's B must be 1, its Sk is ignored, k / v / bias /
 * dk / dv / dbias must be NULL. Query i sits at position p = (n_ori - Sq) + i
 * and selects original rows [p - ori_win_left, p + ori_win_right] clipped to
 * [0, n_ori) (negative bound = unbounded) plus compressed rows:
 *   SCFA (cmp_kv and cmp_idx given): the rows listed in cmp_idx[i, g, :]
 *     (-1 = unused slot; indices may repeat and then count twice);
 *   CFA (cmp_kv given, cmp_idx == NULL): every compressed row c whose block
 *     of cmp_ratio original positions ends at or before p, i.e.
 *     c < min(n_cmp, (p + 1) / cmp_ratio) (cmp_ratio >= 1 required; topk is
 *     ignored);
 *   SWA (cmp_kv == NULL, cmp_idx == NULL): none.
 * All arrays contiguous: ori_kv bf16 [n_ori, Hk, D], cmp_kv bf16
 * [n_cmp, Hk, D], cmp_idx int32 [Sq, Hk, topk]; gradients d_ori_kv fp32
 * [n_ori, Hk, D] and d_cmp_kv fp32 [n_cmp, Hk, D] receive dKV = dK + dV,
 * summed over every query and head that selected the row. */
typedef struct attn_sparse {
  const void* ori_kv;
  const void* cmp_kv;
  const int32_t* cmp_idx;
  int32_t n_ori, n_cmp, topk;
  int32_t ori_win_left, ori_win_right;
  float* d_ori_kv;
  float* d_cmp_kv;
  int32_t cmp_ratio; /* CFA only: original positions per compressed row */
} attn_sparse_t;

/* Forward with log-sum-exp, used to produce the backward's O and LSE inputs
 * ("34_bwd_gqa_fmha.py" cpu_fwd_with_intermediates, "28_backward_dbias_fmha.py"
 * cpu_attention_fwd_bias, "22_sink_tokens_fmha.py" cpu_attention_fwd_masked).
 * Writes o (bf16, o_stride layout) and lse (fp32 [B, Hq, Sq], natural log).
 * sparse != NULL selects the sparse variant (k, v, bias must then be NULL).
 * Dense problems with D in {64, 128} whose q / k / v rows are evenly spaced
 * over (batch, position) (stride[0] == S * stride[1], or B == 1) run on the
 * tensor cores: bf16 operands, one pass over the live key tiles (online
 * softmax with a lazily rescaled fp32 O accumulator, divided by the row sum
 * at the end), P rounded to bf16 for its MMA; LSE = max + log(sum) in fp32.
 * Other shapes (this producer of the backward's inputs has no other
 * implementation for them), and ATTN_FLAG_CUDA_CORES, run the fp32
 * CUDA-core forward. A variable-length batch returns ATTN_ERR_UNSUPPORTED. */
attn_status_t attn_fwd_lse(const attn_problem_t* prob, const attn_mask_t* mask,
                           const attn_sparse_t* sparse,
                           const void* q, const void* k, const void* v,
                           const float* bias, void* o, float* lse,
                           cudaStream_t stream);

/* Bytes of device workspace that attn_bwd_preprocess and attn_bwd need for
 * this problem: a status record, the fp16 staging of the operands of the
 * tensor-core path (lengths rounded up to whole 128-row tiles), and with
 * ATTN_FLAG_DETERMINISTIC the per-batch dbias slices (dense, B > 1, outside
 * the D = 64 batch-inner case above) or the per-slot dKV rows (sparse).
 * Returns 0 if the arguments are invalid or the problem needs the CUDA-core
 * kernels without ATTN_FLAG_CUDA_CORES. */
size_t attn_bwd_workspace_size(const attn_problem_t* prob, const attn_mask_t* mask,
                               const attn_sparse_t* sparse);

/* Backward pre-pass ("34_bwd_gqa_fmha.py" cpu_bwd_gqa: D = rowsum(dO * O);
 * Ascend formula phase 2: SoftmaxGrad(dO, O)):
 *  - delta[b, h, i] = sum_d dO[b, i, h, d] * O[b, i, h, d] in fp32;
 *  - zeroes the outputs attn_bwd accumulates into: dbias (if non-NULL and
 *    not in the D = 64 batch-inner case, where attn_bwd stores every entry;
 *    in the deterministic mode with B > 1, the per-batch dbias slices of the
 *    workspace instead, which attn_bwd then sums into dbias), for the sparse
 *    variant sparse->d_ori_kv / d_cmp_kv, and dk / dv when the tensor-core
 *    path splits a KV head's query-head group over several CTAs that add
 *    their partial sums (small problems);
 *  - clears the workspace status record;
 *  - when attn_bwd will take the tensor-core path, writes fp16 copies of q,
 *    k, v and dO into the workspace (head-major rows, each head's length
 *    rounded up to whole 128-row tiles with zero rows) for it.
 *    Every bf16 value of magnitude in [2^-14, 65504] converts exactly; a
 *    larger one is recorded as ATTN_ERR_RANGE.
 * q, k, v, dbias, dk and dv are the same tensors later passed to attn_bwd
 * (k, v, dk, dv NULL for the sparse variant; for a dense problem dk and dv
 * must be given, fp32 [B, Sk, Hk, D] contiguous, 16-byte aligned). Must
 * precede attn_bwd on the same stream with the same workspace, and the inputs
 * must not change in between; attn_bwd reports ATTN_ERR_INVALID_ARG through
 * the status record (and leaves dk / dv unwritten) if it receives dk / dv
 * buffers other than the ones this call prepared. */
attn_status_t attn_bwd_preprocess(const attn_problem_t* prob, const attn_sparse_t* sparse,
                                  const void* q, const void* k, const void* v,
                                  const void* o, const void* dO, float* delta,
                                  float* dbias, float* dk, float* dv,
                                  void* workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/* The fused backward ("34_bwd_gqa_fmha.py" docstring and cpu_bwd_gqa;
 * "28_backward_dbias_fmha.py" cpu_attention_bwd_dbias; Ascend
 * "sparse_flash_mla_grad" phases 1-3). P is rebuilt from lse; delta comes
 * from attn_bwd_preprocess, which also zeroed dbias, the sparse gradients
 * and (when needed) dk / dv that this call accumulates into; dq, dk and dv
 * hold the complete gradients afterwards. dbias may be non-NULL without bias (gradient of a zero
 * bias). Returns ATTN_ERR_UNSUPPORTED for D outside {64, 128, 512} or the
 * sparse variant with D != 512 when no fallback kernel covers it. */
attn_status_t attn_bwd(const attn_problem_t* prob, const attn_mask_t* mask,
                       const attn_sparse_t* sparse,
                       const void* q, const void* k, const void* v, const void* dO,
                       const float* lse, const float* delta, const float* bias,
                       float* dq, float* dk, float* dv, float* dbias,
                       void* workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Gradient of learnable sink logits (one per query head): a sink logit s_h
 * joins every softmax denominator of head h without a value vector, so it is
 * already inside the LSE the forward returned, and P, dS, dq, dk, dv of
 * attn_bwd are unchanged by it. Its own gradient (Ascend
 * "sparse_flash_mla_grad" formula, phase 3: dSinks = ReduceSum(-P x dP x
 * SimpleSoftmax(sinks, lse))) is
 *   dsinks[h] = -sum over b, i of exp(sinks[h] - lse[b, h, i]) * delta[b, h, i]
 * with delta the attn_bwd_preprocess output; rows with lse = -inf add nothing.
 * sinks, dsinks fp32 [Hq]; lse, delta fp32 [B, Hq, Sq] (B = 1 for the sparse
 * variant); all device memory, 4-byte aligned. dsinks is overwritten. One CTA
 * per head sums in a fixed order: the result is bitwise reproducible.
 * Call after attn_bwd_preprocess on the same stream. Returns
 * ATTN_ERR_INVALID_ARG for null pointers or non-positive B, Hq, Sq. */
attn_status_t attn_bwd_dsinks(const attn_problem_t* prob, const float* sinks,
                              const float* lse, const float* delta, float* dsinks,
                              cudaStream_t stream);

/* Synchronises `stream`, then returns the first device-side condition
 * recorded in the workspace status record since the last
 * attn_bwd_preprocess (ATTN_OK if none). *detail (may be NULL) receives a
 * condition-specific integer (e.g. the offending query row). */
attn_status_t attn_read_device_status(const void* workspace, cudaStream_t stream,
                                      int32_t* detail);

/* Static, human-readable name of a status code. */
const char* attn_status_string(attn_status_t status);

/* Backward without any device allocation by the caller or the library.
 * The source pages have no counterpart of this entry point: it exists for
 * callers that cannot call cudaMalloc -- code running inside a framework hook
 * that must not re-enter the framework's allocator, deployments whose device
 * memory is fixed at start-up, or paths that must not stall other streams
 * (cudaMalloc can synchronise the device).
 *
 * It runs attn_bwd_preprocess and attn_bwd (same arguments and results as
 * those two calls) with their workspace placed in a fixed 32 MiB array that
 * the library keeps in the device memory of every GPU it is used on, for as
 * long as the library is loaded. Inputs and outputs stay caller-owned device
 * memory; delta is an output here (the pre-pass's rowsum(dO * O)).
 * - Returns ATTN_ERR_WORKSPACE, before enqueuing anything, when the problem
 *   needs more than 32 MiB of workspace (attn_bwd_workspace_size).
 * - The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any
 *   stream capture. The address belongs to the device's context: if that
 *   context is replaced (cudaDeviceReset), the next call looks it up again,
 *   and that call too should come before any stream capture.
 * - All calls share the array and it keeps the last call's contents (the
 *   pre-pass rewrites everything the backward reads). Calls whose work
 *   overlaps on the GPU race on it: order them on one stream or synchronise.
 * - device_status may be NULL. Otherwise the call synchronises `stream` and
 *   stores the device-side status code in device_status[0] and its detail in
 *   device_status[1] (as attn_read_device_status would). If the status
 *   record cannot be read back (the synchronisation or the copy fails), the
 *   call returns ATTN_ERR_CUDA and leaves device_status unwritten. */
attn_status_t attn_bwd_noalloc(const attn_problem_t* prob, const attn_mask_t* mask,
                               const attn_sparse_t* sparse,
                               const void* q, const void* k, const void* v,
                               const void* o, const void* dO, const float* lse,
                               const float* bias, float* delta,
                               float* dq, float* dk, float* dv, float* dbias,
                               cudaStream_t stream, int32_t* device_status);

/* Tile classes of a mask ("22_sink_tokens_fmha.py" mask builders applied to
 * tiles): out[mt * ceil(Sk / tile_k) + nt] = 0 if the tile rows
 * [mt tile_q, ...) x keys [nt tile_k, ...) (clipped to Sq, Sk) hold no live
 * entry, 2 if every entry is live, 1 otherwise. Host-only (the same
 * classification the kernels use to skip tiles and to mask partial ones);
 * out holds ceil(Sq / tile_q) * ceil(Sk / tile_k) bytes. Returns
 * ATTN_ERR_INVALID_ARG for non-positive sizes or a NULL out. */
attn_status_t attn_mask_tile_classes(const attn_mask_t* mask, int32_t Sq, int32_t Sk,
                                     int32_t tile_q, int32_t tile_k, int8_t* out);

/* Diagnostic (tests): the per-element live sets of the dense tensor-core
 * backward, read back from the device. For one sequence of Sq queries and Sk
 * keys under `mask` (NULL = every entry live; bottom_right honoured), a kernel
 * walks the live tiles and applies the per-element predicate exactly as the
 * backward's two kinds of CTA do: the key-major CTAs (dK, dV; a thread per key
 * row) and the query-major CTAs (dQ; a thread per query row). For every entry
 * it treats as live it adds 1 to kv_live[i * Sk + j] (key-major view) or
 * q_live[i * Sk + j] (query-major view); a live entry outside the lengths
 * adds 1 to *outside instead. With a correct mask both arrays equal the mask
 * ("22_sink_tokens_fmha.py" mask builders) as 0 / 1 bytes and *outside stays
 * 0; a 2 would mean a tile visited twice.
 * kv_live, q_live: device uint8 [Sq, Sk]; outside: device int32 [1]; all
 * zeroed by the caller, written on `stream`. aligned_variant = 1 probes the
 * kernel instantiation that assumes whole 128-row tiles (Sq and Sk must then
 * be multiples of 128), 0 the one that handles any lengths. Returns
 * ATTN_ERR_INVALID_ARG for non-positive sizes, NULL outputs or a bad variant. */
attn_status_t attn_debug_mask_live(const attn_mask_t* mask, int32_t Sq, int32_t Sk,
                                   int32_t aligned_variant, uint8_t* kv_live, uint8_t* q_live,
                                   int32_t* outside, cudaStream_t stream);

/* Diagnostic (tests): the selected-row lists of the sparse tensor-core
 * backward (Ascend "sparse_flash_mla_grad" formula, phase 1), built on the
 * device by the same routine the backward kernel runs. For every item =
 * i * Hk + g (query token i, KV head g) it writes the item's rows, in the
 * order the kernel processes them (the original-KV window ascending, then
 * the valid top-k entries in slot order, or every eligible compressed row
 * for CFA), to rows[item * max_rows + 0 .. n - 1] and n to counts[item]. A
 * row is an index into [ori rows ; cmp rows] x Hk: original row r of KV
 * head g is r * Hk + g, compressed row c is (n_ori + c) * Hk + g. Indices
 * that are -1 or out of range are skipped. rows: device int32
 * [Sq * Hk, max_rows]; counts: device int32 [Sq * Hk]. prob / sparse as for
 * attn_bwd (gradient pointers unused). Returns ATTN_ERR_INVALID_ARG when
 * max_rows is below the per-item bound (window + topk, or window + n_cmp
 * for CFA) and ATTN_ERR_UNSUPPORTED when that bound exceeds 1024 (the
 * tensor-core kernel's limit). */
attn_status_t attn_debug_sparse_rows(const attn_problem_t* prob, const attn_sparse_t* sparse,
                                     int32_t* rows, int32_t* counts, int32_t max_rows,
                                     cudaStream_t stream);

/* Which backward kernel attn_bwd would launch for these arguments:
 * 0 = none (invalid, unsupported, or outside the tensor-core shapes without
 * ATTN_FLAG_CUDA_CORES), 1 = tcgen05 tensor-core kernel, 2 = SIMT kernels
 * (ATTN_FLAG_CUDA_CORES). For tests and benchmarks. */
int32_t attn_bwd_path(const attn_problem_t* prob, const attn_mask_t* mask,
                      const attn_sparse_t* sparse);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_BWD_H */
