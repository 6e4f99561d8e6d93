// Backward pre-pass and operand staging.
//
// D = rowsum(dO * O) ("34_bwd_gqa_fmha.py" cpu_bwd_gqa; Ascend
// "sparse_flash_mla_grad" phase 2, SoftmaxGrad(dO, O)), computed in fp32 from
// the bf16 rows, one warp per (b, i, h) row. The same pass zeroes the row of
// dq that the backward accumulates into and, for the tensor-core path, writes
// dO once as an fp16 head-major copy. All of it is HBM-bound streaming.
//
// The tensor-core backward feeds fp16 operands to kind::f16 MMAs: the
// probabilities P and the gradient dS are rounded to fp16 (11 significant
// bits) instead of bf16 (8 bits), which keeps the rounding of the gradient
// operands well inside the parity tolerance, and the other operand of each
// of those MMAs must then be fp16 as well. bf16 -> fp16 is exact for every
// bf16 value of magnitude in [2^-14, 65504]; larger magnitudes are reported as
// ATTN_ERR_RANGE, smaller ones lose low bits (absolute error below 2^-25).

#include "internal.h"

namespace attn {
namespace {

using bf16 = __nv_bfloat16;
constexpr int kWarps = 8;

__device__ __forceinline__ void zero_range(float* a, int64_t n, int64_t tid, int64_t stride) {
  // a is 16-byte aligned (checked on the host); float4 body, scalar tail.
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  float4* a4 = reinterpret_cast<float4*>(a);
  for (int64_t t = tid; t < n / 4; t += stride) a4[t] = z;
  for (int64_t t = (n / 4) * 4 + tid; t < n; t += stride) a[t] = 0.f;
}

__global__ void clear_kernel(DevStatus* st, float* a, int64_t na, float* b, int64_t nb,
                             float* c, int64_t nc) {
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  if (tid == 0 && st != nullptr) {
    st->code = 0;
    st->detail = 0;
  }
  zero_range(a, na, tid, stride);
  zero_range(b, nb, tid, stride);
  zero_range(c, nc, tid, stride);
}

template <int EPL>
__device__ __forceinline__ bool store_half_checked(__half* dst, const float* x) {
  bool bad = false;
#pragma unroll
  for (int e = 0; e < EPL; e += 2) {
    __half2 h = __floats2half2_rn(x[e], x[e + 1]);
    bad |= __hisinf(__low2half(h)) | __hisinf(__high2half(h));
    *reinterpret_cast<__half2*>(dst + e) = h;
  }
  return bad;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
preprocess_kernel(int B, int Hq, int Sq, int64_t o0, int64_t o1, int64_t o2, int64_t d0,
                  int64_t d1, int64_t d2, const bf16* __restrict__ o,
                  const bf16* __restrict__ dO, float* __restrict__ delta,
                  float* __restrict__ dq, __half* __restrict__ do16, DevStatus* st) {
  constexpr int EPL = D / 32;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (int64_t)B * Hq * Sq) return;
  // Rows in memory order of dq ([B, Sq, Hq, D]) so the zeroing streams.
  const int h = (int)(warp % Hq);
  const int i = (int)((warp / Hq) % Sq);
  const int b = (int)(warp / ((int64_t)Hq * Sq));
  float ov[EPL], dv[EPL];
  load_bf16<EPL>(o + b * o0 + i * o1 + h * o2 + lane * EPL, ov);
  load_bf16<EPL>(dO + b * d0 + i * d1 + h * d2 + lane * EPL, dv);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) s = fmaf(ov[e], dv[e], s);
  s = warp_sum(s);
  const int64_t r = ((int64_t)b * Hq + h) * Sq + i;
  if (lane == 0) delta[r] = s;
  float z[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) z[e] = 0.f;
  store_f32<EPL>(dq + warp * D + lane * EPL, z);
  if (do16 != nullptr) {
    if (store_half_checked<EPL>(do16 + r * D + lane * EPL, dv)) report(st, ATTN_ERR_RANGE, 3);
  }
}

// fp16 head-major copies of q (which = 0), k (1), v (2): warp per source row.
template <int D>
__global__ void __launch_bounds__(kWarps * 32)
stage_kernel(int B, int Hq, int Hk, int Sq, int Sk, int64_t q0, int64_t q1, int64_t q2, int64_t k0, int64_t k1, int64_t k2,
             int64_t v0, int64_t v1, int64_t v2, const bf16* __restrict__ q,
             const bf16* __restrict__ k, const bf16* __restrict__ v, __half* __restrict__ q16,
             __half* __restrict__ k16, __half* __restrict__ v16, DevStatus* st) {
  constexpr int EPL = D / 32;
  int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t nq = (int64_t)B * Hq * Sq;
  const int64_t nk = (int64_t)B * Hk * Sk;
  const bf16* src;
  __half* dst;
  int which;
  if (warp < nq) {
    // destination order [B, Hq, Sq]
    const int i = (int)(warp % Sq);
    const int h = (int)((warp / Sq) % Hq);
    const int b = (int)(warp / ((int64_t)Sq * Hq));
    src = q + b * q0 + i * q1 + h * q2;
    dst = q16 + warp * D;
    which = 0;
  } else {
    warp -= nq;
    which = 1;
    if (warp >= nk) {
      warp -= nk;
      which = 2;
      if (warp >= nk) return;
    }
    const int j = (int)(warp % Sk);
    const int g = (int)((warp / Sk) % Hk);
    const int b = (int)(warp / ((int64_t)Sk * Hk));
    src = (which == 1) ? k + b * k0 + j * k1 + g * k2 : v + b * v0 + j * v1 + g * v2;
    dst = ((which == 1) ? k16 : v16) + warp * D;
  }
  float x[EPL];
  load_bf16<EPL>(src + lane * EPL, x);
  if (store_half_checked<EPL>(dst + lane * EPL, x)) report(st, ATTN_ERR_RANGE, which);
}

inline unsigned blocks_for(int64_t warps) { return (unsigned)((warps + kWarps - 1) / kWarps); }

}  // namespace

cudaError_t launch_preprocess(const Problem& p, const void* o, const void* dO, float* delta,
                              float* dq, float* dbias, float* d_ori, float* d_cmp,
                              __half* do16, DevStatus* st, cudaStream_t stream) {
  // 1) status record + buffers accumulated with atomics
  const int64_t nbias = dbias ? (int64_t)p.Hq * p.Sq * p.Sk : 0;
  const int64_t nori = d_ori ? (int64_t)p.n_ori * p.Hk * p.D : 0;
  const int64_t ncmp = d_cmp ? (int64_t)p.n_cmp * p.Hk * p.D : 0;
  const int64_t work = (nbias + nori + ncmp) / 4;
  int64_t g = (work + 255) / 256;
  g = g < 1 ? 1 : (g > 152 * 16 ? 152 * 16 : g);
  clear_kernel<<<(unsigned)g, 256, 0, stream>>>(st, dbias, nbias, d_ori, nori, d_cmp, ncmp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // 2) delta, dq zeroing, dO staging
  const int64_t rows = (int64_t)p.B * p.Hq * p.Sq;
  if (rows == 0) return cudaSuccess;
  const bf16* ob = static_cast<const bf16*>(o);
  const bf16* db = static_cast<const bf16*>(dO);
#define ATTN_PRE(DD)                                                                        \
  preprocess_kernel<DD><<<blocks_for(rows), kWarps * 32, 0, stream>>>(                      \
      p.B, p.Hq, p.Sq, p.os[0], p.os[1], p.os[2], p.dos[0], p.dos[1], p.dos[2], ob, db, delta, \
      dq, do16, st)
  switch (p.D) {
    case 64: ATTN_PRE(64); break;
    case 128: ATTN_PRE(128); break;
    case 512: ATTN_PRE(512); break;
    default: return cudaErrorInvalidValue;
  }
#undef ATTN_PRE
  return cudaGetLastError();
}

cudaError_t launch_stage_qkv(const Problem& p, const void* q, const void* k, const void* v,
                             __half* q16, __half* k16, __half* v16, DevStatus* st,
                             cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.Hq * p.Sq + 2 * (int64_t)p.B * p.Hk * p.Sk;
  if (rows == 0) return cudaSuccess;
#define ATTN_STAGE(DD)                                                                      \
  stage_kernel<DD><<<blocks_for(rows), kWarps * 32, 0, stream>>>(                           \
      p.B, p.Hq, p.Hk, p.Sq, p.Sk, p.qs[0], p.qs[1], p.qs[2], p.ks[0], p.ks[1],     \
      p.ks[2], p.vs[0], p.vs[1], p.vs[2], static_cast<const bf16*>(q),                      \
      static_cast<const bf16*>(k), static_cast<const bf16*>(v), q16, k16, v16, st)
  switch (p.D) {
    case 64: ATTN_STAGE(64); break;
    case 128: ATTN_STAGE(128); break;
    case 512: ATTN_STAGE(512); break;
    default: return cudaErrorInvalidValue;
  }
#undef ATTN_STAGE
  return cudaGetLastError();
}

}  // namespace attn
