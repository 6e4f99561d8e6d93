// SIMT (CUDA-core) kernels: the attention forward that produces O / LSE, and a
// general backward used for shapes the tensor-core kernel does not cover
// (the selected-KV sparse variant, head dim 512, ragged sequence lengths).
//
// One warp owns one output row; each lane holds D / 32 consecutive elements of
// the row, so every row load is one coalesced 2*D-byte transaction and a dot
// product is a lane-local FMA chain plus a 5-step butterfly reduction.
//
// Formulas: composable_kernel "34_bwd_gqa_fmha.py" (forward with LSE,
// cpu_bwd_gqa), "28_backward_dbias_fmha.py" (bias, dbias),
// "22_sink_tokens_fmha.py" (masks), Ascend "sparse_flash_mla_grad" (selected
// shared KV, phases 1-3).

#include "internal.h"

#include <math.h>

namespace attn {
namespace {

using bf16 = __nv_bfloat16;

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ int64_t row_off(const int64_t* s, int b, int i, int h) {
  return (int64_t)b * s[0] + (int64_t)i * s[1] + (int64_t)h * s[2];
}

struct Strides {
  int64_t q[3], k[3], v[3], o[3], dO[3];
};

// Online-softmax accumulator for one row.
template <int EPL>
struct RowSoftmax {
  float m = -INFINITY, l = 0.f, acc[EPL];
  __device__ RowSoftmax() {
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  }
  __device__ __forceinline__ void add(float s, const float* vv) {
    float m_new = fmaxf(m, s);
    float corr = expf(m - m_new);
    float w = expf(s - m_new);
    l = l * corr + w;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = acc[e] * corr + w * vv[e];
    m = m_new;
  }
};

// ----------------------------------------------------------------- forward --

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
fwd_dense_kernel(int B, int Hq, int Hk, int Sq, int Sk, float scale, MaskSpec mask,
                 Strides st, const bf16* __restrict__ q, const bf16* __restrict__ k,
                 const bf16* __restrict__ v, const float* __restrict__ bias,
                 bf16* __restrict__ o, float* __restrict__ lse) {
  constexpr int EPL = D / 32;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (int64_t)B * Hq * Sq) return;
  const int i = (int)(warp % Sq);
  const int h = (int)((warp / Sq) % Hq);
  const int b = (int)(warp / ((int64_t)Sq * Hq));
  const int g = h / (Hq / Hk);

  float qv[EPL];
  load_bf16<EPL>(q + row_off(st.q, b, i, h) + lane * EPL, qv);
  RowSoftmax<EPL> rs;
  const float* brow = bias ? bias + ((int64_t)h * Sq + i) * Sk : nullptr;
  auto visit = [&](int j) {
    float kv[EPL], vv[EPL];
    load_bf16<EPL>(k + row_off(st.k, b, j, g) + lane * EPL, kv);
    load_bf16<EPL>(v + row_off(st.v, b, j, g) + lane * EPL, vv);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) s = fmaf(qv[e], kv[e], s);
    s = warp_sum(s) * scale;
    if (brow) s += brow[j];
    rs.add(s, vv);
  };
  const int ns = min(mask.sink, Sk);
  for (int j = 0; j < ns; ++j) visit(j);
  int lo, hi;
  mask_row_range(mask, i, Sk, &lo, &hi);
  for (int j = max(lo, ns); j <= hi; ++j) visit(j);

  float out[EPL];
  const bool live = rs.l > 0.f;
  const float inv = live ? 1.f / rs.l : 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) out[e] = rs.acc[e] * inv;
  store_bf16<EPL>(o + row_off(st.o, b, i, h) + lane * EPL, out);
  if (lane == 0) lse[((int64_t)b * Hq + h) * Sq + i] = live ? rs.m + logf(rs.l) : -INFINITY;
}

// Selected rows of query i (Ascend phase 1): the original-KV window, then the
// listed compressed rows. Calls f(row_pointer) for each; reports bad indices.
struct SparseSel {
  const bf16* ori;
  const bf16* cmp;
  const int32_t* idx;
  int Sq, Hk, D, n_ori, n_cmp, topk, wl, wr, ratio;  // ratio > 0: CFA (no index list)
};

template <typename F>
__device__ __forceinline__ void for_each_selected(const SparseSel& s, int i, int g,
                                                  DevStatus* st, F&& f) {
  const int pos = (s.n_ori - s.Sq) + i;
  int lo = s.wl >= 0 ? pos - s.wl : 0;
  int hi = s.wr >= 0 ? pos + s.wr : s.n_ori - 1;
  lo = max(lo, 0);
  hi = min(hi, s.n_ori - 1);
  for (int j = lo; j <= hi; ++j) f(s.ori + ((int64_t)j * s.Hk + g) * s.D, 0, j);
  if (s.cmp == nullptr) return;
  if (s.ratio > 0) {  // CFA: every compressed row whose block ends at or before pos
    const int nc = min(s.n_cmp, max(pos + 1, 0) / s.ratio);
    for (int c = 0; c < nc; ++c) f(s.cmp + ((int64_t)c * s.Hk + g) * s.D, 1, c);
    return;
  }
  const int32_t* row = s.idx + ((int64_t)i * s.Hk + g) * s.topk;
  for (int t = 0; t < s.topk; ++t) {
    const int c = __ldg(row + t);
    if (c < 0) {
      if (c != -1) report(st, ATTN_ERR_INDEX_OOB, i);
      continue;
    }
    if (c >= s.n_cmp) {
      report(st, ATTN_ERR_INDEX_OOB, i);
      continue;
    }
    f(s.cmp + ((int64_t)c * s.Hk + g) * s.D, 1, c);
  }
}

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
fwd_sparse_kernel(int Hq, float scale, Strides st, SparseSel sel, const bf16* __restrict__ q,
                  bf16* __restrict__ o, float* __restrict__ lse, DevStatus* status) {
  constexpr int EPL = D / 32;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (int64_t)sel.Sq * Hq) return;
  const int h = (int)(warp % Hq);
  const int i = (int)(warp / Hq);
  const int g = h / (Hq / sel.Hk);
  float qv[EPL];
  load_bf16<EPL>(q + row_off(st.q, 0, i, h) + lane * EPL, qv);
  RowSoftmax<EPL> rs;
  for_each_selected(sel, i, g, status, [&](const bf16* row, int, int) {
    float kv[EPL];
    load_bf16<EPL>(row + lane * EPL, kv);
    float s = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) s = fmaf(qv[e], kv[e], s);
    rs.add(warp_sum(s) * scale, kv);
  });
  float out[EPL];
  const bool live = rs.l > 0.f;
  const float inv = live ? 1.f / rs.l : 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) out[e] = rs.acc[e] * inv;
  store_bf16<EPL>(o + row_off(st.o, 0, i, h) + lane * EPL, out);
  if (lane == 0) lse[(int64_t)h * sel.Sq + i] = live ? rs.m + logf(rs.l) : -INFINITY;
}

// ---------------------------------------------------------------- backward --

// dQ rows (and dbias): warp per (b, h, i), loop over live keys.
template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_dq_kernel(int B, int Hq, int Hk, int Sq, int Sk, float scale, MaskSpec mask, Strides st,
              const bf16* __restrict__ q, const bf16* __restrict__ k,
              const bf16* __restrict__ v, const bf16* __restrict__ dO,
              const float* __restrict__ lse, const float* __restrict__ delta,
              const float* __restrict__ bias, float* __restrict__ dq,
              float* __restrict__ dbias, int64_t dbias_bstride) {
  constexpr int EPL = D / 32;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (int64_t)B * Hq * Sq) return;
  const int i = (int)(warp % Sq);
  const int h = (int)((warp / Sq) % Hq);
  const int b = (int)(warp / ((int64_t)Sq * Hq));
  const int g = h / (Hq / Hk);
  const int64_t r = ((int64_t)b * Hq + h) * Sq + i;
  const float L = lse[r];
  const float Dl = delta[r];
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  if (L != -INFINITY) {
    float qv[EPL], dov[EPL];
    load_bf16<EPL>(q + row_off(st.q, b, i, h) + lane * EPL, qv);
    load_bf16<EPL>(dO + row_off(st.dO, b, i, h) + lane * EPL, dov);
    const int64_t brow = ((int64_t)h * Sq + i) * Sk;
    auto visit = [&](int j) {
      float kv[EPL], vv[EPL];
      load_bf16<EPL>(k + row_off(st.k, b, j, g) + lane * EPL, kv);
      load_bf16<EPL>(v + row_off(st.v, b, j, g) + lane * EPL, vv);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        s = fmaf(qv[e], kv[e], s);
        dp = fmaf(dov[e], vv[e], dp);
      }
      s = warp_sum(s) * scale;
      dp = warp_sum(dp);
      if (bias) s += bias[brow + j];
      const float p = expf(s - L);
      const float ds = p * (dp - Dl);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(ds, kv[e], acc[e]);
      if (dbias && lane == 0) atomicAdd(dbias + b * dbias_bstride + brow + j, ds);
    };
    const int ns = min(mask.sink, Sk);
    for (int j = 0; j < ns; ++j) visit(j);
    int lo, hi;
    mask_row_range(mask, i, Sk, &lo, &hi);
    for (int j = max(lo, ns); j <= hi; ++j) visit(j);
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] *= scale;
  store_f32<EPL>(dq + (((int64_t)b * Sq + i) * Hq + h) * D + lane * EPL, acc);
}

// dK / dV rows: warp per (b, g, j), loop over the group's heads and live queries.
template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_dkdv_kernel(int B, int Hq, int Hk, int Sq, int Sk, float scale, MaskSpec mask, Strides st,
                const bf16* __restrict__ q, const bf16* __restrict__ k,
                const bf16* __restrict__ v, const bf16* __restrict__ dO,
                const float* __restrict__ lse, const float* __restrict__ delta,
                const float* __restrict__ bias, float* __restrict__ dk,
                float* __restrict__ dv) {
  constexpr int EPL = D / 32;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (int64_t)B * Hk * Sk) return;
  const int j = (int)(warp % Sk);
  const int g = (int)((warp / Sk) % Hk);
  const int b = (int)(warp / ((int64_t)Sk * Hk));
  const int ratio = Hq / Hk;
  float kv[EPL], vv[EPL], ak[EPL], av[EPL];
  load_bf16<EPL>(k + row_off(st.k, b, j, g) + lane * EPL, kv);
  load_bf16<EPL>(v + row_off(st.v, b, j, g) + lane * EPL, vv);
#pragma unroll
  for (int e = 0; e < EPL; ++e) ak[e] = av[e] = 0.f;
  int lo = 0, hi = Sq - 1;
  if (j >= mask.sink) mask_col_range(mask, j, Sq, &lo, &hi);
  for (int h = g * ratio; h < (g + 1) * ratio; ++h) {
    for (int i = lo; i <= hi; ++i) {
      const int64_t r = ((int64_t)b * Hq + h) * Sq + i;
      const float L = lse[r];
      if (L == -INFINITY) continue;
      float qv[EPL], dov[EPL];
      load_bf16<EPL>(q + row_off(st.q, b, i, h) + lane * EPL, qv);
      load_bf16<EPL>(dO + row_off(st.dO, b, i, h) + lane * EPL, dov);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        s = fmaf(qv[e], kv[e], s);
        dp = fmaf(dov[e], vv[e], dp);
      }
      s = warp_sum(s) * scale;
      dp = warp_sum(dp);
      if (bias) s += bias[((int64_t)h * Sq + i) * Sk + j];
      const float p = expf(s - L);
      const float ds = p * (dp - delta[r]);
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        ak[e] = fmaf(ds, qv[e], ak[e]);
        av[e] = fmaf(p, dov[e], av[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) ak[e] *= scale;
  const int64_t out = (((int64_t)b * Sk + j) * Hk + g) * D + lane * EPL;
  store_f32<EPL>(dk + out, ak);
  store_f32<EPL>(dv + out, av);
}

// Sparse dQ: warp per (i, h) over the selected shared-KV rows.
template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_sparse_dq_kernel(int Hq, float scale, Strides st, SparseSel sel,
                     const bf16* __restrict__ q, const bf16* __restrict__ dO,
                     const float* __restrict__ lse, const float* __restrict__ delta,
                     float* __restrict__ dq, DevStatus* status) {
  constexpr int EPL = D / 32;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= (int64_t)sel.Sq * Hq) return;
  const int h = (int)(warp % Hq);
  const int i = (int)(warp / Hq);
  const int g = h / (Hq / sel.Hk);
  const int64_t r = (int64_t)h * sel.Sq + i;
  const float L = lse[r];
  const float Dl = delta[r];
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  if (L != -INFINITY) {
    float qv[EPL], dov[EPL];
    load_bf16<EPL>(q + row_off(st.q, 0, i, h) + lane * EPL, qv);
    load_bf16<EPL>(dO + row_off(st.dO, 0, i, h) + lane * EPL, dov);
    for_each_selected(sel, i, g, status, [&](const bf16* row, int, int) {
      float kv[EPL];
      load_bf16<EPL>(row + lane * EPL, kv);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        s = fmaf(qv[e], kv[e], s);
        dp = fmaf(dov[e], kv[e], dp);
      }
      s = warp_sum(s) * scale;
      dp = warp_sum(dp);
      const float p = expf(s - L);
      const float ds = p * (dp - Dl);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = fmaf(ds, kv[e], acc[e]);
    });
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] *= scale;
  store_f32<EPL>(dq + ((int64_t)i * Hq + h) * D + lane * EPL, acc);
}

// Sparse dKV: block per (i, g). For each selected row the warps split the
// group's heads, sum scale*dS*q + P*dO over them, reduce across warps in
// shared memory and add the row's contribution with one atomic per element.
template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_sparse_dkv_kernel(int Hq, float scale, Strides st, SparseSel sel,
                      const bf16* __restrict__ q, const bf16* __restrict__ dO,
                      const float* __restrict__ lse, const float* __restrict__ delta,
                      float* __restrict__ d_ori, float* __restrict__ d_cmp,
                      DevStatus* status) {
  constexpr int EPL = D / 32;
  __shared__ float red[kWarpsPerBlock][D];
  const int i = blockIdx.x / sel.Hk;
  const int g = blockIdx.x % sel.Hk;
  const int w = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ratio = Hq / sel.Hk;
  for_each_selected(sel, i, g, w == 0 ? status : nullptr, [&](const bf16* row, int src, int j) {
    float kv[EPL], c[EPL];
    load_bf16<EPL>(row + lane * EPL, kv);
#pragma unroll
    for (int e = 0; e < EPL; ++e) c[e] = 0.f;
    for (int h = g * ratio + w; h < (g + 1) * ratio; h += kWarpsPerBlock) {
      const int64_t r = (int64_t)h * sel.Sq + i;
      const float L = lse[r];
      if (L == -INFINITY) continue;
      float qv[EPL], dov[EPL];
      load_bf16<EPL>(q + row_off(st.q, 0, i, h) + lane * EPL, qv);
      load_bf16<EPL>(dO + row_off(st.dO, 0, i, h) + lane * EPL, dov);
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        s = fmaf(qv[e], kv[e], s);
        dp = fmaf(dov[e], kv[e], dp);
      }
      s = warp_sum(s) * scale;
      dp = warp_sum(dp);
      const float p = expf(s - L);
      const float sds = scale * p * (dp - delta[r]);
#pragma unroll
      for (int e = 0; e < EPL; ++e) c[e] = fmaf(sds, qv[e], fmaf(p, dov[e], c[e]));
    }
#pragma unroll
    for (int e = 0; e < EPL; ++e) red[w][lane * EPL + e] = c[e];
    __syncthreads();
    float* dst = (src == 0 ? d_ori : d_cmp) + ((int64_t)j * sel.Hk + g) * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
      float t = 0.f;
#pragma unroll
      for (int u = 0; u < kWarpsPerBlock; ++u) t += red[u][d];
      atomicAdd(dst + d, t);
    }
    __syncthreads();
  });
}

Strides strides_of(const Problem& p) {
  Strides s;
  for (int t = 0; t < 3; ++t) {
    s.q[t] = p.qs[t];
    s.k[t] = p.ks[t];
    s.v[t] = p.vs[t];
    s.o[t] = p.os[t];
    s.dO[t] = p.dos[t];
  }
  return s;
}

SparseSel sel_of(const Problem& p, const void* ori, const void* cmp, const int32_t* idx) {
  SparseSel s;
  s.ori = static_cast<const bf16*>(ori);
  s.cmp = static_cast<const bf16*>(cmp);
  s.idx = idx;
  s.Sq = p.Sq;
  s.Hk = p.Hk;
  s.D = p.D;
  s.n_ori = p.n_ori;
  s.n_cmp = p.n_cmp;
  s.topk = p.topk;
  s.wl = p.ori_wl;
  s.wr = p.ori_wr;
  s.ratio = p.cmp_ratio;
  return s;
}

inline unsigned blocks_for_warps(int64_t warps) {
  return (unsigned)((warps + kWarpsPerBlock - 1) / kWarpsPerBlock);
}

template <int D>
cudaError_t fwd_impl(const Problem& p, const void* q, const void* k, const void* v,
                     const float* bias, const void* ori, const void* cmp, const int32_t* idx,
                     void* o, float* lse, DevStatus* status, cudaStream_t stream) {
  const Strides st = strides_of(p);
  const dim3 block(kWarpsPerBlock * 32);
  if (p.sparse) {
    const int64_t warps = (int64_t)p.Sq * p.Hq;
    if (warps == 0) return cudaSuccess;
    fwd_sparse_kernel<D><<<blocks_for_warps(warps), block, 0, stream>>>(
        p.Hq, p.scale, st, sel_of(p, ori, cmp, idx), static_cast<const bf16*>(q),
        static_cast<bf16*>(o), lse, status);
  } else {
    const int64_t warps = (int64_t)p.B * p.Hq * p.Sq;
    if (warps == 0) return cudaSuccess;
    fwd_dense_kernel<D><<<blocks_for_warps(warps), block, 0, stream>>>(
        p.B, p.Hq, p.Hk, p.Sq, p.Sk, p.scale, p.mask, st, static_cast<const bf16*>(q),
        static_cast<const bf16*>(k), static_cast<const bf16*>(v), bias,
        static_cast<bf16*>(o), lse);
  }
  return cudaGetLastError();
}

template <int D>
cudaError_t bwd_impl(const Problem& p, const void* q, const void* k, const void* v,
                     const void* dO, const float* lse, const float* delta, const float* bias,
                     float* dq, float* dk, float* dv, float* dbias, const void* ori,
                     const void* cmp, const int32_t* idx, float* d_ori, float* d_cmp,
                     DevStatus* status, cudaStream_t stream) {
  const Strides st = strides_of(p);
  const dim3 block(kWarpsPerBlock * 32);
  const bf16* qb = static_cast<const bf16*>(q);
  const bf16* dob = static_cast<const bf16*>(dO);
  if (p.sparse) {
    const SparseSel sel = sel_of(p, ori, cmp, idx);
    const int64_t warps = (int64_t)p.Sq * p.Hq;
    if (warps == 0) return cudaSuccess;
    bwd_sparse_dq_kernel<D><<<blocks_for_warps(warps), block, 0, stream>>>(
        p.Hq, p.scale, st, sel, qb, dob, lse, delta, dq, status);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_sparse_dkv_kernel<D><<<(unsigned)((int64_t)p.Sq * p.Hk), block, 0, stream>>>(
        p.Hq, p.scale, st, sel, qb, dob, lse, delta, d_ori, d_cmp, status);
    return cudaGetLastError();
  }
  const bf16* kb = static_cast<const bf16*>(k);
  const bf16* vb = static_cast<const bf16*>(v);
  const int64_t qwarps = (int64_t)p.B * p.Hq * p.Sq;
  if (qwarps > 0) {
    bwd_dq_kernel<D><<<blocks_for_warps(qwarps), block, 0, stream>>>(
        p.B, p.Hq, p.Hk, p.Sq, p.Sk, p.scale, p.mask, st, qb, kb, vb, dob, lse, delta, bias,
        dq, dbias, p.dbias_bstride);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t kwarps = (int64_t)p.B * p.Hk * p.Sk;
  if (kwarps > 0) {
    bwd_dkdv_kernel<D><<<blocks_for_warps(kwarps), block, 0, stream>>>(
        p.B, p.Hq, p.Hk, p.Sq, p.Sk, p.scale, p.mask, st, qb, kb, vb, dob, lse, delta, bias,
        dk, dv);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

}  // namespace

cudaError_t launch_fwd_simt(const Problem& p, const void* q, const void* k, const void* v,
                            const float* bias, const void* ori_kv, const void* cmp_kv,
                            const int32_t* cmp_idx, void* o, float* lse, DevStatus* st,
                            cudaStream_t stream) {
  switch (p.D) {
    case 64: return fwd_impl<64>(p, q, k, v, bias, ori_kv, cmp_kv, cmp_idx, o, lse, st, stream);
    case 128: return fwd_impl<128>(p, q, k, v, bias, ori_kv, cmp_kv, cmp_idx, o, lse, st, stream);
    case 512: return fwd_impl<512>(p, q, k, v, bias, ori_kv, cmp_kv, cmp_idx, o, lse, st, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bwd_simt(const Problem& p, const void* q, const void* k, const void* v,
                            const void* dO, const float* lse, const float* delta,
                            const float* bias, float* dq, float* dk, float* dv, float* dbias,
                            const void* ori_kv, const void* cmp_kv, const int32_t* cmp_idx,
                            float* d_ori, float* d_cmp, DevStatus* st, cudaStream_t stream) {
  switch (p.D) {
    case 64:
      return bwd_impl<64>(p, q, k, v, dO, lse, delta, bias, dq, dk, dv, dbias, ori_kv, cmp_kv,
                          cmp_idx, d_ori, d_cmp, st, stream);
    case 128:
      return bwd_impl<128>(p, q, k, v, dO, lse, delta, bias, dq, dk, dv, dbias, ori_kv, cmp_kv,
                           cmp_idx, d_ori, d_cmp, st, stream);
    case 512:
      return bwd_impl<512>(p, q, k, v, dO, lse, delta, bias, dq, dk, dv, dbias, ori_kv, cmp_kv,
                           cmp_idx, d_ori, d_cmp, st, stream);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace attn
