// Backward pre-pass: one fused, HBM-streaming kernel.
//
// D = rowsum(dO * O) ("34_bwd_gqa_fmha.py" cpu_bwd_gqa; Ascend
// "sparse_flash_mla_grad" phase 2, SoftmaxGrad(dO, O)), computed in fp32 from
// the bf16 rows. The same pass zeroes dbias / the sparse dKV buffers that the
// backward accumulates into, clears the status record, and
// for the tensor-core path writes fp16 head-major copies of q, k, v and dO
// (dense) or one fp16 copy of the original and compressed KV rows (sparse).
//
// Why fp16 copies: the tensor-core backward feeds kind::f16 MMAs, and rounds
// P and dS to fp16 (11 significant bits) instead of bf16 (8), which keeps the
// rounding of the gradient operands well inside the parity tolerance; the
// other operand of each of those MMAs must then be fp16 as well. bf16 -> fp16
// is exact for every bf16 value of magnitude in [2^-14, 65504]; larger ones
// set a range flag that attn_bwd turns into ATTN_ERR_RANGE, smaller ones lose
// low bits (absolute error below 2^-25).
//
// Layout of the work: a row of D elements is split into 16-byte chunks of 8
// values; LPR = min(D / 8, 32) lanes cover a row, so a warp streams
// 32 / LPR rows at once with 16-byte loads and stores; a grid-stride loop
// keeps every SM's memory pipe full. Rows are visited in blocks of 8 per head
// (see decompose) so that both the reads and the head-major writes stream.

#include "internal.h"
#include "tc_ptx.cuh"

namespace attn {
namespace {

using bf16 = __nv_bfloat16;
constexpr int kThreads = 256;
// Resident blocks per SM (32 warps) for the HBM latency.
constexpr int kPreBlocksPerSM = 4;

struct PreParams {
  int B, Hq, Hk, Sq, Sk;
  int Sqs, Sks;  // rows per head of the fp16 copies (tile-rounded; zero past Sq / Sk)
  // variable-length batch: sequence bounds (nullptr: fixed lengths Sq, Sk)
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k;
  int64_t o0, o1, o2, d0, d1, d2, q0, q1, q2, k0, k1, k2, v0, v1, v2;
  const bf16* o;
  const bf16* dO;
  const bf16* q;
  const bf16* k;
  const bf16* v;
  float* delta;
  __half* q16;
  __half* k16;
  __half* v16;
  __half* do16;  // nullptr: no staging (SIMT path)
  const bf16* ori;  // sparse shared KV: fp16 copy [ori rows ; cmp rows] into kv16
  const bf16* cmp;
  int64_t kv_ori_rows, kv_cmp_rows;
  __half* kv16;     // nullptr: no KV staging
  float* zero_a;
  int64_t zero_na;
  float* zero_b;
  int64_t zero_nb;
  float* zero_c;
  int64_t zero_nc;
  float* zero_d;
  int64_t zero_nd;
  float* zero_e;
  int64_t zero_ne;
  float* dk;  // recorded for the backward's check
  float* dv;
  DevStatus* st;
};

__device__ __forceinline__ uint4 load_raw(const bf16* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ void unpack8(const uint4& raw, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float2 x = __bfloat1622float2(h[t]);
    f[2 * t] = x.x;
    f[2 * t + 1] = x.y;
  }
}

// fp16 copy of 8 values; returns their largest magnitude (the caller checks
// the fp16 range once at the end).
__device__ __forceinline__ float store8_half(__half* p, const float* f) {
  uint4 raw;
  __half2* h = reinterpret_cast<__half2*>(&raw);
  float m = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    h[t] = __floats2half2_rn(f[2 * t], f[2 * t + 1]);
    m = fmaxf(m, fmaxf(fabsf(f[2 * t]), fabsf(f[2 * t + 1])));
  }
  *reinterpret_cast<uint4*>(p) = raw;
  return m;
}

// Work order over (batch, block of kIB rows, head, row in block): a warp step
// covers rows of one head that are contiguous in the head-major fp16 copies
// (2 KiB runs at D = 128), and the heads of one row block together read a
// contiguous span of the [B, S, H, D] input.
constexpr int kIB = 8;

// 32-bit index math (the host rejects problems with 2^31 or more rows): a
// 64-bit division is a long software sequence on the GPU.
__device__ __forceinline__ void decompose(int64_t f64, int H, int S, int* b, int* h, int* i) {
  const uint32_t f = (uint32_t)f64;
  const uint32_t ii = f % kIB;
  const uint32_t g = f / kIB;
  *h = (int)(g % (uint32_t)H);
  const uint32_t blk = g / (uint32_t)H;
  const uint32_t nblk = (uint32_t)(S + kIB - 1) / kIB;
  *i = (int)((blk % nblk) * kIB + ii);
  *b = (int)(blk / nblk);
}

__device__ __forceinline__ void zero_range(float* a, int64_t n, int64_t tid, int64_t stride) {
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  float4* a4 = reinterpret_cast<float4*>(a);
  for (int64_t t = tid; t < n / 4; t += stride) a4[t] = z;
  for (int64_t t = (n / 4) * 4 + tid; t < n; t += stride) a[t] = 0.f;
}

template <int D>
__global__ void __launch_bounds__(kThreads, kPreBlocksPerSM)
preprocess_kernel(const PreParams p) {
  constexpr int CH = D / 8;                 // 16-byte chunks per row
  constexpr int LPR = CH < 32 ? CH : 32;    // lanes per row
  constexpr int CPL = CH / LPR;             // chunks per lane
  constexpr int RPW = 32 / LPR;             // rows per warp step
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR;               // row slot within the warp
  const int cl = lane % LPR;                // lane within the row
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;

  // the backward launched after this kernel may start its set-up now; it waits
  // for this grid's completion before it reads anything written here
  ptx::grid_launch_dependents();
  if (tid == 0) {
    p.st->code = 0;
    p.st->detail = 0;
    p.st->reserved[1] = (int32_t)gridDim.x;  // number of flag slots written below
    uint64_t* rec = reinterpret_cast<uint64_t*>(&p.st->reserved[2]);
    rec[0] = reinterpret_cast<uint64_t>(p.dk);
    rec[1] = reinterpret_cast<uint64_t>(p.dv);
  }
  int range_bits = 0;

  // ---- query-side rows (b, i, h): delta, staging; key-side rows (k, v) ----
  // One loop over the steps of both kinds, so that each warp waits for about
  // one round of loads. A step covers RPW * U rows (a divisor of kIB, aligned)
  // of one head inside one block of kIB rows: the index split is done once per
  // step, and all of the step's loads are issued before any dependent work.
  constexpr int U = D >= 512 ? 1 : 2;  // D = 512 rows are 1 KiB: one slot keeps registers in budget
  static_assert(kIB % (RPW * U) == 0, "a warp step stays inside one row block");
  float amax_q = 0.f, amax_do = 0.f, amax_k = 0.f, amax_v = 0.f;
  // query rows visited: the staged rows per head when staging (their tail past
  // Sq is written as zeros), else the rows themselves
  const int sq_it = p.do16 != nullptr ? p.Sqs : p.Sq;
  const int64_t nq = (int64_t)p.B * ((sq_it + kIB - 1) / kIB) * kIB * p.Hq;
  const int64_t nk = (int64_t)p.B * ((p.Sks + kIB - 1) / kIB) * kIB * p.Hk;
  const int64_t nq_steps = nq / (RPW * U);
  const int64_t n_steps = nq_steps + (p.do16 != nullptr ? 2 * nk / (RPW * U) : 0);
  for (int64_t step = warp0; step < n_steps; step += nwarps) {
    if (step < nq_steps) {
      const int64_t r0 = step * RPW * U;
      int h, i0, b;
      decompose(r0, p.Hq, sq_it, &b, &h, &i0);
      // rows of this sequence: [0, len) at token offsets tok + i (varlen) or
      // batch offsets b * stride[0]
      int tok = 0, len = p.Sq;
      if (p.cu_q != nullptr) seq_span(p.cu_q, b, p.total_q, p.Sq, &tok, &len);
      const bf16* ob = p.o + (p.cu_q ? tok * p.o1 : b * p.o0) + h * p.o2;
      const bf16* dob = p.dO + (p.cu_q ? tok * p.d1 : b * p.d0) + h * p.d2;
      const bf16* qb = p.q + (p.cu_q ? tok * p.q1 : b * p.q0) + h * p.q2;
      const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
      uint4 of[U][CPL], df[U][CPL], qf[U][CPL];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * RPW + sub;
#pragma unroll
        for (int c = 0; c < CPL; ++c) of[u][c] = df[u][c] = qf[u][c] = z4;
        if (i < len) {
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const int e0 = (cl + c * LPR) * 8;
            of[u][c] = load_raw(ob + i * p.o1 + e0);
            df[u][c] = load_raw(dob + i * p.d1 + e0);
            if (p.do16 != nullptr) qf[u][c] = load_raw(qb + i * p.q1 + e0);
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * RPW + sub;
        const bool valid = i < len;
        float s = 0.f;
        if (i < sq_it) {  // a real row, or a zero row of the staged tail
          const int64_t hm = ((int64_t)b * p.Hq + h) * sq_it + i;  // head-major row
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const int e0 = (cl + c * LPR) * 8;
            float ov[8], dv[8];
            unpack8(of[u][c], ov);
            unpack8(df[u][c], dv);
#pragma unroll
            for (int t = 0; t < 8; ++t) s = fmaf(ov[t], dv[t], s);
            if (p.do16 != nullptr) {
              float qv[8];
              unpack8(qf[u][c], qv);
              amax_do = fmaxf(amax_do, store8_half(p.do16 + hm * D + e0, dv));
              amax_q = fmaxf(amax_q, store8_half(p.q16 + hm * D + e0, qv));
            }
          }
        }
#pragma unroll
        for (int o = LPR / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (valid && cl == 0) p.delta[((int64_t)b * p.Hq + h) * p.Sq + i] = s;
      }
    } else {
      // nk is a multiple of kIB, so a step never straddles the k / v boundary
      const int64_t r0 = (step - nq_steps) * RPW * U;
      const bool is_v = r0 >= nk;
      int g, j0, b;
      decompose(is_v ? r0 - nk : r0, p.Hk, p.Sks, &b, &g, &j0);
      int tok = 0, len = p.Sk;
      if (p.cu_k != nullptr) seq_span(p.cu_k, b, p.total_k, p.Sk, &tok, &len);
      const int64_t s1 = is_v ? p.v1 : p.k1;
      const int64_t bo = p.cu_k ? tok * s1 : b * (is_v ? p.v0 : p.k0);
      const bf16* src0 = (is_v ? p.v + p.v2 * g : p.k + p.k2 * g) + bo;
      __half* dst0 = (is_v ? p.v16 : p.k16) + (((int64_t)b * p.Hk + g) * p.Sks) * D;
      uint4 f[U][CPL];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * RPW + sub;
#pragma unroll
        for (int c = 0; c < CPL; ++c) f[u][c] = make_uint4(0u, 0u, 0u, 0u);
        if (j < len) {
#pragma unroll
          for (int c = 0; c < CPL; ++c) f[u][c] = load_raw(src0 + j * s1 + (cl + c * LPR) * 8);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int j = j0 + u * RPW + sub;
        if (j >= p.Sks) continue;  // rows in [len, Sks) are written as zeros
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          float x[8];
          unpack8(f[u][c], x);
          const float m = store8_half(dst0 + (int64_t)j * D + (cl + c * LPR) * 8, x);
          if (is_v) amax_v = fmaxf(amax_v, m); else amax_k = fmaxf(amax_k, m);
        }
      }
    }
  }
  // ---- sparse shared KV rows, staged as one fp16 [ori ; cmp] matrix ----
  if (p.kv16 != nullptr) {
    const int64_t nkv = p.kv_ori_rows + p.kv_cmp_rows;
    for (int64_t r0 = warp0 * RPW * U; r0 < nkv; r0 += nwarps * RPW * U) {
      uint4 f[U][CPL];
      int64_t rows[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        rows[u] = r0 + u * RPW + sub;
        if (rows[u] < nkv) {
          const bf16* src = rows[u] < p.kv_ori_rows ? p.ori + rows[u] * D
                                                    : p.cmp + (rows[u] - p.kv_ori_rows) * D;
#pragma unroll
          for (int c = 0; c < CPL; ++c) f[u][c] = load_raw(src + (cl + c * LPR) * 8);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (rows[u] >= nkv) continue;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          float x[8];
          unpack8(f[u][c], x);
          amax_k = fmaxf(amax_k, store8_half(p.kv16 + rows[u] * D + (cl + c * LPR) * 8, x));
        }
      }
    }
  }

  // a bf16 value overflows fp16 exactly when its magnitude is at least 65520
  range_bits |= (amax_q >= 65520.f ? 1 : 0) | (amax_k >= 65520.f ? 2 : 0) |
                (amax_v >= 65520.f ? 4 : 0) | (amax_do >= 65520.f ? 8 : 0);

  // ---- buffers accumulated with atomics: dbias, sparse dKV ----
  zero_range(p.zero_a, p.zero_na, tid, nthreads);
  zero_range(p.zero_b, p.zero_nb, tid, nthreads);
  zero_range(p.zero_c, p.zero_nc, tid, nthreads);
  zero_range(p.zero_d, p.zero_nd, tid, nthreads);
  zero_range(p.zero_e, p.zero_ne, tid, nthreads);

  // Range overflow is handed to attn_bwd through this block's flag slot: a
  // report straight into the status record could race with the reset above.
  __shared__ int block_bits;
  if (threadIdx.x == 0) block_bits = 0;
  __syncthreads();
  if (range_bits) atomicOr(&block_bits, range_bits);
  __syncthreads();
  if (threadIdx.x == 0) reinterpret_cast<int32_t*>(p.st + 1)[blockIdx.x] = block_bits;
}

// Sink-logit gradient: one CTA per query head; each thread sums its strided
// share of the (batch, query) rows in double, then a fixed tree over the
// block, so the result does not depend on scheduling.
constexpr int kSinkThreads = 256;
__global__ void __launch_bounds__(kSinkThreads)
dsinks_kernel(int B, int Hq, int Sq, const float* __restrict__ sinks,
              const float* __restrict__ lse, const float* __restrict__ delta,
              float* __restrict__ dsinks) {
  const int h = blockIdx.x;
  const float s = sinks[h];
  const int64_t n = (int64_t)B * Sq;
  double acc = 0.0;
  for (int64_t r = threadIdx.x; r < n; r += kSinkThreads) {
    const int64_t b = r / Sq, i = r % Sq;
    const int64_t row = (b * Hq + h) * Sq + i;
    const float L = lse[row];
    if (L != -INFINITY) acc -= (double)expf(s - L) * (double)delta[row];
  }
  __shared__ double part[kSinkThreads];
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int w = kSinkThreads / 2; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) dsinks[h] = (float)part[0];
}

// Deterministic sum of per-batch slices: each thread adds its elements over
// the slices in slice order (4 at a time when the slices are 16-byte apart).
__global__ void __launch_bounds__(256)
sum_slices_kernel(const float* __restrict__ slices, int n, int64_t stride,
                  float* __restrict__ out) {
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if ((stride & 3) == 0) {
    for (int64_t e = t0; e < stride / 4; e += step) {
      float4 acc = reinterpret_cast<const float4*>(slices)[e];
      for (int b = 1; b < n; ++b) {
        const float4 v = reinterpret_cast<const float4*>(slices + b * stride)[e];
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
      reinterpret_cast<float4*>(out)[e] = acc;
    }
  } else {
    for (int64_t e = t0; e < stride; e += step) {
      float acc = slices[e];
      for (int b = 1; b < n; ++b) acc += slices[b * stride + e];
      out[e] = acc;
    }
  }
}

}  // namespace

cudaError_t launch_sum_slices(const float* slices, int n, int64_t stride, float* out,
                              cudaStream_t stream) {
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  sum_slices_kernel<<<sms * 8, 256, 0, stream>>>(slices, n, stride, out);
  return cudaGetLastError();
}

cudaError_t launch_dsinks(int B, int Hq, int Sq, const float* sinks, const float* lse,
                          const float* delta, float* dsinks, cudaStream_t stream) {
  dsinks_kernel<<<Hq, kSinkThreads, 0, stream>>>(B, Hq, Sq, sinks, lse, delta, dsinks);
  return cudaGetLastError();
}

cudaError_t launch_preprocess(const Problem& pr, const void* q, const void* k, const void* v,
                              const void* o, const void* dO, float* delta,
                              float* dbias, float* d_ori, float* d_cmp, __half* q16, __half* k16,
                              __half* v16, __half* do16, const void* ori_kv, const void* cmp_kv,
                              __half* kv16, float* dk_zero, float* dv_zero, float* dk,
                              float* dv, DevStatus* st, cudaStream_t stream) {
  PreParams p;
  p.B = pr.B;
  p.Hq = pr.Hq;
  p.Hk = pr.Hk;
  p.Sq = pr.Sq;
  p.Sk = pr.Sk;
  p.Sqs = do16 != nullptr ? tc_rows(pr.Sq) : pr.Sq;
  p.Sks = do16 != nullptr ? tc_rows(pr.Sk) : pr.Sk;
  p.cu_q = pr.varlen ? pr.cu_q : nullptr;
  p.cu_k = pr.varlen ? pr.cu_k : nullptr;
  p.total_q = pr.total_q;
  p.total_k = pr.total_k;
  p.o0 = pr.os[0]; p.o1 = pr.os[1]; p.o2 = pr.os[2];
  p.d0 = pr.dos[0]; p.d1 = pr.dos[1]; p.d2 = pr.dos[2];
  p.q0 = pr.qs[0]; p.q1 = pr.qs[1]; p.q2 = pr.qs[2];
  p.k0 = pr.ks[0]; p.k1 = pr.ks[1]; p.k2 = pr.ks[2];
  p.v0 = pr.vs[0]; p.v1 = pr.vs[1]; p.v2 = pr.vs[2];
  p.o = static_cast<const bf16*>(o);
  p.dO = static_cast<const bf16*>(dO);
  p.q = static_cast<const bf16*>(q);
  p.k = static_cast<const bf16*>(k);
  p.v = static_cast<const bf16*>(v);
  p.delta = delta;
  p.q16 = q16;
  p.k16 = k16;
  p.v16 = v16;
  p.do16 = do16;
  p.ori = static_cast<const bf16*>(ori_kv);
  p.cmp = static_cast<const bf16*>(cmp_kv);
  p.kv_ori_rows = kv16 ? (int64_t)pr.n_ori * pr.Hk : 0;
  p.kv_cmp_rows = kv16 && cmp_kv ? (int64_t)pr.n_cmp * pr.Hk : 0;
  p.kv16 = kv16;
  p.zero_a = dbias;
  p.zero_na = dbias ? (pr.dbias_bstride > 0 ? pr.B * pr.dbias_bstride
                                             : (int64_t)pr.Hq * pr.Sq * pr.Sk)
                    : 0;
  p.zero_b = d_ori;
  p.zero_nb = d_ori ? (int64_t)pr.n_ori * pr.Hk * pr.D : 0;
  p.zero_c = d_cmp;
  p.zero_nc = d_cmp ? (int64_t)pr.n_cmp * pr.Hk * pr.D : 0;
  const int64_t nkd = (pr.varlen ? (int64_t)pr.total_k : (int64_t)pr.B * pr.Sk) * pr.Hk * pr.D;
  p.zero_d = dk_zero;
  p.zero_nd = dk_zero ? nkd : 0;
  p.zero_e = dv_zero;
  p.zero_ne = dv_zero ? nkd : 0;
  p.dk = dk;
  p.dv = dv;
  p.st = st;
  // Enough resident warps to keep HBM busy; the loops stride over the rest.
  int dev = 0, sms = 152;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int want = sms * kPreBlocksPerSM;
  const unsigned grid = (unsigned)(want < kPreMaxBlocks ? want : kPreMaxBlocks);
  switch (pr.D) {
    case 64: preprocess_kernel<64><<<grid, kThreads, 0, stream>>>(p); break;
    case 128: preprocess_kernel<128><<<grid, kThreads, 0, stream>>>(p); break;
    case 512: preprocess_kernel<512><<<grid, kThreads, 0, stream>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace attn
