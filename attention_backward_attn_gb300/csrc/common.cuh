// Internal helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "attn_bwd.h"
#include "mask.h"

namespace attn {

// Status record at the start of every workspace. Kernels record the first
// device-side condition; attn_read_device_status copies it back.
struct DevStatus {
  int32_t code;
  int32_t detail;
  int32_t reserved[62];
};
static_assert(sizeof(DevStatus) == 256, "status record is 256 bytes");

// Per-block flag slots of the pre-pass follow the status record: every block
// of the pre-pass writes its slot on every call (so stale or uninitialised
// workspace contents never leak into a report); the backward ORs them.
constexpr int kPreMaxBlocks = 2048;
constexpr size_t kStatusBytes = sizeof(DevStatus) + kPreMaxBlocks * sizeof(int32_t);

__device__ __forceinline__ void report(DevStatus* st, int32_t code, int32_t detail) {
  if (st == nullptr) return;
  if (atomicCAS(&st->code, 0, code) == 0) {
    atomicExch(&st->detail, detail);
  }
}

// Rows [*start, *start + *len) of sequence b of a variable-length batch
// (cumulative lengths cu); false (and an empty span) when the bounds are out
// of order, past `total` rows, or longer than max_len.
__device__ __forceinline__ bool seq_span(const int32_t* cu, int b, int total, int max_len,
                                         int* start, int* len) {
  const int a = cu[b], e = cu[b + 1];
  if (a < 0 || e < a || e > total || e - a > max_len) {
    *start = 0;
    *len = 0;
    return false;
  }
  *start = a;
  *len = e - a;
  return true;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Load EPL consecutive bf16 values (EPL in {2, 4, 8, 16}) as floats.
template <int EPL>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16* p, float* out) {
  if constexpr (EPL == 2) {
    __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(p);
    float2 f = __bfloat1622float2(v);
    out[0] = f.x; out[1] = f.y;
  } else if constexpr (EPL == 4) {
    uint2 raw = *reinterpret_cast<const uint2*>(p);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      float2 f = __bfloat1622float2(h[t]);
      out[2 * t] = f.x; out[2 * t + 1] = f.y;
    }
  } else {
    static_assert(EPL % 8 == 0, "EPL must be 2, 4 or a multiple of 8");
#pragma unroll
    for (int c = 0; c < EPL / 8; ++c) {
      uint4 raw = *reinterpret_cast<const uint4*>(p + 8 * c);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        float2 f = __bfloat1622float2(h[t]);
        out[8 * c + 2 * t] = f.x; out[8 * c + 2 * t + 1] = f.y;
      }
    }
  }
}

template <int EPL>
__device__ __forceinline__ void store_bf16(__nv_bfloat16* p, const float* in) {
#pragma unroll
  for (int t = 0; t < EPL; t += 2) {
    *reinterpret_cast<__nv_bfloat162*>(p + t) = __floats2bfloat162_rn(in[t], in[t + 1]);
  }
}

template <int EPL>
__device__ __forceinline__ void store_f32(float* p, const float* in) {
  if constexpr (EPL % 4 == 0) {
#pragma unroll
    for (int t = 0; t < EPL; t += 4)
      *reinterpret_cast<float4*>(p + t) = make_float4(in[t], in[t + 1], in[t + 2], in[t + 3]);
  } else {
#pragma unroll
    for (int t = 0; t < EPL; t += 2)
      *reinterpret_cast<float2*>(p + t) = make_float2(in[t], in[t + 1]);
  }
}

// Host-side view of a launch: validated problem plus derived values.
struct Problem {
  int B, Hq, Hk, Sq, Sk, D;
  float scale;
  int64_t qs[3], ks[3], vs[3], os[3], dos[3];
  MaskSpec mask;
  bool sparse;
  bool deterministic;  // ATTN_FLAG_DETERMINISTIC
  bool cuda_cores;     // ATTN_FLAG_CUDA_CORES
  // variable-length batch: per-sequence bounds on the device (Sq, Sk are
  // upper bounds); the mask is then top-left and br asks for bottom-right
  // alignment per sequence
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k;
  bool varlen, br;
  // > 0: dbias is accumulated into per-batch slices this many floats apart
  // (deterministic mode, B > 1), summed in batch order afterwards
  int64_t dbias_bstride;
  // sparse fields (cmp_ratio > 0 only in the CFA case: no index list, every
  // compressed row whose block ends at or before the query is selected)
  int n_ori, n_cmp, topk, ori_wl, ori_wr, cmp_ratio;
};

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace attn
