// Internal helpers shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "attn_bwd.h"

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

// live(i, j) = j < sink || (i - wl <= j <= i + wr); negative bound = unbounded
// ("22_sink_tokens_fmha.py" mask builders, top-left aligned).
// Key mask over (query i, key j): live when j < sink or -wl <= j - i <= wr.
// The bounds are relative to the diagonal j = i; kMaskUnbounded leaves that
// side open. They may be negative: a bottom-right aligned mask is a top-left
// one with both bounds shifted by Sk - Sq. Bounds are clamped to
// [-kMaskMaxBound, kMaskMaxBound] and lengths to kMaxMaskedLen, so i +- bound
// stays inside int.
constexpr int kMaskUnbounded = 1 << 29;
constexpr int kMaskMaxBound = 1 << 28;
constexpr int kMaxMaskedLen = 1 << 28;
struct MaskSpec {
  int wl;
  int wr;
  int sink;
};

__host__ __device__ __forceinline__ bool mask_live(const MaskSpec& m, int i, int j) {
  if (j < m.sink) return true;
  return j >= i - m.wl && j <= i + m.wr;
}

// Non-sink key range [lo, hi] (inclusive, clipped to [0, n); empty when
// lo > hi) live for row i.
__host__ __device__ __forceinline__ void mask_row_range(const MaskSpec& m, int i, int n,
                                                        int* lo, int* hi) {
  const int a = i - m.wl, b = i + m.wr;
  *lo = a < 0 ? 0 : a;
  *hi = b > n - 1 ? n - 1 : b;
}

// Non-sink query range [lo, hi] live for key j (j >= sink), clipped to [0, n).
__host__ __device__ __forceinline__ void mask_col_range(const MaskSpec& m, int j, int n,
                                                        int* lo, int* hi) {
  const int a = j - m.wr, b = j + m.wl;
  *lo = a < 0 ? 0 : a;
  *hi = b > n - 1 ? n - 1 : b;
}

// Tile classification over rows [m0, m1) x keys [n0, n1) for the same mask:
// tile_any = at least one live entry, tile_full = every entry live.
__host__ __device__ __forceinline__ bool tile_any(const MaskSpec& m, int m0, int m1, int n0,
                                                  int n1) {
  if (m0 >= m1 || n0 >= n1) return false;
  if (n0 < m.sink) return true;
  const int dmax = (n1 - 1) - m0;  // largest j - i in the tile
  const int dmin = n0 - (m1 - 1);  // smallest j - i in the tile
  return dmax >= -m.wl && dmin <= m.wr;
}

__host__ __device__ __forceinline__ bool tile_full(const MaskSpec& m, int m0, int m1, int n0,
                                                   int n1) {
  const int a = n0 > m.sink ? n0 : m.sink;  // first column not covered by the sinks
  if (a >= n1) return true;
  const int dmax = (n1 - 1) - m0;
  const int dmin = a - (m1 - 1);
  return dmin >= -m.wl && dmax <= m.wr;
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
  // sparse fields (cmp_ratio > 0 only in the CFA case: no index list, every
  // compressed row whose block ends at or before the query is selected)
  int n_ori, n_cmp, topk, ori_wl, ori_wr, cmp_ratio;
};

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace attn
