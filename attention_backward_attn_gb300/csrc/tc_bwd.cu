// Tensor-core (tcgen05 / TMEM / TMA) fused attention backward for sm_103a.
//
// Math (composable_kernel "34_bwd_gqa_fmha.py" docstring and cpu_bwd_gqa,
// "28_backward_dbias_fmha.py" cpu_attention_bwd_dbias):
//   P = exp(scale Q K^T + bias - LSE) on live entries, D = rowsum(dO * O),
//   dP = dO V^T, dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q,
//   dV = P^T dO, dK / dV summed over the query heads of a KV head,
//   dbias = sum over the batch of dS.
//
// Tiling: one CTA owns a 128-row key tile of one (batch, KV head) and loops
// over every query head of the group and every 128-row query tile that has a
// live entry (fully masked tiles are skipped, partial ones get the per-element
// mask). Per tile pair, in a key-major ("transposed") formulation so that the
// softmax warps own one key row each:
//   MMA1  S^T  = K  Q^T      (M = 128 keys,    N = 128 queries, K = D)
//   MMA2  dP^T = V  dO^T     (M = 128 keys,    N = 128 queries, K = D)
//   SFU   P^T = exp2(S^T * scale*log2e + bias*log2e - LSE*log2e),
//         dS^T = P^T (dP^T - D)           -> P^T fp16 into TMEM, dS^T fp16 into SMEM
//   MMA3  dV  += P^T  dO     (A = P^T from TMEM, B = dO  MN-major)
//   MMA4  dK  += dS^T Q      (A = dS^T K-major,  B = Q   MN-major)
//   MMA5  dQ_t = dS   K      (A = dS^T read MN-major, B = K MN-major)
// dK / dV stay in TMEM for the whole group (the GQA reduction happens on
// chip); dQ_t is drained by a second warpgroup with fp32 vector atomics.
//
// TMEM (512 columns x 128 lanes x 32 bit): [0, D) dK, [D, 2D) dV,
// [2D, 2D+128) S^T (P^T fp16 packed into its first 64 columns),
// [2D+128, 2D+256) dP^T, reused for dQ_t once dS^T exists.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer (and TMEM
// owner), warps 4-7 softmax / dS, warps 8-11 dQ drain; warps 4-7 also write
// dK / dV at the end. Every mbarrier wait is bounded: after ~2 s a wait
// records ATTN_ERR_DEVICE_TIMEOUT, raises a CTA-wide abort flag, and the CTA
// drains its in-flight copies / MMAs, frees TMEM and exits.
//
// Operands are fp16 (exact copies of the bf16 inputs, staged by the
// pre-pass): with fp16 P and dS the rounding of the gradient GEMM operands
// has 3 more mantissa bits than bf16, and kind::f16 needs A and B of the same
// type.

#include "internal.h"
#include "tc_ptx.cuh"

#include <mutex>

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // key rows per CTA
constexpr int kThreads = 384;
constexpr int kSlab = 128 * 128;  // one [128 rows][64 fp16] 128B-swizzled slab, bytes
constexpr uint64_t kTimeoutNs = 2000000000ull;

template <int D>
struct Smem {
  static constexpr int kTile = (D / 64) * kSlab;  // a [128][D] fp16 operand tile
  static constexpr int K = 0;
  static constexpr int V = K + kTile;
  static constexpr int Q = V + kTile;        // 2 stages
  static constexpr int dO = Q + 2 * kTile;   // 2 stages
  static constexpr int dS = dO + 2 * kTile;  // [128 keys][128 queries] fp16, 2 slabs
  static constexpr int LSE = dS + 2 * kSlab; // 2 stages x 128 fp32
  static constexpr int DLT = LSE + 1024;     // 2 stages x 128 fp32
  static constexpr int BAR = DLT + 1024;     // mbarriers
  static constexpr int MISC = BAR + 128;     // TMEM base, abort flag
  static constexpr int TOTAL = MISC + 16;
};

enum Bar { kKvFull = 0, kQFull0 = 1, kQEmpty0 = 3, kSFull = 5, kPFull = 6, kDqFull = 7,
           kDqEmpty = 8, kAccFull = 9, kNumBars = 10 };

struct TcParams {
  int B, Hq, Hk, Sq, Sk;
  float scale;
  float scale_log2;
  MaskSpec mask;
  const float* lse;
  const float* delta;
  const float* bias;
  float* dq;
  float* dk;
  float* dv;
  float* dbias;
  DevStatus* status;
};

struct Ctx {
  uint32_t bars;       // shared address of barrier 0
  volatile int* abort; // CTA-wide abort flag
  DevStatus* status;
  __device__ uint32_t bar(int i) const { return bars + 8u * i; }
};

// Bounded mbarrier wait: true when the phase with `parity` completed; false
// if the CTA aborted or ~2 s passed (then the abort flag is raised).
__device__ __noinline__ bool wait_bar(const Ctx& c, int which, uint32_t parity, int where) {
  const uint32_t bar = c.bar(which);
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((n & 31u) == 0) {
      if (*c.abort) return false;
      if (ptx::globaltimer_ns() - t0 > kTimeoutNs) {
        *c.abort = 1;
        report(c.status, ATTN_ERR_DEVICE_TIMEOUT, where);
        return false;
      }
    }
  }
}

// Teardown wait: ignores the abort flag, still bounded.
__device__ __noinline__ void drain_bar(const Ctx& c, int which, uint32_t parity) {
  const uint32_t bar = c.bar(which);
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kTimeoutNs) {
      report(c.status, ATTN_ERR_DEVICE_TIMEOUT, 100 + which);
      return;
    }
  }
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Iterates the live (query head, query tile) pairs of this CTA's key tile.
struct TileIter {
  int r, nmt, n0, hl, mt;
  MaskSpec mask;
  __device__ TileIter(int r_, int nmt_, int n0_, MaskSpec m) : r(r_), nmt(nmt_), n0(n0_), hl(0), mt(-1), mask(m) {}
  __device__ bool next() {
    for (;;) {
      if (++mt >= nmt) {
        mt = 0;
        if (++hl >= r) return false;
      }
      if (tile_any(mask, mt * BM, mt * BM + BM, n0, n0 + BN)) return true;
    }
  }
};

template <int D, bool BIAS, bool DBIAS>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const TcParams p) {
  using L = Smem<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (sbase & 1023u) {  // the 128B-swizzle atoms need 1 KiB alignment
    if (threadIdx.x == 0) report(p.status, ATTN_ERR_UNSUPPORTED, 1);
    return;
  }
  const int nnt = p.Sk / BN;
  const int nt = blockIdx.x % nnt;
  const int g = (blockIdx.x / nnt) % p.Hk;
  const int b = blockIdx.x / (nnt * p.Hk);
  const int n0 = nt * BN;
  const int r = p.Hq / p.Hk;
  const int nmt = p.Sq / BM;

  Ctx c;
  c.bars = sbase + L::BAR;
  c.abort = reinterpret_cast<volatile int*>(smem + L::MISC + 4);
  c.status = p.status;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::MISC);

  if (threadIdx.x == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    ptx::prefetch_tmap(&tmdO);
    ptx::mbar_init(c.bar(kKvFull), 1);
    ptx::mbar_init(c.bar(kQFull0), 1);
    ptx::mbar_init(c.bar(kQFull0 + 1), 1);
    ptx::mbar_init(c.bar(kQEmpty0), 1);
    ptx::mbar_init(c.bar(kQEmpty0 + 1), 1);
    ptx::mbar_init(c.bar(kSFull), 1);
    ptx::mbar_init(c.bar(kPFull), 128);
    ptx::mbar_init(c.bar(kDqFull), 1);
    ptx::mbar_init(c.bar(kDqEmpty), 128);
    ptx::mbar_init(c.bar(kAccFull), 1);
    *c.abort = 0;
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + L::MISC, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  const uint32_t t_dK = tmem;
  const uint32_t t_dV = tmem + D;
  const uint32_t t_S = tmem + 2 * D;
  const uint32_t t_dP = tmem + 2 * D + 128;

  const uint32_t sK = sbase + L::K, sV = sbase + L::V, sDS = sbase + L::dS;
  int n_iters = 0;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      const int krow = (b * p.Hk + g) * p.Sk + n0;
      ptx::mbar_arrive_expect_tx(c.bar(kKvFull), 2 * L::kTile);
#pragma unroll
      for (int hf = 0; hf < D / 64; ++hf) {
        ptx::tma_load_2d(sK + hf * kSlab, &tmK, c.bar(kKvFull), hf * 64, krow);
        ptx::tma_load_2d(sV + hf * kSlab, &tmV, c.bar(kKvFull), hf * 64, krow);
      }
      TileIter it(r, nmt, n0, p.mask);
      int t = 0;
      int issued[2] = {0, 0};
      while (it.next()) {
        const int st = t & 1;
        const int use = t >> 1;
        if (use > 0 && !wait_bar(c, kQEmpty0 + st, (use - 1) & 1, 1)) break;
        const int h = g * r + it.hl;
        const int m0 = it.mt * BM;
        const int64_t row = ((int64_t)b * p.Hq + h) * p.Sq + m0;
        const uint32_t full = c.bar(kQFull0 + st);
        ptx::mbar_arrive_expect_tx(full, 2 * L::kTile + 2 * 512);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf) {
          ptx::tma_load_2d(sbase + L::Q + st * L::kTile + hf * kSlab, &tmQ, full, hf * 64, (int)row);
          ptx::tma_load_2d(sbase + L::dO + st * L::kTile + hf * kSlab, &tmdO, full, hf * 64, (int)row);
        }
        ptx::bulk_load(sbase + L::LSE + st * 512, p.lse + row, 512, full);
        ptx::bulk_load(sbase + L::DLT + st * 512, p.delta + row, 512, full);
        issued[st] = use + 1;
        ++t;
      }
      // make sure no copy is still landing in shared memory when the CTA ends
      drain_bar(c, kKvFull, 0);
      for (int st = 0; st < 2; ++st)
        if (issued[st] > 0) drain_bar(c, kQFull0 + st, (issued[st] - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t id_S = ptx::idesc_f16_f32(128, 128, false, false);
      constexpr uint32_t id_dKV = ptx::idesc_f16_f32(128, D, false, true);
      constexpr uint32_t id_dQ = ptx::idesc_f16_f32(128, D, true, true);
      bool ok = wait_bar(c, kKvFull, 0, 2);
      TileIter it(r, nmt, n0, p.mask);
      int t = 0;
      while (ok && it.next()) {
        const int st = t & 1;
        const uint32_t sQ = sbase + L::Q + st * L::kTile;
        const uint32_t sdO = sbase + L::dO + st * L::kTile;
        if (!wait_bar(c, kQFull0 + st, (t >> 1) & 1, 3)) break;
        if (t > 0 && !wait_bar(c, kDqEmpty, (t - 1) & 1, 4)) break;
        ptx::tc_fence_after();
        // MMA1 S^T = K Q^T and MMA2 dP^T = V dO^T (both operands K-major over d)
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kSlab + (s & 3) * 32;
          ptx::mma_ss(t_S, ptx::smem_desc_sw128(sK + off, 16, 1024),
                      ptx::smem_desc_sw128(sQ + off, 16, 1024), id_S, s > 0);
        }
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kSlab + (s & 3) * 32;
          ptx::mma_ss(t_dP, ptx::smem_desc_sw128(sV + off, 16, 1024),
                      ptx::smem_desc_sw128(sdO + off, 16, 1024), id_S, s > 0);
        }
        ptx::mma_commit(c.bar(kSFull));
        if (!wait_bar(c, kPFull, t & 1, 5)) break;
        ptx::tc_fence_after();
        // MMA3 dV += P^T dO : A = P^T (TMEM, fp16 pairs), B = dO MN-major over d
#pragma unroll
        for (int s = 0; s < BM / 16; ++s) {
          ptx::mma_ts(t_dV, t_S + s * 8, ptx::smem_desc_sw128(sdO + s * 2048, kSlab, 1024),
                      id_dKV, (t > 0 || s > 0) ? 1u : 0u);
        }
        // MMA4 dK += dS^T Q : A = dS^T K-major over queries, B = Q MN-major over d
#pragma unroll
        for (int s = 0; s < BM / 16; ++s) {
          const uint32_t off = (s >> 2) * kSlab + (s & 3) * 32;
          ptx::mma_ss(t_dK, ptx::smem_desc_sw128(sDS + off, 16, 1024),
                      ptx::smem_desc_sw128(sQ + s * 2048, kSlab, 1024), id_dKV,
                      (t > 0 || s > 0) ? 1u : 0u);
        }
        // MMA5 dQ_t = dS K : A = dS^T read MN-major over queries, B = K MN-major over d
#pragma unroll
        for (int s = 0; s < BN / 16; ++s) {
          ptx::mma_ss(t_dP, ptx::smem_desc_sw128(sDS + s * 2048, kSlab, 1024),
                      ptx::smem_desc_sw128(sK + s * 2048, kSlab, 1024), id_dQ, s > 0);
        }
        ptx::mma_commit(c.bar(kDqFull));
        ptx::mma_commit(c.bar(kQEmpty0 + st));
        ++t;
      }
      ptx::mma_commit(c.bar(kAccFull));
    }
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------- softmax / dS warpgroup --
    const int tw = threadIdx.x - 128;          // key row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp - 4) * 32) << 16;
    const int j = n0 + tw;
    TileIter it(r, nmt, n0, p.mask);
    int t = 0;
    bool ok = true;
    while (it.next()) {
      const int st = t & 1;
      if (!wait_bar(c, kQFull0 + st, (t >> 1) & 1, 6)) { ok = false; break; }
      // A row without live keys has LSE = -inf; it can only sit in a partial
      // tile, where the per-element mask below zeroes its probabilities.
      const float* lse_s = reinterpret_cast<const float*>(smem + L::LSE + st * 512);
      const float* dl_s = reinterpret_cast<const float*>(smem + L::DLT + st * 512);
      if (!wait_bar(c, kSFull, t & 1, 7)) { ok = false; break; }
      ptx::tc_fence_after();
      const int h = g * r + it.hl;
      const int m0 = it.mt * BM;
      const bool partial = !tile_full(p.mask, m0, m0 + BM, n0, n0 + BN);
      const float* brow = nullptr;
      if constexpr (BIAS) brow = p.bias + ((int64_t)h * p.Sq + m0) * p.Sk + j;
      float* dbrow = nullptr;
      if constexpr (DBIAS) dbrow = p.dbias + ((int64_t)h * p.Sq + m0) * p.Sk + j;
      const uint32_t ds_row = sDS + tw * 128;
#pragma unroll 1
      for (int cc = 0; cc < BM / 32; ++cc) {
        uint32_t sr[32], dr[32];
        ptx::tmem_ld32(t_S + lane_off + cc * 32, sr);
        ptx::tmem_ld32(t_dP + lane_off + cc * 32, dr);
        float bv[32];
        if constexpr (BIAS) {
#pragma unroll
          for (int e = 0; e < 32; ++e) bv[e] = __ldg(brow + (int64_t)(cc * 32 + e) * p.Sk);
        }
        ptx::tmem_wait_ld();
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float pe[2], de[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int il = cc * 32 + e + u;
            float x = fmaf(__uint_as_float(sr[e + u]), p.scale_log2, lse_s[il] * -kLog2e);
            if constexpr (BIAS) x = fmaf(bv[e + u], kLog2e, x);
            float pv = ptx::ex2(x);
            if (partial && !mask_live(p.mask, m0 + il, j)) pv = 0.f;
            pe[u] = pv;
            de[u] = pv * (__uint_as_float(dr[e + u]) - dl_s[il]);
            if constexpr (DBIAS) atomicAdd(dbrow + (int64_t)il * p.Sk, de[u]);
          }
          pk[e / 2] = pack_half2(pe[0], pe[1]);
          dk[e / 2] = pack_half2(de[0], de[1]);
        }
        // P^T fp16 into the (already read) front of the S^T columns
        ptx::tmem_st16(t_S + lane_off + cc * 16, pk);
        // dS^T fp16 into shared memory, 128B-swizzled K-major rows (one key row per thread)
        const uint32_t slab = ds_row + (cc >> 1) * kSlab;
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t chunk = (uint32_t)((cc & 1) * 4 + q4) ^ (uint32_t)(tw & 7);
          ptx::st_shared_v4(slab + chunk * 16, dk[4 * q4], dk[4 * q4 + 1], dk[4 * q4 + 2],
                            dk[4 * q4 + 3]);
        }
      }
      ptx::tmem_wait_st();
      ptx::fence_async_shared();
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar(kPFull));
      ++t;
    }
    n_iters = t;
    // ------------------------------------------------ dK / dV epilogue --
    if (ok && wait_bar(c, kAccFull, 0, 8)) {
      ptx::tc_fence_after();
      float* dkrow = p.dk + (((int64_t)b * p.Sk + j) * p.Hk + g) * D;
      float* dvrow = p.dv + (((int64_t)b * p.Sk + j) * p.Hk + g) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t kr[32], vr[32];
        if (n_iters > 0) {
          ptx::tmem_ld32(t_dK + lane_off + cc * 32, kr);
          ptx::tmem_ld32(t_dV + lane_off + cc * 32, vr);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) kr[e] = vr[e] = 0u;
        }
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          *reinterpret_cast<float4*>(dkrow + cc * 32 + e) =
              make_float4(__uint_as_float(kr[e]) * p.scale, __uint_as_float(kr[e + 1]) * p.scale,
                          __uint_as_float(kr[e + 2]) * p.scale, __uint_as_float(kr[e + 3]) * p.scale);
          *reinterpret_cast<float4*>(dvrow + cc * 32 + e) =
              make_float4(__uint_as_float(vr[e]), __uint_as_float(vr[e + 1]),
                          __uint_as_float(vr[e + 2]), __uint_as_float(vr[e + 3]));
        }
      }
    }
  } else if (warp >= 8) {
    // ---------------------------------------------------- dQ drain group --
    const int tq = threadIdx.x - 256;  // query row within the tile == TMEM lane
    const uint32_t lane_off = (uint32_t)((warp - 8) * 32) << 16;
    TileIter it(r, nmt, n0, p.mask);
    int t = 0;
    while (it.next()) {
      if (!wait_bar(c, kDqFull, t & 1, 9)) break;
      ptx::tc_fence_after();
      const int h = g * r + it.hl;
      const int i = it.mt * BM + tq;
      float* dst = p.dq + (((int64_t)b * p.Sq + i) * p.Hq + h) * D;
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        ptx::tmem_ld32(t_dP + lane_off + cc * 32, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          atomicAdd(reinterpret_cast<float4*>(dst + cc * 32 + e),
                    make_float4(__uint_as_float(v[e]) * p.scale, __uint_as_float(v[e + 1]) * p.scale,
                                __uint_as_float(v[e + 2]) * p.scale,
                                __uint_as_float(v[e + 3]) * p.scale));
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar(kDqEmpty));
      ++t;
    }
  }

  // ----------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (lane == 0) drain_bar(c, kAccFull, 0);  // every MMA of this CTA has completed
    __syncwarp();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------------ host --

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  });
  return fn;
}

// Row-major [rows][D] fp16 matrix, boxes of 128 rows x 64 columns, 128B swizzle.
bool make_map(CUtensorMap* m, const __half* base, uint64_t rows, int D) {
  EncodeFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * sizeof(__half)};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<__half*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool BIAS, bool DBIAS>
cudaError_t launch_variant(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                           const CUtensorMap& dO, const TcParams& p, int grid,
                           cudaStream_t stream) {
  auto kern = attn_bwd_tc_kernel<D, BIAS, DBIAS>;
  static bool configured = false;  // attribute set once per process and variant
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Smem<D>::TOTAL);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  kern<<<grid, kThreads, Smem<D>::TOTAL, stream>>>(q, k, v, dO, p);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                     const CUtensorMap& dO, const TcParams& p, int grid, cudaStream_t stream) {
  if (p.bias && p.dbias) return launch_variant<D, true, true>(q, k, v, dO, p, grid, stream);
  if (p.bias) return launch_variant<D, true, false>(q, k, v, dO, p, grid, stream);
  if (p.dbias) return launch_variant<D, false, true>(q, k, v, dO, p, grid, stream);
  return launch_variant<D, false, false>(q, k, v, dO, p, grid, stream);
}

}  // namespace

bool tc_supported(const Problem& p) {
  return !p.sparse && (p.D == 64 || p.D == 128) && p.B > 0 && p.Sq > 0 && p.Sk > 0 &&
         p.Sq % BM == 0 && p.Sk % BN == 0 && encode_fn() != nullptr;
}

cudaError_t launch_bwd_tc(const Problem& pr, const __half* q16, const __half* k16,
                          const __half* v16, const __half* do16, const float* lse,
                          const float* delta, const float* bias, float* dq, float* dk,
                          float* dv, float* dbias, DevStatus* st, cudaStream_t stream) {
  CUtensorMap mq, mk, mv, mdo;
  const uint64_t qrows = (uint64_t)pr.B * pr.Hq * pr.Sq;
  const uint64_t krows = (uint64_t)pr.B * pr.Hk * pr.Sk;
  if (!make_map(&mq, q16, qrows, pr.D) || !make_map(&mk, k16, krows, pr.D) ||
      !make_map(&mv, v16, krows, pr.D) || !make_map(&mdo, do16, qrows, pr.D))
    return cudaErrorInvalidValue;
  TcParams p;
  p.B = pr.B;
  p.Hq = pr.Hq;
  p.Hk = pr.Hk;
  p.Sq = pr.Sq;
  p.Sk = pr.Sk;
  p.scale = pr.scale;
  p.scale_log2 = pr.scale * kLog2e;
  p.mask = pr.mask;
  p.lse = lse;
  p.delta = delta;
  p.bias = bias;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.dbias = dbias;
  p.status = st;
  const int grid = pr.B * pr.Hk * (pr.Sk / BN);
  if (pr.D == 64) return launch_d<64>(mq, mk, mv, mdo, p, grid, stream);
  return launch_d<128>(mq, mk, mv, mdo, p, grid, stream);
}

}  // namespace attn
