// Tensor-core forward with log-sum-exp (the inputs O, LSE of the backward).
//
// O = softmax(scale Q K^T + bias, masked) V and LSE = natural log-sum-exp of
// the masked logits (CK "34_bwd_gqa_fmha.py" cpu_fwd_with_intermediates, CK
// "28_backward_dbias_fmha.py" cpu_attention_fwd_bias, CK
// "22_sink_tokens_fmha.py" masked CPU forward), for dense problems with
// D in {64, 128} whose q / k / v rows are packed over (batch, position).
//
// One CTA per (batch, query head, 128-row query tile), one pass over the
// live key tiles of the mask (online softmax): per tile S = Q K^T into one of
// two TMEM buffers; each of the two softmax warpgroups takes 64 keys of every
// row and keeps its own running maximum m, sum and O accumulator for them
// (O_wg += P(:, its keys) V(its keys, :) in TMEM), so the halves never wait
// for each other. The scale m of the accumulated terms moves only when a
// tile's maximum exceeds it by more than 2^8 (lazy rescaling: the row of
// O_wg and the sum are then scaled down once the previous P V has
// completed), so most tiles need no correction. At the end the halves meet
// once: O = (O_0 2^(m_0 - m) + O_1 2^(m_1 - m)) / sum and LSE = m + log2(sum)
// with m = max(m_0, m_1). Operands are the caller's bf16 rows, loaded by TMA
// through 3-D tensor maps (d, head, batch * position), K and V of a tile
// into stages released separately (K once S has read it, V once P V has);
// P is rounded to bf16 for its MMA (O is stored as bf16). On tiles the mask
// leaves whole and without bias the softmax works on the raw scores in the
// registers the TMEM load filled (the scale is folded into the exponent).
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 4-7 / 8-11 two softmax warpgroups (key columns 0-63 / 64-127
// of a tile; thread = query row), which also write O. Every mbarrier wait is
// bounded (the CTA gives up after ~2 s and exits; the forward has no status
// record to report into).

#include "internal.h"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

namespace attn {
namespace {

constexpr int kBM = 128;  // query rows per tile
constexpr int kBN = 128;  // key rows per tile
constexpr int kFwdThreads = 384;
constexpr int kFSlab = 128 * 128;  // [128 rows][64 bf16] 128B-swizzled slab, bytes

template <int D>
struct FwdSmem {
  static constexpr int kTile = (D / 64) * kFSlab;
  static constexpr int Q = 0;
  static constexpr int K = Q + kTile;         // 2 stages
  static constexpr int V = K + 2 * kTile;     // 2 stages
  static constexpr int STAT = V + 2 * kTile;  // [2 warpgroups][128 rows] (max, sum)
  static constexpr int BAR = STAT + 2 * 128 * 8;
  static constexpr int MISC = BAR + 256;      // TMEM base, abort flag
  static constexpr int TOTAL = MISC + 16;
};

// fQFull: Q landed. fKFull / fKEmpty, fVFull / fVEmpty: K and V of a step in
// stage 0 / 1 (K is read by S alone, so its stage frees once S completed; V
// by P V). fSFull: S of a step in TMEM buffer 0 / 1. fPFull: one warpgroup's half of P
// written over S (128 arrivals; [warpgroup][buffer]). fPvDone: both P V
// halves of a step completed (its buffer is free and both O accumulators hold
// its terms). fOFull: every MMA completed.
enum FwdBar { fQFull = 0, fKFull0 = 1, fVFull0 = 3, fKEmpty0 = 5, fVEmpty0 = 7, fSFull0 = 9,
              fPFull0 = 11, fPvDone0 = 15, fOFull = 17, kFwdBars = 18 };

struct FwdParams {
  int B, Hq, Hk, Sq, Sk;
  float scale_log2;
  MaskSpec mask;
  const float* bias;  // [Hq, Sq, Sk] or nullptr
  __nv_bfloat16* o;
  int64_t os0, os1, os2;
  float* lse;  // [B, Hq, Sq]
};

constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  // kind::f16 with A and B of type bf16 (format 1 in the A / B type fields)
  return ptx::idesc_f16_f32(M, N, a_mn, b_mn) | (1u << 7) | (1u << 10);
}

__device__ __forceinline__ uint32_t pack_bf162(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ int imin2(int a, int b) { return a < b ? a : b; }

// The k-th live key tile of a query tile (sink tiles, then the window range).
struct KeyTiles {
  int s_end, w_first, count;
  __device__ KeyTiles(const FwdParams& p, int m0) {
    int w_lo, w_hi;
    live_key_tiles(p.mask, p.Sq, p.Sk, kBM, kBN, m0, &s_end, &w_lo, &w_hi);
    w_first = w_lo > s_end ? w_lo : s_end;
    count = s_end + (w_hi >= w_first ? w_hi - w_first + 1 : 0);
  }
  __device__ int tile(int k) const { return k < s_end ? k : w_first + (k - s_end); }
};

template <int D, bool BIAS>
__global__ void __launch_bounds__(kFwdThreads, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
  using L = FwdSmem<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  if (sbase & 1023u) return;  // 128B-swizzle atoms need 1 KiB alignment (uniform over the grid)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nmt = (p.Sq + kBM - 1) / kBM;
  const int bh = (int)blockIdx.x % (p.B * p.Hq);
  const int mt = nmt - 1 - (int)blockIdx.x / (p.B * p.Hq);  // later query tiles first
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int g = h / (p.Hq / p.Hk);
  const int m0 = mt * kBM;
  const KeyTiles tiles(p, m0);
  const int T = tiles.count;

  Ctx c;
  c.bars = sbase + L::BAR;
  c.abort = reinterpret_cast<volatile int*>(smem + L::MISC + 4);
  c.status = nullptr;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kFwdBars; ++i) {
      const bool many = i >= fPFull0 && i < fPvDone0;  // a warpgroup: 128 arrivals
      ptx::mbar_init(c.bar(i), many ? 128u : 1u);
    }
    *c.abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + L::MISC, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::MISC);
  // O accumulators: warpgroup wg's keys (64 of each tile) in [wg D, wg D + D)
  const uint32_t t_O = tmem;
  const uint32_t t_S0 = tmem + 2 * D;  // S buffers 0 / 1 (128 columns each)

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      const int qrow = b * p.Sq + m0;
      ptx::mbar_arrive_expect_tx(c.bar(fQFull), L::kTile);
#pragma unroll
      for (int hf = 0; hf < D / 64; ++hf)
        ptx::tma_load_3d(sbase + L::Q + hf * kFSlab, &tmQ, c.bar(fQFull), hf * 64, h, qrow);
      // K of step u into stage u & 1 once S(u - 2) read the stage, then V of
      // step u once P V(u - 2) did (loads issued per stage: nk, nv)
      int nk[2] = {0, 0}, nv[2] = {0, 0};
      for (int u = 0; u < T; ++u) {
        const int st = u & 1, use = u >> 1;
        const int krow = b * p.Sk + tiles.tile(u) * kBN;
        if (use > 0 && !wait_bar(c, fKEmpty0 + st, (use - 1) & 1, 1)) break;
        const uint32_t kfull = c.bar(fKFull0 + st);
        ptx::mbar_arrive_expect_tx(kfull, L::kTile);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          ptx::tma_load_3d(sbase + L::K + st * L::kTile + hf * kFSlab, &tmK, kfull, hf * 64, g, krow);
        nk[st] = use + 1;
        if (use > 0 && !wait_bar(c, fVEmpty0 + st, (use - 1) & 1, 7)) break;
        const uint32_t vfull = c.bar(fVFull0 + st);
        ptx::mbar_arrive_expect_tx(vfull, L::kTile);
#pragma unroll
        for (int hf = 0; hf < D / 64; ++hf)
          ptx::tma_load_3d(sbase + L::V + st * L::kTile + hf * kFSlab, &tmV, vfull, hf * 64, g, krow);
        nv[st] = use + 1;
      }
      // no copy may still be landing in shared memory when the CTA ends
      drain_bar(c, fQFull, 0);
      for (int st = 0; st < 2; ++st) {
        if (nk[st] > 0) drain_bar(c, fKFull0 + st, (nk[st] - 1) & 1);
        if (nv[st] > 0) drain_bar(c, fVFull0 + st, (nv[st] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t id_S = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_O = idesc_bf16(128, D, false, true);
      const uint64_t dQ = ptx::smem_desc_sw128(sbase + L::Q, 16, 1024);
      const uint64_t dK = ptx::smem_desc_sw128(sbase + L::K, 16, 1024);
      const uint64_t dVmn = ptx::smem_desc_sw128(sbase + L::V, kFSlab, 1024);
      int n_s[2] = {0, 0}, n_pv[2] = {0, 0};  // S / P V steps issued per stage
      // O_wg += P(:, keys of wg) V(keys of wg, :) of step v, each half once
      // its warpgroup has written its P over S(v) in TMEM
      auto issue_pv = [&](int v) -> bool {
        const int sv = v & 1;
        const uint32_t t_S = t_S0 + sv * 128;
        const uint64_t dv = ptx::desc_add(dVmn, sv * L::kTile);
        if (!wait_bar(c, fVFull0 + sv, (v >> 1) & 1, 5)) return false;
#pragma unroll
        for (int wg = 0; wg < 2; ++wg) {
          if (!wait_bar(c, fPFull0 + wg * 2 + sv, (v >> 1) & 1, 6)) return false;
          ptx::tc_fence_after();
#pragma unroll
          for (int s = 4 * wg; s < 4 * wg + 4; ++s) {
            const uint32_t a_col = t_S + (s >> 2) * 64 + (s & 3) * 8;
            ptx::mma_ts(t_O + wg * D, a_col, ptx::desc_add(dv, s * 2048), id_O,
                        (v > 0 || s > 4 * wg) ? 1u : 0u);
          }
        }
        ptx::mma_commit(c.bar(fVEmpty0 + sv));  // V of the step read
        ptx::mma_commit(c.bar(fPvDone0 + sv));  // its S buffer free again, O up to date
        ++n_pv[sv];
        return true;
      };
      // S(u) first, then the P V of step u - 1 (its P is being written while
      // S(u) runs)
      bool ok = T == 0 || wait_bar(c, fQFull, 0, 2);
      for (int u = 0; ok && u < T; ++u) {
        const int st = u & 1;
        ok = wait_bar(c, fKFull0 + st, (u >> 1) & 1, 3) &&
             (u < 2 || wait_bar(c, fPvDone0 + st, ((u - 2) >> 1) & 1, 4));  // buffer of step u - 2
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t t_S = t_S0 + st * 128;
        const uint64_t dk = ptx::desc_add(dK, st * L::kTile);
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kFSlab + (s & 3) * 32;
          ptx::mma_ss(t_S, ptx::desc_add(dQ, off), ptx::desc_add(dk, off), id_S, s > 0);
        }
        ptx::mma_commit(c.bar(fSFull0 + st));
        ptx::mma_commit(c.bar(fKEmpty0 + st));  // K of the step read
        ++n_s[st];
        if (u > 0) ok = issue_pv(u - 1);
      }
      if (ok && T > 0) issue_pv(T - 1);
      ptx::mma_commit(c.bar(fOFull));
      // commit arrivals no other role waits for: waited here before the CTA exits
      for (int st = 0; st < 2; ++st) {
        if (n_s[st] > 0) drain_bar(c, fKEmpty0 + st, (n_s[st] - 1) & 1);
        if (n_pv[st] > 0) {
          drain_bar(c, fVEmpty0 + st, (n_pv[st] - 1) & 1);
          drain_bar(c, fPvDone0 + st, (n_pv[st] - 1) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ----------------------------------------------- softmax warpgroups --
    const int wg = (warp - 4) >> 2;  // key columns [64 wg, 64 wg + 64) of a tile
    const int lg = warp & 3;
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int il = lg * 32 + lane;  // query row within the tile
    const int i = m0 + il;
    const bool row_in = i < p.Sq;
    const int ic = row_in ? i : p.Sq - 1;
    const float* brow = nullptr;
    if constexpr (BIAS) brow = p.bias + ((int64_t)h * p.Sq + ic) * p.Sk;
    // This thread's 64 keys of step u's tile, as x (fp32 bits in x[]) with
    // the log2-domain logit = x * xs: on a tile where every key is live and
    // there is no bias, x is the raw score as it came from TMEM and xs =
    // scale log2(e) (the scaling folds into the exponent's fma); otherwise x
    // is the logit itself (dead keys -inf) and xs = 1.
    auto scores = [&](int u, uint32_t* x, float& xs) -> bool {
      const int st = u & 1;
      // the tile's mask class (uniform over the CTA), worked out while S(u)
      // may still be running
      const int n0 = tiles.tile(u) * kBN;
      const int kcap = p.Sk - n0;  // keys [0, kcap) of the tile exist
      const bool partial = m0 + kBM > p.Sq || n0 + kBN > p.Sk ||
                           !tile_full(p.mask, m0, m0 + kBM, n0, n0 + kBN);
      int klo = 0, khi = kBN - 1, ksink = 0;
      if (partial) {
        klo = i - p.mask.wl - n0;
        khi = imin2(i + p.mask.wr - n0, kcap - 1);
        ksink = imin2(p.mask.sink - n0, kcap);
      }
      // the row's bias for these keys: 16-byte loads when the tile's keys
      // all exist and the bias rows are 16-byte aligned (Sk a multiple of 4),
      // else clamped scalar loads (keys past Sk are dead). At D = 64 they are
      // issued before S is waited for; at D = 128 after S is in registers (so
      // that the two 64-value arrays are not live across the wait).
      float bv[BIAS ? 64 : 1];
      auto load_bias = [&]() {
        if constexpr (BIAS) {
          if (kcap >= kBN && (p.Sk & 3) == 0) {
            const float4* b4 = reinterpret_cast<const float4*>(brow + n0 + wg * 64);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float4 t4 = __ldg(b4 + e);
              bv[4 * e] = t4.x;
              bv[4 * e + 1] = t4.y;
              bv[4 * e + 2] = t4.z;
              bv[4 * e + 3] = t4.w;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 64; ++e) bv[e] = __ldg(brow + n0 + imin2(wg * 64 + e, kcap - 1));
          }
        }
      };
      if constexpr (D == 64) load_bias();
      // (warp-uniform outcome: the TMEM loads below are warp-collective)
      const bool full = wait_bar(c, fSFull0 + st, (u >> 1) & 1, 10);
      if (!__all_sync(0xffffffffu, full)) return false;
      ptx::tc_fence_after();
      const uint32_t t_S = t_S0 + st * 128 + lane_off + wg * 64;
      ptx::tmem_ld32(t_S, x);
      ptx::tmem_ld32(t_S + 32, x + 32);
      ptx::tmem_wait_ld();
      if (!BIAS && !partial) {
        xs = p.scale_log2;
        return true;
      }
      if constexpr (D != 64) load_bias();
#pragma unroll
      for (int e = 0; e < 64; ++e) {
        const int kk = wg * 64 + e;  // key within the tile
        float xv = __uint_as_float(x[e]) * p.scale_log2;
        if constexpr (BIAS) xv = fmaf(bv[e], kLog2e, xv);
        const bool live = !partial || (kk >= klo && kk <= khi) || kk < ksink;
        x[e] = __float_as_uint(live ? xv : -INFINITY);
      }
      xs = 1.f;
      return true;
    };
    // One pass over the live key tiles. Each warpgroup keeps, per row, its
    // own running maximum m_used, sum l and O accumulator over its 64 keys of
    // every tile, so the two halves of a row never wait for each other; they
    // meet once at the end. P is taken against m_used, the maximum the
    // accumulated terms were scaled with; only when a tile's maximum exceeds
    // it by more than kRescaleLog2 (so P stays below 2^kRescaleLog2) does
    // m_used move up, and then the row of this warpgroup's O and its sum are
    // scaled down by 2^(old - new) once the previous P V has completed.
    constexpr float kRescaleLog2 = 8.f;
    float m_used = -INFINITY, l = 0.f;
    const uint32_t t_Ow = t_O + wg * D + lane_off;  // this warpgroup's O rows
    bool ok = true;
    for (int u = 0; u < T; ++u) {
      uint32_t x[64];
      float xs;
      if (!scores(u, x, xs)) { ok = false; break; }
      // the tile's maximum logit: max(x) xs exactly, xs being positive
      float mx[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        mx[r] = __uint_as_float(x[16 * r]);
#pragma unroll
        for (int e = 1; e < 15; e += 2)
          mx[r] = ptx::max3(mx[r], __uint_as_float(x[16 * r + e]), __uint_as_float(x[16 * r + e + 1]));
        mx[r] = fmaxf(mx[r], __uint_as_float(x[16 * r + 15]));
      }
      const float m_tile = ptx::max3(mx[0], mx[1], fmaxf(mx[2], mx[3])) * xs;
      const bool raise = m_tile > m_used + kRescaleLog2;  // this row's scale moves up
      const bool rescale = raise && m_used != -INFINITY;  // ... and O holds terms of it
      // The TMEM loads / stores are warp-collective: the warp takes the
      // rescale path when any of its rows needs it (factor 1 for the others).
      if (__any_sync(0xffffffffu, rescale)) {
        // once P V(u - 1) (and so every earlier one) completed
        const bool done = wait_bar(c, fPvDone0 + ((u - 1) & 1), ((u - 1) >> 1) & 1, 13);
        if (!__all_sync(0xffffffffu, done)) { ok = false; break; }
        ptx::tc_fence_after();
        const float f = rescale ? ptx::ex2(m_used - m_tile) : 1.f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          uint32_t ov[32];
          ptx::tmem_ld32(t_Ow + cc * 32, ov);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
          ptx::tmem_st16(t_Ow + cc * 32, ov);
          ptx::tmem_st16(t_Ow + cc * 32 + 16, ov + 16);
        }
        l *= f;
      }
      if (raise) m_used = m_tile;
      // P = 2^(x xs - m_used) as bf16 over S. Dead keys give 2^-inf = 0; a
      // row with no live key so far (m_used = -inf, every x -inf) takes 0 as
      // its offset, so its P is 0 too.
      const float nm = m_used == -INFINITY ? 0.f : -m_used;
      uint32_t pk[32];
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int e = 0; e < 64; e += 2) {
        float a0, a1;
        ptx::fma2(a0, a1, __uint_as_float(x[e]), __uint_as_float(x[e + 1]), xs, xs, nm, nm);
        const float p0 = ptx::ex2(a0), p1 = ptx::ex2(a1);
        ptx::add2(s0, s1, s0, s1, p0, p1);
        pk[e / 2] = pack_bf162(p0, p1);
      }
      l += s0 + s1;
      const uint32_t t_S = t_S0 + (u & 1) * 128 + lane_off + wg * 64;
      ptx::tmem_st16(t_S, pk);
      ptx::tmem_st16(t_S + 16, pk + 16);
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar(fPFull0 + wg * 2 + (u & 1)));
    }
    // the two halves of the row meet in shared memory
    float* stat = reinterpret_cast<float*>(smem + L::STAT);
    stat[(wg * 128 + il) * 2] = m_used;
    stat[(wg * 128 + il) * 2 + 1] = l;
    asm volatile("bar.sync 1, 256;" ::: "memory");
    const float m_o = stat[((1 - wg) * 128 + il) * 2];
    const float l_o = stat[((1 - wg) * 128 + il) * 2 + 1];
    const float mm = fmaxf(m_used, m_o);
    const float f0 = m_used == -INFINITY ? 0.f : ptx::ex2(m_used - mm);  // this half
    const float f1 = m_o == -INFINITY ? 0.f : ptx::ex2(m_o - mm);        // the other
    const float lsum = l * f0 + l_o * f1;
    const float lse2 = lsum > 0.f ? mm + log2f(lsum) : -INFINITY;  // log2 domain
    if (wg == 0 && row_in)
      p.lse[((int64_t)b * p.Hq + h) * p.Sq + i] = lse2 == -INFINITY ? -INFINITY : lse2 / kLog2e;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    // O = (O_self f0 + O_other f1) / sum: this warpgroup writes columns
    // [wg D/2, wg D/2 + D/2) of its row
    if (ok && (T == 0 || wait_bar(c, fOFull, 0, 11))) {
      ptx::tc_fence_after();
      __nv_bfloat16* orow = p.o + b * p.os0 + (int64_t)ic * p.os1 + h * p.os2 + wg * (D / 2);
      const float g_self = f0 * inv, g_other = f1 * inv;
#pragma unroll 1
      for (int cc = 0; cc < D / 64; ++cc) {
        uint32_t va[32], vb[32];
        if (T > 0) {
          ptx::tmem_ld32(t_O + wg * D + lane_off + wg * (D / 2) + cc * 32, va);
          ptx::tmem_ld32(t_O + (1 - wg) * D + lane_off + wg * (D / 2) + cc * 32, vb);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) va[e] = vb[e] = 0u;
        }
        if (row_in) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            float o8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              o8[k] = __uint_as_float(va[e + k]) * g_self + __uint_as_float(vb[e + k]) * g_other;
            uint4 w;
            w.x = pack_bf162(o8[0], o8[1]);
            w.y = pack_bf162(o8[2], o8[3]);
            w.z = pack_bf162(o8[4], o8[5]);
            w.w = pack_bf162(o8[6], o8[7]);
            *reinterpret_cast<uint4*>(orow + cc * 32 + e) = w;
          }
        }
      }
    }
  }

  // ----------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (lane == 0) drain_bar(c, fOFull, 0);
    __syncwarp();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// [rows][H][D] bf16 with element strides (row, head): 3-D map (d, head, row),
// boxes of 64 d x 1 head x 128 rows, 128B swizzle.
bool make_map3(CUtensorMap* m, const void* base, int64_t rows, int H, int D, int64_t s_row,
               int64_t s_head) {
  EncodeFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)s_head * 2, (cuuint64_t)s_row * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool BIAS>
cudaError_t launch_fwd_variant(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                               const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = attn_fwd_tc_kernel<D, BIAS>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         FwdSmem<D>::TOTAL);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  kern<<<grid, kFwdThreads, FwdSmem<D>::TOTAL, stream>>>(q, k, v, p);
  return cudaGetLastError();
}

}  // namespace

bool fwd_tc_supported(const Problem& p) {
  // rows of one head must be evenly spaced over (batch, position): the tensor
  // maps view q / k / v as [batch * position][head][d]
  const bool packed_q = p.B == 1 || p.qs[0] == (int64_t)p.Sq * p.qs[1];
  const bool packed_k = p.B == 1 || (p.ks[0] == (int64_t)p.Sk * p.ks[1] &&
                                     p.vs[0] == (int64_t)p.Sk * p.vs[1]);
  return !p.sparse && !p.varlen && !p.cuda_cores && (p.D == 64 || p.D == 128) && p.B > 0 &&
         p.Sq > 0 && p.Sk > 0 && packed_q && packed_k && p.qs[1] > 0 && p.ks[1] > 0 &&
         p.vs[1] > 0 && encode_fn() != nullptr;
}

cudaError_t launch_fwd_tc(const Problem& pr, const void* q, const void* k, const void* v,
                          const float* bias, void* o, float* lse, cudaStream_t stream) {
  CUtensorMap mq, mk, mv;
  if (!make_map3(&mq, q, (int64_t)pr.B * pr.Sq, pr.Hq, pr.D, pr.qs[1], pr.qs[2]) ||
      !make_map3(&mk, k, (int64_t)pr.B * pr.Sk, pr.Hk, pr.D, pr.ks[1], pr.ks[2]) ||
      !make_map3(&mv, v, (int64_t)pr.B * pr.Sk, pr.Hk, pr.D, pr.vs[1], pr.vs[2]))
    return cudaErrorInvalidValue;
  FwdParams p;
  p.B = pr.B;
  p.Hq = pr.Hq;
  p.Hk = pr.Hk;
  p.Sq = pr.Sq;
  p.Sk = pr.Sk;
  p.scale_log2 = pr.scale * kLog2e;
  p.mask = pr.mask;
  p.bias = bias;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.os0 = pr.os[0];
  p.os1 = pr.os[1];
  p.os2 = pr.os[2];
  p.lse = lse;
  const int grid = pr.B * pr.Hq * ((pr.Sq + kBM - 1) / kBM);
  if (pr.D == 64)
    return bias ? launch_fwd_variant<64, true>(mq, mk, mv, p, grid, stream)
                : launch_fwd_variant<64, false>(mq, mk, mv, p, grid, stream);
  return bias ? launch_fwd_variant<128, true>(mq, mk, mv, p, grid, stream)
              : launch_fwd_variant<128, false>(mq, mk, mv, p, grid, stream);
}

}  // namespace attn
