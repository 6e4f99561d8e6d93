// Tensor-core (tcgen05 / TMEM / TMA) fused attention backward for sm_103a.
//
// Math (composable_kernel "34_bwd_gqa_fmha.py" docstring and cpu_bwd_gqa,
// "28_backward_dbias_fmha.py" cpu_attention_bwd_dbias):
//   P = exp(scale Q K^T + bias - LSE) on live entries, D = rowsum(dO * O),
//   dP = dO V^T, dS = P (dP - D), dQ = scale dS K, dK = scale dS^T Q,
//   dV = P^T dO, dK / dV summed over the query heads of a KV head,
//   dbias = sum over the batch of dS.
//
// One launch, two kinds of CTA (all tiles 128 x 128, fp16 operands, fp32
// accumulators in TMEM; fully masked tiles are skipped and partial tiles get
// a per-element mask):
//
// Key-major CTAs (dK, dV, dbias). cs CTAs share one 128-row key tile of one
// (batch, KV head); CTA `rank` takes r / cs of the r query heads that share
// the KV head and loops over their live query tiles, accumulating its partial
// dK / dV in TMEM over the group. At the end each CTA adds its partial rows
// into dK / dV with TMA bulk reductions (the pre-pass zeroes the buffers when
// cs > 1), so no post-pass over per-head gradients exists. Trailing key tiles
// with fewer live query tiles may use a smaller split (cs_lo, down to one CTA
// that stores its rows), so that no CTA runs longer than the longest split
// one while fewer CTAs pay the fixed costs. Per
// tile, so that one thread owns one key row of the softmax:
//   MMA1  S^T  = K  Q^T      (M = keys, N = queries, K = D; both K-major)
//   MMA2  dP^T = V  dO^T     (into the same TMEM columns, once S^T was read)
//   SFU   phase 1: P^T = exp2(S^T scale log2e + bias log2e - LSE log2e),
//                  kept in fp32 registers
//         phase 2: dS^T = P^T (dP^T - D); dS^T and P^T go as fp16 pairs into
//                  the columns of dP^T just read (A operands of MMA3 / MMA4)
//   MMA3  dV += P^T dO       (A = P^T in TMEM, B = dO MN-major)
//   MMA4  dK += dS^T Q       (A = dS^T in TMEM, B = Q MN-major)
// TMEM holds dK, dV and two 128-column buffers; tile t uses buffer t & 1
// for S^T, then dP^T, then dS^T / P^T. Issue order per tile: dP(t) (as soon
// as the softmax has copied S^T(t) into registers), S(t+1) into the other
// buffer (free once dV / dK(t-1) have read it), dV(t), dK(t). No MMA has to
// wait for an earlier one to complete, so the tensor pipe runs while the
// softmax works on the same tile.
//
// Query-major CTAs (dQ): one CTA per (batch, query head, 128-row query tile)
// loops over the live key tiles of its KV head, recomputing S and dP:
//   MMA1' S  = Q  K^T        (M = queries, N = keys)
//   MMA2' dP = dO V^T        (into the same TMEM columns, once S was read)
//   SFU   dS = exp2(...) (dP - D), fp16 into TMEM over dP
//   MMA3' dQ += dS K         (A = dS in TMEM, B = K MN-major)
// dQ accumulates in TMEM over all key tiles and is written once: no atomics
// and no zero-filled accumulation buffer. Tile t uses TMEM buffer t % 3 of
// three, so S(t+1) goes out right after dP(t) and the softmax never waits for
// the next S.
//
// dbias at D = 64 (B <= 4, whole tiles, fixed lengths): batch-inner
// query-major CTAs instead, one per (query head, query tile) over all
// batches, batch innermost; each sums dS over the batches in registers and
// stores every dbias element of a live tile once, and the key-major CTAs run
// without dbias (details at qb_cta). Otherwise the key-major softmax adds dS
// into dbias with fp32 reductions.
//
// Lengths need not be whole tiles: the pre-pass stages every head's rows
// rounded up to 128 with zero rows past the length, a tile that crosses a
// length takes the per-element mask, and rows past the lengths are not
// stored. A variable-length batch gives every CTA its sequence's bounds,
// output rows and mask alignment (Seq). Live tiles come from closed-form
// ranges (mask.h), so the walk never visits a dead tile.
//
// Warp roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 4-7 and 8-11 two softmax warpgroups (columns 0-63 / 64-127 of
// the tile), which also run the epilogue. Every mbarrier wait is bounded:
// after ~2 s it records ATTN_ERR_DEVICE_TIMEOUT, raises a CTA-wide abort
// flag, and the CTA drains its copies / MMAs, frees TMEM and exits.
//
// Operands are fp16 (exact copies of the bf16 inputs, staged by the
// pre-pass): P and dS rounded to fp16 keep 3 more mantissa bits than bf16,
// and kind::f16 needs A and B of the same type.

#include "internal.h"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

#include <algorithm>
#include <mutex>
#include <vector>

namespace attn {
namespace {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // key rows per tile
constexpr int kThreads = 384;
constexpr int kSlab = 128 * 128;  // one [128 rows][64 fp16] 128B-swizzled slab, bytes

// Shared memory of a key-major CTA.
template <int D>
struct SmemKV {
  static constexpr int kTile = (D / 64) * kSlab;  // a [128][D] fp16 operand tile
  static constexpr int K = 0;
  static constexpr int V = K + kTile;
  static constexpr int Q = V + kTile;        // 3 stages
  static constexpr int dO = Q + 3 * kTile;   // 2 stages
  static constexpr int LSE = dO + 2 * kTile; // 2 stages x 128 fp32 (with the dO stage)
  static constexpr int DLT = LSE + 1024;     // 2 stages x 128 fp32
  static constexpr int BAR = DLT + 1024;     // mbarriers (up to 32)
  static constexpr int MISC = BAR + 256;     // TMEM base, abort flag
  // D = 64 with a bias: the tile's bias [128 queries][128 keys] fp32 as four
  // TMA boxes of 32 keys (128B-swizzled 128-byte rows), one stage
  static constexpr int BIAS = (MISC + 16 + 1023) / 1024 * 1024;
  static constexpr int TOTAL = D == 64 ? BIAS + 4 * kSlab : MISC + 16;
  // end-of-kernel staging of dK / dV rows for the bulk reductions (reuses Q, dO)
  static constexpr int kStageRow = D * 4 + 16;  // padded fp32 row: conflict-free v4 stores
  static constexpr int STAGE = Q;
  static_assert(2 * 128 * kStageRow <= 5 * kTile, "staging fits");
};

// Shared memory of a query-major CTA.
template <int D>
struct SmemQ {
  static constexpr int kTile = (D / 64) * kSlab;
  static constexpr int kKS = D == 128 ? 3 : 2;  // K stages (the bias stages take the room at D = 64)
  static constexpr int Q = 0;
  static constexpr int dO = Q + kTile;
  static constexpr int K = dO + kTile;          // kKS stages
  static constexpr int V = K + kKS * kTile;     // 2 stages
  static constexpr int BAR = V + 2 * kTile;     // mbarriers (up to 32)
  static constexpr int MISC = BAR + 256;
  // D = 64 with a bias: two stages of the tile's bias [128 queries][128 keys]
  // fp32 (four 128B-swizzled TMA boxes of 32 keys each)
  static constexpr int BIAS = (MISC + 16 + 1023) / 1024 * 1024;
  static constexpr int TOTAL = D == 64 ? BIAS + 2 * 4 * kSlab : MISC + 16;
  // end-of-kernel staging of dQ rows for the copy-engine stores (reuses K, V)
  static constexpr int kStageRow = D * 4 + 16;  // padded fp32 row: conflict-free v4 stores
  static constexpr int STAGE = K;
  static_assert(128 * kStageRow <= (kKS + 2) * kTile, "staging fits");
};

static_assert(SmemKV<64>::TOTAL <= 232448 && SmemQ<64>::TOTAL <= 232448 &&
                  SmemKV<128>::TOTAL <= 232448 && SmemQ<128>::TOTAL <= 232448,
              "shared memory per CTA");

// Bias tiles through TMA (D = 64, whole tiles): a box is [128 rows][32 fp32]
// with the 128-byte swizzle, so the 16-byte chunk c of row r sits at chunk
// c ^ (r & 7). Byte offset of element (row r, column k) of a [128][128] tile
// stored as four such boxes.
__device__ __forceinline__ uint32_t bias_off(int r, int k) {
  return (uint32_t)((k >> 5) * kSlab + r * 128 + ((((k & 31) >> 2) ^ (r & 7)) << 4) +
                    (k & 3) * 4);
}

// Whether a kernel instantiation reads its bias tiles through TMA into
// shared memory (room for them at D = 64; whole tiles only, so that every
// box is inside the bias tensor and its rows are 16-byte aligned).
template <int D, bool BIAS, bool RB>
constexpr bool tma_bias() {
  return BIAS && !RB && D == 64;
}

template <int D>
constexpr int smem_total() {
  return SmemKV<D>::TOTAL > SmemQ<D>::TOTAL ? SmemKV<D>::TOTAL : SmemQ<D>::TOTAL;
}

// barrier indices, key-major CTA
// Tile t works in TMEM buffer t & 1: MMA1 writes S^T there (kSFull0 + (t & 1)),
// the softmax copies it out (kSFree), MMA2 writes dP^T over it (kdPFull), the
// softmax writes dS^T and P^T back into the same columns (kP2Full, 256
// arrivals) and MMA3 / MMA4 read them (kMma40 + (t & 1): that buffer is free
// again). Q(t) uses stage t % 3 (kQFull0.., kQEmpty0.. once dK(t) read it),
// dO(t) with LSE / delta stage t & 1 (kOFull0.., kOEmpty0.. once dV(t) read
// it). kBiasFull / kBiasEmpty: the tile's bias landed in shared memory / was
// read by the softmax (256 arrivals), on the TMA bias path.
enum BarKV { kKvFull = 0, kQFull0 = 1, kQEmpty0 = 4, kOFull0 = 7, kOEmpty0 = 9, kSFull0 = 11,
             kSFree = 13, kdPFull = 14, kP2Full = 15, kMma40 = 16, kAccFull = 18,
             kBiasFull = 19, kBiasEmpty = 20, kKvBars = 21 };
// barrier indices, query-major CTA
// Tile t works in TMEM buffer t % 3: MMA1' writes S there (qSFull0 + t % 3),
// the softmax copies it out (qSFree), MMA2' writes dP over it (qdPFull), the
// softmax writes dS back into the same columns (qDsFull, 256 arrivals) and
// MMA3' reads it (qMma30 + t % 3: that buffer is free again). One S-ready and
// one MMA3'-done barrier per buffer, so that no barrier can complete two
// phases before its waiter polls the first. K(t) uses stage t % kKS
// (qKFull0.., qKEmpty0.. once dQ(t) read it), V(t) stage t & 1 (qVFull0..,
// qVEmpty0.. once dP(t) read it); qBiasFull0/1 / qBiasEmpty0/1: the two bias
// stages (TMA bias path).
enum BarQ { qQdoFull = 0, qKFull0 = 1, qKEmpty0 = 4, qVFull0 = 7, qVEmpty0 = 9, qSFull0 = 11,
            qSFree = 14, qdPFull = 15, qDsFull = 16, qMma30 = 17, qAccFull = 20,
            qBiasFull0 = 21, qBiasEmpty0 = 23, kQBars = 25 };

struct TcParams {
  int B, Hq, Hk, Sq, Sk;
  int Sqs, Sks;    // rows per head of the fp16 copies: Sq, Sk rounded up to whole tiles
  int ragged;      // Sq or Sk is not a whole number of tiles, or a variable-length batch
  // variable-length batch (cu_q == nullptr: fixed lengths Sq, Sk): sequence
  // bounds, and bottom-right alignment per sequence (br) of the top-left mask
  const int32_t* cu_q;
  const int32_t* cu_k;
  int total_q, total_k;
  int br;
  int cs;          // key-major CTAs per key tile (query-head split) of key tiles [0, n_split)
  int n_split;     // key tiles from n_split on have fewer live query tiles and
  int cs_lo;       // split over cs_lo CTAs only
  int kv_ctas;     // blocks [0, kv_ctas) are key-major, the rest query-major
  int qb_ctas;     // batch-inner dbias mode: blocks [0, qb_ctas) are batch-inner
                   // query-major, the rest key-major (without dbias)
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
  int64_t dbias_bstride;  // > 0: batch b adds into its own dbias slice, b dbias_bstride floats on
  DevStatus* status;
};

// Bits [a, b) of a 32-bit mask, clipped to [0, 32).
__device__ __forceinline__ uint32_t bits_between(int a, int b) {
  a = a < 0 ? 0 : a;
  b = b > 32 ? 32 : b;
  if (b <= a) return 0u;
  const uint32_t below_b = b >= 32 ? 0xffffffffu : ((1u << b) - 1u);
  return below_b & ~((1u << a) - 1u);
}

__device__ __forceinline__ int imin(int a, int b) { return a < b ? a : b; }

// One sequence of the batch as a CTA sees it: its lengths, the first rows of
// its dq and dk / dv in the outputs, and the mask aligned to it.
struct Seq {
  int lq, lk;
  int64_t oq, ok;
  MaskSpec mask;
};

// False (nothing to do; bad bounds are recorded) when the varlen bounds of
// sequence b are out of order or out of range.
__device__ __forceinline__ bool seq_of(const TcParams& p, int b, Seq* s) {
  if (p.cu_q == nullptr) {
    s->lq = p.Sq;
    s->lk = p.Sk;
    s->oq = (int64_t)b * p.Sq;
    s->ok = (int64_t)b * p.Sk;
    s->mask = p.mask;
    return true;
  }
  int tq, tk;
  const bool okq = seq_span(p.cu_q, b, p.total_q, p.Sq, &tq, &s->lq);
  const bool okk = seq_span(p.cu_k, b, p.total_k, p.Sk, &tk, &s->lk);
  if (!okq || !okk) {
    if (threadIdx.x == 0) report(p.status, ATTN_ERR_INVALID_ARG, b);
    return false;
  }
  s->oq = tq;
  s->ok = tk;
  s->mask = p.br ? mask_aligned(p.mask, s->lk - s->lq) : p.mask;
  return true;
}

// Whether some entry of the tile rows [m0, m0 + BM) x keys [n0, n0 + BN) is
// dead (masked, or past the end of the queries or keys), so that the tile
// needs the per-element mask.
__device__ __forceinline__ bool tile_cut(const Seq& s, int m0, int n0) {
  return m0 + BM > s.lq || n0 + BN > s.lk || !tile_full(s.mask, m0, m0 + BM, n0, n0 + BN);
}

// Per-element mask of one row of a tile, as both kinds of CTA apply it. The
// tile at (m0, n0) needs it when the mask cuts the tile (or, kMayBeRagged,
// the tile crosses a length); the return value says so. Otherwise every
// entry of the tile is live and the ranges are the whole tile.
//
// Key-major view, key row j: the live queries of the tile are [*qlo, *qhi]
// (tile-relative, may reach outside [0, BM): the chunk bits clip them). A
// sink key is live for every query; queries past the length and a key past
// its length are dead.
template <bool kMayBeRagged>
__device__ __forceinline__ bool kv_row_live(const Seq& s, int m0, int n0, int j, int* qlo,
                                            int* qhi) {
  const bool partial = kMayBeRagged ? tile_cut(s, m0, n0)
                                    : !tile_full(s.mask, m0, m0 + BM, n0, n0 + BN);
  int lo = 0, hi = BM - 1;
  if (partial) {
    if (j >= s.mask.sink) {
      lo = j - s.mask.wr - m0;
      hi = j + s.mask.wl - m0;
    }
    if constexpr (kMayBeRagged) {
      hi = imin(hi, s.lq - 1 - m0);
      if (j >= s.lk) hi = lo - 1;
    }
  }
  *qlo = lo;
  *qhi = hi;
  return partial;
}

// Live queries [q0, q0 + 32) of a key row: bit u for query q0 + u.
__device__ __forceinline__ uint32_t kv_chunk_bits(int qlo, int qhi, int q0) {
  return bits_between(qlo - q0, qhi - q0 + 1);
}

// Query-major view, query row i: the live keys of the tile are the window
// [*klo, *khi] plus the sink keys [0, *ksink) (tile-relative); keys past the
// length are dead. (Rows past the query length are padding: their staged
// Q / dO rows are zero, so dS is zero there whatever the mask says, and they
// are not stored.)
template <bool kMayBeRagged>
__device__ __forceinline__ bool q_row_live(const Seq& s, int m0, int n0, int i, int* klo,
                                           int* khi, int* ksink) {
  const bool partial = kMayBeRagged ? tile_cut(s, m0, n0)
                                    : !tile_full(s.mask, m0, m0 + BM, n0, n0 + BN);
  int lo = 0, hi = BN - 1, sk = 0;
  if (partial) {
    lo = i - s.mask.wl - n0;
    hi = i + s.mask.wr - n0;
    sk = s.mask.sink - n0;
    if constexpr (kMayBeRagged) {
      hi = imin(hi, s.lk - n0 - 1);
      sk = imin(sk, s.lk - n0);
    }
  }
  *klo = lo;
  *khi = hi;
  *ksink = sk;
  return partial;
}

// Live keys [k0, k0 + 32) of a query row: bit u for key k0 + u.
__device__ __forceinline__ uint32_t q_chunk_bits(int klo, int khi, int ksink, int k0) {
  return bits_between(klo - k0, khi - k0 + 1) | bits_between(-k0, ksink - k0);
}

// Live (query head, query tile) pairs of a key tile, heads outer: the live
// query tiles form one range (live_query_tiles), so the walk touches live
// tiles only.
struct QTileIter {
  int hpc, lo, hi, hl, mt;
  __device__ QTileIter(int hpc_, int n0, const Seq& s) : hpc(hpc_), hl(0) {
    live_query_tiles(s.mask, s.lq, s.lk, BM, BN, n0, &lo, &hi);
    mt = lo - 1;
  }
  __device__ bool next() {
    if (lo > hi) return false;
    if (++mt > hi) {
      mt = lo;
      if (++hl >= hpc) return false;
    }
    return true;
  }
};

// Live key tiles of a query tile, ascending: the sink tiles, then the window
// tiles (live_key_tiles).
struct KTileIter {
  int s_end, w_lo, w_hi, nt;
  __device__ KTileIter(int m0, const Seq& s) : nt(-1) {
    live_key_tiles(s.mask, s.lq, s.lk, BM, BN, m0, &s_end, &w_lo, &w_hi);
  }
  __device__ bool next() {
    if (++nt < s_end) return true;
    if (nt < w_lo) nt = w_lo;
    return nt <= w_hi;
  }
};

// Eight fp32 values as one 32-byte store (one full sector: half the store
// instructions of 16-byte stores when each thread writes its own row). The
// output buffers need only be 16-byte aligned: where dst is not 32-byte
// aligned the values go out as two 16-byte stores.
__device__ __forceinline__ void put8(float* dst, const float* v) {
  if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
    asm volatile("st.global.v8.f32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst),
                 "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
                 "f"(v[7])
                 : "memory");
  } else {
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(v[0]), "f"(v[1]),
                 "f"(v[2]), "f"(v[3])
                 : "memory");
    asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4), "f"(v[4]),
                 "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
  }
}

// Barrier set-up by thread 0 (the producer), which then issues the CTA's
// first copies at once (`early`: they complete on the barriers it has just
// initialised), so that their latency overlaps the TMEM allocation and the
// CTA-wide barrier.
template <typename Early>
__device__ __forceinline__ void init_common(const Ctx& c, uint32_t tmem_slot_addr, int nbars,
                                            const uint32_t* counts, int warp, Early&& early) {
  if (threadIdx.x == 0) {
    for (int i = 0; i < nbars; ++i) ptx::mbar_init(c.bar(i), counts[i]);
    *c.abort = 0;
    ptx::fence_mbar_init();
    early();
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot_addr, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
}

// ======================================================= key-major CTA ====
// RB: bias / dbias accesses clamped or predicated for ragged lengths (a
// separate instantiation, so that aligned problems keep unconditional,
// freely scheduled loads and reductions)
template <int D, bool BIAS, bool DBIAS, bool RB>
__device__ __forceinline__ void kv_cta(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                       const CUtensorMap* tmV, const CUtensorMap* tmdO,
                                       const CUtensorMap* tmB, const TcParams& p, uint8_t* smem,
                                       uint32_t sbase, int kvi) {
  using L = SmemKV<D>;
  // The bias variants run ragged lengths only as RB instantiations; the others
  // take both and test the lengths at run time.
  constexpr bool kMayBeRagged = RB || (!BIAS && !DBIAS);
  constexpr bool kTB = tma_bias<D, BIAS, RB>();  // bias tiles through TMA (whole tiles)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // key tiles [0, n_split) over cs CTAs each, the rest over cs_lo
  const int bhk = p.B * p.Hk;
  const int n_hi = p.n_split * bhk * p.cs;  // CTAs of the first n_split key tiles
  const bool lo_part = kvi >= n_hi;
  const int cs = lo_part ? p.cs_lo : p.cs;
  const int kk = lo_part ? kvi - n_hi : kvi;
  const int rank = kk % cs;
  const int ci = kk / cs;
  const int bg = ci % bhk;  // (batch, KV head); key tile slowest = heaviest first when causal
  const int nt = (lo_part ? p.n_split : 0) + ci / bhk;
  const int g = bg % p.Hk;
  const int b = bg / p.Hk;
  const int n0 = nt * BN;
  const int r = p.Hq / p.Hk;
  const int hpc = r / cs;
  const int h_first = g * r + rank * hpc;
  Seq sq;
  if (!seq_of(p, b, &sq) || n0 >= sq.lk) return;  // a key tile past this sequence's keys

  Ctx c;
  c.bars = sbase + L::BAR;
  c.abort = reinterpret_cast<volatile int*>(smem + L::MISC + 4);
  c.status = p.status;
  // a ragged problem's dO barriers take one more arrival: the producer warp's
  // plain copy of LSE / delta (the TMA bulk copy needs whole 16-byte-aligned
  // tiles)
  const uint32_t of = p.ragged ? 2u : 1u;
  // kKvFull, kQFull0-2, kQEmpty0-2, kOFull0/1, kOEmpty0/1, kSFull0/1, kSFree, kdPFull,
  // kP2Full, kMma40/1, kAccFull, kBiasFull, kBiasEmpty
  const uint32_t counts[kKvBars] = {1, 1, 1, 1, 1, 1, 1, of, of, 1, 1, 1, 1,
                                    256, 1, 256, 1, 1, 1, 1, 256};
  const uint32_t sK = sbase + L::K, sV = sbase + L::V;
  init_common(c, sbase + L::MISC, kKvBars, counts, warp, [&] {
    // K / V of the key tile, and Q of its first live tile (stage 0)
    const int krow = (b * p.Hk + g) * p.Sks + n0;
    ptx::mbar_arrive_expect_tx(c.bar(kKvFull), 2 * L::kTile);
#pragma unroll
    for (int hf = 0; hf < D / 64; ++hf) {
      ptx::tma_load_2d(sK + hf * kSlab, tmK, c.bar(kKvFull), hf * 64, krow);
      ptx::tma_load_2d(sV + hf * kSlab, tmV, c.bar(kKvFull), hf * 64, krow);
    }
    QTileIter it0(hpc, n0, sq);
    if (it0.next()) {
      const int row = (b * p.Hq + h_first + it0.hl) * p.Sqs + it0.mt * BM;
      ptx::mbar_arrive_expect_tx(c.bar(kQFull0), L::kTile);
#pragma unroll
      for (int hf = 0; hf < D / 64; ++hf)
        ptx::tma_load_2d(sbase + L::Q + hf * kSlab, tmQ, c.bar(kQFull0), hf * 64, row);
    }
  });
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::MISC);
  const uint32_t t_dK = tmem;
  const uint32_t t_dV = tmem + D;
  const uint32_t t_buf0 = tmem + 2 * D;  // tile t: S^T / dP^T / (dS^T, P^T) at t_buf0 + (t & 1) 128
  bool epi_ok = false;
  int n_iters = 0;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    // lane 0 waits and issues the copies; with ragged lengths the whole warp
    // also copies the tile's LSE / delta rows (zero past Sq). Q stages rotate
    // over three buffers, dO (with LSE / delta) over two.
    // (K / V and the first Q went out with the barrier set-up)
    int q_issued[3] = {0, 0, 0};
    int o_issued[2] = {0, 0};
    int bias_issued = 0;
    if (lane == 0 || p.ragged) {  // warp-uniform when ragged
      QTileIter it(hpc, n0, sq);
      int t = 0;
      while (it.next()) {
        const int qs = t % 3, qu = t / 3;  // Q stage and its use count
        const int os = t & 1, ou = t >> 1; // dO stage and its use count
        const int h = h_first + it.hl;
        const int m0 = it.mt * BM;
        const int64_t row = ((int64_t)b * p.Hq + h) * p.Sqs + m0;   // staged fp16 rows
        const int64_t lrow = ((int64_t)b * p.Hq + h) * p.Sq + m0;   // LSE / delta rows
        bool go = true;
        if (lane == 0) {
          // Q(t) once dK(t-3) released its stage (Q(0): already issued)
          if (qu > 0) go = wait_bar(c, kQEmpty0 + qs, (qu - 1) & 1, 1);
          if (go && t == 0) {
            q_issued[0] = 1;
          } else if (go) {
            const uint32_t qfull = c.bar(kQFull0 + qs);
            ptx::mbar_arrive_expect_tx(qfull, L::kTile);
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf)
              ptx::tma_load_2d(sbase + L::Q + qs * L::kTile + hf * kSlab, tmQ, qfull, hf * 64,
                               (int)row);
            q_issued[qs] = qu + 1;
          }
          // dO(t), LSE(t), delta(t) once dV(t-2) released the stage
          if (go && ou > 0) go = wait_bar(c, kOEmpty0 + os, (ou - 1) & 1, 16);
          if (go) {
            const uint32_t ofull = c.bar(kOFull0 + os);
            ptx::mbar_arrive_expect_tx(ofull, L::kTile + (p.ragged ? 0 : 2 * 512));
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf)
              ptx::tma_load_2d(sbase + L::dO + os * L::kTile + hf * kSlab, tmdO, ofull, hf * 64,
                               (int)row);
            if (!p.ragged) {
              ptx::bulk_load(sbase + L::LSE + os * 512, p.lse + lrow, 512, ofull);
              ptx::bulk_load(sbase + L::DLT + os * 512, p.delta + lrow, 512, ofull);
            }
            o_issued[os] = ou + 1;
          }
          if constexpr (kTB) {
            // the tile's bias rows (one stage: once the softmax read tile t - 1's)
            if (go && t > 0) go = wait_bar(c, kBiasEmpty, (t - 1) & 1, 14);
            if (go) {
              const uint32_t bfull = c.bar(kBiasFull);
              ptx::mbar_arrive_expect_tx(bfull, 4 * kSlab);
#pragma unroll
              for (int bx = 0; bx < 4; ++bx)
                ptx::tma_load_2d(sbase + L::BIAS + bx * kSlab, tmB, bfull, n0 + 32 * bx,
                                 h * p.Sq + m0);
              ++bias_issued;
            }
          }
        }
        if (p.ragged) {
          __syncwarp();
          if (!__shfl_sync(0xffffffffu, go, 0)) break;
          float* lse_s = reinterpret_cast<float*>(smem + L::LSE + os * 512);
          float* dl_s = reinterpret_cast<float*>(smem + L::DLT + os * 512);
#pragma unroll
          for (int u = 0; u < BM / 32; ++u) {
            const int q = u * 32 + lane;
            const bool in = m0 + q < sq.lq;
            lse_s[q] = in ? p.lse[lrow + q] : 0.f;
            dl_s[q] = in ? p.delta[lrow + q] : 0.f;
          }
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive(c.bar(kOFull0 + os));
        } else if (!go) {
          break;
        }
        ++t;
      }
    }
    if (lane == 0) {
      // no copy may still be landing in shared memory when the CTA ends
      drain_bar(c, kKvFull, 0);
      for (int s = 0; s < 3; ++s)
        if (q_issued[s] > 0) drain_bar(c, kQFull0 + s, (q_issued[s] - 1) & 1);
      for (int s = 0; s < 2; ++s)
        if (o_issued[s] > 0) drain_bar(c, kOFull0 + s, (o_issued[s] - 1) & 1);
      if (bias_issued > 0) drain_bar(c, kBiasFull, (bias_issued - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t id_S = ptx::idesc_f16_f32(128, 128, false, false);
      constexpr uint32_t id_KV = ptx::idesc_f16_f32(128, D, false, true);
      // operand descriptors, built once (K steps add their offsets)
      const uint64_t dK = ptx::smem_desc_sw128(sK, 16, 1024);
      const uint64_t dV = ptx::smem_desc_sw128(sV, 16, 1024);
      // stage 0 of Q / dO in K-major and MN-major views (stage s: + s kTile)
      const uint64_t dQk = ptx::smem_desc_sw128(sbase + L::Q, 16, 1024);
      const uint64_t ddOk = ptx::smem_desc_sw128(sbase + L::dO, 16, 1024);
      const uint64_t dQmn = ptx::smem_desc_sw128(sbase + L::Q, kSlab, 1024);
      const uint64_t ddOmn = ptx::smem_desc_sw128(sbase + L::dO, kSlab, 1024);
      auto issue_S = [&](int t) {  // MMA1 S^T = K Q^T (both K-major over d) into buffer t & 1
        const uint64_t dq = ptx::desc_add(dQk, (t % 3) * L::kTile);
        const uint32_t dst = t_buf0 + (t & 1) * 128;
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kSlab + (s & 3) * 32;
          ptx::mma_ss(dst, ptx::desc_add(dK, off), ptx::desc_add(dq, off), id_S, s > 0);
        }
      };
      auto issue_dP = [&](int t) {  // MMA2 dP^T = V dO^T over S^T(t)
        const uint64_t ddo = ptx::desc_add(ddOk, (t & 1) * L::kTile);
        const uint32_t dst = t_buf0 + (t & 1) * 128;
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kSlab + (s & 3) * 32;
          ptx::mma_ss(dst, ptx::desc_add(dV, off), ptx::desc_add(ddo, off), id_S, s > 0);
        }
      };
      // MMA3 dV += P^T dO and MMA4 dK += dS^T Q, A operands from the tile's
      // TMEM buffer: the 16 queries of K step s sit in chunk ((s & 3) >> 1) of
      // warpgroup (s >> 2)'s 64 columns, dS^T in its first 16 columns and P^T
      // in the next 16, 8 columns (fp16 pairs) per step. B = dO / Q MN-major.
      auto issue_dVdK = [&](int t) {
        const uint32_t buf = t_buf0 + (t & 1) * 128;
        const uint64_t ddo_mn = ptx::desc_add(ddOmn, (t & 1) * L::kTile);
        const uint64_t dq_mn = ptx::desc_add(dQmn, (t % 3) * L::kTile);
#pragma unroll
        for (int s = 0; s < BM / 16; ++s) {
          const uint32_t col = buf + (s >> 2) * 64 + ((s >> 1) & 1) * 32 + (s & 1) * 8;
          ptx::mma_ts(t_dV, col + 16, ptx::desc_add(ddo_mn, s * 2048), id_KV,
                      (t > 0 || s > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int s = 0; s < BM / 16; ++s) {
          const uint32_t col = buf + (s >> 2) * 64 + ((s >> 1) & 1) * 32 + (s & 1) * 8;
          ptx::mma_ts(t_dK, col, ptx::desc_add(dq_mn, s * 2048), id_KV,
                      (t > 0 || s > 0) ? 1u : 0u);
        }
      };
      // Per tile t (TMEM buffer t & 1): dP(t) over S^T(t) as soon as the
      // softmax has copied S^T(t) into its registers (kSFree); then S(t+1)
      // into the other buffer (once dV / dK of tile t - 1 have read it and
      // Q(t+1) has landed), then dV(t), dK(t) (once P^T(t) and dS^T(t) are in
      // TMEM). The softmax computes the exponentials of tile t while dP(t),
      // S(t+1) and dV / dK(t-1) run. Waits suspend the thread (mbarrier
      // try_wait), so the MMA warp takes no issue slots from the softmax
      // warps that share its SM sub-partition.
      bool ok = wait_bar(c, kKvFull, 0, 2);
      int n_tiles = 0;  // tiles whose dV / dK MMAs were issued
      QTileIter it(hpc, n0, sq);
      bool have = ok && it.next();
      if (have) {
        have = wait_bar(c, kQFull0, 0, 3);
        if (have) {
          ptx::tc_fence_after();
          issue_S(0);
          ptx::mma_commit(c.bar(kSFull0));
        }
      }
      int t = 0;
      while (have) {
        const int b2 = t & 1;
        if (!wait_bar(c, kSFree, t & 1, 13)) break;
        if (!wait_bar(c, kOFull0 + b2, (t >> 1) & 1, 5)) break;
        ptx::tc_fence_after();
        issue_dP(t);
        ptx::mma_commit(c.bar(kdPFull));
        const bool have1 = it.next();
        const int n1 = b2 ^ 1;                                   // buffer of tile t + 1
        const uint32_t qpar = ((t + 1) / 3) & 1;                 // fill of Q stage (t+1) % 3
        const uint32_t mpar = t > 0 ? ((t - 1) >> 1) & 1 : 0u;  // dV / dK(t-1) done
        if (have1) {
          if (t > 0 && !wait_bar(c, kMma40 + n1, mpar, 6)) break;
          if (!wait_bar(c, kQFull0 + (t + 1) % 3, qpar, 5)) break;
          ptx::tc_fence_after();
          issue_S(t + 1);
          ptx::mma_commit(c.bar(kSFull0 + n1));
        }
        if (!wait_bar(c, kP2Full, t & 1, 7)) break;
        ptx::tc_fence_after();
        issue_dVdK(t);
        ptx::mma_commit(c.bar(kOEmpty0 + b2));     // dO(t) read by dP(t) and dV(t)
        ptx::mma_commit(c.bar(kQEmpty0 + t % 3));  // Q(t) read by S(t) and dK(t)
        ptx::mma_commit(c.bar(kMma40 + b2));       // buffer t & 1 free again
        ++n_tiles;
        if (!ok) break;
        have = have1;
        ++t;
      }
      ptx::mma_commit(c.bar(kAccFull));
      // The last commits of the stage and buffer barriers are waited by nobody
      // else: wait for them here, so that no commit arrival is still in flight
      // when the CTA exits (a late one would land on the barriers of the next
      // CTA on this SM). Buffer / dO stage b took the commits of tiles b,
      // b + 2, ...; Q stage s those of tiles s, s + 3, ...
      for (int bb = 0; bb < 2; ++bb) {
        const int n_b = (n_tiles + 1 - bb) >> 1;
        if (n_b > 0) {
          drain_bar(c, kMma40 + bb, (n_b - 1) & 1);
          drain_bar(c, kOEmpty0 + bb, (n_b - 1) & 1);
        }
      }
      for (int s = 0; s < 3; ++s) {
        const int n_s = (n_tiles + 2 - s) / 3;
        if (n_s > 0) drain_bar(c, kQEmpty0 + s, (n_s - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------- softmax / dS warpgroups --
    const int wg = (warp - 4) >> 2;                  // 0: queries 0-63, 1: 64-127
    const int lg = warp & 3;                         // TMEM lane quarter
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int jl = lg * 32 + lane;                   // key row within the tile
    const int j = n0 + jl;
    QTileIter it(hpc, n0, sq);
    int t = 0;
    bool ok = true;
    while (it.next()) {
      const int b2 = t & 1;
      if (!wait_bar(c, kOFull0 + b2, (t >> 1) & 1, 8)) { ok = false; break; }  // LSE / delta
      const float* lse_s = reinterpret_cast<const float*>(smem + L::LSE + b2 * 512);
      const float* dl_s = reinterpret_cast<const float*>(smem + L::DLT + b2 * 512);
      if (!wait_bar(c, kSFull0 + b2, (t >> 1) & 1, 9)) { ok = false; break; }
      ptx::tc_fence_after();
      const uint32_t buf = t_buf0 + b2 * 128;  // this tile's TMEM buffer
      const int h = h_first + it.hl;
      const int m0 = it.mt * BM;
      // Live queries of this key row within the tile, [qlo, qhi]. A row
      // without live keys has LSE = -inf; it can only sit in a partial tile,
      // where this mask zeroes its probabilities. So do the rows past Sq and
      // a key row past Sk (zero operands in the staged copies).
      int qlo, qhi;
      const bool partial = kv_row_live<kMayBeRagged>(sq, m0, n0, j, &qlo, &qhi);
      const int qcap = sq.lq - 1 - m0;       // last query of the tile
      // bias / dbias element (query m0 + q, key j); reads of rows and keys
      // past the lengths are clamped into the tensor (their P is zero)
      const int jc = kMayBeRagged ? imin(j, sq.lk - 1) : j;
      const float* brow = nullptr;
      if constexpr (BIAS && !kTB) brow = p.bias + ((int64_t)h * p.Sq + m0) * p.Sk + jc;
      if constexpr (kTB) {
        if (!wait_bar(c, kBiasFull, t & 1, 15)) { ok = false; break; }
      }
      float* dbrow = nullptr;
      if constexpr (DBIAS)
        dbrow = p.dbias + b * p.dbias_bstride + ((int64_t)h * p.Sq + m0) * p.Sk + j;
      // phase 1: P^T from S^T, fp32 in registers (one key row per thread)
      float pv[64];
      {
        uint32_t sr[64];
        ptx::tmem_ld32(buf + lane_off + wg * 64, sr);
        ptx::tmem_ld32(buf + lane_off + wg * 64 + 32, sr + 32);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(c.bar(kSFree));  // S^T(t) is in registers: MMA2 may overwrite it
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int q0 = wg * 64 + cc * 32;  // first query of this chunk within the tile
          const uint32_t live = kv_chunk_bits(qlo, qhi, q0);
#pragma unroll
          for (int e4 = 0; e4 < 32; e4 += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(lse_s + q0 + e4);
            const float lv[4] = {l4.x, l4.y, l4.z, l4.w};
            float bv[4];
            if constexpr (BIAS && RB) {
#pragma unroll
              for (int u = 0; u < 4; ++u)
                bv[u] = __ldg(brow + (int64_t)imin(q0 + e4 + u, qcap) * p.Sk);
            } else if constexpr (kTB) {
              // bias (query q0 + e4 + u, key jl) of the tile in shared memory
#pragma unroll
              for (int u = 0; u < 4; ++u)
                bv[u] = *reinterpret_cast<const float*>(smem + L::BIAS +
                                                        bias_off(q0 + e4 + u, jl));
            } else if constexpr (BIAS) {
#pragma unroll
              for (int u = 0; u < 4; ++u) bv[u] = __ldg(brow + (int64_t)(q0 + e4 + u) * p.Sk);
            }
            // x = S scale log2e - LSE log2e (+ bias log2e), two queries per instruction
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              float n0, n1;
              ptx::mul2(n0, n1, lv[u], lv[u + 1], -kLog2e, -kLog2e);
              ptx::fma2(x[u], x[u + 1], __uint_as_float(sr[cc * 32 + e4 + u]),
                        __uint_as_float(sr[cc * 32 + e4 + u + 1]), p.scale_log2, p.scale_log2,
                        n0, n1);
              if constexpr (BIAS)
                ptx::fma2(x[u], x[u + 1], bv[u], bv[u + 1], kLog2e, kLog2e, x[u], x[u + 1]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) pv[cc * 32 + e4 + u] = ptx::ex2(x[u]);
            if (partial) {  // warp-uniform: only tiles the mask cuts need the per-query test
#pragma unroll
              for (int u = 0; u < 4; ++u)
                if (!((live >> (e4 + u)) & 1u)) pv[cc * 32 + e4 + u] = 0.f;
            }
          }
        }
        if constexpr (kTB) ptx::mbar_arrive(c.bar(kBiasEmpty));  // bias tile read
      }
      // phase 2: dS^T = P^T (dP^T - D). Each 32-query chunk of dP^T, once
      // read, takes dS^T (16 columns of fp16 pairs, A operand of dK) and P^T
      // (the next 16 columns, A operand of dV) in its place.
      if (!wait_bar(c, kdPFull, t & 1, 10)) { ok = false; break; }
      ptx::tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int q0 = wg * 64 + cc * 32;
        uint32_t live_d = 0xffffffffu;
        if constexpr (DBIAS && RB) live_d = partial ? kv_chunk_bits(qlo, qhi, q0) : live_d;
        uint32_t dr[32];
        ptx::tmem_ld32(buf + lane_off + wg * 64 + cc * 32, dr);
        ptx::tmem_wait_ld();
        uint32_t dk[16], pk[16];
#pragma unroll
        for (int e4 = 0; e4 < 32; e4 += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(dl_s + q0 + e4);
          const float dv[4] = {d4.x, d4.y, d4.z, d4.w};
          float de[4];
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            float t0, t1;
            ptx::sub2(t0, t1, __uint_as_float(dr[e4 + u]), __uint_as_float(dr[e4 + u + 1]), dv[u],
                      dv[u + 1]);
            ptx::mul2(de[u], de[u + 1], pv[cc * 32 + e4 + u], pv[cc * 32 + e4 + u + 1], t0, t1);
          }
          if constexpr (DBIAS && RB) {
            // live entries only: rows past Sq and a key past Sk have no dbias
            // element (and a dead entry's dS is zero)
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if ((live_d >> (e4 + u)) & 1u) atomicAdd(dbrow + (int64_t)(q0 + e4 + u) * p.Sk, de[u]);
          } else if constexpr (DBIAS) {
#pragma unroll
            for (int u = 0; u < 4; ++u) atomicAdd(dbrow + (int64_t)(q0 + e4 + u) * p.Sk, de[u]);
          }
          dk[e4 / 2] = pack_half2(de[0], de[1]);
          dk[e4 / 2 + 1] = pack_half2(de[2], de[3]);
          pk[e4 / 2] = pack_half2(pv[cc * 32 + e4], pv[cc * 32 + e4 + 1]);
          pk[e4 / 2 + 1] = pack_half2(pv[cc * 32 + e4 + 2], pv[cc * 32 + e4 + 3]);
        }
        // this chunk's 32 columns were read above
        ptx::tmem_st16(buf + lane_off + wg * 64 + cc * 32, dk);
        ptx::tmem_st16(buf + lane_off + wg * 64 + cc * 32 + 16, pk);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar(kP2Full));
      ++t;
    }
    n_iters = t;
    epi_ok = ok && wait_bar(c, kAccFull, 0, 11);
  }

  // ------------------------------------------------- dK / dV epilogue --
  // Warpgroup 0 owns dK (scaled), warpgroup 1 dV; thread = key row.
  ptx::tc_fence_before();
  __syncthreads();
  const bool epi_thread = warp >= 4;
  const int ewg = (warp - 4) >> 2;
  const int ejl = (warp & 3) * 32 + lane;
  if (epi_thread) {
    ptx::tc_fence_after();
    const uint32_t t_acc = ewg == 0 ? t_dK : t_dV;
    const float mul = ewg == 0 ? p.scale : 1.f;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    float* grow = (ewg == 0 ? p.dk : p.dv) + ((sq.ok + n0 + ejl) * p.Hk + g) * D;
    const uint32_t srow = sbase + L::STAGE + (ewg * 128 + ejl) * L::kStageRow;
    if (epi_ok) {
#pragma unroll 1
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t v[32];
        if (n_iters > 0) {
          ptx::tmem_ld32(t_acc + lane_off + cc * 32, v);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float a0 = __uint_as_float(v[e]) * mul, a1 = __uint_as_float(v[e + 1]) * mul;
          const float a2 = __uint_as_float(v[e + 2]) * mul, a3 = __uint_as_float(v[e + 3]) * mul;
          ptx::st_shared_v4f(srow + (cc * 32 + e) * 4, a0, a1, a2, a3);
        }
      }
      if (n0 + ejl >= sq.lk) {
        // a padding row past Sk: nothing to write (the TMEM loads above are
        // warp-wide, so the row still took part in them)
      } else if (cs == 1) {
        // the whole row goes out as one copy-engine store
        ptx::fence_async_shared();
        ptx::bulk_store(grow, srow, D * 4);
        ptx::bulk_commit();
        ptx::bulk_wait_all();
      } else {
        // The cs head-split CTAs of this key tile add their partial rows into
        // dK / dV (zeroed by the pre-pass, which recorded which buffers) with
        // one TMA bulk reduction per row; the shared-memory row must stay
        // until the copy engine read it.
        const uint64_t* rec = reinterpret_cast<const uint64_t*>(&p.status->reserved[2]);
        if (rec[0] == reinterpret_cast<uint64_t>(p.dk) &&
            rec[1] == reinterpret_cast<uint64_t>(p.dv)) {
          ptx::fence_async_shared();
          ptx::bulk_reduce_add_f32(grow, srow, D * 4);
          ptx::bulk_commit();
          ptx::bulk_wait_all();
        } else if (ejl == 0) {
          report(p.status, ATTN_ERR_INVALID_ARG, 3);  // dk / dv not prepared by the pre-pass
        }
      }
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

// ===================================================== query-major CTA ====
template <int D, bool BIAS, bool RB>
__device__ __forceinline__ void q_cta(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                      const CUtensorMap* tmV, const CUtensorMap* tmdO,
                                      const CUtensorMap* tmB, const TcParams& p, uint8_t* smem,
                                      uint32_t sbase, int qi) {
  using L = SmemQ<D>;
  constexpr bool kMayBeRagged = RB || !BIAS;  // as in the key-major CTA (dbias is not used here)
  constexpr bool kTB = tma_bias<D, BIAS, RB>();  // bias tiles through TMA (whole tiles)
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nmt = p.Sqs / BM;
  const int bh = qi % (p.B * p.Hq);
  const int mt = nmt - 1 - qi / (p.B * p.Hq);  // later query tiles first (heavier when causal)
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int g = h / (p.Hq / p.Hk);
  const int m0 = mt * BM;
  Seq sq;
  if (!seq_of(p, b, &sq) || m0 >= sq.lq) return;  // a query tile past this sequence's queries

  Ctx c;
  c.bars = sbase + L::BAR;
  c.abort = reinterpret_cast<volatile int*>(smem + L::MISC + 4);
  c.status = p.status;
  // qQdoFull, qKFull0-2, qKEmpty0-2, qVFull0/1, qVEmpty0/1, qSFull0-2, qSFree, qdPFull,
  // qDsFull, qMma30-2, qAccFull, qBiasFull0/1, qBiasEmpty0/1
  const uint32_t counts[kQBars] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1,
                                   256, 1, 256, 1, 1, 1, 1, 1, 1, 256, 256};
  const uint32_t sQ = sbase + L::Q, sdO = sbase + L::dO;
  init_common(c, sbase + L::MISC, kQBars, counts, warp, [&] {
    // Q / dO of the query tile, and K / V of its first live key tile (stage 0)
    const int qrow = (b * p.Hq + h) * p.Sqs + m0;
    ptx::mbar_arrive_expect_tx(c.bar(qQdoFull), 2 * L::kTile);
#pragma unroll
    for (int hf = 0; hf < D / 64; ++hf) {
      ptx::tma_load_2d(sQ + hf * kSlab, tmQ, c.bar(qQdoFull), hf * 64, qrow);
      ptx::tma_load_2d(sdO + hf * kSlab, tmdO, c.bar(qQdoFull), hf * 64, qrow);
    }
    KTileIter it0(m0, sq);
    if (it0.next()) {
      const int krow = (b * p.Hk + g) * p.Sks + it0.nt * BN;
      ptx::mbar_arrive_expect_tx(c.bar(qKFull0), L::kTile);
      ptx::mbar_arrive_expect_tx(c.bar(qVFull0), L::kTile);
#pragma unroll
      for (int hf = 0; hf < D / 64; ++hf) {
        ptx::tma_load_2d(sbase + L::K + hf * kSlab, tmK, c.bar(qKFull0), hf * 64, krow);
        ptx::tma_load_2d(sbase + L::V + hf * kSlab, tmV, c.bar(qVFull0), hf * 64, krow);
      }
    }
  });
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::MISC);
  // TMEM: [0, D) dQ, then three 128-column buffers; tile t works in buffer
  // t % 3 (S, then dP over it, then dS over the front half of each
  // warpgroup's columns)
  const uint32_t t_dQ = tmem;
  const uint32_t t_buf0 = tmem + 128;
  bool epi_ok = false;
  int n_iters = 0;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      // (Q / dO and the first K / V went out with the barrier set-up)
      // K(t) rotates over kKS stages (released by dQ(t)), V(t) over two
      // (released by dP(t)), the bias (TMA bias path) over two (released by
      // the softmax's phase 1)
      KTileIter it(m0, sq);
      int t = 0;
      int k_issued[3] = {0, 0, 0}, v_issued[2] = {0, 0}, b_issued[2] = {0, 0};
      while (it.next()) {
        const int ks = t % L::kKS, ku = t / L::kKS;
        const int vs = t & 1, vu = t >> 1;
        const int krow = (b * p.Hk + g) * p.Sks + it.nt * BN;
        if (t > 0) {
          if (ku > 0 && !wait_bar(c, qKEmpty0 + ks, (ku - 1) & 1, 21)) break;
          const uint32_t kfull = c.bar(qKFull0 + ks);
          ptx::mbar_arrive_expect_tx(kfull, L::kTile);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf)
            ptx::tma_load_2d(sbase + L::K + ks * L::kTile + hf * kSlab, tmK, kfull, hf * 64, krow);
          if (vu > 0 && !wait_bar(c, qVEmpty0 + vs, (vu - 1) & 1, 20)) break;
          const uint32_t vfull = c.bar(qVFull0 + vs);
          ptx::mbar_arrive_expect_tx(vfull, L::kTile);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf)
            ptx::tma_load_2d(sbase + L::V + vs * L::kTile + hf * kSlab, tmV, vfull, hf * 64, krow);
        }
        k_issued[ks] = ku + 1;
        v_issued[vs] = vu + 1;
        if constexpr (kTB) {
          if (vu > 0 && !wait_bar(c, qBiasEmpty0 + vs, (vu - 1) & 1, 19)) break;
          const uint32_t bfull = c.bar(qBiasFull0 + vs);
          ptx::mbar_arrive_expect_tx(bfull, 4 * kSlab);
#pragma unroll
          for (int bx = 0; bx < 4; ++bx)
            ptx::tma_load_2d(sbase + L::BIAS + vs * 4 * kSlab + bx * kSlab, tmB, bfull,
                             it.nt * BN + 32 * bx, h * p.Sq + m0);
          b_issued[vs] = vu + 1;
        }
        ++t;
      }
      // no copy may still be landing in shared memory when the CTA ends
      drain_bar(c, qQdoFull, 0);
      for (int s = 0; s < L::kKS; ++s)
        if (k_issued[s] > 0) drain_bar(c, qKFull0 + s, (k_issued[s] - 1) & 1);
      for (int s = 0; s < 2; ++s) {
        if (v_issued[s] > 0) drain_bar(c, qVFull0 + s, (v_issued[s] - 1) & 1);
        if (b_issued[s] > 0) drain_bar(c, qBiasFull0 + s, (b_issued[s] - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t id_S = ptx::idesc_f16_f32(128, 128, false, false);
      constexpr uint32_t id_dQ = ptx::idesc_f16_f32(128, D, false, true);
      // operand descriptors, built once (K steps add their offsets)
      const uint64_t dQ = ptx::smem_desc_sw128(sQ, 16, 1024);
      const uint64_t ddO = ptx::smem_desc_sw128(sdO, 16, 1024);
      // stage 0 of K / V (stage st: + st kTile)
      const uint64_t dKk = ptx::smem_desc_sw128(sbase + L::K, 16, 1024);
      const uint64_t dVk = ptx::smem_desc_sw128(sbase + L::V, 16, 1024);
      const uint64_t dKmn = ptx::smem_desc_sw128(sbase + L::K, kSlab, 1024);
      auto issue_S = [&](int t) {  // MMA1' S = Q K^T into buffer t % 3 (K stage t % kKS)
        const uint64_t dk = ptx::desc_add(dKk, (t % L::kKS) * L::kTile);
        const uint32_t dst = t_buf0 + (t % 3) * 128;
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kSlab + (s & 3) * 32;
          ptx::mma_ss(dst, ptx::desc_add(dQ, off), ptx::desc_add(dk, off), id_S, s > 0);
        }
      };
      auto issue_dP = [&](int t) {  // MMA2' dP = dO V^T over S(t) in buffer t % 3
        const uint64_t dv = ptx::desc_add(dVk, (t & 1) * L::kTile);
        const uint32_t dst = t_buf0 + (t % 3) * 128;
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kSlab + (s & 3) * 32;
          ptx::mma_ss(dst, ptx::desc_add(ddO, off), ptx::desc_add(dv, off), id_S, s > 0);
        }
      };
      auto issue_dQ = [&](int t) {  // MMA3' dQ += dS K : A = dS (TMEM fp16 pairs), B = K MN-major
        const uint64_t dk = ptx::desc_add(dKmn, (t % L::kKS) * L::kTile);
        const uint32_t src = t_buf0 + (t % 3) * 128;
#pragma unroll
        for (int s = 0; s < BN / 16; ++s) {
          const uint32_t a_col = src + (s >> 2) * 64 + (s & 3) * 8;
          ptx::mma_ts(t_dQ, a_col, ptx::desc_add(dk, s * 2048), id_dQ,
                      (t > 0 || s > 0) ? 1u : 0u);
        }
      };
      // Per tile t (TMEM buffer t % 3): dP(t) over S(t) as soon as the softmax
      // has copied S(t) into its registers (qSFree); then S(t+1), which needs
      // its K stage and buffer (t+1) % 3, last read by dQ(t-2); then dQ(t)
      // once dS(t) is in TMEM. The softmax's exponentials of tile t overlap
      // dP(t), S(t+1) and dQ(t-1); S(t+1) is ready before the softmax
      // finishes tile t.
      bool ok = wait_bar(c, qQdoFull, 0, 22);
      int n_tiles = 0;  // tiles whose dQ MMAs were issued
      int n_dp = 0;     // tiles whose dP MMAs were issued
      KTileIter it(m0, sq);
      bool have = ok && it.next();
      if (have) {
        have = wait_bar(c, qKFull0, 0, 23);
        if (have) {
          ptx::tc_fence_after();
          issue_S(0);
          ptx::mma_commit(c.bar(qSFull0));
        }
      }
      int t = 0;
      while (have) {
        const int st = t & 1, bt = t % 3;
        if (!wait_bar(c, qSFree, t & 1, 24)) break;
        if (!wait_bar(c, qVFull0 + st, (t >> 1) & 1, 29)) break;
        ptx::tc_fence_after();
        issue_dP(t);
        ptx::mma_commit(c.bar(qdPFull));
        ptx::mma_commit(c.bar(qVEmpty0 + st));  // V(t) read by dP(t) only
        ++n_dp;
        const bool have1 = it.next();
        const int b1 = (t + 1) % 3;
        const int k1 = (t + 1) % L::kKS;                        // K stage of tile t + 1
        const uint32_t kpar = ((t + 1) / L::kKS) & 1;           // its fill for tile t + 1
        const uint32_t mpar = t >= 2 ? ((t - 2) / 3) & 1 : 0u;  // dQ(t-2) on qMma30 + b1
        if (have1) {
          if (t >= 2 && !wait_bar(c, qMma30 + b1, mpar, 25)) break;
          if (!wait_bar(c, qKFull0 + k1, kpar, 23)) break;
          ptx::tc_fence_after();
          issue_S(t + 1);
          ptx::mma_commit(c.bar(qSFull0 + b1));
        }
        if (!wait_bar(c, qDsFull, t & 1, 26)) break;
        ptx::tc_fence_after();
        issue_dQ(t);
        ptx::mma_commit(c.bar(qMma30 + bt));
        ptx::mma_commit(c.bar(qKEmpty0 + t % L::kKS));  // K(t) read by S(t) and dQ(t)
        ++n_tiles;
        if (!ok) break;
        have = have1;
        ++t;
      }
      ptx::mma_commit(c.bar(qAccFull));
      // the last dQ / K-V-stage commits: waited here (see the key-major CTA);
      // buffer b took the dQ commits of tiles b, b + 3, ..., stage s those of
      // tiles s, s + 2, ...
      for (int b3 = 0; b3 < 3; ++b3) {
        const int n_b = (n_tiles - b3 + 2) / 3;
        if (n_b > 0) drain_bar(c, qMma30 + b3, (n_b - 1) & 1);
      }
      for (int s2 = 0; s2 < L::kKS; ++s2) {
        const int n_s = (n_tiles + L::kKS - 1 - s2) / L::kKS;
        if (n_s > 0) drain_bar(c, qKEmpty0 + s2, (n_s - 1) & 1);
      }
      for (int s2 = 0; s2 < 2; ++s2) {  // dP commits: one per tile whose dP went out
        const int n_s = (n_dp + 1 - s2) >> 1;
        if (n_s > 0) drain_bar(c, qVEmpty0 + s2, (n_s - 1) & 1);
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax / dS groups --
    const int wg = (warp - 4) >> 2;                  // 0: keys 0-63, 1: keys 64-127
    const int lg = warp & 3;
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int il = lg * 32 + lane;                   // query row within the tile
    const int i = m0 + il;
    const bool row_in = i < sq.lq;                   // rows past the length: padding (not stored)
    const int ic = row_in ? i : sq.lq - 1;
    const int64_t row = ((int64_t)b * p.Hq + h) * p.Sq + ic;
    const float nl = row_in ? p.lse[row] * -kLog2e : 0.f;  // -inf rows: see the partial-tile mask
    const float dl = row_in ? p.delta[row] : 0.f;
    const float* brow = nullptr;
    if constexpr (BIAS && !kTB) brow = p.bias + ((int64_t)h * p.Sq + ic) * p.Sk;
    // TMA bias: this row's 128-byte rows of the four boxes (chunk c of the
    // row sits at chunk c ^ (il & 7))
    const uint32_t brow_s = L::BIAS + il * 128;
    KTileIter it(m0, sq);
    int t = 0;
    bool ok = true;
    while (it.next()) {
      if (!wait_bar(c, qSFull0 + t % 3, (t / 3) & 1, 27)) { ok = false; break; }
      ptx::tc_fence_after();
      const int n0 = it.nt * BN;
      const int kcap = sq.lk - n0;  // keys [0, kcap) of the tile exist
      int klo, khi, ksink;
      const bool partial = q_row_live<kMayBeRagged>(sq, m0, n0, i, &klo, &khi, &ksink);
      const uint32_t t_S = t_buf0 + (t % 3) * 128;  // this tile's TMEM buffer
      if constexpr (kTB) {
        if (!wait_bar(c, qBiasFull0 + (t & 1), (t >> 1) & 1, 30)) { ok = false; break; }
      }
      // phase 1: P from S (registers)
      float pv[64];
      {
        uint32_t sr[64];
        ptx::tmem_ld32(t_S + lane_off + wg * 64, sr);
        ptx::tmem_ld32(t_S + lane_off + wg * 64 + 32, sr + 32);
        ptx::tmem_wait_ld();
        ptx::tc_fence_before();
        ptx::mbar_arrive(c.bar(qSFree));  // S(t) is in registers: MMA2' may overwrite it
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int k0 = wg * 64 + cc * 32;  // first key of this chunk within the tile
          const uint32_t live = q_chunk_bits(klo, khi, ksink, k0);
#pragma unroll
          for (int e4 = 0; e4 < 32; e4 += 4) {
            float bv[4];
            if constexpr (BIAS && RB) {
              // keys past Sk read the last one (their P is zero); a bias row
              // of ragged length is not 16-byte aligned
#pragma unroll
              for (int u = 0; u < 4; ++u) bv[u] = __ldg(brow + n0 + imin(k0 + e4 + u, kcap - 1));
            } else if constexpr (kTB) {
              // keys k0 + e4 .. + 3: box k0 / 32, 16-byte chunk e4 / 4 of the row
              const float4 b4 = *reinterpret_cast<const float4*>(
                  smem + brow_s + (t & 1) * 4 * kSlab + (k0 >> 5) * kSlab +
                  ((((uint32_t)e4 >> 2) ^ ((uint32_t)il & 7u)) << 4));
              bv[0] = b4.x;
              bv[1] = b4.y;
              bv[2] = b4.z;
              bv[3] = b4.w;
            } else if constexpr (BIAS) {
              const float4 b4 = __ldg(reinterpret_cast<const float4*>(brow + n0 + k0 + e4));
              bv[0] = b4.x;
              bv[1] = b4.y;
              bv[2] = b4.z;
              bv[3] = b4.w;
            }
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              ptx::fma2(x[u], x[u + 1], __uint_as_float(sr[cc * 32 + e4 + u]),
                        __uint_as_float(sr[cc * 32 + e4 + u + 1]), p.scale_log2, p.scale_log2,
                        nl, nl);
              if constexpr (BIAS)
                ptx::fma2(x[u], x[u + 1], bv[u], bv[u + 1], kLog2e, kLog2e, x[u], x[u + 1]);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) pv[cc * 32 + e4 + u] = ptx::ex2(x[u]);
            if (partial) {  // warp-uniform: only tiles the mask cuts need the per-key test
#pragma unroll
              for (int u = 0; u < 4; ++u)
                if (!((live >> (e4 + u)) & 1u)) pv[cc * 32 + e4 + u] = 0.f;
            }
          }
        }
      }
      if constexpr (kTB) ptx::mbar_arrive(c.bar(qBiasEmpty0 + (t & 1)));  // bias stage read
      // phase 2: dS = P (dP - D), fp16 pairs over the (already read) front
      // half of this group's dP columns in the tile's buffer (A operand of dQ)
      if (!wait_bar(c, qdPFull, t & 1, 29)) { ok = false; break; }
      ptx::tc_fence_after();
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t dr[32];
        ptx::tmem_ld32(t_S + lane_off + wg * 64 + cc * 32, dr);
        ptx::tmem_wait_ld();
        uint32_t dk[16];
#pragma unroll
        for (int e4 = 0; e4 < 32; e4 += 4) {
          float de[4];
#pragma unroll
          for (int u = 0; u < 4; u += 2) {
            float t0, t1;
            ptx::sub2(t0, t1, __uint_as_float(dr[e4 + u]), __uint_as_float(dr[e4 + u + 1]), dl,
                      dl);
            ptx::mul2(de[u], de[u + 1], pv[cc * 32 + e4 + u], pv[cc * 32 + e4 + u + 1], t0, t1);
          }
          dk[e4 / 2] = pack_half2(de[0], de[1]);
          dk[e4 / 2 + 1] = pack_half2(de[2], de[3]);
        }
        ptx::tmem_st16(t_S + lane_off + wg * 64 + cc * 16, dk);
      }
      ptx::tmem_wait_st();
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar(qDsFull));
      ++t;
    }
    n_iters = t;
    epi_ok = ok && wait_bar(c, qAccFull, 0, 28);
    // ---------------------------------------------------- dQ epilogue --
    // thread = query row; warpgroup wg writes columns [wg D/2, wg D/2 + D/2)
    if (epi_ok) {
      ptx::tc_fence_after();
      // staged in the (idle) K / V stages, then one copy-engine store per half
      // row (rows past Sq are not stored)
      float* grow = p.dq + ((sq.oq + ic) * p.Hq + h) * D + wg * (D / 2);
      const uint32_t srow = sbase + L::STAGE + il * L::kStageRow + wg * (D / 2) * 4;
      uint32_t v[D / 2];
      if (n_iters > 0) {
#pragma unroll
        for (int cc = 0; cc < D / 64; ++cc)
          ptx::tmem_ld32(t_dQ + lane_off + wg * (D / 2) + cc * 32, v + cc * 32);
        ptx::tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < D / 2; ++e) v[e] = 0u;
      }
#pragma unroll
      for (int e = 0; e < D / 2; e += 4)
        ptx::st_shared_v4f(srow + e * 4, __uint_as_float(v[e]) * p.scale,
                           __uint_as_float(v[e + 1]) * p.scale, __uint_as_float(v[e + 2]) * p.scale,
                           __uint_as_float(v[e + 3]) * p.scale);
      if (row_in) {
        ptx::fence_async_shared();
        ptx::bulk_store(grow, srow, D / 2 * 4);
        ptx::bulk_commit();
        ptx::bulk_wait_all();
      }
    }
  }

  // ----------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (lane == 0) drain_bar(c, qAccFull, 0);
    __syncwarp();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ============================================ batch-inner query-major CTA ====
// Dense problems with a dbias output at D = 64 (whole tiles, fixed lengths,
// B <= 4): the query-major CTA of (query head h, query tile) takes every
// batch of that tile, batch innermost. For each live key tile it computes
// S, dP and dS of every batch (dQ of batch b accumulating in its own TMEM
// columns), sums dS over the batches in registers and stores that sum, the
// tile of dbias = sum over b of dS, once: no atomics, no zero-filled dbias,
// and a fixed summation order. The key-major CTAs then run without dbias.
//
// Shared memory: two sub-tile stages (Q, dO, K, V of one (key tile, batch))
// and one bias tile (shared by the batches of a key tile). TMEM: dQ of
// batch b in columns [b D, b D + D), two 128-column S / dP / dS buffers from
// column 256. Sub-tile number T = key tile index x B + batch.
template <int D>
struct SmemQB {
  static constexpr int kTile = (D / 64) * kSlab;
  static constexpr int kStage = 4 * kTile;       // Q, dO, K, V of one sub-tile
  static constexpr int ST = 0;                   // two stages
  static constexpr int BIAS = ST + 2 * kStage;   // [128 queries][128 keys] fp32, four boxes of 32 keys
  static constexpr int BAR = BIAS + 4 * kSlab;   // mbarriers (up to 32)
  static constexpr int MISC = BAR + 256;         // TMEM base, abort flag
  static constexpr int TOTAL = MISC + 16;
};
static_assert(SmemQB<64>::TOTAL <= 232448, "shared memory per CTA");

// barrier indices, batch-inner query-major CTA: stage s full / released (by
// dQ of its sub-tile), bias tile full / read (phase 1 of the key tile's last
// batch, 256 arrivals), S of sub-tile T in buffer T & 1, S read, dP ready,
// dS written (256), dQ of sub-tile T done (buffer T & 1 free), all dQ done.
enum BarQB { bStFull0 = 0, bStEmpty0 = 2, bBiasFull = 4, bBiasEmpty = 5, bSFull0 = 6, bSFree = 8,
             bdPFull = 9, bDsFull = 10, bMma0 = 11, bAccFull = 13, kQBBars = 14 };

template <int D, bool BIAS>
__device__ __forceinline__ void qb_cta(const CUtensorMap* tmQ, const CUtensorMap* tmK,
                                       const CUtensorMap* tmV, const CUtensorMap* tmdO,
                                       const CUtensorMap* tmB, const TcParams& p, uint8_t* smem,
                                       uint32_t sbase, int qi) {
  using L = SmemQB<D>;
  static_assert(D == 64, "batch-inner CTA: dQ of four batches and two buffers fill TMEM at D = 64");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nmt = p.Sqs / BM;
  const int h = qi % p.Hq;
  const int m0 = (nmt - 1 - qi / p.Hq) * BM;
  const int g = h / (p.Hq / p.Hk);
  const int B = p.B;
  Seq sq;
  if (!seq_of(p, 0, &sq)) return;  // fixed lengths: every batch has the same sequence view

  Ctx c;
  c.bars = sbase + L::BAR;
  c.abort = reinterpret_cast<volatile int*>(smem + L::MISC + 4);
  c.status = p.status;
  // bStFull0/1, bStEmpty0/1, bBiasFull, bBiasEmpty, bSFull0/1, bSFree, bdPFull, bDsFull,
  // bMma0/1, bAccFull
  const uint32_t counts[kQBBars] = {1, 1, 1, 1, 1, 256, 1, 1, 256, 1, 256, 1, 1, 1};
  init_common(c, sbase + L::MISC, kQBBars, counts, warp, [] {});
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::MISC);
  const uint32_t t_dQ = tmem;          // batch b: [b D, b D + D)
  const uint32_t t_buf0 = tmem + 256;  // sub-tile T: t_buf0 + (T & 1) 128
  int n_live = 0;                      // live key tiles of this query tile
  {
    KTileIter it(m0, sq);
    while (it.next()) ++n_live;
  }
  const int n_sub = n_live * B;
  bool epi_ok = false;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer --
    if (lane == 0) {
      KTileIter it(m0, sq);
      int t = 0;
      int st_issued[2] = {0, 0};
      bool go = true;
      while (go && it.next()) {
        const int n0 = it.nt * BN;
        // the key tile's bias, once the previous key tile's batches read theirs
        if (t > 0 && !(go = wait_bar(c, bBiasEmpty, (t - 1) & 1, 50))) break;
        ptx::mbar_arrive_expect_tx(c.bar(bBiasFull), 4 * kSlab);
#pragma unroll
        for (int bx = 0; bx < 4; ++bx)
          ptx::tma_load_2d(sbase + L::BIAS + bx * kSlab, tmB, c.bar(bBiasFull), n0 + 32 * bx,
                           h * p.Sq + m0);
        for (int b = 0; b < B; ++b) {
          const int T = t * B + b;
          const int s = T & 1, u = T >> 1;
          if (u > 0 && !(go = wait_bar(c, bStEmpty0 + s, (u - 1) & 1, 51))) break;
          const uint32_t full = c.bar(bStFull0 + s);
          const uint32_t st = sbase + L::ST + s * L::kStage;
          const int qrow = (b * p.Hq + h) * p.Sqs + m0;
          const int krow = (b * p.Hk + g) * p.Sks + n0;
          ptx::mbar_arrive_expect_tx(full, L::kStage);
#pragma unroll
          for (int hf = 0; hf < D / 64; ++hf) {
            ptx::tma_load_2d(st + hf * kSlab, tmQ, full, hf * 64, qrow);
            ptx::tma_load_2d(st + L::kTile + hf * kSlab, tmdO, full, hf * 64, qrow);
            ptx::tma_load_2d(st + 2 * L::kTile + hf * kSlab, tmK, full, hf * 64, krow);
            ptx::tma_load_2d(st + 3 * L::kTile + hf * kSlab, tmV, full, hf * 64, krow);
          }
          st_issued[s] = u + 1;
        }
        ++t;
      }
      // no copy may still be landing in shared memory when the CTA ends
      if (t > 0) drain_bar(c, bBiasFull, (t - 1) & 1);
      for (int s = 0; s < 2; ++s)
        if (st_issued[s] > 0) drain_bar(c, bStFull0 + s, (st_issued[s] - 1) & 1);
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t id_S = ptx::idesc_f16_f32(128, 128, false, false);
      constexpr uint32_t id_dQ = ptx::idesc_f16_f32(128, D, false, true);
      // stage 0 views (stage s: + s kStage): Q, dO, K K-major; K MN-major
      const uint64_t dQs = ptx::smem_desc_sw128(sbase + L::ST, 16, 1024);
      const uint64_t ddOs = ptx::smem_desc_sw128(sbase + L::ST + L::kTile, 16, 1024);
      const uint64_t dKs = ptx::smem_desc_sw128(sbase + L::ST + 2 * L::kTile, 16, 1024);
      const uint64_t dVs = ptx::smem_desc_sw128(sbase + L::ST + 3 * L::kTile, 16, 1024);
      const uint64_t dKmn = ptx::smem_desc_sw128(sbase + L::ST + 2 * L::kTile, kSlab, 1024);
      auto issue_S = [&](int T) {  // S = Q K^T of sub-tile T into buffer T & 1
        const uint32_t so = (T & 1) * L::kStage;
        const uint32_t dst = t_buf0 + (T & 1) * 128;
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kSlab + (s & 3) * 32;
          ptx::mma_ss(dst, ptx::desc_add(dQs, so + off), ptx::desc_add(dKs, so + off), id_S, s > 0);
        }
      };
      auto issue_dP = [&](int T) {  // dP = dO V^T over S(T)
        const uint32_t so = (T & 1) * L::kStage;
        const uint32_t dst = t_buf0 + (T & 1) * 128;
#pragma unroll
        for (int s = 0; s < D / 16; ++s) {
          const uint32_t off = (s >> 2) * kSlab + (s & 3) * 32;
          ptx::mma_ss(dst, ptx::desc_add(ddOs, so + off), ptx::desc_add(dVs, so + off), id_S, s > 0);
        }
      };
      // dQ_b += dS K (A = dS, fp16 pairs over the front half of each
      // warpgroup's columns; B = K MN-major); the batch's first key tile
      // (first) overwrites its accumulator
      auto issue_dQ = [&](int T, int b, bool first) {
        const uint64_t dk = ptx::desc_add(dKmn, (T & 1) * L::kStage);
        const uint32_t src = t_buf0 + (T & 1) * 128;
#pragma unroll
        for (int s = 0; s < BN / 16; ++s) {
          const uint32_t a_col = src + (s >> 2) * 64 + (s & 3) * 8;
          ptx::mma_ts(t_dQ + b * D, a_col, ptx::desc_add(dk, s * 2048), id_dQ,
                      (!first || s > 0) ? 1u : 0u);
        }
      };
      // Per sub-tile T (buffer T & 1): dP(T) once the softmax has copied S(T)
      // out; S(T+1) once dQ(T-1) has read its buffer and its stage landed;
      // dQ(T) once dS(T) is in TMEM.
      int n_done = 0;  // sub-tiles whose dQ went out
      bool ok = n_sub == 0 || wait_bar(c, bStFull0, 0, 52);
      if (ok && n_sub > 0) {
        ptx::tc_fence_after();
        issue_S(0);
        ptx::mma_commit(c.bar(bSFull0));
      }
      for (int T = 0; ok && T < n_sub; ++T) {
        ok = wait_bar(c, bSFree, T & 1, 53);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_dP(T);
        ptx::mma_commit(c.bar(bdPFull));
        if (T + 1 < n_sub) {
          const int n1 = (T + 1) & 1;
          ok = (T < 1 || wait_bar(c, bMma0 + n1, ((T - 1) >> 1) & 1, 54)) &&
               wait_bar(c, bStFull0 + n1, ((T + 1) >> 1) & 1, 52);
          if (!ok) break;
          ptx::tc_fence_after();
          issue_S(T + 1);
          ptx::mma_commit(c.bar(bSFull0 + n1));
        }
        ok = wait_bar(c, bDsFull, T & 1, 55);
        if (!ok) break;
        ptx::tc_fence_after();
        issue_dQ(T, T % B, T < B);
        ptx::mma_commit(c.bar(bMma0 + (T & 1)));
        ptx::mma_commit(c.bar(bStEmpty0 + (T & 1)));  // Q / K read by S and dQ, dO / V by dP
        ++n_done;
      }
      ptx::mma_commit(c.bar(bAccFull));
      // the last buffer / stage releases, waited here (see the key-major CTA)
      for (int bb = 0; bb < 2; ++bb) {
        const int n_b = (n_done + 1 - bb) >> 1;
        if (n_b > 0) {
          drain_bar(c, bMma0 + bb, (n_b - 1) & 1);
          drain_bar(c, bStEmpty0 + bb, (n_b - 1) & 1);
        }
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------ softmax / dS groups --
    const int wg = (warp - 4) >> 2;  // 0: keys 0-63, 1: keys 64-127
    const int lg = warp & 3;
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int il = lg * 32 + lane;   // query row within the tile
    const int i = m0 + il;
    // the bias tile's row il: chunk c of a box row sits at chunk c ^ (il & 7)
    const uint32_t brow_s = L::BIAS + il * 128;
    float* dbrow = p.dbias + ((int64_t)h * p.Sq + i) * p.Sk + wg * 64;
    KTileIter it(m0, sq);
    int t = 0;
    bool ok = true;
    while (ok && it.next()) {
      const int n0 = it.nt * BN;
      int klo, khi, ksink;
      const bool partial = q_row_live<false>(sq, m0, n0, i, &klo, &khi, &ksink);
      if (!wait_bar(c, bBiasFull, t & 1, 56)) { ok = false; break; }
      float acc[64];  // sum over the batches of dS for keys n0 + wg 64 + [0, 64)
#pragma unroll
      for (int e = 0; e < 64; ++e) acc[e] = 0.f;
      for (int b = 0; b < B; ++b) {
        const int T = t * B + b;
        const uint32_t t_S = t_buf0 + (T & 1) * 128;
        // -LSE log2e and delta of this row in batch b (fixed lengths: every
        // row exists), read before the wait for S
        const int64_t row = ((int64_t)b * p.Hq + h) * p.Sq + i;
        const float nlb = __ldg(p.lse + row) * -kLog2e;
        const float dlb = __ldg(p.delta + row);
        if (!wait_bar(c, bSFull0 + (T & 1), (T >> 1) & 1, 57)) { ok = false; break; }
        ptx::tc_fence_after();
        // phase 1: P as fp16 pairs (the A operand precision of dQ)
        uint32_t pk[32];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t sr[32];
          ptx::tmem_ld32(t_S + lane_off + wg * 64 + cc * 32, sr);
          ptx::tmem_wait_ld();
          if (cc == 1) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(c.bar(bSFree));  // S(T) is in registers: dP may overwrite it
          }
          const int k0 = wg * 64 + cc * 32;
          const uint32_t live = q_chunk_bits(klo, khi, ksink, k0);
#pragma unroll
          for (int e4 = 0; e4 < 32; e4 += 4) {
            float bv[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (BIAS) {
              const float4 b4 = *reinterpret_cast<const float4*>(
                  smem + brow_s + (k0 >> 5) * kSlab +
                  ((((uint32_t)e4 >> 2) ^ ((uint32_t)il & 7u)) << 4));
              bv[0] = b4.x;
              bv[1] = b4.y;
              bv[2] = b4.z;
              bv[3] = b4.w;
            }
            float x[4];
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
              ptx::fma2(x[u], x[u + 1], __uint_as_float(sr[e4 + u]), __uint_as_float(sr[e4 + u + 1]),
                        p.scale_log2, p.scale_log2, nlb, nlb);
              if constexpr (BIAS)
                ptx::fma2(x[u], x[u + 1], bv[u], bv[u + 1], kLog2e, kLog2e, x[u], x[u + 1]);
            }
            float pv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) pv[u] = ptx::ex2(x[u]);
            if (partial) {  // warp-uniform: only tiles the mask cuts need the per-key test
#pragma unroll
              for (int u = 0; u < 4; ++u)
                if (!((live >> (e4 + u)) & 1u)) pv[u] = 0.f;
            }
            pk[cc * 16 + e4 / 2] = pack_half2(pv[0], pv[1]);
            pk[cc * 16 + e4 / 2 + 1] = pack_half2(pv[2], pv[3]);
          }
        }
        if (b == B - 1) ptx::mbar_arrive(c.bar(bBiasEmpty));  // the key tile's bias is read
        // phase 2: dS = P (dP - D) as fp16 pairs over the front half of this
        // group's dP columns (A operand of dQ), and into the batch sum
        if (!wait_bar(c, bdPFull, T & 1, 58)) { ok = false; break; }
        ptx::tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t dr[32];
          ptx::tmem_ld32(t_S + lane_off + wg * 64 + cc * 32, dr);
          ptx::tmem_wait_ld();
          uint32_t dk[16];
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            const float2 pf = __half22float2(*reinterpret_cast<const __half2*>(&pk[cc * 16 + e2]));
            float t0, t1, d0, d1;
            ptx::sub2(t0, t1, __uint_as_float(dr[2 * e2]), __uint_as_float(dr[2 * e2 + 1]), dlb,
                      dlb);
            ptx::mul2(d0, d1, pf.x, pf.y, t0, t1);
            acc[cc * 32 + 2 * e2] += d0;
            acc[cc * 32 + 2 * e2 + 1] += d1;
            dk[e2] = pack_half2(d0, d1);
          }
          ptx::tmem_st16(t_S + lane_off + wg * 64 + cc * 16, dk);
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(c.bar(bDsFull));
      }
      if (!ok) break;
      // this key tile's dbias: row i, keys n0 + wg 64 + [0, 64), the batch
      // sum in batch order (dead entries have dS = 0)
#pragma unroll
      for (int e = 0; e < 64; e += 8) put8(dbrow + n0 + e, acc + e);
      ++t;
    }
    epi_ok = ok && wait_bar(c, bAccFull, 0, 59);
    // ---------------------------------------------------- dQ epilogue --
    // batch b: row i, columns [wg D/2, wg D/2 + D/2) of dQ_b
    if (epi_ok) {
      ptx::tc_fence_after();
      for (int b = 0; b < B; ++b) {
        uint32_t v[D / 2];
        if (n_sub > 0) {
#pragma unroll
          for (int cc = 0; cc < D / 64; ++cc)
            ptx::tmem_ld32(t_dQ + b * D + lane_off + wg * (D / 2) + cc * 32, v + cc * 32);
          ptx::tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < D / 2; ++e) v[e] = 0u;
        }
        float* grow = p.dq + (((int64_t)b * p.Sq + i) * p.Hq + h) * D + wg * (D / 2);
#pragma unroll
        for (int e = 0; e < D / 2; e += 8) {
          float o8[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) o8[u] = __uint_as_float(v[e + u]) * p.scale;
          put8(grow + e, o8);
        }
      }
    }
  }

  // ----------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (lane == 0) drain_bar(c, bAccFull, 0);
    __syncwarp();
    ptx::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool BIAS, bool DBIAS, bool RB, bool QB>
__global__ void __launch_bounds__(kThreads, 1)
attn_bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                   const __grid_constant__ CUtensorMap tmB, const TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  // 1 KiB alignment of the 128B-swizzle atoms (uniform over the grid)
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report(p.status, ATTN_ERR_UNSUPPORTED, 1);
    return;
  }
  if (threadIdx.x == 0) {
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmK);
    ptx::prefetch_tmap(&tmV);
    ptx::prefetch_tmap(&tmdO);
    if constexpr (tma_bias<D, BIAS, RB>()) ptx::prefetch_tmap(&tmB);
  }
  // everything below reads what the pre-pass wrote (launched as its
  // programmatic dependent, this grid may start before the pre-pass ends)
  ptx::grid_dependency_wait();
  if (blockIdx.x == 0) {
    // fp16 overflow found while staging the operands: OR of the pre-pass's
    // per-block flag slots
    const int nslots = min(max(p.status->reserved[1], 0), kPreMaxBlocks);
    const int32_t* slots = reinterpret_cast<const int32_t*>(p.status + 1);
    int bits = 0;
    for (int i = threadIdx.x; i < nslots; i += blockDim.x) bits |= slots[i];
    bits = __reduce_or_sync(0xffffffffu, bits);
    if (bits && (threadIdx.x & 31) == 0) report(p.status, ATTN_ERR_RANGE, bits);
  }
  if constexpr (QB) {
    // batch-inner query-major CTAs first (the longest), then key-major ones
    // without dbias
    if ((int)blockIdx.x < p.qb_ctas)
      qb_cta<D, BIAS>(&tmQ, &tmK, &tmV, &tmdO, &tmB, p, smem, sbase, (int)blockIdx.x);
    else
      kv_cta<D, BIAS, false, RB>(&tmQ, &tmK, &tmV, &tmdO, &tmB, p, smem, sbase,
                                 (int)blockIdx.x - p.qb_ctas);
  } else if ((int)blockIdx.x < p.kv_ctas) {
    kv_cta<D, BIAS, DBIAS, RB>(&tmQ, &tmK, &tmV, &tmdO, &tmB, p, smem, sbase, (int)blockIdx.x);
  } else {
    const int qi = (int)blockIdx.x - p.kv_ctas;
    q_cta<D, BIAS, RB>(&tmQ, &tmK, &tmV, &tmdO, &tmB, p, smem, sbase, qi);
  }
}

// ------------------------------------------------------------ mask probe --
// The per-element live sets the two kinds of CTA compute for one sequence,
// through the same tile walks (QTileIter / KTileIter) and row predicates
// (kv_row_live / q_row_live and their chunk bits) as the backward kernel.
// Blocks [0, nkt) take the key-major view (thread = key row of a key tile)
// and add 1 to kv_live[i][j] for every entry they treat as live; blocks
// [nkt, nkt + nqt) take the query-major view (thread = query row) and add 1
// to q_live[i][j]. A live entry outside [0, lq) x [0, lk) (key-major), or at
// a key past lk (query-major), is counted in *outside instead. A tile the
// walk visited twice shows up as 2.
template <bool kMayBeRagged>
__global__ void __launch_bounds__(128)
mask_probe_kernel(const Seq s, int nkt, uint8_t* kv_live, uint8_t* q_live, int* outside) {
  const int t = (int)threadIdx.x;
  if ((int)blockIdx.x < nkt) {
    const int n0 = (int)blockIdx.x * BN;
    const int j = n0 + t;
    QTileIter it(1, n0, s);
    while (it.next()) {
      const int m0 = it.mt * BM;
      int qlo, qhi;
      const bool partial = kv_row_live<kMayBeRagged>(s, m0, n0, j, &qlo, &qhi);
      for (int q0 = 0; q0 < BM; q0 += 32) {
        const uint32_t live = partial ? kv_chunk_bits(qlo, qhi, q0) : 0xffffffffu;
        for (int u = 0; u < 32; ++u) {
          if (!((live >> u) & 1u)) continue;
          const int i = m0 + q0 + u;
          if (i >= s.lq || j >= s.lk) atomicAdd(outside, 1);
          else kv_live[(int64_t)i * s.lk + j] += 1;
        }
      }
    }
  } else {
    const int m0 = ((int)blockIdx.x - nkt) * BM;
    const int i = m0 + t;
    if (i >= s.lq) return;  // padding rows: not stored, dS zero (see q_row_live)
    KTileIter it(m0, s);
    while (it.next()) {
      const int n0 = it.nt * BN;
      int klo, khi, ksink;
      const bool partial = q_row_live<kMayBeRagged>(s, m0, n0, i, &klo, &khi, &ksink);
      for (int k0 = 0; k0 < BN; k0 += 32) {
        const uint32_t live = partial ? q_chunk_bits(klo, khi, ksink, k0) : 0xffffffffu;
        for (int u = 0; u < 32; ++u) {
          if (!((live >> u) & 1u)) continue;
          const int j = n0 + k0 + u;
          if (j >= s.lk) atomicAdd(outside, 1);
          else q_live[(int64_t)i * s.lk + j] += 1;
        }
      }
    }
  }
}

// ------------------------------------------------------------------ host --

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

// Zeros over n fp32 values (n a multiple of 4, p 16-byte aligned): dbias
// entries of tiles the mask leaves dead (batch-inner dbias mode, which stores
// only the tiles it visits), and the gradients of an empty problem.
__global__ void zero_fill_kernel(float* p, int64_t n) {
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n / 4;
       i += (int64_t)gridDim.x * blockDim.x)
    reinterpret_cast<float4*>(p)[i] = z;
}

// The kernel's tensor maps: fp16 staged q, k, v, dO, and the fp32 bias (TMA
// bias path only; a copy of q otherwise, never read).
struct TcMaps {
  CUtensorMap q, k, v, dO, bias;
};

// Row-major [rows][cols] fp32 bias (rows = heads x queries), boxes of 128
// rows x 32 columns (128 bytes), 128B swizzle: the tiles the TMA bias path
// loads (cols a multiple of 4, so that rows are 16-byte aligned).
bool make_bias_map(CUtensorMap* m, const float* base, uint64_t rows, int cols) {
  EncodeFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * sizeof(float)};
  cuuint32_t box[2] = {32, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, bool BIAS, bool DBIAS, bool RB, bool QB = false>
cudaError_t launch_variant(const TcMaps& m, const TcParams& p, int grid, cudaStream_t stream) {
  auto kern = attn_bwd_tc_kernel<D, BIAS, DBIAS, RB, QB>;
  int smem = smem_total<D>();
  if constexpr (QB) smem = smem > SmemQB<D>::TOTAL ? smem : SmemQB<D>::TOTAL;
  static bool configured = false;  // attribute set once per process and variant
  if (!configured) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  return launch_dependent(kern, dim3(grid), dim3(kThreads), (size_t)smem, stream, m.q, m.k, m.v,
                          m.dO, m.bias, p);
}

template <int D>
cudaError_t launch_d(const TcMaps& m, const TcParams& p, int grid, cudaStream_t stream) {
  if constexpr (D == 64) {
    if (p.qb_ctas > 0) {
      if (p.bias) return launch_variant<D, true, true, false, true>(m, p, grid, stream);
      return launch_variant<D, false, true, false, true>(m, p, grid, stream);
    }
  }
  // without bias and dbias, ragged lengths need no separate instantiation
  if (p.ragged) {
    if (p.bias && p.dbias) return launch_variant<D, true, true, true>(m, p, grid, stream);
    if (p.bias) return launch_variant<D, true, false, true>(m, p, grid, stream);
    if (p.dbias) return launch_variant<D, false, true, true>(m, p, grid, stream);
  }
  if (p.bias && p.dbias) return launch_variant<D, true, true, false>(m, p, grid, stream);
  if (p.bias) return launch_variant<D, true, false, false>(m, p, grid, stream);
  if (p.dbias) return launch_variant<D, false, true, false>(m, p, grid, stream);
  return launch_variant<D, false, false, false>(m, p, grid, stream);
}

// Query heads per KV head are split over cs key-major CTAs. Every CTA pays a
// fixed cost (K / V load, TMEM set-up, the dK / dV epilogue) and a split adds
// a bulk reduction of its partial rows, so the split is the smallest divisor
// of the group size that still gives about three quarters of a wave of
// key-major CTAs (measured: 64 key tiles on 152 SMs run best with 2, 512 with 1).
int head_split(int ratio, int key_tiles, int sms) {
  for (int c = 1; c < ratio; ++c)
    if (ratio % c == 0 && (int64_t)key_tiles * c * 4 >= (int64_t)sms * 3) return c;
  return ratio;
}

int sm_count() {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

}  // namespace

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

// The key tiles that need less splitting: with the uniform split cs, a
// key-major CTA takes at most (r / cs) max_n L_n query tiles (L_n = live query
// tiles of key tile n, r = query heads per KV head). The trailing key tiles
// whose (r / c) L_n stays within that bound can run as c < cs CTAs each (no
// longer than the longest CTA, fewer fixed costs); of the divisors c of cs,
// the one that removes the most CTAs is taken. Lengths of a variable-length
// batch are taken at their maxima (a schedule choice only).
static void tail_split(const Problem& pr, int cs, int* n_split, int* cs_lo) {
  const int nkt = tc_rows(pr.Sk) / BN;
  *n_split = nkt;
  *cs_lo = cs;
  if (cs == 1 || nkt == 0) return;
  const int r = pr.Hq / pr.Hk;
  std::vector<int> live(nkt);
  int lmax = 0;
  for (int n = 0; n < nkt; ++n) {
    int lo, hi;
    live_query_tiles(pr.mask, pr.Sq, pr.Sk, BM, BN, n * BN, &lo, &hi);
    live[n] = hi >= lo ? hi - lo + 1 : 0;
    lmax = std::max(lmax, live[n]);
  }
  const int64_t cap = (int64_t)(r / cs) * lmax;
  int64_t best = 0;
  for (int c = 1; c < cs; ++c) {
    if (cs % c != 0) continue;
    int ns = nkt;
    while (ns > 0 && (int64_t)(r / c) * live[ns - 1] <= cap) --ns;
    const int64_t saved = (int64_t)(nkt - ns) * (cs - c);
    if (saved > best) {
      best = saved;
      *n_split = ns;
      *cs_lo = c;
    }
  }
}

int tc_head_split(const Problem& p) {
  // deterministic: one CTA per key tile writes dK / dV (no partial sums added
  // in arrival order)
  if (p.deterministic) return 1;
  return head_split(p.Hq / p.Hk, p.B * p.Hk * (tc_rows(p.Sk) / BN), sm_count());
}

bool tc_dbias_in_q(const Problem& p) {
  // dQ of B batches (B D columns) and two S / dP buffers fit TMEM at D = 64;
  // whole tiles and fixed lengths (the CTA's sub-tiles share one sequence view)
  return tc_supported(p) && !p.cuda_cores && p.D == 64 && p.B <= 4 && !p.varlen &&
         p.Sq % BM == 0 && p.Sk % BN == 0;
}

// A shape decision only: a driver without cuTensorMapEncodeTiled makes the
// launch fail (ATTN_ERR_CUDA) rather than move the problem to other kernels.
bool tc_supported(const Problem& p) {
  return !p.sparse && (p.D == 64 || p.D == 128) && p.B > 0 && p.Sq >= 0 && p.Sk >= 0;
}

cudaError_t launch_mask_probe(const MaskSpec& m, int Sq, int Sk, bool aligned_variant,
                              uint8_t* kv_live, uint8_t* q_live, int32_t* outside,
                              cudaStream_t stream) {
  Seq s;
  s.lq = Sq;
  s.lk = Sk;
  s.oq = 0;
  s.ok = 0;
  s.mask = m;
  const int nkt = tc_rows(Sk) / BN, nqt = tc_rows(Sq) / BM;
  if (aligned_variant)
    mask_probe_kernel<false><<<nkt + nqt, 128, 0, stream>>>(s, nkt, kv_live, q_live, outside);
  else
    mask_probe_kernel<true><<<nkt + nqt, 128, 0, stream>>>(s, nkt, kv_live, q_live, outside);
  return cudaGetLastError();
}

cudaError_t launch_bwd_tc(const Problem& pr, const __half* q16, const __half* k16,
                          const __half* v16, const __half* do16, const float* lse,
                          const float* delta, const float* bias, float* dq, float* dk,
                          float* dv, float* dbias, DevStatus* st, cudaStream_t stream) {
  if (pr.Sq == 0 || pr.Sk == 0) {
    // nothing to differentiate: the gradients are zero (dbias has no entry)
    const int64_t rq = pr.varlen ? pr.total_q : (int64_t)pr.B * pr.Sq;
    const int64_t rk = pr.varlen ? pr.total_k : (int64_t)pr.B * pr.Sk;
    const int64_t n[3] = {rq * pr.Hq * pr.D, rk * pr.Hk * pr.D, rk * pr.Hk * pr.D};
    float* out[3] = {dq, dk, dv};
    for (int i = 0; i < 3; ++i) {
      if (n[i] == 0) continue;
      zero_fill_kernel<<<(unsigned)std::min<int64_t>((n[i] / 4 + 255) / 256, 4096), 256, 0,
                         stream>>>(out[i], n[i]);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  CUtensorMap mq, mk, mv, mdo;
  const uint64_t qrows = (uint64_t)pr.B * pr.Hq * tc_rows(pr.Sq);
  const uint64_t krows = (uint64_t)pr.B * pr.Hk * tc_rows(pr.Sk);
  if (!make_map(&mq, q16, qrows, pr.D) || !make_map(&mk, k16, krows, pr.D) ||
      !make_map(&mv, v16, krows, pr.D) || !make_map(&mdo, do16, qrows, pr.D))
    return cudaErrorInvalidValue;
  TcParams p;
  p.B = pr.B;
  p.Hq = pr.Hq;
  p.Hk = pr.Hk;
  p.Sq = pr.Sq;
  p.Sk = pr.Sk;
  p.Sqs = tc_rows(pr.Sq);
  p.Sks = tc_rows(pr.Sk);
  p.cu_q = pr.varlen ? pr.cu_q : nullptr;
  p.cu_k = pr.varlen ? pr.cu_k : nullptr;
  p.total_q = pr.total_q;
  p.total_k = pr.total_k;
  p.br = pr.br ? 1 : 0;
  p.ragged = (p.Sqs != p.Sq || p.Sks != p.Sk || pr.varlen) ? 1 : 0;
  p.cs = tc_head_split(pr);
  tail_split(pr, p.cs, &p.n_split, &p.cs_lo);
  p.kv_ctas = pr.B * pr.Hk * (p.n_split * p.cs + (p.Sks / BN - p.n_split) * p.cs_lo);
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
  p.dbias_bstride = pr.dbias_bstride;
  p.status = st;
  // dbias in batch-inner query-major CTAs (one per query head and query
  // tile) when it applies; then the tiles the mask leaves dead are never
  // visited, and their dbias entries are zeroed first
  const bool qb = dbias != nullptr && tc_dbias_in_q(pr);
  p.qb_ctas = qb ? pr.Hq * (p.Sqs / BM) : 0;
  const int q_ctas = qb ? p.qb_ctas : pr.B * pr.Hq * (p.Sqs / BM);
  const int grid = p.kv_ctas + q_ctas;
  if (qb) {
    bool any_dead = false;
    for (int n0 = 0; n0 < p.Sks && !any_dead; n0 += BN) {
      int lo, hi;
      live_query_tiles(pr.mask, pr.Sq, pr.Sk, BM, BN, n0, &lo, &hi);
      any_dead = lo != 0 || hi != p.Sqs / BM - 1;
    }
    if (any_dead) {
      const int64_t n = (int64_t)pr.Hq * pr.Sq * pr.Sk;
      zero_fill_kernel<<<std::min<int64_t>((n / 4 + 255) / 256, 4096), 256, 0, stream>>>(dbias, n);
      const cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  TcMaps maps;
  maps.q = mq;
  maps.k = mk;
  maps.v = mv;
  maps.dO = mdo;
  maps.bias = mq;
  if (pr.D == 64 && bias != nullptr && !p.ragged &&
      !make_bias_map(&maps.bias, bias, (uint64_t)pr.Hq * pr.Sq, pr.Sk))
    return cudaErrorInvalidValue;
  if (pr.D == 64) return launch_d<64>(maps, p, grid, stream);
  return launch_d<128>(maps, p, grid, stream);
}

}  // namespace attn
