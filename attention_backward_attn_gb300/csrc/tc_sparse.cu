// Tensor-core (tcgen05 / TMEM) backward of the selected-KV sparse attention
// with one shared latent KV per KV head (Ascend "sparse_flash_mla_grad",
// formula section, phases 1-3):
//   selKv(i) = original rows in the window of query i, then the compressed
//              rows listed in topk[i] (-1 = empty slot);  K = V = selKv;
//   P = exp(scale Q selKv^T - LSE) (the given LSE);  dP = dO selKv^T;
//   dS = P (dP - D) with D = rowsum(dO * O);  dQ = scale dS selKv;
//   dKV = scale dS^T Q + P^T dO, added into the rows it was gathered from.
//
// One work item per (query token i, KV head g); a persistent CTA per SM takes
// items in a fixed stride. The r = 64 query heads of the KV
// head and their 64 dO rows are stacked into one 128-row operand
// X = [Q_i ; dO_i] (fp16, eight 128B-swizzled slabs of 64 columns), so S and
// dP come out of one MMA and the thread that owns a selected row sees S and
// dP of every head for it. The selected rows are processed in tiles of 128:
//   MMA-A  [S^T | dP^T] = KV X^T     M = 128 rows, N = 128 (64 S + 64 dP), K = 512
//   SFU    P^T = exp2(S^T scale log2e - LSE log2e), dS^T = P^T (dP^T - D);
//          G = [scale dS^T | P^T] as fp16 in shared memory ([128 rows][128])
//   MMA-B  dQ^T += KV^T (scale dS^T) M = 128 d (4 chunks), N = 64 heads, K = 128 rows
//   MMA-C  dKV^T = X^T G             M = 128 d (4 chunks), N = 128 rows, K = 128
//   drain  every dKV^T block: TMEM -> registers -> red.global.add.f32 into the
//          original / compressed gradient rows (each warp instruction adds
//          one 128-byte run of one row)
// dQ^T accumulates in TMEM over all tiles of the token and is written once.
// The dKV reductions (D fp32 per selected row and token, from every token
// that selected the row) are the bulk of the memory traffic, so the drain
// has two warpgroups (one per 64-row half) and its own TMEM columns: a drain
// warpgroup copies its half of a block into registers and releases it at
// once, so the next block's MMAs run while it reduces, and the next tile's
// MMA-A, softmax and MMA-B run while the previous tile drains.
//
// KV rows come from an fp16 copy of [ori_kv ; cmp_kv] made by the pre-pass.
// Two loader warps copy them with cp.async (16 bytes per thread, written in
// the 128-byte swizzled layout the MMAs read) into a ring of 16 KB slots.
// Every tile streams twice: 8 slots of [128 rows x 64 d] (K-major A of
// MMA-A), then 8 slots of [64 rows x 128 d] (MN-major A of MMA-B: two
// 64-column halves 8 KB apart); X takes 128 KB of shared memory, which leaves
// no room to keep a whole [128 x 512] KV tile between the two.
//
// TMEM (512 columns): [0, 128) S^T|dP^T, [128, 256) a dKV^T block (column n =
// row n of the tile), [256, 512) dQ^T (chunk c of 128 d at 256 + 64 c, one
// column per head).
//
// Warp roles (512 threads): warp 0 builds the selected-row list of each
// token (two buffers, so the list of the next token is ready early) and
// issues the TMA copies of X; warp 1 owns TMEM and lane 0 issues the MMAs;
// warps 2-3 load KV rows (they run on into the next token's tiles while the
// current one finishes); warps 4-7 convert X from bf16 to fp16 in place and
// run the softmax (thread = selected row); warps 8-11 / 12-15 drain rows
// 0-63 / 64-127 of each dKV^T block and write dQ (thread = column d). Between tokens the drain
// is still reducing the last tile while X of the next token loads and
// converts. Every wait is bounded (tc_util.cuh).

#include "internal.h"
#include "tc_ptx.cuh"
#include "tc_util.cuh"

#include <math.h>

#include <algorithm>

namespace attn {
namespace {

constexpr int kSpThreads = 512;
constexpr int kSpD = 512;         // head dim (latent KV width)
constexpr int kSpR = 64;          // query heads per KV head
constexpr int kSpMaxRows = 1024;  // selected rows per (token, KV head)
constexpr int kSpSlots = 3;       // KV ring depth
constexpr int kSpSlot = 16384;    // bytes per slot / per X or G slab

struct SpSmem {
  static constexpr int X = 0;                          // 8 slabs: rows 0-63 Q, 64-127 dO
  static constexpr int KV = X + 8 * kSpSlot;           // ring of kSpSlots slots
  static constexpr int G = KV + kSpSlots * kSpSlot;    // slab 0 scale dS^T, slab 1 P^T
  static constexpr int ROWS = G + 2 * kSpSlot;         // 2 buffers: int32 row ids of a token
  static constexpr int LSE = ROWS + 2 * 4 * kSpMaxRows;  // 2 x 64 fp32: LSE log2e (+inf if not finite)
  static constexpr int DLT = LSE + 2 * 4 * kSpR;       // 2 x 64 fp32: D
  static constexpr int BAR = DLT + 2 * 4 * kSpR;       // mbarriers
  static constexpr int MISC = BAR + 256;               // TMEM base, abort flag, 2 row counts
  static constexpr int TOTAL = MISC + 16;
};
static_assert(SpSmem::TOTAL <= 227 * 1024, "shared memory budget");

// mbarriers. Per token: sXFull, sXReady, sXFree, sRowsReady/sRowsFree (one
// pair per row-list buffer, tokens alternate), sDqFull, sDqFree. Per tile
// (running counters across the tokens of the CTA): the ring, sStFull, sGFull,
// sGFree, sDkvFull / sDkvEmpty (four dKV^T blocks per tile).
enum SpBar {
  sXFull = 0,        // X landed (TMA transaction count)
  sXReady = 1,       // X converted to fp16 (128 softmax threads)
  sXFree = 2,        // the MMAs of the token stopped reading X
  sRowsReady0 = 3,   // row list, N, LSE and D of a token written (x2, 32 lanes)
  sRowsFree0 = 5,    // every role is done with the token's row list (x2, 449 arrivals)
  sKvFull0 = 7,      // ring slot filled (x3, 64 loader arrivals)
  sKvEmpty0 = 10,    // ring slot consumed by its MMAs (x3)
  sStFull = 13,      // S^T | dP^T of the tile in TMEM
  sGFull = 14,       // G written, S^T | dP^T read (128 arrivals)
  sGFree = 15,       // the MMAs of the tile stopped reading G
  sDkvFull = 16,     // a dKV^T block (one d chunk, all 128 rows) is in TMEM
  sDkvEmpty = 17,    // both drain warpgroups have read it (256 arrivals)
  sDqFull = 18,      // dQ^T of the token complete
  sDqFree = 19,      // the drain has read dQ^T (256 arrivals)
  sDone = 20,        // every MMA of the CTA completed (teardown)
  kSpBars = 21
};

struct SpParams {
  int Sq, Hq, Hk, n_ori, n_cmp, topk, wl, wr;
  int ratio;  // > 0: CFA (no index list; every compressed row whose block ends by the query)
  float scale;
  float scale_log2;
  const __half* kv16;  // [(n_ori + n_cmp) * Hk][512] fp16 copy of [ori_kv ; cmp_kv]
  const int32_t* idx;  // [Sq][Hk][topk] or nullptr
  const float* lse;    // [Hq][Sq]
  const float* delta;  // [Hq][Sq]
  float* dq;           // [Sq][Hq][512]
  float* d_ori;        // [n_ori][Hk][512]
  float* d_cmp;        // [n_cmp][Hk][512]
  DevStatus* status;
  // Deterministic mode (det_part != nullptr): each item's dKV rows are stored
  // to det_part[(item det_stride + slot)][512] instead of being added into
  // d_ori / d_cmp; det_rows holds the item's row list (same slots) and
  // det_meta[3 item .. +2] = {row count, window rows, first window row}.
  // item = token Hk + KV head. attn_bwd then adds them per row in token order.
  float* det_part;
  int32_t* det_rows;
  int32_t* det_meta;
  int det_stride;
};

// Selected rows of (token i, KV head g) as row ids of the fp16 copy
// [ori rows ; cmp rows] viewed as [(n_ori + n_cmp) * Hk][512]: the window
// first, then the valid top-k entries in slot order (SCFA) or every compressed
// row whose block ends at or before the query (CFA). Returns the count; the
// list is padded to a multiple of 128 with its first entry (masked later).
// Run by one full warp.
__device__ int build_rows(const SpParams& p, int i, int g, int32_t* rows, int lane,
                          int* nwin_out, int* lo_out) {
  const int pos = (p.n_ori - p.Sq) + i;
  int lo = p.wl >= 0 ? pos - p.wl : 0;
  int hi = p.wr >= 0 ? pos + p.wr : p.n_ori - 1;
  lo = max(lo, 0);
  hi = min(hi, p.n_ori - 1);
  const int nwin = hi >= lo ? hi - lo + 1 : 0;
  *nwin_out = nwin;
  *lo_out = lo;
  for (int j = lane; j < nwin; j += 32) rows[j] = (lo + j) * p.Hk + g;
  int n = nwin;
  if (p.ratio > 0) {  // CFA
    const int nc = min(p.n_cmp, max(pos + 1, 0) / p.ratio);
    for (int c = lane; c < nc; c += 32) rows[n + c] = (p.n_ori + c) * p.Hk + g;
    n += nc;
  } else if (p.idx != nullptr) {
    const int32_t* ir = p.idx + ((int64_t)i * p.Hk + g) * p.topk;
    bool bad = false;
    for (int t0 = 0; t0 < p.topk; t0 += 32) {
      const int t = t0 + lane;
      const int cidx = t < p.topk ? __ldg(ir + t) : -1;
      bad |= cidx < -1 || cidx >= p.n_cmp;
      const bool ok = cidx >= 0 && cidx < p.n_cmp;
      const uint32_t m = __ballot_sync(0xffffffffu, ok);
      if (ok) rows[n + __popc(m & ((1u << lane) - 1u))] = (p.n_ori + cidx) * p.Hk + g;
      n += __popc(m);
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) report(p.status, ATTN_ERR_INDEX_OOB, i);
  }
  __syncwarp();
  const int padded = (n + 127) / 128 * 128;
  const int32_t first = n > 0 ? rows[0] : 0;
  __syncwarp();
  for (int j = n + lane; j < padded; j += 32) rows[j] = first;
  return n;
}

// 8 bf16 -> 8 fp16 in place; returns the largest magnitude seen (a bf16
// value overflows fp16 exactly when its magnitude is at least 65520).
__device__ __forceinline__ float bf16x8_to_half(uint4* v, float amax) {
  uint32_t w[4] = {v->x, v->y, v->z, v->w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float lo = __uint_as_float(w[t] << 16);
    const float hi = __uint_as_float(w[t] & 0xffff0000u);
    amax = fmaxf(amax, fmaxf(fabsf(lo), fabsf(hi)));
    w[t] = pack_half2(lo, hi);
  }
  *v = make_uint4(w[0], w[1], w[2], w[3]);
  return amax;
}

__global__ void __launch_bounds__(kSpThreads, 1)
attn_bwd_sparse_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
                          const __grid_constant__ CUtensorMap tmdO, const SpParams p) {
  using L = SpSmem;
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) report(p.status, ATTN_ERR_UNSUPPORTED, 2);
    return;
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Persistent: this CTA takes work items u = blockIdx.x + k gridDim.x, item
  // u = (token Sq - 1 - u / Hk, KV head u % Hk): later tokens select more rows
  // and go first, and a strided share keeps the CTAs balanced.
  const int n_items = p.Sq * p.Hk;
  const int n_tok = ((int)blockIdx.x < n_items)
                        ? (n_items - 1 - (int)blockIdx.x) / (int)gridDim.x + 1
                        : 0;
  auto item_i = [&](int k) { return p.Sq - 1 - ((int)blockIdx.x + k * (int)gridDim.x) / p.Hk; };
  auto item_g = [&](int k) { return ((int)blockIdx.x + k * (int)gridDim.x) % p.Hk; };

  // everything below reads what the pre-pass wrote (launched as its
  // programmatic dependent, this grid may start before the pre-pass ends)
  ptx::grid_dependency_wait();
  if (blockIdx.x == 0) {
    // fp16 overflow found while staging the KV copy: OR of the pre-pass's
    // per-block flag slots
    const int nslots = min(max(p.status->reserved[1], 0), kPreMaxBlocks);
    const int32_t* slots = reinterpret_cast<const int32_t*>(p.status + 1);
    int bits = 0;
    for (int s = threadIdx.x; s < nslots; s += blockDim.x) bits |= slots[s];
    bits = __reduce_or_sync(0xffffffffu, bits);
    if (bits && lane == 0) report(p.status, ATTN_ERR_RANGE, bits);
  }

  Ctx c;
  c.bars = sbase + L::BAR;
  c.abort = reinterpret_cast<volatile int*>(smem + L::MISC + 4);
  c.status = p.status;
  volatile int* nrows_s = reinterpret_cast<volatile int*>(smem + L::MISC + 8);  // [2]

  if (threadIdx.x == 0) {
    uint32_t counts[kSpBars];
    for (int b = 0; b < kSpBars; ++b) counts[b] = 1;
    counts[sXReady] = 128;
    counts[sRowsReady0] = counts[sRowsReady0 + 1] = 32;
    // drain 256 + loaders 64 + softmax 128 + MMA thread 1: once all of them
    // arrived, every role has also passed the token's sRowsReady phase
    counts[sRowsFree0] = counts[sRowsFree0 + 1] = 449;
    for (int s = 0; s < kSpSlots; ++s) counts[sKvFull0 + s] = 64;
    counts[sGFull] = 128;
    counts[sDkvEmpty] = 256;
    counts[sDqFree] = 256;
    for (int b = 0; b < kSpBars; ++b) ptx::mbar_init(c.bar(b), counts[b]);
    *c.abort = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tmQ);
    ptx::prefetch_tmap(&tmdO);
  }
  if (warp == 1) {
    ptx::tmem_alloc(sbase + L::MISC, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::MISC);
  const uint32_t sX = sbase + L::X, sKV = sbase + L::KV, sG = sbase + L::G;
  // tcgen05.commit arrivals the MMA thread sent to each barrier (counted so
  // that the teardown can wait for the last phase of every one of them: an
  // arrival still in flight at exit would land on the barriers of the next
  // CTA this SM runs, which belongs to another launch since the CTAs are
  // persistent)
  int n_ring = 0, n_st = 0, n_gfree = 0, n_dkv = 0, n_xfree = 0, n_dq = 0;
  auto rows_of = [&](int b) { return reinterpret_cast<int32_t*>(smem + L::ROWS + b * 4 * kSpMaxRows); };
  auto rows_addr = [&](int b) { return sbase + L::ROWS + b * 4 * kSpMaxRows; };
  auto lse_of = [&](int b) { return reinterpret_cast<float*>(smem + L::LSE + b * 4 * kSpR); };
  auto dlt_of = [&](int b) { return reinterpret_cast<float*>(smem + L::DLT + b * 4 * kSpR); };

  if (warp == 0) {
    // ------------------------- per token: row list, LSE / D, X TMA copies --
    int x_issued = 0;
    for (int k = 0; k < n_tok; ++k) {
      const int b = k & 1, i = item_i(k), g = item_g(k);
      if (k >= 2 && !wait_bar(c, sRowsFree0 + b, (uint32_t)((k - 2) >> 1) & 1u, 30)) break;
      int nwin, wlo;
      const int n = build_rows(p, i, g, rows_of(b), lane, &nwin, &wlo);
      if (p.det_part != nullptr) {  // the row list of the item's stored dKV rows
        const int64_t item = (int64_t)i * p.Hk + g;
        for (int j = lane; j < n; j += 32) p.det_rows[item * p.det_stride + j] = rows_of(b)[j];
        if (lane == 0) {
          p.det_meta[3 * item] = n;
          p.det_meta[3 * item + 1] = nwin;
          p.det_meta[3 * item + 2] = wlo;
        }
      }
      for (int h = lane; h < kSpR; h += 32) {
        const int64_t r = (int64_t)(g * kSpR + h) * p.Sq + i;
        const float lv = p.lse[r];
        lse_of(b)[h] = isfinite(lv) ? lv * kLog2e : INFINITY;  // +inf: P = 0 for the head
        dlt_of(b)[h] = p.delta[r];
      }
      if (lane == 0) nrows_s[b] = n;
      __syncwarp();
      ptx::mbar_arrive(c.bar(sRowsReady0 + b));
      // X of this token once the previous token's MMAs stopped reading X
      if (k >= 1 && !wait_bar(c, sXFree, (uint32_t)(k - 1) & 1u, 31)) break;
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(c.bar(sXFull), 8 * kSpSlot);
        for (int s = 0; s < 8; ++s) {
          ptx::tma_load_3d(sX + s * kSpSlot, &tmQ, c.bar(sXFull), 64 * s, g * kSpR, i);
          ptx::tma_load_3d(sX + s * kSpSlot + kSpSlot / 2, &tmdO, c.bar(sXFull), 64 * s,
                           g * kSpR, i);
        }
      }
      ++x_issued;
    }
    // the last X copy lands before the CTA moves on, whatever else happened
    if (lane == 0 && x_issued > 0) drain_bar(c, sXFull, (uint32_t)(x_issued - 1) & 1u);
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      constexpr uint32_t idA = ptx::idesc_f16_f32(128, 128, false, false);
      constexpr uint32_t idB = ptx::idesc_f16_f32(128, 64, true, true);
      constexpr uint32_t idC = ptx::idesc_f16_f32(128, 128, true, false);
      const uint32_t tS = tmem, tQ = tmem + 256;
      bool ok = true;
      int slot = 0;
      uint32_t ph = 0;
      int issued = 0, freed = 0;  // dKV^T blocks issued / read by the drain
      int gt = 0;  // tiles of this CTA so far (all tokens)
      // operand descriptors, built once (slots and K steps add their offsets)
      const uint64_t dKV = ptx::smem_desc_sw128(sKV, 16, 1024);               // K-major
      const uint64_t dKVmn = ptx::smem_desc_sw128(sKV, kSpSlot / 2, 1024);    // MN-major
      const uint64_t dX = ptx::smem_desc_sw128(sX, 16, 1024);                 // K-major
      const uint64_t dXmn = ptx::smem_desc_sw128(sX, kSpSlot, 1024);          // MN-major
      const uint64_t dG = ptx::smem_desc_sw128(sG, 16, 1024);                 // K-major
      const uint64_t dGmn = ptx::smem_desc_sw128(sG, kSpSlot, 1024);          // MN-major
      // One ring slot of MMA-A: [S^T | dP^T] (+)= KV X^T over column slab s.
      auto a_slab = [&](int s) {
        if (!wait_bar(c, sKvFull0 + slot, ph, 42)) return false;
        ptx::fence_async_shared();  // cp.async data -> async proxy
        ptx::tc_fence_after();
        const uint64_t a0 = ptx::desc_add(dKV, slot * kSpSlot);
        const uint64_t b0 = ptx::desc_add(dX, s * kSpSlot);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          ptx::mma_ss(tS, ptx::desc_add(a0, 32 * k), ptx::desc_add(b0, 32 * k), idA, (s | k) != 0);
        ptx::mma_commit(c.bar(sKvEmpty0 + slot));
        ++n_ring;
        if (++slot == kSpSlots) { slot = 0; ph ^= 1u; }
        return true;
      };
      // One ring slot of MMA-B: dQ^T (d chunk j / 2) += KV^T (scale dS^T) over
      // the 64 selected rows of half j % 2, 16 per K step (slot data landed).
      auto b_slot = [&](int t, int j) {
        const int cc = j >> 1, nh = j & 1;
        const uint64_t a0 = ptx::desc_add(dKVmn, slot * kSpSlot);
        const uint64_t b0 = ptx::desc_add(dGmn, 64 * nh * 128);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_ss(tQ + 64 * cc, ptx::desc_add(a0, 2048 * kk), ptx::desc_add(b0, 2048 * kk),
                      idB, (t | nh | kk) != 0);
      };
      // One ring slot of MMA-A for the next tile (slot data landed).
      auto a_next = [&](int s) {
        const uint64_t a0 = ptx::desc_add(dKV, slot * kSpSlot);
        const uint64_t b0 = ptx::desc_add(dX, s * kSpSlot);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          ptx::mma_ss(tS, ptx::desc_add(a0, 32 * k), ptx::desc_add(b0, 32 * k), idA, (s | k) != 0);
      };
      // One MMA-C block: dKV^T (d chunk cc, all 128 rows of the tile) =
      // X^T G (the drain has read the previous block).
      auto c_block = [&](int cc) {
        const uint64_t a0 = ptx::desc_add(dXmn, 2 * cc * kSpSlot);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          ptx::mma_ss(tmem + 128, ptx::desc_add(a0, 2048 * kk),
                      ptx::desc_add(dG, (kk >> 2) * kSpSlot + (kk & 3) * 32), idC, kk != 0);
        ptx::mma_commit(c.bar(sDkvFull));
        ++n_dkv;
        ++issued;
      };
      // After sGFull of tile t: two independent streams. The MMA-C blocks go
      // out as the drain frees a dKV^T buffer; the ring slots (MMA-B of this
      // tile interleaved with MMA-A of the next, in fill order) as their data
      // lands. Neither waits for the other: the thread polls both.
      auto tile_streams = [&](int t, bool next) {
        const int nr = next ? 16 : 8;
        int r = 0, cb = 0;
        uint64_t t0 = 0;
        for (uint32_t idle = 0; r < nr || cb < 4;) {
          bool did = false;
          // ring slots first: a slot returns to the loaders only once its MMAs
          // complete, and the next tile's MMA-A and softmax wait on the ring
          if (r < nr && ptx::mbar_test_wait(c.bar(sKvFull0 + slot), ph)) {
            ptx::fence_async_shared();  // cp.async data -> async proxy
            ptx::tc_fence_after();
            if (!next || (r & 1) == 0) b_slot(t, next ? r >> 1 : r);
            else a_next(r >> 1);
            ptx::mma_commit(c.bar(sKvEmpty0 + slot));
            ++n_ring;
            if (++slot == kSpSlots) { slot = 0; ph ^= 1u; }
            ++r;
            did = true;
          }
          if (cb < 4) {
            if (freed < issued &&
                ptx::mbar_test_wait(c.bar(sDkvEmpty), (uint32_t)freed & 1u))
              ++freed;
            if (freed >= issued) {
              ptx::tc_fence_after();
              c_block(cb++);
              did = true;
            }
          }
          if (did) {
            idle = 0;
          } else if ((++idle & 63u) == 0) {
            if (*c.abort) return false;
            const uint64_t now = ptx::globaltimer_ns();
            if (t0 == 0 || idle == 64) t0 = now;
            if (now - t0 > kTimeoutNs) {
              *c.abort = 1;
              report(c.status, ATTN_ERR_DEVICE_TIMEOUT, 48);
              return false;
            }
          }
        }
        return true;
      };
      for (int k = 0; k < n_tok && ok; ++k) {
        const int b = k & 1;
        if (!wait_bar(c, sRowsReady0 + b, (uint32_t)(k >> 1) & 1u, 40)) break;
        const int T = (nrows_s[b] + 127) / 128;
        ptx::mbar_arrive(c.bar(sRowsFree0 + b));
        if (!wait_bar(c, sXReady, (uint32_t)k & 1u, 41)) break;
        ptx::tc_fence_after();
        if (T > 0) {
          for (int s = 0; s < 8 && ok; ++s) ok = a_slab(s);
          if (!ok) break;
          ptx::mma_commit(c.bar(sStFull));
          ++n_st;
        }
        for (int t = 0; t < T && ok; ++t, ++gt) {
          if (!wait_bar(c, sGFull, (uint32_t)gt & 1u, 43)) { ok = false; break; }
          // the first dQ^T MMA of a token overwrites what the drain read last token
          if (t == 0 && k > 0 && !wait_bar(c, sDqFree, (uint32_t)(k - 1) & 1u, 46)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          // (the softmax read S^T | dP^T of this tile before sGFull: MMA-A of
          // the next tile may overwrite it)
          const bool next = t + 1 < T;
          if (!(ok = tile_streams(t, next))) break;
          ptx::mma_commit(c.bar(sGFree));
          ++n_gfree;
          if (next) {
            ptx::mma_commit(c.bar(sStFull));
            ++n_st;
          }
        }
        if (!ok) break;
        // with no tiles, dQ^T was not touched, but sDqFull of this token must not
        // complete before the drain consumed the previous one
        if (T == 0 && k > 0 && !wait_bar(c, sDqFree, (uint32_t)(k - 1) & 1u, 47)) break;
        ptx::mma_commit(c.bar(sXFree));  // completes when every MMA reading X did
        ++n_xfree;
        ptx::mma_commit(c.bar(sDqFull));  // dQ^T of the token (T = 0: nothing to wait for)
        ++n_dq;
      }
      ptx::mma_commit(c.bar(sDone));  // completes once every MMA above has
    }
  } else if (warp < 4) {
    // ------------------------------------------- KV rows: cp.async loaders --
    // Thread tl owns rows r0 + 8 k (k < 16) of every tile and the 16-byte
    // chunk c8 of each 128-byte row segment; (r0 + 8 k) & 7 == r0, so the
    // 128B-swizzle position of its chunk is the same for all of them.
    const int tl = (int)threadIdx.x - 64;
    const int c8 = tl & 7, r0 = tl >> 3;
    const uint32_t swz = (uint32_t)((c8 ^ r0) << 4);
    int slot = 0;
    uint32_t ph = 0;
    bool ok = true;
    // Each fill arrives on its slot's sKvFull when its own copies land (the
    // MMA thread fences the async proxy after the wait), so all three slots
    // can be in flight and no fill waits on the loader's next step.
    // Row ids live in registers (this thread's 16 rows r0 + 8 k of a tile):
    // shared-memory loads wait behind the MMAs' operand reads, and a fill
    // must not wait on them.
    auto load_ids = [&](const int32_t* rt, int32_t (&ids)[16]) {
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) ids[kk] = rt[r0 + 8 * kk];
    };
    // MMA-A slot: [128 rows][64 d], columns 64 s of the tile's rows
    auto fill_a = [&](const int32_t (&ids)[16], int s) {
      if (!wait_bar(c, sKvEmpty0 + slot, ph ^ 1u, 31)) return false;
      const uint32_t dst = sKV + slot * kSpSlot + swz;
      const __half* src = p.kv16 + 8 * c8 + 64 * s;
#pragma unroll
      for (int kk = 0; kk < 16; ++kk)
        ptx::cp_async_16(dst + (r0 + 8 * kk) * 128, src + (int64_t)ids[kk] * kSpD);
      ptx::cp_async_arrive_noinc(c.bar(sKvFull0 + slot));
      if (++slot == kSpSlots) { slot = 0; ph ^= 1u; }
      return true;
    };
    // MMA-B slot j: [64 rows][128 d] (rows 64 (j % 2) on, d chunk j / 2) as two
    // [64][64] halves 8 KB apart
    auto fill_b = [&](const int32_t (&ids)[16], int j) {
      const int cc = j >> 1, nh = j & 1;
      if (!wait_bar(c, sKvEmpty0 + slot, ph ^ 1u, 32)) return false;
      const uint32_t dst = sKV + slot * kSpSlot + swz;
      const __half* src = p.kv16 + 8 * c8 + 128 * cc;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const __half* sp = src + (int64_t)(nh ? ids[8 + kk] : ids[kk]) * kSpD;
        ptx::cp_async_16(dst + (r0 + 8 * kk) * 128, sp);
        ptx::cp_async_16(dst + kSpSlot / 2 + (r0 + 8 * kk) * 128, sp + 64);
      }
      ptx::cp_async_arrive_noinc(c.bar(sKvFull0 + slot));
      if (++slot == kSpSlots) { slot = 0; ph ^= 1u; }
      return true;
    };
    int32_t cur[16], nxt[16];
    for (int k = 0; k < n_tok && ok; ++k) {
      const int b = k & 1;
      const uint32_t rph = (uint32_t)(k >> 1) & 1u;
      if (!wait_bar(c, sRowsReady0 + b, rph, 35)) break;
      const int T = (nrows_s[b] + 127) / 128;
      const int32_t* rows = rows_of(b);
      // the order in which the MMA thread consumes the ring
      if (T > 0) {
        load_ids(rows, cur);
        for (int s = 0; s < 8 && ok; ++s) ok = fill_a(cur, s);
      }
      for (int t = 0; t < T && ok; ++t) {
        const bool next = t + 1 < T;
        if (next) load_ids(rows + 128 * (t + 1), nxt);
        for (int j = 0; j < 8 && ok; ++j)
          ok = fill_b(cur, j) && (!next || fill_a(nxt, j));
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) cur[kk] = nxt[kk];
      }
      if (ok) ptx::mbar_arrive(c.bar(sRowsFree0 + b));  // row ids no longer read
    }
    ptx::cp_async_commit();
    ptx::cp_async_wait<0>();  // no copy may still write shared memory at exit
  } else if (warp < 8) {
    // ------------- per token: X bf16 -> fp16 in place, then the softmax --
    const int q4 = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int n = 32 * q4 + lane;  // selected row of a tile
    const uint32_t grow = sG + n * 128;
    const uint32_t sw = (uint32_t)(n & 7);
    int gt = 0;
    bool ok = true;
    for (int k = 0; k < n_tok && ok; ++k) {
      const int b = k & 1;
      if (!wait_bar(c, sXFull, (uint32_t)k & 1u, 50)) break;
      float amax = 0.f;
      {
        // 8192 16-byte chunks over 128 threads; 4 loads in flight per thread
        constexpr int kChunks = 8 * kSpSlot / 16;
        for (int e0 = (int)threadIdx.x - 128; e0 < kChunks; e0 += 4 * 128) {
          uint4 v[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) v[u] = ptx::ld_shared_v4_u32(sX + 16 * (e0 + u * 128));
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            amax = bf16x8_to_half(&v[u], amax);
            ptx::st_shared_v4(sX + 16 * (e0 + u * 128), v[u].x, v[u].y, v[u].z, v[u].w);
          }
        }
      }
      if (__any_sync(0xffffffffu, amax >= 65520.f) && lane == 0)
        report(p.status, ATTN_ERR_RANGE, 16);
      ptx::fence_async_shared();
      ptx::mbar_arrive(c.bar(sXReady));
      if (!wait_bar(c, sRowsReady0 + b, (uint32_t)(k >> 1) & 1u, 51)) break;
      const int N = nrows_s[b];
      const int T = (N + 127) / 128;
      const float* lse_s = lse_of(b);
      const float* dlt_s = dlt_of(b);
      for (int t = 0; t < T; ++t, ++gt) {
        if (!wait_bar(c, sStFull, (uint32_t)gt & 1u, 60)) { ok = false; break; }
        ptx::tc_fence_after();
        const bool valid = 128 * t + n < N;
        uint32_t pk[32], dk[32];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sv[32], dv[32];
          ptx::tmem_ld32(tmem + lane_off + 32 * half, sv);
          ptx::tmem_ld32(tmem + lane_off + 64 + 32 * half, dv);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int h = 32 * half + j;
            float x0, x1, pr0, pr1, t0, t1, d0, d1;
            ptx::fma2(x0, x1, __uint_as_float(sv[j]), __uint_as_float(sv[j + 1]), p.scale_log2,
                      p.scale_log2, -lse_s[h], -lse_s[h + 1]);
            pr0 = valid ? ptx::ex2(x0) : 0.f;
            pr1 = valid ? ptx::ex2(x1) : 0.f;
            ptx::sub2(t0, t1, __uint_as_float(dv[j]), __uint_as_float(dv[j + 1]), dlt_s[h],
                      dlt_s[h + 1]);
            ptx::mul2(d0, d1, pr0, pr1, t0, t1);
            ptx::mul2(d0, d1, d0, d1, p.scale, p.scale);
            pk[h / 2] = pack_half2(pr0, pr1);
            dk[h / 2] = pack_half2(d0, d1);
          }
        }
        ptx::tc_fence_before();
        // G of the previous tile must be out of use
        if (gt > 0 && !wait_bar(c, sGFree, (uint32_t)(gt - 1) & 1u, 61)) { ok = false; break; }
        // head h lives in 16-byte chunk h / 8 of the row (slab 0 dS, slab 1 P)
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t off = (((uint32_t)q) ^ sw) * 16u;
          ptx::st_shared_v4(grow + off, dk[4 * q], dk[4 * q + 1], dk[4 * q + 2], dk[4 * q + 3]);
          ptx::st_shared_v4(grow + kSpSlot + off, pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                            pk[4 * q + 3]);
        }
        ptx::fence_async_shared();
        ptx::mbar_arrive(c.bar(sGFull));
      }
      if (ok) ptx::mbar_arrive(c.bar(sRowsFree0 + b));
    }
  } else {
    // -------------------- per token: dKV^T drain, then dQ: thread = column d --
    const int q4 = warp & 3;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int bb = warp < 12 ? 0 : 1;  // row half of this warpgroup (columns 64 bb of a block)
    const int dl = 32 * q4 + lane;
    const int ori_rows = p.n_ori * p.Hk;
    const uint32_t tbuf = tmem + 128 + 64 * bb + lane_off;
    bool ok = true;
    int used = 0;
    for (int k = 0; k < n_tok && ok; ++k) {
      const int b = k & 1, i = item_i(k), g = item_g(k);
      if (!wait_bar(c, sRowsReady0 + b, (uint32_t)(k >> 1) & 1u, 70)) break;
      const int N = nrows_s[b];
      const int T = (N + 127) / 128;
      for (int t = 0; t < T && ok; ++t) {
        const int nt = min(64, N - 128 * t - 64 * bb);  // valid rows of this half (may be <= 0)
        const uint32_t rt_s = rows_addr(b) + 512 * t + 256 * bb;
        for (int cc = 0; cc < 4; ++cc) {
          if (!wait_bar(c, sDkvFull, (uint32_t)used & 1u, 71)) { ok = false; break; }
          ++used;
          ptx::tc_fence_after();
          uint32_t v[64];
          ptx::tmem_ld32(tbuf, v);
          ptx::tmem_ld32(tbuf + 32, v + 32);
          ptx::tmem_wait_ld();
          ptx::tc_fence_before();
          ptx::mbar_arrive(c.bar(sDkvEmpty));
          float* const ori_base = p.d_ori + 128 * cc + dl;
          float* const cmp_base = p.d_cmp - (int64_t)ori_rows * kSpD + 128 * cc + dl;
          if (p.det_part != nullptr) {
            // deterministic mode: store the rows at their slots (no reduction)
            float* const part = p.det_part +
                                (((int64_t)i * p.Hk + g) * p.det_stride + 128 * t + 64 * bb) * kSpD +
                                128 * cc + dl;
#pragma unroll
            for (int u = 0; u < 64; ++u)
              if (u < nt) part[(int64_t)u * kSpD] = __uint_as_float(v[u]);
            continue;
          }
#pragma unroll
          for (int n0 = 0; n0 < 64; n0 += 8) {
            if (n0 < nt) {
              const int4 ra = ptx::ld_shared_v4_s32(rt_s + 4 * n0);
              const int4 rb = ptx::ld_shared_v4_s32(rt_s + 4 * n0 + 16);
              const int r8[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                if (n0 + u < nt) {
                  float* const base = r8[u] < ori_rows ? ori_base : cmp_base;
                  ptx::red_add_f32_stream(base + (int64_t)r8[u] * kSpD,
                                          __uint_as_float(v[n0 + u]));
                }
              }
            }
          }
        }
      }
      if (!ok) break;
      // dQ of the token: this warpgroup writes d chunks 2 bb and 2 bb + 1
      if (!wait_bar(c, sDqFull, (uint32_t)k & 1u, 72)) break;
      ptx::tc_fence_after();
      float* dq = p.dq + ((int64_t)i * p.Hq + g * kSpR) * kSpD;
      if (T == 0) {
        for (int h = 0; h < kSpR; ++h)
#pragma unroll
          for (int cc = 2 * bb; cc < 2 * bb + 2; ++cc) dq[h * kSpD + 128 * cc + dl] = 0.f;
      } else {
#pragma unroll 1
        for (int cc = 2 * bb; cc < 2 * bb + 2; ++cc) {
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint32_t v[32];
            ptx::tmem_ld32(tmem + lane_off + 256 + 64 * cc + 32 * half, v);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              dq[(32 * half + j) * kSpD + 128 * cc + dl] = __uint_as_float(v[j]);
          }
        }
      }
      // dQ^T read: the next token's MMA-B may overwrite it
      ptx::tc_fence_before();
      ptx::mbar_arrive(c.bar(sDqFree));
      // this token's row list, N, LSE and D are no longer read by anyone
      ptx::mbar_arrive(c.bar(sRowsFree0 + b));
    }
  }

  // ----------------------------------------------------------- teardown --
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (lane == 0) {
      drain_bar(c, sDone, 0);  // every MMA of this CTA has completed
      // and every commit arrival has landed, including those no role waits
      // for (the last ring-slot releases, sGFree, sXFree) and those whose
      // waiter left early on an abort
      auto last = [&](int which, int n) {
        if (n > 0) drain_bar(c, which, (uint32_t)(n - 1) & 1u);
      };
      // ring slot u % kSpSlots took the u-th release
      for (int sl = 0; sl < kSpSlots; ++sl)
        last(sKvEmpty0 + sl, n_ring / kSpSlots + (sl < n_ring % kSpSlots ? 1 : 0));
      last(sStFull, n_st);
      last(sGFree, n_gfree);
      last(sDkvFull, n_dkv);
      last(sXFree, n_xfree);
      last(sDqFull, n_dq);
    }
    __syncwarp();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ------------------------------------------------------------ rows probe --
// The selected-row lists the backward kernel works on: one warp per item
// (token i, KV head g) runs build_rows, as warp 0 of the kernel does, and
// writes the item's list (rows of the fp16 copy [ori ; cmp] viewed as
// [(n_ori + n_cmp) Hk][512], so original row r of KV head g is r Hk + g and
// compressed row c is (n_ori + c) Hk + g) to rows[item][0, n) and n to
// counts[item], item = i Hk + g.
constexpr int kProbeWarps = 4;

__global__ void __launch_bounds__(32 * kProbeWarps)
rows_probe_kernel(const SpParams p, int32_t* rows, int32_t* counts, int stride) {
  __shared__ int32_t buf[kProbeWarps][kSpMaxRows];
  const int w = (int)threadIdx.x >> 5, lane = (int)threadIdx.x & 31;
  const int item = (int)blockIdx.x * kProbeWarps + w;
  if (item >= p.Sq * p.Hk) return;
  const int i = item / p.Hk, g = item % p.Hk;
  int nwin, lo;
  const int n = build_rows(p, i, g, buf[w], lane, &nwin, &lo);
  for (int j = lane; j < n; j += 32) rows[(int64_t)item * stride + j] = buf[w][j];
  if (lane == 0) counts[item] = n;
}

// ------------------------------------------------------------------ host --

// [Sq][H][512] bf16 rows with element strides (token, head): 3-D map, boxes
// of 64 heads x 64 columns, 128B swizzle.
bool make_qmap(CUtensorMap* m, const void* base, int Sq, int H, int64_t s_tok, int64_t s_head) {
  EncodeFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kSpD, (cuuint64_t)H, (cuuint64_t)Sq};
  cuuint64_t strides[2] = {(cuuint64_t)s_head * 2, (cuuint64_t)s_tok * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kSpR, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t max_selected_rows(const Problem& p) {
  const int64_t win = (p.ori_wl >= 0 && p.ori_wr >= 0)
                          ? std::min<int64_t>(p.n_ori, (int64_t)p.ori_wl + p.ori_wr + 1)
                          : p.n_ori;
  return win + (p.n_cmp > 0 ? (p.cmp_ratio > 0 ? p.n_cmp : p.topk) : 0);
}

}  // namespace

int64_t sparse_det_stride(const Problem& p) { return (max_selected_rows(p) + 127) / 128 * 128; }

int64_t sparse_row_bound(const Problem& p) { return max_selected_rows(p); }

cudaError_t launch_rows_probe(const Problem& pr, const int32_t* idx, int32_t* rows,
                              int32_t* counts, int stride, cudaStream_t stream) {
  SpParams p{};
  p.Sq = pr.Sq;
  p.Hq = pr.Hq;
  p.Hk = pr.Hk;
  p.n_ori = pr.n_ori;
  p.n_cmp = pr.n_cmp;
  p.topk = pr.topk;
  p.ratio = pr.cmp_ratio;
  p.wl = pr.ori_wl;
  p.wr = pr.ori_wr;
  p.idx = pr.n_cmp > 0 && pr.cmp_ratio == 0 ? idx : nullptr;
  p.status = nullptr;  // out-of-range indices are skipped, not reported
  const int64_t items = (int64_t)pr.Sq * pr.Hk;
  if (items == 0) return cudaSuccess;
  const unsigned grid = (unsigned)((items + kProbeWarps - 1) / kProbeWarps);
  rows_probe_kernel<<<grid, 32 * kProbeWarps, 0, stream>>>(p, rows, counts, stride);
  return cudaGetLastError();
}

bool tc_sparse_supported(const Problem& p) {
  return p.sparse && p.D == kSpD && p.B == 1 && p.Hq == kSpR * p.Hk && p.Sq > 0 && p.n_ori > 0 &&
         max_selected_rows(p) <= kSpMaxRows &&
         (int64_t)(p.n_ori + p.n_cmp) * p.Hk < (int64_t(1) << 31) && p.qs[1] > 0 &&
         p.qs[2] > 0 && p.dos[1] > 0 && p.dos[2] > 0;  // (shape only, as tc_supported)
}

cudaError_t launch_bwd_sparse_tc(const Problem& pr, const void* q, const void* dO,
                                 const __half* kv16, const int32_t* idx, const float* lse,
                                 const float* delta, float* dq, float* d_ori, float* d_cmp,
                                 const SparseDet& det, DevStatus* st, cudaStream_t stream) {
  CUtensorMap mq, mdo;
  if (!make_qmap(&mq, q, pr.Sq, pr.Hq, pr.qs[1], pr.qs[2]) ||
      !make_qmap(&mdo, dO, pr.Sq, pr.Hq, pr.dos[1], pr.dos[2]))
    return cudaErrorInvalidValue;
  SpParams p;
  p.Sq = pr.Sq;
  p.Hq = pr.Hq;
  p.Hk = pr.Hk;
  p.n_ori = pr.n_ori;
  p.n_cmp = pr.n_cmp;
  p.topk = pr.topk;
  p.ratio = pr.cmp_ratio;
  p.wl = pr.ori_wl;
  p.wr = pr.ori_wr;
  p.scale = pr.scale;
  p.scale_log2 = pr.scale * kLog2e;
  p.kv16 = kv16;
  p.idx = pr.n_cmp > 0 && pr.cmp_ratio == 0 ? idx : nullptr;
  p.lse = lse;
  p.delta = delta;
  p.dq = dq;
  p.d_ori = d_ori;
  p.d_cmp = d_cmp;
  p.status = st;
  p.det_part = det.part;
  p.det_rows = det.rows;
  p.det_meta = det.meta;
  p.det_stride = det.stride;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_sparse_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SpSmem::TOTAL);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
  }
  const int64_t items = (int64_t)pr.Sq * pr.Hk;
  const unsigned grid = (unsigned)(items < sms ? items : sms);  // persistent: one CTA per SM
  return launch_dependent(attn_bwd_sparse_tc_kernel, dim3(grid), dim3(kSpThreads),
                          (size_t)SpSmem::TOTAL, stream, mq, mdo, p);
}

}  // namespace attn
