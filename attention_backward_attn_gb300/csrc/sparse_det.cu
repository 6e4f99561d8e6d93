// Deterministic dKV of the sparse (selected shared-KV) backward.
//
// In the default mode every token adds its dKV rows into d_ori / d_cmp with
// fp32 reductions, so a row's sum depends on the order in which tokens
// arrive (the Ascend "sparse_flash_mla_grad" page notes that its operator is
// not deterministic by default). In deterministic mode the tensor-core kernel
// stores each item's (token, KV head) rows at their slots instead, and this
// file adds them up per row in ascending token order:
//
//   slots   warp per item: for every compressed row of the item's list, the
//           first slot that holds it and how many slots do (a top-k list may
//           repeat an index; each repeat is one more equal term);
//   reduce  block per (row, KV head): the items that selected the row, in
//           token order, found from the window bounds (original rows) or the
//           slot table (compressed rows) and compacted in shared memory; then
//           every thread sums its 4 columns over that list in order, and the
//           row is written (not added).
//
// The same inputs therefore give the same bits on every run, whatever the
// scheduling.

#include "internal.h"

namespace attn {
namespace {

constexpr int kD = 512;           // the sparse variant's head dimension
constexpr int kRedThreads = 128;  // 4 columns each
constexpr int kChunk = 1024;      // tokens examined per compaction round
constexpr int kNoSlot = 0x7f7f7f7f;  // slot table fill (byte 0x7f)

struct DetParams {
  int Sq, Hk, n_ori, n_cmp, wl, wr;
  int64_t stride;
  const float* part;
  const int32_t* rows;
  const int32_t* meta;
  int32_t* slot;
  int32_t* mult;
  float* d_ori;
  float* d_cmp;
};

__global__ void __launch_bounds__(256) det_slots_kernel(const DetParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t items = (int64_t)p.Sq * p.Hk;
  const int64_t ori_rows = (int64_t)p.n_ori * p.Hk;
  for (int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; item < items;
       item += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int n = p.meta[3 * item];
    for (int j = lane; j < n; j += 32) {
      const int r = p.rows[item * p.stride + j];
      if (r < ori_rows) continue;
      const int c = r / p.Hk - p.n_ori;  // r = (n_ori + c) Hk + g
      atomicMin(&p.slot[item * p.n_cmp + c], j);
      atomicAdd(&p.mult[item * p.n_cmp + c], 1);
    }
  }
}

__global__ void __launch_bounds__(kRedThreads) det_reduce_kernel(const DetParams p) {
  __shared__ int2 hits[kChunk];  // (item, slot | multiplicity << 16) in token order
  __shared__ int warp_n[kRedThreads / 32];
  __shared__ int n_hits;
  const int r = blockIdx.x;  // flat row (row Hk + g) of [ori ; cmp]
  const int g = r % p.Hk;
  const int row = r / p.Hk;
  const bool ori = row < p.n_ori;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // tokens that can select the row: an original row o sits in the window of
  // query position pos = (n_ori - Sq) + i when pos - wl <= o <= pos + wr
  int ilo = 0, ihi = p.Sq - 1;
  if (ori) {
    const int d = p.n_ori - p.Sq;
    if (p.wr >= 0) ilo = max(ilo, row - p.wr - d);
    if (p.wl >= 0) ihi = min(ihi, row + p.wl - d);
  }
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int col = 4 * tid;
  for (int i0 = ilo; i0 <= ihi; i0 += kChunk) {
    if (tid == 0) n_hits = 0;
    __syncthreads();
    // ordered compaction: round u examines tokens i0 + 128 u + tid
    for (int u = 0; u < kChunk / kRedThreads; ++u) {
      const int i = i0 + u * kRedThreads + tid;
      int slot = -1, mult = 0;
      const int64_t item = (int64_t)i * p.Hk + g;
      if (i <= ihi) {
        if (ori) {
          const int nwin = p.meta[3 * item + 1], lo = p.meta[3 * item + 2];
          if (row >= lo && row < lo + nwin) {
            slot = row - lo;
            mult = 1;
          }
        } else {
          const int64_t e = item * p.n_cmp + (row - p.n_ori);
          const int s = p.slot[e];
          if (s != kNoSlot) {
            slot = s;
            mult = p.mult[e];
          }
        }
      }
      const uint32_t m = __ballot_sync(0xffffffffu, slot >= 0);
      if (lane == 0) warp_n[warp] = __popc(m);
      __syncthreads();
      int before = n_hits;
      for (int w = 0; w < warp; ++w) before += warp_n[w];
      if (slot >= 0)
        hits[before + __popc(m & ((1u << lane) - 1u))] = make_int2((int)item, slot | (mult << 16));
      __syncthreads();
      if (tid == 0) {
        int total = n_hits;
        for (int w = 0; w < kRedThreads / 32; ++w) total += warp_n[w];
        n_hits = total;
      }
      __syncthreads();
    }
    // the chunk's terms in token order; four rows in flight per step
    const int nh = n_hits;
    int h = 0;
    for (; h + 4 <= nh; h += 4) {
      float4 v[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int2 e = hits[h + k];
        v[k] = *reinterpret_cast<const float4*>(
            p.part + ((int64_t)e.x * p.stride + (e.y & 0xffff)) * kD + col);
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int reps = hits[h + k].y >> 16;
        for (int t = 0; t < reps; ++t) {
          acc.x += v[k].x;
          acc.y += v[k].y;
          acc.z += v[k].z;
          acc.w += v[k].w;
        }
      }
    }
    for (; h < nh; ++h) {
      const int2 e = hits[h];
      const float4 v = *reinterpret_cast<const float4*>(
          p.part + ((int64_t)e.x * p.stride + (e.y & 0xffff)) * kD + col);
      for (int t = 0; t < (e.y >> 16); ++t) {
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
    }
    __syncthreads();  // hits is rewritten by the next chunk
  }
  const int64_t ori_rows = (int64_t)p.n_ori * p.Hk;
  float* out = ori ? p.d_ori + (int64_t)r * kD : p.d_cmp + ((int64_t)r - ori_rows) * kD;
  *reinterpret_cast<float4*>(out + col) = acc;
}

}  // namespace

cudaError_t launch_sparse_det_reduce(const Problem& pr, const SparseDet& det, float* d_ori,
                                     float* d_cmp, cudaStream_t stream) {
  DetParams p;
  p.Sq = pr.Sq;
  p.Hk = pr.Hk;
  p.n_ori = pr.n_ori;
  p.n_cmp = pr.n_cmp;
  p.wl = pr.ori_wl;
  p.wr = pr.ori_wr;
  p.stride = det.stride;
  p.part = det.part;
  p.rows = det.rows;
  p.meta = det.meta;
  p.slot = det.slot;
  p.mult = det.mult;
  p.d_ori = d_ori;
  p.d_cmp = d_cmp;
  const int64_t items = (int64_t)pr.Sq * pr.Hk;
  if (pr.n_cmp > 0) {
    const size_t n = (size_t)items * pr.n_cmp * sizeof(int32_t);
    cudaError_t e = cudaMemsetAsync(det.slot, 0x7f, n, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(det.mult, 0, n, stream);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (items + 7) / 8;  // 8 warps per block, one item each
    det_slots_kernel<<<(unsigned)(blocks < 65535 ? blocks : 65535), 256, 0, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t flat_rows = (int64_t)(pr.n_ori + pr.n_cmp) * pr.Hk;
  det_reduce_kernel<<<(unsigned)flat_rows, kRedThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
