// Pieces shared by the tensor-core kernels: bounded mbarrier waits with a
// CTA-wide abort flag, fp16 packing, and the host-side tensor-map encoder.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace attn {

// Upper bound on any single mbarrier wait. A wait that runs out records
// ATTN_ERR_DEVICE_TIMEOUT and raises the CTA's abort flag; the CTA then
// drains its copies and MMAs, frees TMEM and exits.
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct Ctx {
  uint32_t bars;        // shared address of barrier 0
  volatile int* abort;  // CTA-wide abort flag
  DevStatus* status;
  __device__ uint32_t bar(int i) const { return bars + 8u * i; }
};

// Slow path of wait_bar (out of line: the caller's registers are saved only
// when the barrier was not already complete).
static __device__ __noinline__ bool wait_bar_slow(const Ctx& c, int which, uint32_t parity,
                                                  int where) {
  const uint32_t bar = c.bar(which);
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

// Bounded mbarrier wait: true when the phase with `parity` completed; false
// if the CTA aborted or ~2 s passed (then the abort flag is raised).
static __device__ __forceinline__ bool wait_bar(const Ctx& c, int which, uint32_t parity,
                                                int where) {
  if (ptx::mbar_try_wait(c.bar(which), parity)) return true;
  return wait_bar_slow(c, which, parity, where);
}

// Teardown wait: ignores the abort flag, still bounded.
static __device__ __noinline__ void drain_bar(const Ctx& c, int which, uint32_t parity) {
  const uint32_t bar = c.bar(which);
  const uint64_t t0 = ptx::globaltimer_ns();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (ptx::globaltimer_ns() - t0 > kTimeoutNs) {
      report(c.status, ATTN_ERR_DEVICE_TIMEOUT, 100 + which);
      return;
    }
  }
}

static __device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link-time
// dependency on libcuda); nullptr if the driver does not provide it.
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeFn encode_fn();

// Launches `kern` as a programmatic dependent of the previous kernel in the
// stream (the pre-pass): its CTAs may be scheduled while that kernel drains,
// and they call grid_dependency_wait() before reading its outputs.
template <typename Kern, typename... Args>
cudaError_t launch_dependent(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace attn
