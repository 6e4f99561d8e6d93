// attn_bwd_noalloc: the whole backward (pre-pass + backward kernel) for
// callers that must not allocate device memory.
//
// Who needs it: code that runs where cudaMalloc is not an option, for example
// inside a framework hook that may not re-enter the framework's allocator,
// in a deployment whose device memory is fixed at start-up (real-time or
// certified systems), or on a path that must not stall other streams
// (cudaMalloc can synchronise the device). Such callers still own their
// inputs and outputs; only the workspace (status record, fp16 operand
// staging) moves into a fixed array that this file places in device memory.
//
// The array lives as long as the library is loaded, on every GPU the process
// uses it on. All calls share it: two calls whose work overlaps on the GPU (on
// different streams, or on one stream from different host threads without
// ordering) race on it and give undefined results. Its contents persist
// between calls; the pre-pass rewrites every part the backward reads (status
// record, flag slots, staged operands), so stale data from an earlier call is
// never used.

#include "internal.h"

#include <mutex>

namespace attn {
namespace {

// Largest workspace a no-allocation call can use: enough for the fp16
// staging of, e.g., B=2, Hq=16, Hk=4, S=1024, D=128 (about 20 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array for the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace attn

extern "C" attn_status_t attn_bwd_noalloc(const attn_problem_t* prob, const attn_mask_t* mask,
                                          const attn_sparse_t* sparse, const void* q,
                                          const void* k, const void* v, const void* o,
                                          const void* dO, const float* lse, const float* bias,
                                          float* delta, float* dq, float* dk, float* dv,
                                          float* dbias, cudaStream_t stream,
                                          int32_t* device_status) {
  const size_t need = attn_bwd_workspace_size(prob, mask, sparse);
  if (need == 0) return ATTN_ERR_INVALID_ARG;
  if (need > attn::kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
  void* ws = nullptr;
  if (attn::scratch_address(&ws) != cudaSuccess) return ATTN_ERR_CUDA;
  attn_status_t s = attn_bwd_preprocess(prob, sparse, q, k, v, o, dO, delta, dbias, dk, dv, ws,
                                        attn::kNoAllocScratchBytes, stream);
  if (s != ATTN_OK) return s;
  s = attn_bwd(prob, mask, sparse, q, k, v, dO, lse, delta, bias, dq, dk, dv, dbias, ws,
               attn::kNoAllocScratchBytes, stream);
  if (s != ATTN_OK || device_status == nullptr) return s;
  int32_t detail = 0;
  device_status[0] = (int32_t)attn_read_device_status(ws, stream, &detail);
  device_status[1] = detail;
  return ATTN_OK;
}
