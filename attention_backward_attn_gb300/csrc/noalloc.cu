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

#include <cuda.h>

#include <mutex>

namespace attn {
namespace {

// Largest workspace a no-allocation call can use: enough for the fp16
// staging of, e.g., B=2, Hq=16, Hk=4, S=1024, D=128 (about 20 MiB).
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// The driver's context queries, looked up once through the runtime (no
// link-time dependency on libcuda). Either may be missing on an old driver.
using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Unique id of the calling thread's current context; false if there is none
// (or the driver cannot say).
bool current_context_id(unsigned long long* id) {
  std::call_once(g_ctx_once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<CtxGetIdFn>(f);
  });
  if (g_ctx_current == nullptr || g_ctx_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return g_ctx_id(ctx, id) == CUDA_SUCCESS;
}

struct ScratchSlot {
  bool valid;
  bool have_ctx;
  unsigned long long ctx;  // id of the context the address belongs to
  void* ptr;
};
std::mutex g_scratch_mu;
ScratchSlot g_scratch[kMaxDevices] = {};

// Device address of the array for the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up
// with cudaGetSymbolAddress, with the device current, and cached per device.
// The address belongs to the device's context: when the calling thread's
// current context is a different one (the old one was destroyed by
// cudaDeviceReset, say) or cannot be identified, the lookup runs again, in
// the context the runtime makes current for it.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  unsigned long long ctx = 0;
  const bool have_ctx = current_context_id(&ctx);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchSlot& sl = g_scratch[dev];
  if (!sl.valid || !have_ctx || !sl.have_ctx || sl.ctx != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    sl.valid = true;
    sl.ptr = p;
    sl.have_ctx = current_context_id(&sl.ctx);  // now current, if it was not before
  }
  *out = sl.ptr;
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
  const attn_status_t dev_code = attn_read_device_status(ws, stream, &detail);
  // The kernels never record ATTN_ERR_CUDA: that code means the host could
  // not read the record (the stream synchronisation or the copy failed, e.g.
  // on a sticky error from an earlier launch), and it is this call's result,
  // not a device-side condition.
  if (dev_code == ATTN_ERR_CUDA) return ATTN_ERR_CUDA;
  device_status[0] = (int32_t)dev_code;
  device_status[1] = detail;
  return ATTN_OK;
}
