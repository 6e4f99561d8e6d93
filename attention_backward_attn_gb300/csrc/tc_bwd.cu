// Tensor-core (tcgen05) backward: placeholder until the kernel lands.
#include "internal.h"

namespace attn {

bool tc_supported(const Problem&) { return false; }

cudaError_t launch_bwd_tc(const Problem&, const __half*, const __half*, const __half*,
                          const __half*, const float*, const float*, const float*, float*,
                          float*, float*, float*, DevStatus*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace attn
