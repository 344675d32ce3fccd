// Tensor-core verify attention (placeholder until the tcgen05 kernel lands).
#include "splash_common.cuh"

namespace splash {

bool tc_supported(int) { return false; }

cudaError_t launch_verify_tc(const AttnParams&, int, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace splash
