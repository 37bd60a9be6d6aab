// bwd_bf16.cu -- ring-order backward (placeholder until the kernels land).
#include "common.cuh"

namespace ra {
cudaError_t launch_bwd_bf16(const BwdArgs&, const void*, const void*, const void*, const void*) {
  return cudaErrorNotSupported;
}
}  // namespace ra
