// Tensor-core expert FFN: not available in this build; the CUDA-core path runs.
#include "internal.h"
namespace moe {
cudaError_t launch_ffn_tc(const Shape&, int64_t, const void*, const int32_t*, const void*, const float*,
                          const void*, const float*, void*, void*, int*, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace moe
