// Cast kernels for BF16 master values with word-aligned outputs (the templates live in
// cast_impl.cuh).
#include "cast_impl.cuh"

namespace mxfp8 {

cudaError_t launch_partial_cast_bf16(const CastParams* jobs, int n, bool shifted, int model,
                                     const DeviceInfo& dev, cudaStream_t stream) {
  return launch_for_dtype<BF16T, true>(jobs, n, shifted, model, dev, stream);
}

}  // namespace mxfp8
