// Cast kernels for FP32 master values with outputs that are not word-aligned
// (fragment-sized outputs of fragments that start inside an output word).
#include "cast_impl.cuh"

namespace mxfp8 {

cudaError_t launch_partial_cast_f32_unaligned(const CastParams* jobs, int n, bool shifted, int model,
                                              const DeviceInfo& dev, cudaStream_t stream) {
  return launch_for_dtype<F32T, false>(jobs, n, shifted, model, dev, stream);
}

}  // namespace mxfp8
