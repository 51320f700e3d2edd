// Cast kernels for BF16 master values with outputs that are not word-aligned
// (fragment-sized outputs of fragments that start inside an output word), BF16 model
// dtype; the FP16-model kernels are in cast_bf16_unaligned_f16.cu (the two halves compile
// in parallel).
#include "cast_impl.cuh"

namespace mxfp8 {

cudaError_t launch_partial_cast_bf16_unaligned(const CastParams* jobs, int n, bool shifted, int model,
                                              const DeviceInfo& dev, cudaStream_t stream) {
  if (model == kModelF16) return launch_partial_cast_bf16_unaligned_f16(jobs, n, shifted, dev, stream);
  return launch_for_model<BF16T, false, kModelBF16>(jobs, n, shifted, dev, stream);
}

}  // namespace mxfp8
