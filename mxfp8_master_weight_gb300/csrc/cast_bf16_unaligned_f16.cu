// Cast kernels for BF16 master values with outputs that are not word-aligned, FP16 model
// dtype (the BF16-model half is in cast_bf16_unaligned.cu).
#include "cast_impl.cuh"

namespace mxfp8 {

cudaError_t launch_partial_cast_bf16_unaligned_f16(const CastParams* jobs, int n, bool shifted,
                                                  const DeviceInfo& dev, cudaStream_t stream) {
  return launch_for_model<BF16T, false, kModelF16>(jobs, n, shifted, dev, stream);
}

}  // namespace mxfp8
