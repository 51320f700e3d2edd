// cast kernels instantiated for BF16 master values (the templates live in
// cast_impl.cuh; one translation unit per input dtype keeps the build parallel).
#include "cast_impl.cuh"

namespace mxfp8 {

cudaError_t launch_partial_cast_bf16(const CastParams* jobs, int n, bool shifted, bool vec_out, int model,
                       const DeviceInfo& dev, cudaStream_t stream) {
  return launch_for_dtype<BF16T>(jobs, n, shifted, vec_out, model, dev, stream);
}

}  // namespace mxfp8
