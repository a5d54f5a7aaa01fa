// GEMV kernels for 128x4-atom pre-permuted scales.
#include "gemv_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_gemv_permuted(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream) {
  return launch_gemv_layout<true>(p, plan, stream);
}

}  // namespace nvfp4
