// GEMV kernels for plain [L][M][K/16] scales, plus the occupancy query.
#include "gemv_kernel.cuh"

namespace nvfp4 {

cudaError_t launch_gemv_plain(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream) {
  return launch_gemv_layout<false>(p, plan, stream);
}

// Both GEMV kernels run kGemvThreads-thread CTAs under the same
// __launch_bounds__ floor; the pipelined one also needs kAsyncSmemBytes of
// shared memory, which two CTAs per SM still fit.
cudaError_t gemv_ctas_per_sm(int* out) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, nvfp4_gemv_kernel<32, 1, false>,
                                                       kGemvThreads, 0);
}

}  // namespace nvfp4
