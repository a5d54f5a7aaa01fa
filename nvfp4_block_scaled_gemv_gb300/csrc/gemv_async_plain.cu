// Pipelined (cp.async) GEMV kernels for plain [L][M][K/16] scales.
#include "gemv_async.cuh"

namespace nvfp4 {

cudaError_t launch_async_plain(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream) {
  return launch_async_layout<false>(p, plan, stream);
}

}  // namespace nvfp4
