// Pipelined (cp.async) GEMV kernels for 128x4-atom pre-permuted scales.
#include "gemv_async.cuh"

namespace nvfp4 {

cudaError_t launch_async_permuted(const GemvParams& p, const GemvPlan& plan, cudaStream_t stream) {
  return launch_async_layout<true>(p, plan, stream);
}

}  // namespace nvfp4
