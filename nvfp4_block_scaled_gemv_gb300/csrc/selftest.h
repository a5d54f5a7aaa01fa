// Device self-test of the bounded mbarrier wait (selftest.cu).
#pragma once
#include <cstdint>

#include <cuda_runtime.h>

namespace nvfp4 {

// What one run of the self-test kernel saw: the bounded wait on a barrier
// phase that completes returned true (completed = 1); the one on a phase
// that nothing completes returned false (gave_up = 1) after waited_ns of
// global time, and the kernel counted `timeouts` waits that gave up.
struct WaitSelftest {
  int completed;
  int gave_up;
  int timeouts;
  int64_t waited_ns;
};

// Runs the self-test kernel (one warp) on `stream` and synchronises it.
cudaError_t run_wait_selftest(cudaStream_t stream, WaitSelftest* out);

}  // namespace nvfp4
