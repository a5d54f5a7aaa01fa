// Device self-test of the bounded mbarrier wait that the tensor-core and
// block-dot kernels use on their pipeline barriers (tc_ptx.cuh, mbar_wait).
//
// One warp, two barriers in shared memory, both initialised for one arrival:
// `done` receives that arrival, `never` receives none.  Lane 0 waits on
// phase 0 of each with the kernels' own bounded wait.  The first wait must
// return at once; the second must give up after the wait limit (2 s of
// global time), count one timeout and return, leaving the context usable.
// Nothing else runs in the kernel: no copies are in flight, no tensor memory
// is held, there is no cluster, so the only wait that can run out is the one
// under test and it is bounded.
#include "selftest.h"
#include "tc_ptx.cuh"

namespace nvfp4 {
namespace {

__device__ int g_selftest_timeouts;
__device__ long long g_selftest_out[3];  // completed, gave_up, waited_ns

__global__ void __launch_bounds__(32) wait_selftest_kernel() {
  __shared__ __align__(8) uint64_t bars[2];
  if (threadIdx.x != 0) return;
  const uint32_t done = smem_u32(&bars[0]);
  const uint32_t never = smem_u32(&bars[1]);
  tc::mbar_init(done, 1);
  tc::mbar_init(never, 1);
  tc::mbar_arrive(done);  // phase 0 of `done` completes
  bool ok_done = true, ok_never = true;
  tc::mbar_wait<false>(done, 0, ok_done, &g_selftest_timeouts);
  const uint64_t t0 = tc::global_ns();
  tc::mbar_wait<false>(never, 0, ok_never, &g_selftest_timeouts);
  const uint64_t t1 = tc::global_ns();
  g_selftest_out[0] = ok_done ? 1 : 0;
  g_selftest_out[1] = ok_never ? 0 : 1;
  g_selftest_out[2] = (long long)(t1 - t0);
}

}  // namespace

cudaError_t run_wait_selftest(cudaStream_t stream, WaitSelftest* out) {
  const int zero = 0;
  const long long unset[3] = {-1, -1, -1};
  cudaError_t err = cudaMemcpyToSymbolAsync(g_selftest_timeouts, &zero, sizeof(zero), 0,
                                            cudaMemcpyHostToDevice, stream);
  if (err == cudaSuccess)
    err = cudaMemcpyToSymbolAsync(g_selftest_out, unset, sizeof(unset), 0,
                                  cudaMemcpyHostToDevice, stream);
  if (err != cudaSuccess) return err;
  wait_selftest_kernel<<<1, 32, 0, stream>>>();
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  long long res[3] = {0, 0, 0};
  int timeouts = 0;
  err = cudaMemcpyFromSymbolAsync(res, g_selftest_out, sizeof(res), 0, cudaMemcpyDeviceToHost,
                                  stream);
  if (err == cudaSuccess)
    err = cudaMemcpyFromSymbolAsync(&timeouts, g_selftest_timeouts, sizeof(timeouts), 0,
                                    cudaMemcpyDeviceToHost, stream);
  if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return err;
  out->completed = (int)res[0];
  out->gave_up = (int)res[1];
  out->timeouts = timeouts;
  out->waited_ns = (int64_t)res[2];
  return cudaSuccess;
}

}  // namespace nvfp4
