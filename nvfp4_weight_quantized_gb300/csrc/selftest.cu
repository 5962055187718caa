// selftest.cu -- a self-test of the bounded device-side wait.
//
// Every pipeline wait of the GEMM kernels gives up after a fixed number of SM
// cycles (sm100::kWaitLimitCycles, about 1.5 s at 2 GHz) and records
// NVFP4_ERR_TIMEOUT in the library's status word instead of spinning forever,
// so a stalled pipeline ends with an error the host can read and the CUDA
// context stays usable.  This kernel takes that path on purpose: one thread
// waits on an mbarrier that nothing ever arrives on, gives up after the same
// limit and sets the same status bit.  No trap, no fault, no unbounded loop.
#include "kernels.h"
#include "tcgen05.cuh"

namespace nvfp4 {

namespace {

__global__ void __launch_bounds__(1) wait_timeout_selftest_kernel(unsigned int* __restrict__ status) {
  __shared__ __align__(8) uint64_t bar;
  sm100::mbar_init(&bar, 1);
  sm100::fence_mbar_init();
  if (!sm100::mbar_wait(&bar, 0)) atomicOr(status, kStatusTimeout);
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(unsigned int* status, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 1, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace nvfp4
