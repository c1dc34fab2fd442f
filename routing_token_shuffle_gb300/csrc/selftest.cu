// Device-side failure path, exercised without faulting the GPU: one warp waits on an
// mbarrier that nothing ever arrives at. The wait is the library's bounded wait (2 s of
// %globaltimer time); when it gives up, the kernel records a timeout in the workspace
// status word and returns, exactly as the GEMM kernels do when a pipeline stalls.
#include "tc_common.cuh"

namespace smoe {
namespace {

__global__ void timeout_probe_kernel(DeviceStatus* st) {
  pdl_wait_and_trigger();
  __shared__ uint64_t bar;
  __shared__ int never;
  if (threadIdx.x == 0) {
    never = 0;
    tc::mbar_init(&bar, 1);
    tc::mbar_init_fence();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    volatile int* abort = &never;
    if (!tc::mbar_wait(&bar, 0, abort)) record_error(st, kStatusTimeout, kTimeoutProbe, 0);
  }
}

}  // namespace

cudaError_t launch_timeout_probe(DeviceStatus* st, cudaStream_t s) {
  SMOE_LAUNCH(timeout_probe_kernel, 1, 32, 0, s, st);
  return cudaGetLastError();
}

}  // namespace smoe
