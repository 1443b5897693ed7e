// pa_selftest.cu -- a self-test of the failure path every kernel's waits
// share: one warp waits on an mbarrier phase that nothing completes (a copy
// that never lands), gives up after the library's bounded wait, records
// PA_ERR_TIMEOUT in the device status word and exits.  No fault, no trap: the
// context stays usable.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int *status) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);  // one arrival expected; none will come
    fence_mbar_init();
  }
  __syncthreads();
  const bool done = __all_sync(0xffffffffu, mbar_wait(b, 0));
  if (!done && threadIdx.x == 0) record_error(status, PA_ERR_TIMEOUT);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int pa_selftest_wait_timeout(pa_stream_t stream) {
  int *status = device_status();
  if (!status) return PA_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
