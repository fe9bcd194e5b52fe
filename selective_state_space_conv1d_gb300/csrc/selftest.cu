// selftest.cu - mamba_selftest_bounded_wait: the watchdog path of
// mamba_device_faults, exercised without a fault.
//
// The decode kernels' copy rings hand stages over with mbarriers and never wait
// on one without a limit: a wait that runs out records MAMBA_FAULT_RING_WAIT in
// a device word and the kernel leaves its loop.  This kernel runs that same
// bounded wait (mbar_wait from async_copy.cuh) on a fresh barrier that needs
// one arrival.  With `complete` the CTA arrives first and the wait succeeds at
// once; without it nothing ever arrives, so the wait gives up after `limit`
// cycles, the bit is set and the kernel returns -- the event a ring whose
// copies never land would report, produced with nothing wrong on the device.
#include <cuda_runtime.h>

#include "../../include/mamba_ssm.h"
#include "async_copy.cuh"
#include "launch.h"

namespace mamba {
namespace {

__device__ int g_selftest_faults = 0;

__global__ void __launch_bounds__(32) selftest_wait_kernel(long long limit, int complete) {
  __shared__ __align__(8) unsigned long long bar_word;
  if (threadIdx.x != 0) return;
  const uint32_t bar = smem_u32(&bar_word);
  mbar_init(bar, 1);
  mbar_fence_init();
  if (complete) mbar_arrive(bar);
  if (!mbar_wait(bar, 0, limit)) atomicOr(&g_selftest_faults, MAMBA_FAULT_RING_WAIT);
}

}  // namespace

cudaError_t launch_selftest_wait(long long limit, int complete, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(limit, complete);
  return cudaGetLastError();
}

int read_selftest_faults(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_selftest_faults, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_selftest_faults, &zero, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace mamba
