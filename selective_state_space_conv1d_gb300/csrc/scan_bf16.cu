// scan_bf16.cu - instantiates the selective-scan kernels for bf16 storage.
#include <type_traits>

#include "scan_kernel.cuh"

namespace mamba {
cudaError_t launch_scan_bf16(const ScanArgs& a, const ScanPlan& p, float* ws, cudaStream_t s) {
  return scan::launch_dtype<__nv_bfloat16>(a, p, ws, s);
}
}  // namespace mamba
