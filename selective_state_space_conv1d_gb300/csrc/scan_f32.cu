// scan_f32.cu - instantiates the selective-scan kernels for f32 storage.
#include <type_traits>

#include "scan_kernel.cuh"

namespace mamba {
cudaError_t launch_scan_f32(const ScanArgs& a, const ScanPlan& p, float* ws, cudaStream_t s) {
  return scan::launch_dtype<float>(a, p, ws, s);
}
}  // namespace mamba
