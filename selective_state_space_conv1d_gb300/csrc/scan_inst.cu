// scan_inst.cu - instantiates the selective-scan kernels for one storage dtype
// and one d_state; the build compiles this file once per (SCAN_BF16, SCAN_N)
// pair and names the entry point launch_scan_<dtype>_<N>.
#include "scan_kernel.cuh"

#if !defined(SCAN_N) || !defined(SCAN_BF16)
#error "compile with -DSCAN_N=<d_state> -DSCAN_BF16=<0|1>"
#endif

#define SCAN_CAT2(a, b) a##b
#define SCAN_CAT(a, b) SCAN_CAT2(a, b)
#if SCAN_BF16
#define SCAN_TIN __nv_bfloat16
#define SCAN_FN SCAN_CAT(launch_scan_bf16_, SCAN_N)
#else
#define SCAN_TIN float
#define SCAN_FN SCAN_CAT(launch_scan_f32_, SCAN_N)
#endif

namespace mamba {
cudaError_t SCAN_FN(const ScanArgs& a, const ScanPlan& p, float* ws, cudaStream_t s) {
  return scan::launch_n<SCAN_N, SCAN_TIN>(a, p, ws, s);
}
}  // namespace mamba
