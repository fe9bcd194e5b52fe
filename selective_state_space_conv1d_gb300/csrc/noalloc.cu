// noalloc.cu - mamba_selective_scan_prefill_noalloc: the selective-scan prefill
// for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the point
// where they run the prefill: an engine whose device memory is planned once at
// start-up and must not grow afterwards, a plugin running inside a host
// framework that owns the allocator, or code that has to keep a fixed memory
// footprint.  mamba_selective_scan_prefill needs a caller workspace to split
// long, narrow prefills along T; this entry point takes that scratch from a
// file-scope device array instead, so the caller passes only inputs and
// outputs.  It allocates nothing and frees nothing.
//
// The array is part of the library image: every GPU that loads the library
// holds kNoallocScratchBytes of it until the process exits.  Its device
// address is looked up once per device (cudaGetSymbolAddress, with that device
// current) on the first call made on that device, so that first call should
// happen before any stream capture.  All calls share the one array and it
// keeps the last call's contents; each call clears the few header words it
// needs (an in-stream memset, no allocation) and overwrites every other byte
// before reading it, but calls that overlap on the GPU (two streams, or two
// threads) race on it and must be ordered by the caller.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstdio>

#include "../../include/mamba_ssm.h"
#include "launch.h"

namespace {

constexpr int64_t kNoallocScratchBytes = MAMBA_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scan_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

thread_local char g_noalloc_err[160];

}  // namespace

// Device address of the scratch array on the current device (set up on the
// first call per device); null and an error code on failure.
static int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(g_noalloc_err, sizeof(g_noalloc_err), "cudaGetDevice: %s", cudaGetErrorString(e));
    return MAMBA_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(g_noalloc_err, sizeof(g_noalloc_err), "device ordinal %d out of range", dev);
    return MAMBA_ERR_UNSUPPORTED;
  }
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_scan_scratch);
    if (e != cudaSuccess || !p) {
      snprintf(g_noalloc_err, sizeof(g_noalloc_err), "cudaGetSymbolAddress(scratch): %s",
               cudaGetErrorString(e));
      cudaGetLastError();
      return MAMBA_ERR_CUDA;
    }
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return MAMBA_OK;
}

extern "C" int mamba_selective_scan_prefill_noalloc(
    void* y, int64_t ld_y, int y_dtype, const void* u, int64_t ld_u, const void* dt, int64_t ld_dt,
    const void* z, int64_t ld_z, const void* Bm, int64_t ld_B, const void* Cm, int64_t ld_C,
    int in_dtype, const float* A_log, const float* D, const float* dt_bias,
    const float* ssm_state_in, float* ssm_state_out, int64_t B, int64_t T, int64_t Di, int64_t N,
    void* stream) {
  int64_t need = mamba_selective_scan_workspace_bytes(B, T, Di, N);
  if (need < 0) return (int)need;  // bad sizes or no usable device; message already set
  if (need > kNoallocScratchBytes) {
    // The plan does not fit: the regular entry point, given the array as its
    // workspace, splits a narrow shape into as many parts as the array holds.
    // A narrow shape that does not split at all within the array is refused:
    // run as one sequential pass it would be many times slower than its split.
    mamba::ScanShapePlan full, lim;
    int rc = mamba::plan_scan_for_current_device(B, T, Di, N, INT64_MAX, &full);
    if (rc == MAMBA_OK) rc = mamba::plan_scan_for_current_device(B, T, Di, N, kNoallocScratchBytes, &lim);
    if (rc != MAMBA_OK) return rc;
    if (full.mode == mamba::kScanSplit && lim.mode != mamba::kScanSplit) {
      char msg[200];
      snprintf(msg, sizeof(msg),
               "mamba_selective_scan_prefill_noalloc: splitting this shape along T needs more than the "
               "%lld bytes of scratch the static array holds (the full split needs %lld)",
               (long long)kNoallocScratchBytes, (long long)need);
      return mamba::set_last_error(MAMBA_ERR_UNSUPPORTED, msg);
    }
    need = kNoallocScratchBytes;
  }
  void* scratch = nullptr;
  if (need > 0) {
    const int rc = noalloc_scratch(&scratch);
    if (rc != MAMBA_OK) return mamba::set_last_error(rc, g_noalloc_err);
  }
  return mamba_selective_scan_prefill(y, ld_y, y_dtype, u, ld_u, dt, ld_dt, z, ld_z, Bm, ld_B, Cm,
                                      ld_C, in_dtype, A_log, D, dt_bias, ssm_state_in,
                                      ssm_state_out, B, T, Di, N, scratch, need, stream);
}
