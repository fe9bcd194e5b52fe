// rmsnorm.cu - RMSNorm of the Mamba-1 block's residual stream:
//
//   out[m][j] = x[m][j] / sqrt(mean_j(x[m][j]^2) + eps) * weight[j]
//
// x is the f32 residual stream, out the normalised activations in f32 or bf16
// (rounded once).  (mamba-rs inference.rs step chain F1 "Save residual +
// RmsNorm", and the mixed-precision chain's f32-in / bf16-out RMSNorm that
// prefill.rs `prefill_body` F1 runs over all rows.)
//
// One warp per row, eight rows per CTA.  A row is read twice: once for the sum
// of squares and once to scale it; the second read hits the L1 cache, so HBM
// sees each row once.  The sum is taken in a fixed order (lane-strided partial
// sums, then a butterfly over the warp), so a row's result does not depend on
// the launch shape.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

constexpr int kRowsPerCta = 8;

template <bool OUT_BF16, bool VEC>
__global__ void __launch_bounds__(32 * kRowsPerCta)
    rmsnorm_kernel(void* __restrict__ out, int64_t ld_out, const float* __restrict__ x, int64_t ld_x,
                   const float* __restrict__ w, float eps, int64_t M, int D, int early) {
  // a grid that fits in one wave lets the next kernel start its set-up at
  // once; a many-wave grid must not let it take SMs early
  if (early) grid_dependents_launch();
  grid_dependency_wait();
  const int lane = threadIdx.x % 32;
  const int64_t row = (int64_t)blockIdx.x * kRowsPerCta + threadIdx.x / 32;
  if (row < M) {
    const float* xr = x + row * ld_x;
    float ss = 0.0f;
    if (VEC) {
      for (int j = 4 * lane; j < D; j += 128) {
        const float4 v = *reinterpret_cast<const float4*>(xr + j);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
      }
    } else {
      for (int j = lane; j < D; j += 32) ss = fmaf(xr[j], xr[j], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss / (float)D + eps);
    if (VEC) {
      for (int j = 4 * lane; j < D; j += 128) {
        const float4 v = *reinterpret_cast<const float4*>(xr + j);
        const float4 g = *reinterpret_cast<const float4*>(w + j);
        const float a = v.x * inv * g.x, b = v.y * inv * g.y, c = v.z * inv * g.z, d = v.w * inv * g.w;
        if (OUT_BF16) {
          __nv_bfloat162 lo = __floats2bfloat162_rn(a, b), hi = __floats2bfloat162_rn(c, d);
          uint2 pk;
          pk.x = *reinterpret_cast<uint32_t*>(&lo);
          pk.y = *reinterpret_cast<uint32_t*>(&hi);
          *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(out) + row * ld_out + j) = pk;
        } else {
          *reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + row * ld_out + j) = make_float4(a, b, c, d);
        }
      }
    } else {
      for (int j = lane; j < D; j += 32) {
        const float v = xr[j] * inv * w[j];
        if (OUT_BF16)
          reinterpret_cast<__nv_bfloat16*>(out)[row * ld_out + j] = __float2bfloat16_rn(v);
        else
          reinterpret_cast<float*>(out)[row * ld_out + j] = v;
      }
    }
  }
  if (!early) grid_dependents_launch();
}

template <bool OUT_BF16>
cudaError_t launch_typed(const RmsNormArgs& a, int sms, cudaStream_t stream) {
  const uintptr_t po = reinterpret_cast<uintptr_t>(a.out), px = reinterpret_cast<uintptr_t>(a.x),
                  pw = reinterpret_cast<uintptr_t>(a.w);
  // 4-column vectors: D, the strides and the bases must keep every row's
  // 4-column groups 16-byte (f32) / 8-byte (bf16) aligned
  const bool vec = a.D % 4 == 0 && a.ld_x % 4 == 0 && a.ld_out % 4 == 0 && px % 16 == 0 && pw % 16 == 0 &&
                   po % (OUT_BF16 ? 8 : 16) == 0;
  const dim3 grid((unsigned)((a.M + kRowsPerCta - 1) / kRowsPerCta)), block(32 * kRowsPerCta);
  const int early = (int64_t)grid.x <= (int64_t)sms * 8;  // 8 CTAs of 256 threads per SM
  if (vec)
    return launch_pdl(true, rmsnorm_kernel<OUT_BF16, true>, grid, block, 0, stream, a.out, a.ld_out, a.x, a.ld_x,
                      a.w, a.eps, a.M, (int)a.D, early);
  return launch_pdl(true, rmsnorm_kernel<OUT_BF16, false>, grid, block, 0, stream, a.out, a.ld_out, a.x, a.ld_x,
                    a.w, a.eps, a.M, (int)a.D, early);
}

}  // namespace

cudaError_t launch_rmsnorm(const RmsNormArgs& a, cudaStream_t stream) {
  if (a.M <= 0 || a.D <= 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  return a.out_bf16 ? launch_typed<true>(a, sms, stream) : launch_typed<false>(a, sms, stream);
}

}  // namespace mamba
