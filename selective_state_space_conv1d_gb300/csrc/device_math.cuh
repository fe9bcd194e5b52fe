// device_math.cuh - per-token arithmetic shared by every kernel of the mixer
// core, so that the prefill kernels and the T=1 step kernels evaluate the same
// operations in the same order (one step == a T=1 prefill, bit for bit).
//
// Formulas (mamba-rs inference.rs / prefill.rs source views):
//   A      = -exp(A_log)                         (GpuMambaInference::new, exp_negate)
//   delta  = softplus(dt + dt_bias)              (step chain F7, prefill F4c)
//   h      = exp(delta A) h + delta B u          (Mamba-1 selective scan)
//   y      = C . h + D u,  out = y SiLU(z)       (F9 + F10, fused gate)
//   SiLU(x)= x / (1 + exp(-x))                   (mixed step, F4+F4b comment)
//   conv   = bias + sum_k w[k] s[k]              (F4, shift-register window)
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mamba {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// --- programmatic dependent launch --------------------------------------------
// The decode-step kernels are launched with programmatic stream serialisation
// (the prefill kernels plainly; there both calls below are no-ops).  Every
// kernel calls grid_dependency_wait() before its first global memory access:
// that waits until the previous grid on the stream has completed and its
// memory is visible, so the stream order of the library's calls is kept
// exactly.  grid_dependents_launch() lets the next kernel on the
// stream be scheduled once every CTA of this grid has called it (or exited);
// its CTAs then sit in their own wait while this grid finishes, placed on
// whichever SMs have room.  The decode-step kernels signal at entry (the next
// layer's grid has the same shape, and its launch and CTA set-up overlap this
// grid's tail).  The prefill kernels signal after their main loop: a long
// one-wave scan launched early would be placed unevenly over SMs still busy
// with the previous grid and keep that imbalance for its whole run.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_begin() {
  grid_dependents_launch();
  grid_dependency_wait();
}

// --- single MUFU instructions (PTX), flush-to-zero ---------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float r;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// softplus(v) = max(v, 0) + ln(2) log2(1 + 2^(-|v| log2 e)): 2 MUFU + 5 FP ops,
// overflow-free for any v.  The absolute error (~1e-7, from lg2.approx near 1;
// the rounding of 1 + e is below it) is far inside the parity bound even for
// the smallest deltas the mixer sees; v < -88 gives exactly 0 (e flushes).
__device__ __forceinline__ float softplus_f(float v) {
  const float e = ex2_approx(-fabsf(v) * kLog2e);
  return fmaf(lg2_approx(1.0f + e), kLn2, fmaxf(v, 0.0f));
}

// SiLU(x) = x / (1 + e^-x); e overflows to +inf for x < -88 and the result is -0.
__device__ __forceinline__ float silu_f(float x) {
  return x * rcp_approx(1.0f + ex2_approx(-x * kLog2e));
}

// A in base-2 units: exp(delta * A) == 2^(delta * a2) with a2 = -exp(A_log) log2(e).
__device__ __forceinline__ float a2_from_alog(float a_log) { return -expf(a_log) * kLog2e; }

// --- storage conversions ------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

__device__ __forceinline__ void store_out(void* base, int64_t i, int is_bf16, float v) {
  if (is_bf16)
    reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<float*>(base)[i] = v;
}

// --- conv: bias + sum_k w[k] s[k], s[K-1] the newest input -------------------
template <int K>
__device__ __forceinline__ float conv_taps(const float (&w)[K], const float (&s)[K], float bias) {
  float acc = bias;
#pragma unroll
  for (int k = 0; k < K; ++k) acc = fmaf(w[k], s[k], acc);
  return acc;
}

// --- selective-scan token update on a group of P states ----------------------
// Updates h[0..P) in place for one token and returns this group's partial of
// C . h.  P is 1 or even; even groups use packed f32x2 FMA/MUL (rounding is
// that of the scalar ops, so the packing changes no bits).
template <int P>
__device__ __forceinline__ float ssm_token_group(float* h, const float* a2, float delta, float du,
                                                 const float* Bv, const float* Cv) {
  if constexpr (P == 1) {
    const float dA = ex2_approx(delta * a2[0]);
    h[0] = fmaf(dA, h[0], du * Bv[0]);
    return Cv[0] * h[0];
  } else {
    const float2 d2 = make_float2(delta, delta);
    const float2 u2 = make_float2(du, du);
#pragma unroll
    for (int j = 0; j < P; j += 2) {
      const float2 arg = __fmul2_rn(d2, make_float2(a2[j], a2[j + 1]));
      const float2 dA = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
      const float2 x = __fmul2_rn(u2, make_float2(Bv[j], Bv[j + 1]));
      const float2 hn = __ffma2_rn(dA, make_float2(h[j], h[j + 1]), x);
      h[j] = hn.x;
      h[j + 1] = hn.y;
    }
    float2 acc = __fmul2_rn(make_float2(Cv[0], Cv[1]), make_float2(h[0], h[1]));
#pragma unroll
    for (int j = 2; j < P; j += 2)
      acc = __ffma2_rn(make_float2(Cv[j], Cv[j + 1]), make_float2(h[j], h[j + 1]), acc);
    return acc.x + acc.y;
  }
}

// States are handled in groups of group_size(N) = min(N, 8), one group per
// lane; the groups' partials are summed by a pairwise tree (level s adds
// partial i and i + s), which is the order an xor-shuffle butterfly produces.
__host__ __device__ constexpr int group_size(int N) { return N < 8 ? N : 8; }

template <int NG>
__device__ __forceinline__ float tree_sum(float (&part)[NG]) {
#pragma unroll
  for (int s = 1; s < NG; s *= 2)
#pragma unroll
    for (int i = 0; i + s < NG; i += 2 * s) part[i] = part[i] + part[i + s];
  return part[0];
}

// y = C . h + D u, then the SiLU(z) gate.
__device__ __forceinline__ float ssm_output(float yssm, float Dc, float u, bool gate, float z) {
  float y = fmaf(Dc, u, yssm);
  if (gate) y *= silu_f(z);
  return y;
}

}  // namespace mamba
