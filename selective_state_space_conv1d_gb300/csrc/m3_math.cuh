// m3_math.cuh - the per-token arithmetic of the Mamba-3 SISO step's inputs
// (mamba-rs 0.2.1 mamba3_siso/gpu/inference.rs steps F4c and F5: the angle
// accumulation, the pairwise rotation of B and C, alpha / beta / gamma), written
// once for the preparation kernel and the fused step so that both give the
// same bits.  Every product and sum is spelled out (no contraction left to the
// compiler).
#pragma once

#include <cuda_runtime.h>

namespace mamba {

// theta + dt * angle, rounded once
__device__ __forceinline__ float m3_advance_angle(float theta, float dt, float angle) {
  return fmaf(dt, angle, theta);
}

// sin t and cos t of an accumulated angle of any size.  t is reduced to
// r = t - 2 pi k, k = rint(t / (2 pi)), |r| <= pi, by the two-constant method
// of Cody and Waite: 2 pi split into a float head (its nearest float) and a
// float tail (the rest), each product with k formed exactly inside an FMA, so
// r is within a few float ulps of the exact reduction however large k is.  On
// [-pi, pi] the MUFU sine and cosine are accurate to about 2^-21 absolute.
constexpr float kTwoPiHead = 6.2831854820251465f;     // float(2 pi)
constexpr float kTwoPiTail = -1.7484555314695172e-7f;  // float(2 pi - kTwoPiHead)
constexpr float kInvTwoPi = 0.15915493667125702f;      // float(1 / (2 pi))
__device__ __forceinline__ void m3_sincos(float t, float* sn, float* cs) {
  const float k = rintf(__fmul_rn(t, kInvTwoPi));
  const float r = fmaf(-k, kTwoPiTail, fmaf(-k, kTwoPiHead, t));
  *sn = __sinf(r);
  *cs = __cosf(r);
}

// the pair (e, o) turned by +t, given sin t and cos t: (cos t e - sin t o, sin t e + cos t o)
__device__ __forceinline__ void m3_rotate(float sn, float cs, float& e, float& o) {
  const float e2 = fmaf(cs, e, -__fmul_rn(sn, o));
  const float o2 = fmaf(sn, e, __fmul_rn(cs, o));
  e = e2;
  o = o2;
}

// the exponential-trapezoidal weights: alpha = exp(dt A) (the decay over the
// step), beta = (1 - lam) dt alpha (the previous token's input, decayed),
// gamma = lam dt (the current one)
struct M3Weights {
  float alpha, beta, gamma;
};
__device__ __forceinline__ M3Weights m3_weights(float dt, float A, float lam) {
  const float al = expf(__fmul_rn(dt, A));
  return {al, __fmul_rn(__fmul_rn(1.0f - lam, dt), al), __fmul_rn(lam, dt)};
}

}  // namespace mamba
