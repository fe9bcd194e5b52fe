// m3_step.cu - batched T=1 step of the Mamba-3 SISO mixer (the trapezoidal
// SSM recurrence), in place on one layer's slabs of its persistent states.
//
// mamba-rs 0.2.1 mamba3_siso/gpu/inference.rs: `Mamba3GpuInferenceState` keeps
// per layer an SSM state [batch][nh][hd][ds], a k state (the previous token's
// B after RoPE) [batch][nh][ds] and a v state (the previous x) [batch][nh][hd];
// step F6 `m3_step_fwd` takes them with the current x, k (B after RoPE) and q
// (C after RoPE), the per-(batch, head) alpha / beta / gamma of F5, and D, on a
// (batch, head) grid with one thread per head-dim row.  The page does not print
// the kernel body; the update read off those arguments is
//   h[p][n] = alpha h[p][n] + beta k_prev[n] v_prev[p] + gamma k[n] x[p]
//   y[p]    = sum_n q[n] h[p][n] + D x[p]
// after which the k state holds k and the v state holds x.
//
// Design (GB300): the step streams the f32 state once in and once out
// (2 * 4 * ds bytes per (batch, head, row)).  One CTA per (batch, head) stages
// the head's vectors (k_prev, k, q over ds; v_prev, x over hd) in shared memory,
// so every thread reads them from there; each thread owns groups of 8
// consecutive states of one row (ds / 8 adjacent threads per row, y summed by
// an xor butterfly) and issues the state loads of all its groups before any
// arithmetic.  The k and v states are rewritten only after a CTA barrier: every
// row of the head reads k_prev and v_prev first.
#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

constexpr int kM3Threads = 256;
constexpr int kM3Group = 8;        // states per thread and row
constexpr int kM3MaxItems = 8;     // (row, group) items per thread: hd * ds / 8 <= 2048

// ITEMS: (row, group) items per thread, all loaded before any arithmetic
template <int N, typename Tin, typename Tout, int ITEMS>
__global__ void __launch_bounds__(kM3Threads) m3_step_kernel(M3StepArgs a) {
  grid_dependency_begin();
  constexpr int NG = N / kM3Group;  // threads per row
  const int P = a.P;
  const int64_t bh = blockIdx.x;    // batch * H + head
  const int head = (int)(bh % a.H);
  __shared__ __align__(16) float s_kp[N], s_k[N], s_q[N];
  extern __shared__ __align__(16) float s_px[];  // v_prev [P], x [P]
  float* s_vp = s_px;
  float* s_x = s_px + P;
  const Tin* X = reinterpret_cast<const Tin*>(a.x);
  const Tin* K = reinterpret_cast<const Tin*>(a.k);
  const Tin* Q = reinterpret_cast<const Tin*>(a.q);
  float* ks = a.k_state + bh * N;
  float* vs = a.v_state + bh * P;
  for (int i = threadIdx.x; i < N; i += kM3Threads) {
    s_kp[i] = ks[i];
    s_k[i] = to_f32(K[bh * N + i]);
    s_q[i] = to_f32(Q[bh * N + i]);
  }
  for (int i = threadIdx.x; i < P; i += kM3Threads) {
    s_vp[i] = vs[i];
    s_x[i] = to_f32(X[bh * P + i]);
  }
  const float alpha = a.alpha[bh], beta = a.beta[bh], gamma = a.gamma[bh];
  const float Dh = a.D ? a.D[head] : 0.0f;
  __syncthreads();

  // items (row p, group q), q fastest; the stride keeps a row's groups in
  // adjacent lanes of one warp (kM3Threads is a multiple of NG)
  const int items = P * NG;
  float* hs = a.ssm_state + bh * (int64_t)P * N;
  float h[ITEMS][kM3Group];
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int idx = threadIdx.x + it * kM3Threads;
    if (idx < items) {
      const float4* src = reinterpret_cast<const float4*>(hs + (int64_t)idx * kM3Group);
      const float4 v0 = src[0], v1 = src[1];
      h[it][0] = v0.x; h[it][1] = v0.y; h[it][2] = v0.z; h[it][3] = v0.w;
      h[it][4] = v1.x; h[it][5] = v1.y; h[it][6] = v1.z; h[it][7] = v1.w;
    }
  }
#pragma unroll
  for (int it = 0; it < ITEMS; ++it) {
    const int idx0 = it * kM3Threads;
    if (idx0 >= items) break;  // uniform over the CTA
    const int idx = threadIdx.x + idx0;
    const bool valid = idx < items;
    const int p = valid ? idx / NG : 0;
    const int q = idx % NG;
    const float xp = s_x[p];
    const float bv = beta * s_vp[p];  // beta v_prev[p]
    const float gx = gamma * xp;      // gamma x[p]
    const int n0 = q * kM3Group;
    float part = 0.0f;
#pragma unroll
    for (int j = 0; j < kM3Group; j += 2) {
      const float2 hn = __ffma2_rn(make_float2(alpha, alpha), make_float2(h[it][j], h[it][j + 1]),
                                   __ffma2_rn(make_float2(bv, bv), make_float2(s_kp[n0 + j], s_kp[n0 + j + 1]),
                                              __fmul2_rn(make_float2(gx, gx),
                                                         make_float2(s_k[n0 + j], s_k[n0 + j + 1]))));
      h[it][j] = hn.x;
      h[it][j + 1] = hn.y;
    }
    float2 acc = __fmul2_rn(make_float2(s_q[n0], s_q[n0 + 1]), make_float2(h[it][0], h[it][1]));
#pragma unroll
    for (int j = 2; j < kM3Group; j += 2)
      acc = __ffma2_rn(make_float2(s_q[n0 + j], s_q[n0 + j + 1]), make_float2(h[it][j], h[it][j + 1]), acc);
    part = acc.x + acc.y;
#pragma unroll
    for (int sft = 1; sft < NG; sft *= 2) part = part + __shfl_xor_sync(0xffffffffu, part, sft);
    if (valid) {
      float4* dst = reinterpret_cast<float4*>(hs + (int64_t)idx * kM3Group);
      __stcs(dst, make_float4(h[it][0], h[it][1], h[it][2], h[it][3]));
      __stcs(dst + 1, make_float4(h[it][4], h[it][5], h[it][6], h[it][7]));
      if (q == 0) reinterpret_cast<Tout*>(a.y)[bh * P + p] = from_f32<Tout>(fmaf(Dh, xp, part));
    }
  }
  // every row has read k_prev and v_prev: hand the current k and x on
  __syncthreads();
  for (int i = threadIdx.x; i < N; i += kM3Threads) ks[i] = s_k[i];
  for (int i = threadIdx.x; i < P; i += kM3Threads) vs[i] = s_x[i];
}

template <int N, typename Tin, typename Tout, int ITEMS>
cudaError_t launch_m3_i(const M3StepArgs& a, cudaStream_t s) {
  const int64_t blocks = a.B * a.H;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const size_t smem = 2 * (size_t)a.P * sizeof(float);
  return launch_pdl(true, m3_step_kernel<N, Tin, Tout, ITEMS>, dim3((unsigned)blocks), dim3(kM3Threads), smem, s, a);
}

template <int N, typename Tin, typename Tout>
cudaError_t launch_m3_o(const M3StepArgs& a, cudaStream_t s) {
  const int64_t per_thread = ((int64_t)a.P * (N / kM3Group) + kM3Threads - 1) / kM3Threads;
  if (per_thread <= 1) return launch_m3_i<N, Tin, Tout, 1>(a, s);
  if (per_thread <= 2) return launch_m3_i<N, Tin, Tout, 2>(a, s);
  if (per_thread <= 4) return launch_m3_i<N, Tin, Tout, 4>(a, s);
  if (per_thread <= kM3MaxItems) return launch_m3_i<N, Tin, Tout, kM3MaxItems>(a, s);
  return cudaErrorInvalidValue;
}

template <int N, typename Tin>
cudaError_t launch_m3_t(const M3StepArgs& a, cudaStream_t s) {
  return a.y_bf16 ? launch_m3_o<N, Tin, __nv_bfloat16>(a, s) : launch_m3_o<N, Tin, float>(a, s);
}

template <typename Tin>
cudaError_t launch_m3_n(const M3StepArgs& a, cudaStream_t s) {
  switch (a.N) {
    case 16: return launch_m3_t<16, Tin>(a, s);
    case 32: return launch_m3_t<32, Tin>(a, s);
    case 64: return launch_m3_t<64, Tin>(a, s);
    case 128: return launch_m3_t<128, Tin>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int m3_max_items() { return kM3MaxItems * kM3Threads; }

cudaError_t launch_m3_step_batched(const M3StepArgs& a, cudaStream_t stream) {
  return a.in_bf16 ? launch_m3_n<__nv_bfloat16>(a, stream) : launch_m3_n<float>(a, stream);
}

}  // namespace mamba
