// ssm_step.cu - batched T=1 selective-SSM step with fused softplus, D skip and
// SiLU(z) gate, in place on one layer's slab of the persistent state.
//
// mamba-rs inference.rs step chain F9 (SSM step) + F10 (y * gate), fused as in
// the mixed engine's gather + step + gate kernel; the state slab of layer l
// starts at l * batch * d_inner * d_state (`GpuInferenceState::ssm_offset`).
//
// Design (GB300): the step is pure streaming of the f32 state (read once,
// written once: 2 * 4 * N bytes per (batch, channel)).  Each lane owns one
// group of P = min(N, 8) consecutive states of one (batch, channel) row and
// moves them with 16-byte loads / stores; the N/P lanes of a row are adjacent,
// so a warp touches one contiguous span of the state.  A CTA covers 32
// channels x bt batch rows: A2 = -exp(A_log) log2(e) for its channels is
// computed once into shared memory instead of once per batch row.  The lanes'
// partial C . h are combined with an xor butterfly, the same pairwise tree the
// prefill kernel uses, so one step equals a T=1 prefill bit for bit.
#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

constexpr int kThreads = 256;
constexpr int kChannels = 32;  // channels per CTA

template <int P>
__device__ __forceinline__ void load_f32_group(const float* p, float (&o)[P], bool vec) {
  if constexpr (P % 4 == 0) {
    if (vec) {
#pragma unroll
      for (int j = 0; j < P; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(p + j);
        o[j] = v.x; o[j + 1] = v.y; o[j + 2] = v.z; o[j + 3] = v.w;
      }
      return;
    }
  }
#pragma unroll
  for (int j = 0; j < P; ++j) o[j] = p[j];
}
template <int P>
__device__ __forceinline__ void store_f32_group(float* p, const float (&o)[P], bool vec) {
  if constexpr (P % 4 == 0) {
    if (vec) {
#pragma unroll
      for (int j = 0; j < P; j += 4)
        *reinterpret_cast<float4*>(p + j) = make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]);
      return;
    }
  }
#pragma unroll
  for (int j = 0; j < P; ++j) p[j] = o[j];
}

template <int N, typename Tin>
__global__ void __launch_bounds__(kThreads) ssm_step_kernel(SsmStepArgs a, int bt, int64_t n_cblk,
                                                            int state_vec) {
  constexpr int P = group_size(N);
  constexpr int NG = N / P;
  __shared__ float s_a2[kChannels * N];

  const int64_t cblk = blockIdx.x % n_cblk;
  const int64_t bblk = blockIdx.x / n_cblk;
  const int64_t c0 = cblk * kChannels;
  const int64_t Di = a.Di;

  // A2 for this CTA's channels, once
  for (int i = threadIdx.x; i < kChannels * N; i += kThreads) {
    const int64_t ch = c0 + i / N;
    s_a2[i] = ch < Di ? a2_from_alog(a.A_log[ch * N + (i % N)]) : 0.0f;
  }
  __syncthreads();

  // lane -> (batch row, channel, state group); groups fastest, then channels
  const int q = threadIdx.x % NG;
  const int cl = (threadIdx.x / NG) % kChannels;
  const int bl = threadIdx.x / (NG * kChannels);
  const int64_t b = bblk * bt + bl;
  const int64_t c = c0 + cl;
  const bool valid = (bl < bt) && (b < a.B) && (c < Di);
  // invalid lanes still join the butterfly (full-warp shuffles); they read row 0
  const int64_t row = valid ? b * Di + c : 0;
  const int64_t bb = valid ? b : 0;
  const int64_t ccl = valid ? c : 0;

  float* st = a.state + row * N + q * P;
  float h[P], a2[P], Bv[P], Cv[P];
  load_f32_group<P>(st, h, state_vec != 0);
#pragma unroll
  for (int j = 0; j < P; ++j) a2[j] = s_a2[cl * N + q * P + j];
  const Tin* Bm = reinterpret_cast<const Tin*>(a.Bm) + bb * N + q * P;
  const Tin* Cm = reinterpret_cast<const Tin*>(a.Cm) + bb * N + q * P;
#pragma unroll
  for (int j = 0; j < P; ++j) {
    Bv[j] = to_f32(Bm[j]);
    Cv[j] = to_f32(Cm[j]);
  }
  const float uv = to_f32(reinterpret_cast<const Tin*>(a.u)[row]);
  const float dtv = to_f32(reinterpret_cast<const Tin*>(a.dt)[row]);
  const float dtb = a.dt_bias ? a.dt_bias[ccl] : 0.0f;
  const float Dc = a.D ? a.D[ccl] : 0.0f;

  const float delta = softplus_f(dtv + dtb);
  const float du = delta * uv;
  float part = ssm_token_group<P>(h, a2, delta, du, Bv, Cv);
#pragma unroll
  for (int s = 1; s < NG; s *= 2) part = part + __shfl_xor_sync(0xffffffffu, part, s);

  if (valid) {
    store_f32_group<P>(st, h, state_vec != 0);
    if (q == 0) {
      const bool gate = a.z != nullptr;
      const float zv = gate ? to_f32(reinterpret_cast<const Tin*>(a.z)[row]) : 0.0f;
      store_out(a.y, row, a.y_bf16, ssm_output(part, Dc, uv, gate, zv));
    }
  }
}

template <int N, typename Tin>
cudaError_t launch_n(const SsmStepArgs& a, cudaStream_t stream) {
  constexpr int NG = N / group_size(N);
  const int per_b = NG * kChannels;
  const int bt = kThreads / per_b;
  const int64_t n_cblk = (a.Di + kChannels - 1) / kChannels;
  const int64_t n_bblk = (a.B + bt - 1) / bt;
  const int64_t blocks = n_cblk * n_bblk;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const int state_vec = (reinterpret_cast<uintptr_t>(a.state) & 15) == 0;
  ssm_step_kernel<N, Tin><<<(unsigned)blocks, kThreads, 0, stream>>>(a, bt, n_cblk, state_vec);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const SsmStepArgs& a, cudaStream_t s) {
  switch (a.N) {
    case 1: return launch_n<1, Tin>(a, s);
    case 2: return launch_n<2, Tin>(a, s);
    case 4: return launch_n<4, Tin>(a, s);
    case 8: return launch_n<8, Tin>(a, s);
    case 16: return launch_n<16, Tin>(a, s);
    case 32: return launch_n<32, Tin>(a, s);
    case 64: return launch_n<64, Tin>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_ssm_step_batched(const SsmStepArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream) {
  (void)dev;
  return a.in_bf16 ? launch_t<__nv_bfloat16>(a, stream) : launch_t<float>(a, stream);
}

}  // namespace mamba
