// ssm_step.cu - batched T=1 selective-SSM step with fused softplus, D skip and
// SiLU(z) gate, in place on one layer's slab of the persistent state.
//
// mamba-rs inference.rs step chain F9 (SSM step) + F10 (y * gate), fused as in
// the mixed engine's gather + step + gate kernel; the state slab of layer l
// starts at l * batch * d_inner * d_state (`GpuInferenceState::ssm_offset`).
//
// Design (GB300): the step is pure streaming of the f32 state (read once,
// written once: 2 * 4 * N bytes per (batch, channel)).  Each lane owns one
// group of P = min(N, 16) consecutive states of one channel and moves them with
// 16-byte loads / stores; the N/P lanes of a row are adjacent, so a warp
// touches one contiguous span of the state.  A lane serves 4 batch rows of its
// channel: A2 = -exp(A_log) log2(e) is computed once for them, and the loads of
// all 4 rows are issued before any arithmetic (one memory round trip with
// 4 x 32 B of state in flight per lane); B / C rows are 16-byte loads shared
// through L1.  The lanes' partial C . h are combined with an xor butterfly,
// the same pairwise tree the prefill kernel uses, so one step equals a T=1
// prefill bit for bit.
#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

constexpr int kMaxThreads = 256;
constexpr int kChannels = 32;  // channels per CTA
constexpr int kRows = 4;       // batch rows per thread (loads of all rows issued together)

// P consecutive values at p (16-byte vector loads when `vec`), widened to f32.
template <int P, typename T>
__device__ __forceinline__ void load_group(const T* p, float (&o)[P], bool vec) {
  if constexpr (sizeof(T) == 4 && P % 4 == 0) {
    if (vec) {
#pragma unroll
      for (int j = 0; j < P; j += 4) {
        const float4 v = *reinterpret_cast<const float4*>(p + j);
        o[j] = v.x; o[j + 1] = v.y; o[j + 2] = v.z; o[j + 3] = v.w;
      }
      return;
    }
  } else if constexpr (sizeof(T) == 2 && P % 8 == 0) {
    if (vec) {
#pragma unroll
      for (int g = 0; g < P; g += 8) {
        const uint4 v = *reinterpret_cast<const uint4*>(p + g);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          o[g + 2 * i] = __uint_as_float(w[i] << 16);
          o[g + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
      }
      return;
    }
  }
#pragma unroll
  for (int j = 0; j < P; ++j) o[j] = to_f32(p[j]);
}

template <int P>
__device__ __forceinline__ void store_group(float* p, const float (&o)[P], bool vec) {
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

// grid: (channel block, batch block); a CTA covers 32 channels x (bt * kRows)
// batch rows; lane -> (batch sub-row, channel, state group), groups fastest.
template <int N, typename Tin>
__global__ void __launch_bounds__(kMaxThreads) ssm_step_kernel(SsmStepArgs a, int bt, int64_t n_cblk,
                                                            int state_vec, int bc_vec) {
  constexpr int P = group_size(N);
  constexpr int NG = N / P;
  const int64_t cblk = blockIdx.x % n_cblk;
  const int64_t bblk = blockIdx.x / n_cblk;
  const int q = threadIdx.x % NG;
  const int cl = (threadIdx.x / NG) % kChannels;
  const int bl = threadIdx.x / (NG * kChannels);
  const int64_t Di = a.Di;
  const int64_t c = cblk * kChannels + cl;
  const bool cvalid = (bl < bt) && (c < Di);
  const int64_t cc = cvalid ? c : 0;

  float a2[P];
#pragma unroll
  for (int j = 0; j < P; ++j) a2[j] = a2_from_alog(a.A_log[cc * N + q * P + j]);
  const float dtb = a.dt_bias ? a.dt_bias[cc] : 0.0f;
  const float Dc = a.D ? a.D[cc] : 0.0f;
  const bool gate = a.z != nullptr;
  const Tin* U = reinterpret_cast<const Tin*>(a.u);
  const Tin* DT = reinterpret_cast<const Tin*>(a.dt);
  const Tin* Z = reinterpret_cast<const Tin*>(a.z);
  const Tin* Bm = reinterpret_cast<const Tin*>(a.Bm);
  const Tin* Cm = reinterpret_cast<const Tin*>(a.Cm);

  // the state (the HBM traffic) of all kRows rows is requested first, in one
  // round trip; B / C rows, shared by every channel of a batch row, are L1/L2
  // hits and are loaded per row just before use
  float h[kRows][P], uv[kRows], dtv[kRows], zv[kRows];
  int64_t row[kRows], brow[kRows];
  bool valid[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int64_t b = (bblk * bt + bl) * kRows + i;
    valid[i] = cvalid && b < a.B;
    // invalid lanes still join the butterfly (full-warp shuffles); they read row 0
    brow[i] = valid[i] ? b : 0;
    row[i] = brow[i] * Di + cc;
    load_group<P>(a.state + row[i] * N + q * P, h[i], state_vec);
    uv[i] = to_f32(U[row[i]]);
    dtv[i] = to_f32(DT[row[i]]);
    zv[i] = gate ? to_f32(Z[row[i]]) : 0.0f;
  }
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    float Bv[P], Cv[P];
    load_group<P>(Bm + brow[i] * N + q * P, Bv, bc_vec);
    load_group<P>(Cm + brow[i] * N + q * P, Cv, bc_vec);
    const float delta = softplus_f(dtv[i] + dtb);
    const float du = delta * uv[i];
    float part = ssm_token_group<P>(h[i], a2, delta, du, Bv, Cv);
#pragma unroll
    for (int s = 1; s < NG; s *= 2) part = part + __shfl_xor_sync(0xffffffffu, part, s);
    if (valid[i]) {
      store_group<P>(a.state + row[i] * N + q * P, h[i], state_vec);
      if (q == 0) store_out(a.y, row[i], a.y_bf16, ssm_output(part, Dc, uv[i], gate, zv[i]));
    }
  }
}

template <int N, typename Tin>
cudaError_t launch_n(const SsmStepArgs& a, cudaStream_t stream) {
  constexpr int NG = N / group_size(N);
  // 128-thread CTAs (256 when a channel needs 8 lanes): ~5 resident per SM
  const int per_b = NG * kChannels;
  const int bt = per_b >= 128 ? 1 : 128 / per_b;
  const int threads = per_b * bt;
  const int64_t n_cblk = (a.Di + kChannels - 1) / kChannels;
  const int64_t rows_per_cta = (int64_t)bt * kRows;
  const int64_t n_bblk = (a.B + rows_per_cta - 1) / rows_per_cta;
  const int64_t blocks = n_cblk * n_bblk;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const int es = sizeof(Tin);
  const int state_vec = (reinterpret_cast<uintptr_t>(a.state) & 15) == 0;
  const int bc_vec = ((reinterpret_cast<uintptr_t>(a.Bm) | reinterpret_cast<uintptr_t>(a.Cm)) & 15) == 0 &&
                     (N * es) % 16 == 0;
  ssm_step_kernel<N, Tin><<<(unsigned)blocks, threads, 0, stream>>>(a, bt, n_cblk, state_vec, bc_vec);
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
