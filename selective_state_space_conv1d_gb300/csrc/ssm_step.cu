// ssm_step.cu - batched T=1 decode step: the SSM step alone, and the fused
// mixer step (conv1d + SiLU step, then SSM step), in place on one layer's slab
// of the persistent states.
//
// mamba-rs inference.rs step chain F4/F4b (conv1d step + SiLU) and F9/F10 (SSM
// step + y * gate); the mixed engine fuses each pair (conv1d step with epilogue
// SiLU; gather + SSM step + gate).  The state slab of layer l starts at
// l * batch * d_inner * {d_conv, d_state} (`GpuInferenceState::conv_offset`,
// `ssm_offset`).  The fused entry point goes one step further and runs both in
// one kernel, so u never leaves registers.
//
// Design (GB300): the step streams the f32 state once in and once out
// (2 * 4 * N bytes per (batch, channel), plus 2 * 4 * K for the conv window when
// fused).  Each lane owns a group of P = min(N, 8) consecutive states of one
// channel (N/P lanes per channel, adjacent) and serves kRows batch rows of it.
// All HBM traffic of those rows -- state groups, conv windows, u/x, dt, z -- is
// requested before any arithmetic (one memory round trip, ~200 B in flight per
// lane); B / C rows, shared by every channel of a batch row, are L1/L2 hits
// fetched one row ahead.  The lanes' partial C . h are summed with an xor
// butterfly in the prefill's order, so one step equals a T=1 prefill bit for
// bit, and the fused step equals conv step + SSM step bit for bit (u is
// rounded to the storage dtype exactly as the separate conv step stores it).
#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

constexpr int kMaxThreads = 256;
constexpr int kChannels = 32;  // channels per CTA
constexpr int kRows = 4;       // batch rows per lane

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

struct StepArgs {
  SsmStepArgs s;
  // fused conv step: x replaces u; conv window slab [B][Di][K]
  const void* x;
  float* conv_state;
  const float* conv_w;
  const float* conv_b;
};

// grid: (channel block, batch block); a CTA covers 32 channels x (bt * kRows)
// batch rows; lane -> (batch sub-row, channel, state group), groups fastest.
template <int N, int K, typename Tin, bool FUSE>
__global__ void __launch_bounds__(kMaxThreads) step_kernel(StepArgs args, int bt, int64_t n_cblk,
                                                           int state_vec, int bc_vec) {
  constexpr int P = group_size(N);
  constexpr int NG = N / P;
  constexpr int KK = FUSE ? K : 1;
  const SsmStepArgs& a = args.s;
  const int64_t cblk = blockIdx.x % n_cblk;
  const int64_t bblk = blockIdx.x / n_cblk;
  const int q = threadIdx.x % NG;
  const int cl = (threadIdx.x / NG) % kChannels;
  const int bl = threadIdx.x / (NG * kChannels);
  const int64_t Di = a.Di;
  const int64_t c = cblk * kChannels + cl;
  const bool cvalid = (bl < bt) && (c < Di);
  const int64_t cc = cvalid ? c : 0;
  const bool gate = a.z != nullptr;
  const Tin* UX = reinterpret_cast<const Tin*>(FUSE ? args.x : a.u);
  const Tin* DT = reinterpret_cast<const Tin*>(a.dt);
  const Tin* Z = reinterpret_cast<const Tin*>(a.z);
  const Tin* Bm = reinterpret_cast<const Tin*>(a.Bm);
  const Tin* Cm = reinterpret_cast<const Tin*>(a.Cm);

  // ---- every HBM access of the kRows rows first: one round trip ----
  float h[kRows][P], win[kRows][KK], uxv[kRows], dtv[kRows], zv[kRows];
  int64_t brow[kRows];
  bool valid[kRows];
#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    const int64_t b = (bblk * bt + bl) * kRows + i;
    valid[i] = cvalid && b < a.B;
    // invalid lanes still join the butterfly (full-warp shuffles); they read row 0
    brow[i] = valid[i] ? b : 0;
    const int64_t row = brow[i] * Di + cc;
    load_group<P>(a.state + row * N + q * P, h[i], state_vec);
    if constexpr (FUSE) load_group<KK>(args.conv_state + row * K, win[i], (K % 4 == 0) && state_vec);
    uxv[i] = to_f32(UX[row]);
    dtv[i] = to_f32(DT[row]);
    zv[i] = gate ? to_f32(Z[row]) : 0.0f;
  }
  float Bn[P], Cn[P];  // B / C of the next row, fetched one row ahead
  load_group<P>(Bm + brow[0] * N + q * P, Bn, bc_vec);
  load_group<P>(Cm + brow[0] * N + q * P, Cn, bc_vec);

  // per-channel parameters (L2-resident), after the loads are in flight
  float a2[P], w[KK];
  const float* al = a.A_log + cc * N + q * P;
#pragma unroll
  for (int j = 0; j < P; ++j) a2[j] = a2_from_alog(al[j]);
  const float dtb = a.dt_bias ? a.dt_bias[cc] : 0.0f;
  const float Dc = a.D ? a.D[cc] : 0.0f;
  float cb = 0.0f;
  if constexpr (FUSE) {
#pragma unroll
    for (int k = 0; k < K; ++k) w[k] = args.conv_w[cc * K + k];
    cb = args.conv_b ? args.conv_b[cc] : 0.0f;
  }

#pragma unroll
  for (int i = 0; i < kRows; ++i) {
    float Bv[P], Cv[P];
#pragma unroll
    for (int j = 0; j < P; ++j) {
      Bv[j] = Bn[j];
      Cv[j] = Cn[j];
    }
    if (i + 1 < kRows) {
      load_group<P>(Bm + brow[i + 1] * N + q * P, Bn, bc_vec);
      load_group<P>(Cm + brow[i + 1] * N + q * P, Cn, bc_vec);
    }
    const int64_t row = brow[i] * Di + cc;
    float uv = uxv[i];
    if constexpr (FUSE) {
      // conv1d step: shift the K-slot window, append x, taps + bias, SiLU; u
      // takes the storage dtype's rounding, as the separate conv step stores it
      float s[KK];
#pragma unroll
      for (int k = 0; k + 1 < K; ++k) s[k] = win[i][k + 1];
      s[K - 1] = uxv[i];
      uv = to_f32(from_f32<Tin>(silu_f(conv_taps<KK>(w, s, cb))));
      if (valid[i] && q == 0) store_group<KK>(args.conv_state + row * K, s, (K % 4 == 0) && state_vec);
    }
    const float delta = softplus_f(dtv[i] + dtb);
    const float du = delta * uv;
    float part = ssm_token_group<P>(h[i], a2, delta, du, Bv, Cv);
#pragma unroll
    for (int sft = 1; sft < NG; sft *= 2) part = part + __shfl_xor_sync(0xffffffffu, part, sft);
    if (valid[i]) {
      store_group<P>(a.state + row * N + q * P, h[i], state_vec);
      if (q == 0) store_out(a.y, row, a.y_bf16, ssm_output(part, Dc, uv, gate, zv[i]));
    }
  }
}

template <int N, int K, typename Tin, bool FUSE>
cudaError_t launch_nk(const StepArgs& a, cudaStream_t stream) {
  constexpr int NG = N / group_size(N);
  // 128-thread CTAs (256 when a channel needs 8 lanes)
  const int per_b = NG * kChannels;
  const int bt = per_b >= 128 ? 1 : 128 / per_b;
  const int threads = per_b * bt;
  const int64_t n_cblk = (a.s.Di + kChannels - 1) / kChannels;
  const int64_t rows_per_cta = (int64_t)bt * kRows;
  const int64_t n_bblk = (a.s.B + rows_per_cta - 1) / rows_per_cta;
  const int64_t blocks = n_cblk * n_bblk;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const int es = sizeof(Tin);
  int state_vec = (reinterpret_cast<uintptr_t>(a.s.state) & 15) == 0;
  if (FUSE) state_vec = state_vec && (reinterpret_cast<uintptr_t>(a.conv_state) & 15) == 0;
  const int bc_vec = ((reinterpret_cast<uintptr_t>(a.s.Bm) | reinterpret_cast<uintptr_t>(a.s.Cm)) & 15) == 0 &&
                     (N * es) % 16 == 0;
  step_kernel<N, K, Tin, FUSE><<<(unsigned)blocks, threads, 0, stream>>>(a, bt, n_cblk, state_vec, bc_vec);
  return cudaGetLastError();
}

template <int N, typename Tin, bool FUSE>
cudaError_t launch_k(const StepArgs& a, int K, cudaStream_t s) {
  if constexpr (!FUSE) {
    (void)K;
    return launch_nk<N, 1, Tin, false>(a, s);
  } else {
    switch (K) {
      case 1: return launch_nk<N, 1, Tin, true>(a, s);
      case 2: return launch_nk<N, 2, Tin, true>(a, s);
      case 3: return launch_nk<N, 3, Tin, true>(a, s);
      case 4: return launch_nk<N, 4, Tin, true>(a, s);
      case 5: return launch_nk<N, 5, Tin, true>(a, s);
      case 6: return launch_nk<N, 6, Tin, true>(a, s);
      case 7: return launch_nk<N, 7, Tin, true>(a, s);
      case 8: return launch_nk<N, 8, Tin, true>(a, s);
    }
    return cudaErrorInvalidValue;
  }
}

template <typename Tin, bool FUSE>
cudaError_t launch_t(const StepArgs& a, int K, cudaStream_t s) {
  switch (a.s.N) {
    case 1: return launch_k<1, Tin, FUSE>(a, K, s);
    case 2: return launch_k<2, Tin, FUSE>(a, K, s);
    case 4: return launch_k<4, Tin, FUSE>(a, K, s);
    case 8: return launch_k<8, Tin, FUSE>(a, K, s);
    case 16: return launch_k<16, Tin, FUSE>(a, K, s);
    case 32: return launch_k<32, Tin, FUSE>(a, K, s);
    case 64: return launch_k<64, Tin, FUSE>(a, K, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_ssm_step_batched(const SsmStepArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream) {
  (void)dev;
  StepArgs s{a, nullptr, nullptr, nullptr, nullptr};
  return a.in_bf16 ? launch_t<__nv_bfloat16, false>(s, 1, stream) : launch_t<float, false>(s, 1, stream);
}

cudaError_t launch_mixer_step_batched(const MixerStepArgs& m, const DeviceInfo& dev,
                                      cudaStream_t stream) {
  (void)dev;
  StepArgs s{m.ssm, m.x, m.conv_state, m.conv_w, m.conv_b};
  return m.ssm.in_bf16 ? launch_t<__nv_bfloat16, true>(s, m.K, stream)
                       : launch_t<float, true>(s, m.K, stream);
}

}  // namespace mamba
