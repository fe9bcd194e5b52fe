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
// fused).  A thread owns a group of P = min(N, 8) consecutive states of one
// channel (N/P adjacent threads per channel).  Two kernels share that mapping
// and the arithmetic:
//  * ring_step_kernel (the main path): a persistent grid of SMs x resident CTAs;
//    each CTA walks a contiguous range of (channel block, batch row) tiles.  One
//    producer thread streams every tile's state, conv window, x/u, dt, z and
//    B/C rows into a ring of shared-memory stages with bulk asynchronous copies
//    (cp.async.bulk, completion on an mbarrier per stage); four consumer warps
//    take each stage into registers, release it, compute and store.  Bytes in
//    flight are set by the ring size, not by registers or by waves of CTAs.
//  * step_kernel (any alignment / shape): each thread serves kRows batch rows
//    and issues all their loads before any arithmetic (one memory round trip).
// The threads' partial C . h are summed with an xor butterfly in the prefill's
// order, so one step equals a T=1 prefill bit for bit, and the fused step equals
// conv step + SSM step bit for bit (u is rounded to the storage dtype exactly as
// the separate conv step stores it).
#include <atomic>

#include "../../include/mamba_ssm.h"
#include "async_copy.cuh"
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
  grid_dependency_begin();
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
    uxv[i] = to_f32(UX[brow[i] * a.ld_ux + cc]);
    dtv[i] = to_f32(DT[brow[i] * a.ld_dt + cc]);
    zv[i] = gate ? to_f32(Z[brow[i] * a.ld_z + cc]) : 0.0f;
  }
  float Bn[P], Cn[P];  // B / C of the next row, fetched one row ahead
  load_group<P>(Bm + brow[0] * a.ld_B + q * P, Bn, bc_vec);
  load_group<P>(Cm + brow[0] * a.ld_C + q * P, Cn, bc_vec);

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
      load_group<P>(Bm + brow[i + 1] * a.ld_B + q * P, Bn, bc_vec);
      load_group<P>(Cm + brow[i + 1] * a.ld_C + q * P, Cn, bc_vec);
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

// ------------------------------------------------------------ ring path --
namespace ring {
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp (lane 0 issues)
constexpr int kMaxStages = 16;
constexpr int kBarBytes = 2 * kMaxStages * 8;  // full[kMaxStages], empty[kMaxStages]
constexpr long long kWaitLimit = 1ll << 31;    // SM cycles (about a second)
// shared memory per CTA for the stages: 32 KB (5 stages of the 6 KB decode
// tile).  Measured on the 24-layer batch-128 fused decode: 24-48 KB rings run
// a layer in 7.03-7.09 us, 64 KB in 7.14, 96 KB in 7.9 (fewer CTAs per SM),
// 12-16 KB in 7.29 (too few bytes in flight per CTA)
#ifndef MAMBA_STEP_RING_BYTES
#define MAMBA_STEP_RING_BYTES (32 * 1024)
#endif
constexpr int kRingBytes = MAMBA_STEP_RING_BYTES;
}  // namespace ring

__host__ __device__ constexpr int align16(int x) { return (x + 15) & ~15; }

// One stage = one (channel block, batch row) tile: byte offsets of its parts.
template <int N, int K, typename Tin, bool FUSE>
struct RingTile {
  static constexpr int P = group_size(N);
  static constexpr int NG = N / P;
  static constexpr int CB = ring::kConsumers / NG;  // channels per tile
  static constexpr int es = sizeof(Tin);
  static constexpr int kState = 0;                               // [CB][N] f32
  static constexpr int kConv = kState + CB * N * 4;              // [CB][K] f32 (fused)
  static constexpr int kUX = kConv + (FUSE ? CB * K * 4 : 0);    // x (fused) or u: [CB]
  static constexpr int kDT = kUX + align16(CB * es);
  static constexpr int kZ = kDT + align16(CB * es);
  static constexpr int kB = kZ + align16(CB * es);               // B row: [N]
  static constexpr int kC = kB + align16(N * es);                // C row: [N]
  static constexpr int kBytes = (kC + align16(N * es) + 127) & ~127;
  // stages in the ring: as many as fit ring::kRingBytes, 2..kMaxStages
  static constexpr int kStages = ring::kRingBytes / kBytes < 2 ? 2
                                 : (ring::kRingBytes / kBytes > ring::kMaxStages ? ring::kMaxStages
                                                                                 : ring::kRingBytes / kBytes);
  static constexpr int kSmem = ring::kBarBytes + kStages * kBytes;
};

__device__ int g_device_faults = 0;  // MAMBA_FAULT_* bits, set by bounded waits that gave up

__device__ __forceinline__ void flag_fault(int bit) { atomicOr(&g_device_faults, bit); }

template <int P>
__device__ __forceinline__ void store_group_cs(float* p, const float (&o)[P]) {
  if constexpr (P % 4 == 0) {
#pragma unroll
    for (int j = 0; j < P; j += 4)
      __stcs(reinterpret_cast<float4*>(p + j), make_float4(o[j], o[j + 1], o[j + 2], o[j + 3]));
  } else {
#pragma unroll
    for (int j = 0; j < P; ++j) __stcs(p + j, o[j]);
  }
}

// Tiles are numbered cblk * B + b; CTA i takes the contiguous range
// [n_tiles * i / grid, n_tiles * (i + 1) / grid), so consecutive tiles of a CTA
// share a channel block and its parameters stay in registers.
template <int N, int K, typename Tin, bool FUSE>
__global__ void __launch_bounds__(ring::kThreads) ring_step_kernel(StepArgs args, int64_t n_tiles) {
  using L = RingTile<N, K, Tin, FUSE>;
  constexpr int stages = L::kStages;
  constexpr int P = L::P, NG = L::NG, CB = L::CB, es = L::es;
  constexpr int KK = FUSE ? K : 1;
  extern __shared__ __align__(128) unsigned char smem[];
  const SsmStepArgs& a = args.s;
  const uint32_t bars = smem_u32(smem);
  const auto full = [&](int s) { return bars + 8u * s; };
  const auto empty = [&](int s) { return bars + 8u * (ring::kMaxStages + s); };
  const int64_t t_begin = n_tiles * blockIdx.x / gridDim.x;
  const int n_my = (int)(n_tiles * (blockIdx.x + 1) / gridDim.x - t_begin);
  const int64_t Bsz = a.B, Di = a.Di;
  const bool gate = a.z != nullptr;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), ring::kConsumerWarps);
    }
    mbar_fence_init();
  }
  grid_dependency_begin();
  __syncthreads();

  if (warp == ring::kConsumerWarps) {
    // ---- producer: one thread streams the tiles into the ring ----
    if (lane != 0) return;
    const char* UX = reinterpret_cast<const char*>(FUSE ? args.x : a.u);
    const char* DT = reinterpret_cast<const char*>(a.dt);
    const char* Z = reinterpret_cast<const char*>(a.z);
    const char* BM = reinterpret_cast<const char*>(a.Bm);
    const char* CM = reinterpret_cast<const char*>(a.Cm);
    const uint32_t ring0 = bars + ring::kBarBytes;
    int issued = 0;
    int64_t cblk = t_begin / Bsz, b = t_begin - cblk * Bsz;  // walked, not divided, per tile
    int s = 0;
    uint32_t phase = 0;  // parity of this pass over the ring
    for (int i = 0; i < n_my; ++i, b = (b + 1 == Bsz) ? (++cblk, 0) : b + 1) {
      if (i >= stages && !mbar_wait(empty(s), phase ^ 1u, ring::kWaitLimit)) {
        flag_fault(MAMBA_FAULT_RING_WAIT);
        break;
      }
      const int64_t c0 = cblk * CB;
      const uint32_t nch = (uint32_t)(Di - c0 < CB ? Di - c0 : CB);
      const int64_t row = b * Di + c0;
      const uint32_t st = ring0 + (uint32_t)(s * L::kBytes), fb = full(s);
      const uint32_t act = nch * es;
      const uint32_t bytes = nch * N * 4 + (FUSE ? nch * K * 4 : 0) + (gate ? 3 : 2) * act + 2 * N * es;
      mbar_arrive_expect_tx(fb, bytes);
      bulk_g2s(st + L::kState, a.state + row * N, nch * N * 4, fb);
      if constexpr (FUSE) bulk_g2s(st + L::kConv, args.conv_state + row * K, nch * K * 4, fb);
      bulk_g2s(st + L::kUX, UX + (b * a.ld_ux + c0) * es, act, fb);
      bulk_g2s(st + L::kDT, DT + (b * a.ld_dt + c0) * es, act, fb);
      if (gate) bulk_g2s(st + L::kZ, Z + (b * a.ld_z + c0) * es, act, fb);
      bulk_g2s(st + L::kB, BM + b * a.ld_B * es, N * es, fb);
      bulk_g2s(st + L::kC, CM + b * a.ld_C * es, N * es, fb);
      issued = i + 1;
      if (++s == stages) {
        s = 0;
        phase ^= 1u;
      }
    }
    // every issued copy lands before this thread leaves
    for (int i = issued > stages ? issued - stages : 0; i < issued; ++i)
      if (!mbar_wait(full(i % stages), (i / stages) & 1, ring::kWaitLimit)) flag_fault(MAMBA_FAULT_RING_WAIT);
    return;
  }

  // ---- consumers: 128 threads, thread -> (channel cl, state group q) ----
  const int q = threadIdx.x % NG;
  const int cl = threadIdx.x / NG;
  int64_t cur_cblk = -1;
  float a2[P], w[KK], dtb = 0.0f, Dc = 0.0f, cb = 0.0f;
  int64_t cblk = t_begin / Bsz, b = t_begin - cblk * Bsz;  // walked, not divided, per tile
  int s = 0;
  uint32_t phase = 0;
  for (int i = 0; i < n_my; ++i, b = (b + 1 == Bsz) ? (++cblk, 0) : b + 1, s = (s + 1 == stages) ? (phase ^= 1u, 0) : s + 1) {
    const int64_t c = cblk * CB + cl;
    const bool valid = c < Di;
    if (cblk != cur_cblk) {  // per-channel parameters (L2), loaded while the stage lands
      cur_cblk = cblk;
      const int64_t cc = valid ? c : Di - 1;
      const float* al = a.A_log + cc * N + q * P;
#pragma unroll
      for (int j = 0; j < P; ++j) a2[j] = a2_from_alog(al[j]);
      dtb = a.dt_bias ? a.dt_bias[cc] : 0.0f;
      Dc = a.D ? a.D[cc] : 0.0f;
      if constexpr (FUSE) {
#pragma unroll
        for (int k = 0; k < K; ++k) w[k] = args.conv_w[cc * K + k];
        cb = args.conv_b ? args.conv_b[cc] : 0.0f;
      }
    }
    if (!__all_sync(0xffffffffu, mbar_wait(full(s), phase, ring::kWaitLimit))) {
      if (lane == 0) flag_fault(MAMBA_FAULT_RING_WAIT);
      break;
    }
    const unsigned char* sp = smem + ring::kBarBytes + s * L::kBytes;
    float h[P], win[KK], Bv[P], Cv[P];
    load_group<P>(reinterpret_cast<const float*>(sp + L::kState) + cl * N + q * P, h, true);
    if constexpr (FUSE) load_group<KK>(reinterpret_cast<const float*>(sp + L::kConv) + cl * K, win, K % 4 == 0);
    const float uxv = to_f32(reinterpret_cast<const Tin*>(sp + L::kUX)[cl]);
    const float dtv = to_f32(reinterpret_cast<const Tin*>(sp + L::kDT)[cl]);
    const float zv = gate ? to_f32(reinterpret_cast<const Tin*>(sp + L::kZ)[cl]) : 0.0f;
    load_group<P>(reinterpret_cast<const Tin*>(sp + L::kB) + q * P, Bv, true);
    load_group<P>(reinterpret_cast<const Tin*>(sp + L::kC) + q * P, Cv, true);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));  // the stage is in registers: hand it back

    const int64_t row = b * Di + c;
    float uv = uxv;
    if constexpr (FUSE) {
      float sw[KK];
#pragma unroll
      for (int k = 0; k + 1 < K; ++k) sw[k] = win[k + 1];
      sw[K - 1] = uxv;
      uv = to_f32(from_f32<Tin>(silu_f(conv_taps<KK>(w, sw, cb))));
      if (valid && q == 0) store_group<KK>(args.conv_state + row * K, sw, K % 4 == 0);
    }
    const float delta = softplus_f(dtv + dtb);
    const float du = delta * uv;
    float part = ssm_token_group<P>(h, a2, delta, du, Bv, Cv);
#pragma unroll
    for (int sft = 1; sft < NG; sft *= 2) part = part + __shfl_xor_sync(0xffffffffu, part, sft);
    if (valid) {
      store_group_cs<P>(a.state + row * N + q * P, h);
      if (q == 0) store_out(a.y, row, a.y_bf16, ssm_output(part, Dc, uv, gate, zv));
    }
  }
}

// The ring path needs every bulk copy 16-byte aligned and a multiple of 16
// bytes: Di % 8 == 0 (tile offsets and lengths are multiples of 8 channels),
// N * es % 16 == 0 (B / C rows), 16-byte aligned base pointers and row
// strides.
bool ring_eligible(const StepArgs& a, bool fuse) {
  const int es = a.s.in_bf16 ? 2 : 4;
  const auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (a.s.Di % 8 != 0 || (a.s.N * es) % 16 != 0) return false;
  // every row of every input starts on a 16-byte boundary
  for (int64_t ld : {a.s.ld_ux, a.s.ld_dt, a.s.ld_B, a.s.ld_C})
    if ((ld * es) % 16 != 0) return false;
  if (a.s.z && (a.s.ld_z * es) % 16 != 0) return false;
  if (!al(a.s.state) || !al(a.s.dt) || !al(a.s.Bm) || !al(a.s.Cm)) return false;
  if (a.s.z && !al(a.s.z)) return false;
  return fuse ? (al(a.x) && al(a.conv_state)) : al(a.s.u);
}

template <int N, int K, typename Tin, bool FUSE>
cudaError_t launch_ring(const StepArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  using L = RingTile<N, K, Tin, FUSE>;
  constexpr int kSmem = L::kSmem;
  static std::atomic<int> occ_cache[64];
  int dev_id = 0;
  cudaError_t e = cudaGetDevice(&dev_id);
  if (e != cudaSuccess) return e;
  if (dev_id < 0 || dev_id >= 64) return cudaErrorInvalidDevice;
  int occ = occ_cache[dev_id].load(std::memory_order_relaxed);
  if (occ == 0) {
    if (kSmem > 48 * 1024 &&
        (e = cudaFuncSetAttribute(ring_step_kernel<N, K, Tin, FUSE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kSmem)) != cudaSuccess)
      return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, ring_step_kernel<N, K, Tin, FUSE>, ring::kThreads,
                                                           kSmem)) != cudaSuccess)
      return e;
    occ = occ < 1 ? 1 : occ;
    occ_cache[dev_id].store(occ, std::memory_order_relaxed);
  }
  const int64_t n_cblk = (a.s.Di + L::CB - 1) / L::CB;
  const int64_t n_tiles = n_cblk * a.s.B;
  const int64_t resident = (int64_t)dev.sm_count * occ;
  const int64_t grid = n_tiles < resident ? n_tiles : resident;
  return launch_pdl(true, ring_step_kernel<N, K, Tin, FUSE>, dim3((unsigned)grid), dim3(ring::kThreads), kSmem,
                    stream, a, n_tiles);
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
                     (N * es) % 16 == 0 && (a.s.ld_B * es) % 16 == 0 && (a.s.ld_C * es) % 16 == 0;
  return launch_pdl(true, step_kernel<N, K, Tin, FUSE>, dim3((unsigned)blocks), dim3(threads), 0, stream, a, bt,
                    n_cblk, state_vec, bc_vec);
}

template <int N, int K, typename Tin, bool FUSE>
cudaError_t launch_nk_any(const StepArgs& a, const DeviceInfo& dev, bool use_ring, cudaStream_t s) {
  if constexpr ((N * sizeof(Tin)) % 16 == 0) {
    if (use_ring) return launch_ring<N, K, Tin, FUSE>(a, dev, s);
  }
  return launch_nk<N, K, Tin, FUSE>(a, s);
}

template <int N, typename Tin, bool FUSE>
cudaError_t launch_k(const StepArgs& a, const DeviceInfo& dev, int K, bool r, cudaStream_t s) {
  if constexpr (!FUSE) {
    (void)K;
    return launch_nk_any<N, 1, Tin, false>(a, dev, r, s);
  } else {
    switch (K) {
      case 1: return launch_nk_any<N, 1, Tin, true>(a, dev, r, s);
      case 2: return launch_nk_any<N, 2, Tin, true>(a, dev, r, s);
      case 3: return launch_nk_any<N, 3, Tin, true>(a, dev, r, s);
      case 4: return launch_nk_any<N, 4, Tin, true>(a, dev, r, s);
      case 5: return launch_nk_any<N, 5, Tin, true>(a, dev, r, s);
      case 6: return launch_nk_any<N, 6, Tin, true>(a, dev, r, s);
      case 7: return launch_nk_any<N, 7, Tin, true>(a, dev, r, s);
      case 8: return launch_nk_any<N, 8, Tin, true>(a, dev, r, s);
    }
    return cudaErrorInvalidValue;
  }
}

template <typename Tin, bool FUSE>
cudaError_t launch_t(const StepArgs& a, const DeviceInfo& dev, int K, cudaStream_t s) {
  const bool r = ring_eligible(a, FUSE);
  switch (a.s.N) {
    case 1: return launch_k<1, Tin, FUSE>(a, dev, K, r, s);
    case 2: return launch_k<2, Tin, FUSE>(a, dev, K, r, s);
    case 4: return launch_k<4, Tin, FUSE>(a, dev, K, r, s);
    case 8: return launch_k<8, Tin, FUSE>(a, dev, K, r, s);
    case 16: return launch_k<16, Tin, FUSE>(a, dev, K, r, s);
    case 32: return launch_k<32, Tin, FUSE>(a, dev, K, r, s);
    case 64: return launch_k<64, Tin, FUSE>(a, dev, K, r, s);
  }
  return cudaErrorInvalidValue;
}

// zero strides mean dense rows
SsmStepArgs with_strides(SsmStepArgs a) {
  if (a.ld_ux == 0) a.ld_ux = a.Di;
  if (a.ld_dt == 0) a.ld_dt = a.Di;
  if (a.ld_z == 0) a.ld_z = a.Di;
  if (a.ld_B == 0) a.ld_B = a.N;
  if (a.ld_C == 0) a.ld_C = a.N;
  return a;
}

}  // namespace

cudaError_t launch_ssm_step_batched(const SsmStepArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream) {
  StepArgs s{with_strides(a), nullptr, nullptr, nullptr, nullptr};
  return a.in_bf16 ? launch_t<__nv_bfloat16, false>(s, dev, 1, stream)
                   : launch_t<float, false>(s, dev, 1, stream);
}

cudaError_t launch_mixer_step_batched(const MixerStepArgs& m, const DeviceInfo& dev,
                                      cudaStream_t stream) {
  StepArgs s{with_strides(m.ssm), m.x, m.conv_state, m.conv_w, m.conv_b};
  return m.ssm.in_bf16 ? launch_t<__nv_bfloat16, true>(s, dev, m.K, stream)
                       : launch_t<float, true>(s, dev, m.K, stream);
}

int read_device_faults(bool clear, cudaError_t* err) {
  int v = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&v, g_device_faults, sizeof(int));
  if (e == cudaSuccess && clear && v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_faults, &zero, sizeof(int));
  }
  *err = e;
  return e == cudaSuccess ? v : -1;
}

}  // namespace mamba
