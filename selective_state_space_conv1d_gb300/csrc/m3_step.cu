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
#include <atomic>

#include "../../include/mamba_ssm.h"
#include "async_copy.cuh"
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

// ------------------------------------------------------------ ring path --
// A persistent grid walks (batch, head) tiles; one producer thread per CTA
// streams each tile's state block [P][N], k and v state rows, and x, k, q rows
// into a ring of shared-memory stages with bulk asynchronous copies (one
// mbarrier per stage); four consumer warps compute from the stage and hand it
// back.  Bytes in flight are set by the ring, not by registers or CTA waves.
namespace m3ring {
constexpr int kConsumerWarps = 4;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxStages = 4;
constexpr int kBarBytes = 2 * kMaxStages * 8;
constexpr int kRingBytes = 64 * 1024;     // shared memory per CTA for the stages
constexpr long long kWaitLimit = 1ll << 31;  // SM cycles (about a second)
}  // namespace m3ring

__device__ int g_m3_faults = 0;

__host__ __device__ constexpr int m3_align16(int x) { return (x + 15) & ~15; }

// byte offsets of one stage's parts for headdim P, d_state N, input size es
struct M3Tile {
  int state, kprev, vprev, x, k, q, bytes;
  __host__ __device__ static M3Tile make(int P, int N, int es) {
    M3Tile t{};
    t.state = 0;
    t.kprev = t.state + P * N * 4;
    t.vprev = t.kprev + N * 4;
    t.x = t.vprev + P * 4;
    t.k = t.x + m3_align16(P * es);
    t.q = t.k + m3_align16(N * es);
    t.bytes = (t.q + m3_align16(N * es) + 127) & ~127;
    return t;
  }
};

template <int N, typename Tin, typename Tout>
__global__ void __launch_bounds__(m3ring::kThreads) m3_ring_kernel(M3StepArgs a, int stages, int64_t n_tiles) {
  constexpr int NG = N / kM3Group;
  constexpr int es = sizeof(Tin);
  extern __shared__ __align__(128) unsigned char smem[];
  const int P = a.P;
  const M3Tile L = M3Tile::make(P, N, es);
  const uint32_t bars = smem_u32(smem);
  const auto full = [&](int s) { return bars + 8u * s; };
  const auto empty = [&](int s) { return bars + 8u * (m3ring::kMaxStages + s); };
  const int64_t t_begin = n_tiles * blockIdx.x / gridDim.x;
  const int n_my = (int)(n_tiles * (blockIdx.x + 1) / gridDim.x - t_begin);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), m3ring::kConsumerWarps);
    }
    mbar_fence_init();
  }
  grid_dependency_begin();
  __syncthreads();

  if (warp == m3ring::kConsumerWarps) {
    // ---- producer ----
    if (lane != 0) return;
    const char* X = reinterpret_cast<const char*>(a.x);
    const char* K = reinterpret_cast<const char*>(a.k);
    const char* Q = reinterpret_cast<const char*>(a.q);
    const uint32_t ring0 = bars + m3ring::kBarBytes;
    int issued = 0, s = 0;
    uint32_t phase = 0;
    for (int i = 0; i < n_my; ++i) {
      if (i >= stages && !mbar_wait(empty(s), phase ^ 1u, m3ring::kWaitLimit)) {
        atomicOr(&g_m3_faults, MAMBA_FAULT_RING_WAIT);
        break;
      }
      const int64_t bh = t_begin + i;
      const uint32_t st = ring0 + (uint32_t)(s * L.bytes), fb = full(s);
      const uint32_t bytes = P * N * 4 + N * 4 + P * 4 + P * es + 2 * N * es;
      mbar_arrive_expect_tx(fb, bytes);
      bulk_g2s(st + L.state, a.ssm_state + bh * (int64_t)P * N, P * N * 4, fb);
      bulk_g2s(st + L.kprev, a.k_state + bh * N, N * 4, fb);
      bulk_g2s(st + L.vprev, a.v_state + bh * P, P * 4, fb);
      bulk_g2s(st + L.x, X + bh * P * es, P * es, fb);
      bulk_g2s(st + L.k, K + bh * N * es, N * es, fb);
      bulk_g2s(st + L.q, Q + bh * N * es, N * es, fb);
      issued = i + 1;
      if (++s == stages) {
        s = 0;
        phase ^= 1u;
      }
    }
    for (int i = issued > stages ? issued - stages : 0; i < issued; ++i)
      if (!mbar_wait(full(i % stages), (i / stages) & 1, m3ring::kWaitLimit))
        atomicOr(&g_m3_faults, MAMBA_FAULT_RING_WAIT);
    return;
  }

  // ---- consumers: items (row p, 8-state group q), q fastest ----
  const int items = P * NG;
  int s = 0;
  uint32_t phase = 0;
  for (int i = 0; i < n_my; ++i) {
    const int64_t bh = t_begin + i;
    const int head = (int)(bh % a.H);
    // per-(batch, head) scalars, fetched while the stage lands
    const float alpha = a.alpha[bh], beta = a.beta[bh], gamma = a.gamma[bh];
    const float Dh = a.D ? a.D[head] : 0.0f;
    if (!__all_sync(0xffffffffu, mbar_wait(full(s), phase, m3ring::kWaitLimit))) {
      if (lane == 0) atomicOr(&g_m3_faults, MAMBA_FAULT_RING_WAIT);
      break;
    }
    const unsigned char* sp = smem + m3ring::kBarBytes + s * L.bytes;
    const float* s_h = reinterpret_cast<const float*>(sp + L.state);
    const float* s_kp = reinterpret_cast<const float*>(sp + L.kprev);
    const float* s_vp = reinterpret_cast<const float*>(sp + L.vprev);
    const Tin* s_x = reinterpret_cast<const Tin*>(sp + L.x);
    const Tin* s_k = reinterpret_cast<const Tin*>(sp + L.k);
    const Tin* s_q = reinterpret_cast<const Tin*>(sp + L.q);
    float* hs = a.ssm_state + bh * (int64_t)P * N;
    for (int idx0 = 0; idx0 < items; idx0 += m3ring::kConsumers) {  // uniform over the warps
      const int idx = idx0 + threadIdx.x;
      const bool valid = idx < items;
      const int p = valid ? idx / NG : 0;
      const int q = idx % NG;
      const int n0 = q * kM3Group;
      float h[kM3Group];
      {
        const float4 v0 = reinterpret_cast<const float4*>(s_h + (p * N + n0))[0];
        const float4 v1 = reinterpret_cast<const float4*>(s_h + (p * N + n0))[1];
        h[0] = v0.x; h[1] = v0.y; h[2] = v0.z; h[3] = v0.w;
        h[4] = v1.x; h[5] = v1.y; h[6] = v1.z; h[7] = v1.w;
      }
      const float xp = to_f32(s_x[p]);
      const float bv = beta * s_vp[p];
      const float gx = gamma * xp;
      float kp[kM3Group], kc[kM3Group], qc[kM3Group];
#pragma unroll
      for (int j = 0; j < kM3Group; ++j) {
        kp[j] = s_kp[n0 + j];
        kc[j] = to_f32(s_k[n0 + j]);
        qc[j] = to_f32(s_q[n0 + j]);
      }
#pragma unroll
      for (int j = 0; j < kM3Group; j += 2) {
        const float2 hn = __ffma2_rn(make_float2(alpha, alpha), make_float2(h[j], h[j + 1]),
                                     __ffma2_rn(make_float2(bv, bv), make_float2(kp[j], kp[j + 1]),
                                                __fmul2_rn(make_float2(gx, gx), make_float2(kc[j], kc[j + 1]))));
        h[j] = hn.x;
        h[j + 1] = hn.y;
      }
      float2 acc = __fmul2_rn(make_float2(qc[0], qc[1]), make_float2(h[0], h[1]));
#pragma unroll
      for (int j = 2; j < kM3Group; j += 2)
        acc = __ffma2_rn(make_float2(qc[j], qc[j + 1]), make_float2(h[j], h[j + 1]), acc);
      float part = acc.x + acc.y;
#pragma unroll
      for (int sft = 1; sft < NG; sft *= 2) part = part + __shfl_xor_sync(0xffffffffu, part, sft);
      if (valid) {
        float4* dst = reinterpret_cast<float4*>(hs + (int64_t)p * N + n0);
        __stcs(dst, make_float4(h[0], h[1], h[2], h[3]));
        __stcs(dst + 1, make_float4(h[4], h[5], h[6], h[7]));
        if (q == 0) reinterpret_cast<Tout*>(a.y)[bh * P + p] = from_f32<Tout>(fmaf(Dh, xp, part));
      }
    }
    // hand the current k and x on (read from the stage, before releasing it)
    for (int j = threadIdx.x; j < N; j += m3ring::kConsumers) a.k_state[bh * N + j] = to_f32(s_k[j]);
    for (int j = threadIdx.x; j < P; j += m3ring::kConsumers) a.v_state[bh * P + j] = to_f32(s_x[j]);
    __syncwarp();
    if (lane == 0) mbar_arrive(empty(s));
    if (++s == stages) {
      s = 0;
      phase ^= 1u;
    }
  }
}

bool m3_ring_eligible(const M3StepArgs& a) {
  const int es = a.in_bf16 ? 2 : 4;
  const auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if ((a.P * 4) % 16 || (a.P * es) % 16 || (a.N * es) % 16) return false;
  if (!al(a.ssm_state) || !al(a.k_state) || !al(a.v_state) || !al(a.x) || !al(a.k) || !al(a.q)) return false;
  return 2 * M3Tile::make(a.P, a.N, es).bytes + m3ring::kBarBytes <= 200 * 1024;
}

template <int N, typename Tin, typename Tout>
cudaError_t launch_m3_ring(const M3StepArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const int es = sizeof(Tin);
  const M3Tile L = M3Tile::make(a.P, N, es);
  int stages = m3ring::kRingBytes / L.bytes;
  stages = stages < 2 ? 2 : (stages > m3ring::kMaxStages ? m3ring::kMaxStages : stages);
  const int smem = m3ring::kBarBytes + stages * L.bytes;
  static std::atomic<int> attr_set[64];
  int dev_id = 0;
  cudaError_t e = cudaGetDevice(&dev_id);
  if (e != cudaSuccess) return e;
  if (dev_id < 0 || dev_id >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev_id].load(std::memory_order_relaxed)) {
    if ((e = cudaFuncSetAttribute(m3_ring_kernel<N, Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  200 * 1024)) != cudaSuccess)
      return e;
    attr_set[dev_id].store(1, std::memory_order_relaxed);
  }
  int occ = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, m3_ring_kernel<N, Tin, Tout>, m3ring::kThreads,
                                                         smem)) != cudaSuccess)
    return e;
  occ = occ < 1 ? 1 : occ;
  const int64_t n_tiles = a.B * a.H;
  const int64_t resident = (int64_t)dev.sm_count * occ;
  const int64_t grid = n_tiles < resident ? n_tiles : resident;
  return launch_pdl(true, m3_ring_kernel<N, Tin, Tout>, dim3((unsigned)grid), dim3(m3ring::kThreads), smem, stream, a,
                    stages, n_tiles);
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
cudaError_t launch_m3_t(const M3StepArgs& a, const DeviceInfo& dev, bool ring, cudaStream_t s) {
  if (ring)
    return a.y_bf16 ? launch_m3_ring<N, Tin, __nv_bfloat16>(a, dev, s) : launch_m3_ring<N, Tin, float>(a, dev, s);
  return a.y_bf16 ? launch_m3_o<N, Tin, __nv_bfloat16>(a, s) : launch_m3_o<N, Tin, float>(a, s);
}

template <typename Tin>
cudaError_t launch_m3_n(const M3StepArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  const bool ring = m3_ring_eligible(a);
  switch (a.N) {
    case 16: return launch_m3_t<16, Tin>(a, dev, ring, s);
    case 32: return launch_m3_t<32, Tin>(a, dev, ring, s);
    case 64: return launch_m3_t<64, Tin>(a, dev, ring, s);
    case 128: return launch_m3_t<128, Tin>(a, dev, ring, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int m3_max_items() { return kM3MaxItems * kM3Threads; }

cudaError_t launch_m3_step_batched(const M3StepArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  return a.in_bf16 ? launch_m3_n<__nv_bfloat16>(a, dev, stream) : launch_m3_n<float>(a, dev, stream);
}

int read_m3_faults(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_m3_faults, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_m3_faults, &zero, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

}  // namespace mamba
