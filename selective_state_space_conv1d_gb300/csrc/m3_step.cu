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
#include "m3_math.cuh"

namespace mamba {
namespace {

constexpr int kM3Threads = 256;
constexpr int kM3Group = 8;        // states per thread and row
constexpr int kM3MaxItems = 8;     // (row, group) items per thread: hd * ds / 8 <= 2048

// The fused form's inputs of one (batch, head): k_in and q_in turned pair by
// pair by the advanced angle state into the staged k and q (the thread of a
// pair reads and writes its own angle), exactly as the preparation kernel does.
template <int N>
__device__ __forceinline__ void m3_stage_rotated(const M3StepArgs& a, int64_t bh, int tid, int nthreads, float* s_k,
                                                 float* s_q) {
  const float d = a.dt[bh];
  const int64_t b = bh / a.H;
  for (int j = tid; j < N / 2; j += nthreads) {
    float ke = a.k_in[bh * N + 2 * j], ko = a.k_in[bh * N + 2 * j + 1];
    float qe = a.q_in[bh * N + 2 * j], qo = a.q_in[bh * N + 2 * j + 1];
    if (j < a.na) {
      const float t = m3_advance_angle(a.theta[bh * a.na + j], d, a.angles[b * a.na + j]);
      a.theta[bh * a.na + j] = t;
      float sn, cs;
      m3_sincos(t, &sn, &cs);
      m3_rotate(sn, cs, ke, ko);
      m3_rotate(sn, cs, qe, qo);
    }
    s_k[2 * j] = ke;
    s_k[2 * j + 1] = ko;
    s_q[2 * j] = qe;
    s_q[2 * j + 1] = qo;
  }
}

// ITEMS: (row, group) items per thread, all loaded before any arithmetic;
// PREP: the fused form (k, q and alpha / beta / gamma made here)
template <int N, typename Tin, typename Tout, int ITEMS, bool PREP>
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
  if constexpr (PREP) {
    m3_stage_rotated<N>(a, bh, threadIdx.x, kM3Threads, s_k, s_q);
    for (int i = threadIdx.x; i < N; i += kM3Threads) s_kp[i] = ks[i];
  } else {
    for (int i = threadIdx.x; i < N; i += kM3Threads) {
      s_kp[i] = ks[i];
      s_k[i] = to_f32(K[bh * N + i]);
      s_q[i] = to_f32(Q[bh * N + i]);
    }
  }
  for (int i = threadIdx.x; i < P; i += kM3Threads) {
    s_vp[i] = vs[i];
    s_x[i] = to_f32(X[bh * P + i]);
  }
  float alpha, beta, gamma;
  if constexpr (PREP) {
    const M3Weights w = m3_weights(a.dt[bh], a.A[bh], a.lam[bh]);
    alpha = w.alpha;
    beta = w.beta;
    gamma = w.gamma;
  } else {
    alpha = a.alpha[bh];
    beta = a.beta[bh];
    gamma = a.gamma[bh];
  }
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
// shared memory per CTA for the stages: 36 KB (two 17 KB stages of the bench's
// headdim 64 x d_state 64 tile, six CTAs per SM).  Measured on the 24-layer
// batch-128 decode: 18.5 us per layer (fused form 20.1) at 36 KB, 19.2 (20.7)
// at 64 KB, 19.2 (21.2) at 72 KB, 20.3 (21.9) at 104 KB with six stages
constexpr int kRingBytes = 36 * 1024;
constexpr long long kWaitLimit = 1ll << 31;  // SM cycles (about a second)
}  // namespace m3ring

__device__ int g_m3_faults = 0;

__host__ __device__ constexpr int m3_align16(int x) { return (x + 15) & ~15; }

// byte offsets of one stage's parts for headdim P, d_state N, x of es bytes,
// k and q of kq_es bytes, and na angles (the fused form's angle state)
struct M3Tile {
  int state, kprev, vprev, x, k, q, th, bytes;
  __host__ __device__ static M3Tile make(int P, int N, int es, int kq_es, int na) {
    M3Tile t{};
    t.state = 0;
    t.kprev = t.state + P * N * 4;
    t.vprev = t.kprev + N * 4;
    t.x = t.vprev + P * 4;
    t.k = t.x + m3_align16(P * es);
    t.q = t.k + m3_align16(N * kq_es);
    t.th = t.q + m3_align16(N * kq_es);
    t.bytes = (t.th + m3_align16(na * 4) + 127) & ~127;
    return t;
  }
};

// PREP: the fused form.  The stage then carries k_in and q_in (f32) and the
// tile's angles; every consumer thread keeps the same 8-state group for all
// its items (the consumer count is a multiple of N / 8), so it turns that
// group's pairs once per tile from the staged angles, and the first thread of
// each group writes the advanced angles back (nothing reads them from global
// memory in this launch after the stage is filled).
template <int N, typename Tin, typename Tout, bool PREP>
__global__ void __launch_bounds__(m3ring::kThreads) m3_ring_kernel(M3StepArgs a, int stages, int64_t n_tiles) {
  constexpr int NG = N / kM3Group;
  constexpr int es = sizeof(Tin);
  constexpr int kq_es = PREP ? 4 : es;
  static_assert(m3ring::kConsumers % NG == 0, "a consumer thread keeps one 8-state group");
  extern __shared__ __align__(128) unsigned char smem[];
  const int P = a.P;
  const int na = PREP ? a.na : 0;
  const M3Tile L = M3Tile::make(P, N, es, kq_es, na);
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
    const char* K = reinterpret_cast<const char*>(PREP ? static_cast<const void*>(a.k_in) : a.k);
    const char* Q = reinterpret_cast<const char*>(PREP ? static_cast<const void*>(a.q_in) : a.q);
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
      const uint32_t bytes = P * N * 4 + N * 4 + P * 4 + P * es + 2 * N * kq_es + na * 4;
      mbar_arrive_expect_tx(fb, bytes);
      bulk_g2s(st + L.state, a.ssm_state + bh * (int64_t)P * N, P * N * 4, fb);
      bulk_g2s(st + L.kprev, a.k_state + bh * N, N * 4, fb);
      bulk_g2s(st + L.vprev, a.v_state + bh * P, P * 4, fb);
      bulk_g2s(st + L.x, X + bh * P * es, P * es, fb);
      bulk_g2s(st + L.k, K + bh * N * kq_es, N * kq_es, fb);
      bulk_g2s(st + L.q, Q + bh * N * kq_es, N * kq_es, fb);
      if (na > 0) bulk_g2s(st + L.th, a.theta + bh * na, na * 4, fb);
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
    float alpha, beta, gamma;
    if constexpr (PREP) {
      const M3Weights w = m3_weights(a.dt[bh], a.A[bh], a.lam[bh]);
      alpha = w.alpha;
      beta = w.beta;
      gamma = w.gamma;
    } else {
      alpha = a.alpha[bh];
      beta = a.beta[bh];
      gamma = a.gamma[bh];
    }
    const float Dh = a.D ? a.D[head] : 0.0f;
    // the fused form: lane l turns pairs l, l + 32, ... of the tile (each
    // warp all of them: no exchange between warps); their raw angles and dt
    // are fetched while the stage lands
    constexpr int kPairsPerLane = (N / 2 + 31) / 32;
    float ang[kPairsPerLane];
    float d = 0.0f;
    if constexpr (PREP) {
      d = a.dt[bh];
      const int64_t b = bh / a.H;
#pragma unroll
      for (int r = 0; r < kPairsPerLane; ++r) {
        const int j = lane + 32 * r;
        ang[r] = j < na ? a.angles[b * na + j] : 0.0f;
      }
    }
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
    // the fused form: this thread's group of k and q, turned.  Each lane
    // advances its pairs' angles from the staged ones (warp 0 stores them)
    // and takes their sine and cosine; a thread gathers its group's four
    // pairs from the lanes that own them.
    float kr[kM3Group], qr[kM3Group];
    if constexpr (PREP) {
      const int g0 = (threadIdx.x % NG) * kM3Group;
      const float* s_kf = reinterpret_cast<const float*>(sp + L.k);
      const float* s_qf = reinterpret_cast<const float*>(sp + L.q);
      const float* s_th = reinterpret_cast<const float*>(sp + L.th);
      float sn_l[kPairsPerLane], cs_l[kPairsPerLane];
#pragma unroll
      for (int r = 0; r < kPairsPerLane; ++r) {
        const int j = lane + 32 * r;
        float t = 0.0f;
        if (j < na) {
          t = m3_advance_angle(s_th[j], d, ang[r]);
          if (warp == 0) a.theta[bh * na + j] = t;
        }
        m3_sincos(t, &sn_l[r], &cs_l[r]);
      }
#pragma unroll
      for (int j = 0; j < kM3Group; ++j) {
        kr[j] = s_kf[g0 + j];
        qr[j] = s_qf[g0 + j];
      }
#pragma unroll
      for (int i2 = 0; i2 < kM3Group / 2; ++i2) {
        const int j = g0 / 2 + i2;  // this thread's pair; owned by lane j % 32, slot j / 32
        float sn = 0.0f, cs = 1.0f;
#pragma unroll
        for (int r = 0; r < kPairsPerLane; ++r) {
          const float sr = __shfl_sync(0xffffffffu, sn_l[r], j % 32);
          const float cr = __shfl_sync(0xffffffffu, cs_l[r], j % 32);
          if (j / 32 == r) {
            sn = sr;
            cs = cr;
          }
        }
        if (j < na) {
          m3_rotate(sn, cs, kr[2 * i2], kr[2 * i2 + 1]);
          m3_rotate(sn, cs, qr[2 * i2], qr[2 * i2 + 1]);
        }
      }
    }
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
        if constexpr (PREP) {
          kc[j] = kr[j];
          qc[j] = qr[j];
        } else {
          kc[j] = to_f32(s_k[n0 + j]);
          qc[j] = to_f32(s_q[n0 + j]);
        }
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
    // hand the current k and x on (read from the stage, before releasing it;
    // the fused form's turned k from the first thread of each group)
    if constexpr (PREP) {
      if (threadIdx.x < NG) {
#pragma unroll
        for (int j = 0; j < kM3Group; ++j) a.k_state[bh * N + threadIdx.x * kM3Group + j] = kr[j];
      }
    } else {
      for (int j = threadIdx.x; j < N; j += m3ring::kConsumers) a.k_state[bh * N + j] = to_f32(s_k[j]);
    }
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
  const bool prep = a.k_in != nullptr;
  const int es = a.in_bf16 ? 2 : 4;
  const int kq_es = prep ? 4 : es;
  const int na = prep ? a.na : 0;
  const auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if ((a.P * 4) % 16 || (a.P * es) % 16 || (a.N * kq_es) % 16 || (na * 4) % 16) return false;
  if (!al(a.ssm_state) || !al(a.k_state) || !al(a.v_state) || !al(a.x)) return false;
  if (prep ? (!al(a.k_in) || !al(a.q_in) || (na > 0 && !al(a.theta))) : (!al(a.k) || !al(a.q))) return false;
  return 2 * M3Tile::make(a.P, a.N, es, kq_es, na).bytes + m3ring::kBarBytes <= 200 * 1024;
}

template <int N, typename Tin, typename Tout, bool PREP>
cudaError_t launch_m3_ring(const M3StepArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const int es = sizeof(Tin);
  const M3Tile L = M3Tile::make(a.P, N, es, PREP ? 4 : es, PREP ? a.na : 0);
  int stages = m3ring::kRingBytes / L.bytes;
  stages = stages < 2 ? 2 : (stages > m3ring::kMaxStages ? m3ring::kMaxStages : stages);
  const int smem = m3ring::kBarBytes + stages * L.bytes;
  auto kern = m3_ring_kernel<N, Tin, Tout, PREP>;
  static std::atomic<int> attr_set[64];
  int dev_id = 0;
  cudaError_t e = cudaGetDevice(&dev_id);
  if (e != cudaSuccess) return e;
  if (dev_id < 0 || dev_id >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev_id].load(std::memory_order_relaxed)) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024)) != cudaSuccess)
      return e;
    attr_set[dev_id].store(1, std::memory_order_relaxed);
  }
  int occ = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, m3ring::kThreads, smem)) != cudaSuccess)
    return e;
  occ = occ < 1 ? 1 : occ;
  const int64_t n_tiles = a.B * a.H;
  const int64_t resident = (int64_t)dev.sm_count * occ;
  const int64_t grid = n_tiles < resident ? n_tiles : resident;
  return launch_pdl(true, kern, dim3((unsigned)grid), dim3(m3ring::kThreads), smem, stream, a, stages, n_tiles);
}

template <int N, typename Tin, typename Tout, int ITEMS, bool PREP>
cudaError_t launch_m3_i(const M3StepArgs& a, cudaStream_t s) {
  const int64_t blocks = a.B * a.H;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  const size_t smem = 2 * (size_t)a.P * sizeof(float);
  return launch_pdl(true, m3_step_kernel<N, Tin, Tout, ITEMS, PREP>, dim3((unsigned)blocks), dim3(kM3Threads), smem,
                    s, a);
}

template <int N, typename Tin, typename Tout, bool PREP>
cudaError_t launch_m3_o(const M3StepArgs& a, cudaStream_t s) {
  const int64_t per_thread = ((int64_t)a.P * (N / kM3Group) + kM3Threads - 1) / kM3Threads;
  if (per_thread <= 1) return launch_m3_i<N, Tin, Tout, 1, PREP>(a, s);
  if (per_thread <= 2) return launch_m3_i<N, Tin, Tout, 2, PREP>(a, s);
  if (per_thread <= 4) return launch_m3_i<N, Tin, Tout, 4, PREP>(a, s);
  if (per_thread <= kM3MaxItems) return launch_m3_i<N, Tin, Tout, kM3MaxItems, PREP>(a, s);
  return cudaErrorInvalidValue;
}

template <int N, typename Tin, bool PREP>
cudaError_t launch_m3_t(const M3StepArgs& a, const DeviceInfo& dev, bool ring, cudaStream_t s) {
  if (ring)
    return a.y_bf16 ? launch_m3_ring<N, Tin, __nv_bfloat16, PREP>(a, dev, s)
                    : launch_m3_ring<N, Tin, float, PREP>(a, dev, s);
  return a.y_bf16 ? launch_m3_o<N, Tin, __nv_bfloat16, PREP>(a, s) : launch_m3_o<N, Tin, float, PREP>(a, s);
}

template <typename Tin, bool PREP>
cudaError_t launch_m3_n(const M3StepArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  const bool ring = m3_ring_eligible(a);
  switch (a.N) {
    case 16: return launch_m3_t<16, Tin, PREP>(a, dev, ring, s);
    case 32: return launch_m3_t<32, Tin, PREP>(a, dev, ring, s);
    case 64: return launch_m3_t<64, Tin, PREP>(a, dev, ring, s);
    case 128: return launch_m3_t<128, Tin, PREP>(a, dev, ring, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

int m3_max_items() { return kM3MaxItems * kM3Threads; }

cudaError_t launch_m3_step_batched(const M3StepArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  if (a.k_in != nullptr)
    return a.in_bf16 ? launch_m3_n<__nv_bfloat16, true>(a, dev, stream) : launch_m3_n<float, true>(a, dev, stream);
  return a.in_bf16 ? launch_m3_n<__nv_bfloat16, false>(a, dev, stream) : launch_m3_n<float, false>(a, dev, stream);
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
