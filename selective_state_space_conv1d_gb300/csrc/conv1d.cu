// conv1d.cu - causal depthwise conv1d + SiLU: T-tiled prefill and T=1 step.
//
// Prefill (mamba-rs prefill.rs `prefill_body` F4a, the T-tiled conv burn-in
// with fused SiLU): each thread owns 4 consecutive channels (one 16-byte f32 or
// 8-byte bf16 access) and a tile of `tt` tokens.  It rebuilds the K-1 previous
// inputs (the halo) from x, or from the conv state for the first tile, in the
// same round trip as its first batch of rows, then streams the tile in batches
// of 4 rows, loading batch i+1 while batch i computes, with the window in
// registers.  Accesses are coalesced along the contiguous channel axis (a warp
// moves 512 or 256 contiguous bytes per row).  The thread of tile 0 also writes
// the new state: the last K entries of [state, x_0..x_{T-1}].  Tile 0 is the only
// tile that reads the old state (tt >= K), so in-place state update is safe.
//
// Step (inference.rs step chain F4 + F4b; mixed step "conv1d step with
// epilogue SiLU"): one thread per (batch, channel) shifts its K-slot window
// (slot 0 oldest), appends x, applies the taps and SiLU, and writes the
// window back; K = 4 moves the window as one 16-byte load / store.
#include <type_traits>

#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

// Four consecutive channels as one vector access: 16 bytes of f32 or 8 bytes
// of bf16, held raw in registers until used (keeps the register count, and so
// the number of rows in flight per SM, high).
template <typename T>
struct Raw4;
template <>
struct Raw4<float> {
  float4 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ float get(int i) const {
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
  }
  static __device__ __forceinline__ void store(float* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <>
struct Raw4<__nv_bfloat16> {
  uint2 v;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { v = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ float get(int i) const {
    const uint32_t w = i < 2 ? v.x : v.y;
    return __uint_as_float((i & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&o)[4]) {
    uint32_t w[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(o[2 * i]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(o[2 * i + 1]));
      w[i] = lo | (hi << 16);
    }
    *reinterpret_cast<uint2*>(p) = make_uint2(w[0], w[1]);
  }
};
// One channel per access (misaligned or ragged layouts): same arithmetic.
template <typename T>
struct Raw1 {
  T v;
  __device__ __forceinline__ void load(const T* p) { v = *p; }
  __device__ __forceinline__ float get(int) const { return to_f32(v); }
  static __device__ __forceinline__ void store(T* p, const float (&o)[1]) { *p = from_f32<T>(o[0]); }
};

template <typename T, int V>
using RawV = typename std::conditional<V == 4, Raw4<T>, Raw1<T>>::type;

constexpr int kConvThreads = 128;
constexpr int kConvRows = 4;  // rows per batch; the next batch loads while this one computes

template <int K, typename T, int V>
__global__ void __launch_bounds__(kConvThreads)
    conv1d_silu_prefill_kernel(ConvPrefillArgs a, int tt, int64_t n_cblk, int64_t n_tiles) {
  grid_dependency_wait();
  using R = RawV<T, V>;
  // block -> (batch, tile, channel block); channel blocks fastest
  int64_t blk = blockIdx.x;
  const int64_t cblk = blk % n_cblk;
  blk /= n_cblk;
  const int64_t tile = blk % n_tiles;
  const int64_t b = blk / n_tiles;
  const int64_t c0 = (cblk * kConvThreads + threadIdx.x) * V;
  if (c0 >= a.Di) return;
  const int64_t t0 = tile * tt;
  const int64_t t1 = min(a.T, t0 + (int64_t)tt);
  const int64_t Di = a.Di;

  const T* __restrict__ xb = reinterpret_cast<const T*>(a.x) + b * a.T * a.ld_x + c0;
  T* __restrict__ ub = reinterpret_cast<T*>(a.u) + b * a.T * a.ld_u + c0;

  // window slot k (k < K-1) holds entry t0+1+k of [state_0..state_{K-1}, x_0, ...];
  // its x rows are loaded together with the first batch
  constexpr int KW = K > 1 ? K - 1 : 1;
  R halo[KW];
  R cur[kConvRows], nxt[kConvRows];
#pragma unroll
  for (int k = 0; k < K - 1; ++k) {
    const int64_t j = t0 + 1 + k;
    if (j >= K) halo[k].load(xb + (j - K) * a.ld_x);
  }
#pragma unroll
  for (int r = 0; r < kConvRows; ++r)
    if (t0 + r < t1) cur[r].load(xb + (t0 + r) * a.ld_x);

  float w[V][K], bias[V], win[V][KW];
#pragma unroll
  for (int v = 0; v < V; ++v) {
#pragma unroll
    for (int k = 0; k < K; ++k) w[v][k] = a.w[(c0 + v) * K + k];
    bias[v] = a.bias ? a.bias[c0 + v] : 0.0f;
  }
#pragma unroll
  for (int k = 0; k < K - 1; ++k) {
    const int64_t j = t0 + 1 + k;
#pragma unroll
    for (int v = 0; v < V; ++v)
      win[v][k] = j < K ? (a.state_in ? a.state_in[(b * Di + c0 + v) * K + j] : 0.0f) : halo[k].get(v);
  }

#pragma unroll 1
  for (int64_t t = t0; t < t1; t += kConvRows) {
#pragma unroll
    for (int r = 0; r < kConvRows; ++r)
      if (t + kConvRows + r < t1) nxt[r].load(xb + (t + kConvRows + r) * a.ld_x);
#pragma unroll
    for (int r = 0; r < kConvRows; ++r) {
      if (t + r < t1) {
        float o[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
          const float xv = cur[r].get(v);
          float s[K];
#pragma unroll
          for (int k = 0; k < K - 1; ++k) s[k] = win[v][k];
          s[K - 1] = xv;
          o[v] = silu_f(conv_taps<K>(w[v], s, bias[v]));
#pragma unroll
          for (int k = 0; k + 1 < K - 1; ++k) win[v][k] = win[v][k + 1];
          if (K > 1) win[v][KW - 1] = xv;
        }
        R::store(ub + (t + r) * a.ld_u, o);
      }
    }
#pragma unroll
    for (int r = 0; r < kConvRows; ++r) cur[r] = nxt[r];
  }
  // signal late: a long scan that follows should find the SMs evenly free
  grid_dependents_launch();

  if (tile == 0 && a.state_out) {
    // new state = entries T..T+K-1 of [state_0..state_{K-1}, x_0..x_{T-1}];
    // every read happens before any write (in-place safe)
    float fin[V][K];
#pragma unroll
    for (int k = 0; k < K; ++k) {
      const int64_t j = a.T + k;
      if (j < K) {
#pragma unroll
        for (int v = 0; v < V; ++v)
          fin[v][k] = a.state_in ? a.state_in[(b * Di + c0 + v) * K + j] : 0.0f;
      } else {
        R r;
        r.load(xb + (j - K) * a.ld_x);
#pragma unroll
        for (int v = 0; v < V; ++v) fin[v][k] = r.get(v);
      }
    }
#pragma unroll
    for (int v = 0; v < V; ++v)
#pragma unroll
      for (int k = 0; k < K; ++k) a.state_out[(b * Di + c0 + v) * K + k] = fin[v][k];
  }
}

// K = 4 (and 2) windows move as one vector access when the slab is aligned.
template <int K>
__device__ __forceinline__ void load_window(const float* p, float (&s)[K]) {
  const uintptr_t al = reinterpret_cast<uintptr_t>(p);
  if (K == 4 && (al & 15) == 0) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    s[0] = v.x; s[1] = v.y; s[2] = v.z; s[3] = v.w;
  } else if (K == 2 && (al & 7) == 0) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    s[0] = v.x; s[1] = v.y;
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) s[k] = p[k];
  }
}
template <int K>
__device__ __forceinline__ void store_window(float* p, const float (&s)[K]) {
  const uintptr_t al = reinterpret_cast<uintptr_t>(p);
  if (K == 4 && (al & 15) == 0) {
    *reinterpret_cast<float4*>(p) = make_float4(s[0], s[1], s[2], s[3]);
  } else if (K == 2 && (al & 7) == 0) {
    *reinterpret_cast<float2*>(p) = make_float2(s[0], s[1]);
  } else {
#pragma unroll
    for (int k = 0; k < K; ++k) p[k] = s[k];
  }
}

constexpr int kStepThreads = 256;

template <int K, typename T>
__global__ void __launch_bounds__(kStepThreads) conv1d_silu_step_kernel(ConvStepArgs a) {
  grid_dependency_begin();
  const int64_t i = (int64_t)blockIdx.x * kStepThreads + threadIdx.x;  // b * Di + c
  if (i >= a.B * a.Di) return;
  const int64_t c = (a.B * a.Di < (int64_t(1) << 31)) ? (int64_t)((uint32_t)i % (uint32_t)a.Di) : i % a.Di;
  float* st = a.state + i * K;
  float old[K], s[K], w[K];
  load_window<K>(st, old);
  load_window<K>(a.w + c * K, w);
#pragma unroll
  for (int k = 0; k + 1 < K; ++k) s[k] = old[k + 1];
  s[K - 1] = to_f32(reinterpret_cast<const T*>(a.x)[a.ld_x == a.Di ? i : (i - c) / a.Di * a.ld_x + c]);
  const float bias = a.bias ? a.bias[c] : 0.0f;
  reinterpret_cast<T*>(a.u)[i] = from_f32<T>(silu_f(conv_taps<K>(w, s, bias)));
  store_window<K>(st, s);
}

template <int K, typename T>
cudaError_t prefill_launch(const ConvPrefillArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const int es = sizeof(T);
  const int vb = 4 * es;  // bytes of a 4-channel access
  const bool vec = (reinterpret_cast<uintptr_t>(a.x) % vb == 0) &&
                   (reinterpret_cast<uintptr_t>(a.u) % vb == 0) && ((a.ld_x * es) % vb == 0) &&
                   ((a.ld_u * es) % vb == 0) && (a.Di % 4 == 0);
  const int V = vec ? 4 : 1;
  const int64_t ncv = (a.Di + V - 1) / V;
  // tokens per thread: enough threads for ~2 waves at full occupancy, at least
  // K (tile 0 must be the only reader of the old state), a multiple of the batch
  const int64_t want_threads = (int64_t)dev.sm_count * 2048 * 2;
  int64_t tt = (a.B * a.T * ncv + want_threads - 1) / want_threads;
  tt = ((tt + kConvRows - 1) / kConvRows) * kConvRows;
  tt = tt < 8 ? 8 : (tt > 256 ? 256 : tt);
  if (tt < K) tt = ((K + kConvRows - 1) / kConvRows) * kConvRows;
  const int64_t n_tiles = (a.T + tt - 1) / tt;
  const int64_t n_cblk = (ncv + kConvThreads - 1) / kConvThreads;
  const int64_t blocks = n_cblk * n_tiles * a.B;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  if (vec)
    return launch_pdl(false, conv1d_silu_prefill_kernel<K, T, 4>, dim3((unsigned)blocks), dim3(kConvThreads), 0,
                      stream, a, (int)tt, n_cblk, n_tiles);
  return launch_pdl(false, conv1d_silu_prefill_kernel<K, T, 1>, dim3((unsigned)blocks), dim3(kConvThreads), 0,
                    stream, a, (int)tt, n_cblk, n_tiles);
}

template <int K, typename T>
cudaError_t step_launch(const ConvStepArgs& a, cudaStream_t stream) {
  const int64_t n = a.B * a.Di;
  const int64_t blocks = (n + kStepThreads - 1) / kStepThreads;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  return launch_pdl(true, conv1d_silu_step_kernel<K, T>, dim3((unsigned)blocks), dim3(kStepThreads), 0, stream, a);
}

template <typename T>
cudaError_t prefill_dispatch_k(const ConvPrefillArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  switch (a.K) {
    case 1: return prefill_launch<1, T>(a, dev, s);
    case 2: return prefill_launch<2, T>(a, dev, s);
    case 3: return prefill_launch<3, T>(a, dev, s);
    case 4: return prefill_launch<4, T>(a, dev, s);
    case 5: return prefill_launch<5, T>(a, dev, s);
    case 6: return prefill_launch<6, T>(a, dev, s);
    case 7: return prefill_launch<7, T>(a, dev, s);
    case 8: return prefill_launch<8, T>(a, dev, s);
  }
  return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t step_dispatch_k(const ConvStepArgs& a, cudaStream_t s) {
  switch (a.K) {
    case 1: return step_launch<1, T>(a, s);
    case 2: return step_launch<2, T>(a, s);
    case 3: return step_launch<3, T>(a, s);
    case 4: return step_launch<4, T>(a, s);
    case 5: return step_launch<5, T>(a, s);
    case 6: return step_launch<6, T>(a, s);
    case 7: return step_launch<7, T>(a, s);
    case 8: return step_launch<8, T>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_conv1d_silu_prefill(const ConvPrefillArgs& a, const DeviceInfo& dev,
                                       cudaStream_t stream) {
  return a.bf16 ? prefill_dispatch_k<__nv_bfloat16>(a, dev, stream)
                : prefill_dispatch_k<float>(a, dev, stream);
}

cudaError_t launch_conv1d_silu_step(const ConvStepArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream) {
  (void)dev;
  ConvStepArgs d = a;
  if (d.ld_x == 0) d.ld_x = d.Di;  // dense rows
  return d.bf16 ? step_dispatch_k<__nv_bfloat16>(d, stream) : step_dispatch_k<float>(d, stream);
}

}  // namespace mamba
