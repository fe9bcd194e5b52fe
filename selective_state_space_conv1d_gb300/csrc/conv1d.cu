// conv1d.cu - causal depthwise conv1d + SiLU: T-tiled prefill and T=1 step.
//
// Prefill (mamba-rs prefill.rs `prefill_body` F4a, the T-tiled conv burn-in
// with fused SiLU): each thread owns a vector of V channels (one 16-byte load:
// 4 f32 or 8 bf16) and a tile of `tt` tokens.  It rebuilds the K-1 previous
// inputs (the halo) from x, or from the conv state for the first tile, then
// streams its tile keeping the window in registers.  Loads and stores are
// 16-byte and coalesced along the contiguous channel axis; a warp moves
// 32 x 16 B = 512 contiguous bytes per row.  The thread of tile 0 also writes
// the new state: the last K entries of [state, x_0..x_{T-1}].  Tile 0 is the only
// tile that reads the old state (tt >= K), so in-place state update is safe.
//
// Step (inference.rs step chain F4 + F4b; mixed step "conv1d step with
// epilogue SiLU"): one thread per (batch, channel) shifts its K-slot window
// (slot 0 oldest), appends x, applies the taps and SiLU, and writes the
// window back; K = 4 moves the window as one 16-byte load / store.
#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

template <typename T, int V>
struct Vec;  // V elements of T in one 16-byte (or scalar) access

template <>
struct Vec<float, 4> {
  static __device__ __forceinline__ void load(const float* p, float (&o)[4]) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
  }
  static __device__ __forceinline__ void store(float* p, const float (&o)[4]) {
    *reinterpret_cast<float4*>(p) = make_float4(o[0], o[1], o[2], o[3]);
  }
};
template <>
struct Vec<__nv_bfloat16, 8> {
  static __device__ __forceinline__ void load(const __nv_bfloat16* p, float (&o)[8]) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
  static __device__ __forceinline__ void store(__nv_bfloat16* p, const float (&o)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(o[2 * i]));
      const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(o[2 * i + 1]));
      w[i] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
  }
};
template <typename T>
struct Vec<T, 1> {
  static __device__ __forceinline__ void load(const T* p, float (&o)[1]) { o[0] = to_f32(*p); }
  static __device__ __forceinline__ void store(T* p, const float (&o)[1]) { *p = from_f32<T>(o[0]); }
};

constexpr int kConvThreads = 128;
constexpr int kConvUnroll = 4;

template <int K, typename T, int V>
__global__ void __launch_bounds__(kConvThreads)
    conv1d_silu_prefill_kernel(ConvPrefillArgs a, int tt, int64_t n_cblk, int64_t n_tiles) {
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

  const T* __restrict__ x = reinterpret_cast<const T*>(a.x);
  T* __restrict__ u = reinterpret_cast<T*>(a.u);
  const T* xb = x + b * a.T * a.ld_x + c0;
  T* ub = u + b * a.T * a.ld_u + c0;

  float w[V][K], bias[V];
#pragma unroll
  for (int v = 0; v < V; ++v) {
#pragma unroll
    for (int k = 0; k < K; ++k) w[v][k] = a.w[(c0 + v) * K + k];
    bias[v] = a.bias ? a.bias[c0 + v] : 0.0f;
  }

  // window slot k (k < K-1) holds entry t0+1+k of [state_0..state_{K-1}, x_0, ...]
  constexpr int KW = K > 1 ? K - 1 : 1;
  float win[V][KW];
#pragma unroll
  for (int k = 0; k < K - 1; ++k) {
    const int64_t j = t0 + 1 + k;
    if (j < K) {
#pragma unroll
      for (int v = 0; v < V; ++v)
        win[v][k] = a.state_in ? a.state_in[(b * Di + c0 + v) * K + j] : 0.0f;
    } else {
      float r[V];
      Vec<T, V>::load(xb + (j - K) * a.ld_x, r);
#pragma unroll
      for (int v = 0; v < V; ++v) win[v][k] = r[v];
    }
  }

  for (int64_t t = t0; t < t1; t += kConvUnroll) {
    float xr[kConvUnroll][V];
#pragma unroll
    for (int r = 0; r < kConvUnroll; ++r)
      if (t + r < t1) Vec<T, V>::load(xb + (t + r) * a.ld_x, xr[r]);
#pragma unroll
    for (int r = 0; r < kConvUnroll; ++r) {
      if (t + r < t1) {
        float o[V];
#pragma unroll
        for (int v = 0; v < V; ++v) {
          float s[K];
#pragma unroll
          for (int k = 0; k < K - 1; ++k) s[k] = win[v][k];
          s[K - 1] = xr[r][v];
          o[v] = silu_f(conv_taps<K>(w[v], s, bias[v]));
#pragma unroll
          for (int k = 0; k + 1 < K - 1; ++k) win[v][k] = win[v][k + 1];
          if (K > 1) win[v][KW - 1] = xr[r][v];
        }
        Vec<T, V>::store(ub + (t + r) * a.ld_u, o);
      }
    }
  }

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
        float r[V];
        Vec<T, V>::load(xb + (j - K) * a.ld_x, r);
#pragma unroll
        for (int v = 0; v < V; ++v) fin[v][k] = r[v];
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
  const int64_t i = (int64_t)blockIdx.x * kStepThreads + threadIdx.x;  // b * Di + c
  if (i >= a.B * a.Di) return;
  const int64_t c = i % a.Di;
  float* st = a.state + i * K;
  float old[K], s[K], w[K];
  load_window<K>(st, old);
#pragma unroll
  for (int k = 0; k + 1 < K; ++k) s[k] = old[k + 1];
  s[K - 1] = to_f32(reinterpret_cast<const T*>(a.x)[i]);
#pragma unroll
  for (int k = 0; k < K; ++k) w[k] = a.w[c * K + k];
  const float bias = a.bias ? a.bias[c] : 0.0f;
  reinterpret_cast<T*>(a.u)[i] = from_f32<T>(silu_f(conv_taps<K>(w, s, bias)));
  store_window<K>(st, s);
}

template <int K, typename T>
cudaError_t prefill_launch(const ConvPrefillArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  constexpr int VV = 16 / sizeof(T);
  const int es = sizeof(T);
  const bool vec = (reinterpret_cast<uintptr_t>(a.x) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(a.u) % 16 == 0) && ((a.ld_x * es) % 16 == 0) &&
                   ((a.ld_u * es) % 16 == 0) && (a.Di % VV == 0);
  const int V = vec ? VV : 1;
  const int64_t ncv = (a.Di + V - 1) / V;
  // tokens per thread: enough threads for ~2 full waves, at least K (tile 0
  // must be the only reader of the old state), a multiple of the unroll
  const int64_t want_threads = (int64_t)dev.sm_count * 2048 * 2;
  int64_t tt = (a.B * a.T * ncv + want_threads - 1) / want_threads;
  tt = ((tt + kConvUnroll - 1) / kConvUnroll) * kConvUnroll;
  tt = tt < 8 ? 8 : (tt > 256 ? 256 : tt);
  if (tt < K) tt = ((K + kConvUnroll - 1) / kConvUnroll) * kConvUnroll;
  const int64_t n_tiles = (a.T + tt - 1) / tt;
  const int64_t n_cblk = (ncv + kConvThreads - 1) / kConvThreads;
  const int64_t blocks = n_cblk * n_tiles * a.B;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  if (vec)
    conv1d_silu_prefill_kernel<K, T, VV>
        <<<(unsigned)blocks, kConvThreads, 0, stream>>>(a, (int)tt, n_cblk, n_tiles);
  else
    conv1d_silu_prefill_kernel<K, T, 1>
        <<<(unsigned)blocks, kConvThreads, 0, stream>>>(a, (int)tt, n_cblk, n_tiles);
  return cudaGetLastError();
}

template <int K, typename T>
cudaError_t step_launch(const ConvStepArgs& a, cudaStream_t stream) {
  const int64_t n = a.B * a.Di;
  const int64_t blocks = (n + kStepThreads - 1) / kStepThreads;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  conv1d_silu_step_kernel<K, T><<<(unsigned)blocks, kStepThreads, 0, stream>>>(a);
  return cudaGetLastError();
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
  return a.bf16 ? step_dispatch_k<__nv_bfloat16>(a, stream) : step_dispatch_k<float>(a, stream);
}

}  // namespace mamba
