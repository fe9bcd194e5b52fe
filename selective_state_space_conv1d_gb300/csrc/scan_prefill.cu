// scan_prefill.cu - chunked selective scan with fused softplus, D skip and
// SiLU(z) gate, continuing from (and returning) the SSM state.
//
// mamba-rs prefill.rs `prefill_body` F4c/F4d computes, per (batch, channel),
//   delta_t = softplus(dt_t + dt_bias),  h_t = exp(delta_t A) h_{t-1} + delta_t B_t u_t,
//   y_t = (C_t . h_t + D u_t) SiLU(z_t),  starting from the persistent state
// ("do NOT zero, we build on top"), with A = -exp(A_log) (inference.rs
// `GpuMambaInference::new`).  The reference routes short prompts to a
// sequential kernel and long ones to a parallel one (`use_parallel(t, ds)`);
// here one kernel covers both, picking its T split from the shape.
//
// Design (GB300):
//  * A CTA owns `ct` consecutive channels of one batch row for all T.  Lanes
//    run along the contiguous channel axis, so every global access of u, dt, z
//    and y is coalesced, and B_t / C_t (shared by all channels of a row) are
//    staged once per CTA and read as shared-memory broadcasts.
//  * u, dt, z, B, C arrive in chunks of tc rows through a 3-deep cp.async
//    ring (16-byte copies, L2-only), so HBM traffic is one read of every
//    input and one write of y; state stays in registers (f32) throughout.
//  * A thread keeps all N states of its channel in registers and walks its
//    rows sequentially.  The state math is packed f32x2 (FFMA2 / FMUL2) plus
//    one MUFU ex2 per state and token; no tensor cores (no contraction).
//  * Narrow shapes (few batch*channel rows, e.g. one 130m layer at batch 1)
//    split each chunk into g segments handled by g thread groups:
//      pass 1: every segment but the last scans from a zero state and keeps
//              its end state and total decay exp(A * sum delta);
//      fold:   one thread per (channel, state) chains the segments' carries;
//      pass 2: every segment rescans from its true carry-in and writes y.
//    The split costs a second exp per state and token but no extra HBM traffic.
#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

constexpr int kStages = 3;
constexpr int kMaxThreads = 256;

struct ScanLayout {
  int tc, ct, es, npad, g, n;
  __host__ __device__ int64_t act_tile() const { return (int64_t)tc * ct * es; }
  __host__ __device__ int64_t bc_tile() const { return (int64_t)tc * npad * es; }
  __host__ __device__ int64_t stage_bytes() const { return 3 * act_tile() + 2 * bc_tile(); }
  __host__ __device__ int64_t fold_offset() const { return kStages * stage_bytes(); }
  __host__ __device__ int64_t fold_bytes() const {
    return g > 1 ? (int64_t)(2 * g + 1) * ct * n * 4 : 0;
  }
  __host__ __device__ int64_t total() const { return fold_offset() + fold_bytes(); }
};

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  const uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int Pending>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(Pending) : "memory");
}

// P consecutive elements of a staged row, widened to f32.
template <int P, typename Tin>
__device__ __forceinline__ void load_group(const Tin* p, float (&o)[P]) {
  if constexpr (sizeof(Tin) == 4 && P % 4 == 0) {
#pragma unroll
    for (int j = 0; j < P; j += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + j);
      o[j] = v.x; o[j + 1] = v.y; o[j + 2] = v.z; o[j + 3] = v.w;
    }
  } else if constexpr (sizeof(Tin) == 2 && P == 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int j = 0; j < P; ++j) o[j] = to_f32(p[j]);
  }
}

// State-only update of a group (pass 1: no output needed).
template <int P>
__device__ __forceinline__ void ssm_state_group(float* h, const float* a2, float delta, float du,
                                                const float* Bv) {
  if constexpr (P == 1) {
    h[0] = fmaf(ex2_approx(delta * a2[0]), h[0], du * Bv[0]);
  } else {
    const float2 d2 = make_float2(delta, delta);
    const float2 u2 = make_float2(du, du);
#pragma unroll
    for (int j = 0; j < P; j += 2) {
      const float2 arg = __fmul2_rn(d2, make_float2(a2[j], a2[j + 1]));
      const float2 dA = make_float2(ex2_approx(arg.x), ex2_approx(arg.y));
      const float2 x = __fmul2_rn(u2, make_float2(Bv[j], Bv[j + 1]));
      const float2 hn = __ffma2_rn(dA, make_float2(h[j], h[j + 1]), x);
      h[j] = hn.x;
      h[j + 1] = hn.y;
    }
  }
}

template <int N, typename Tin>
__global__ void __launch_bounds__(kMaxThreads)
    selective_scan_prefill_kernel(ScanArgs a, ScanLayout L, int ls, int act_vec, int bc_vec,
                                  int64_t n_cblk) {
  constexpr int P = group_size(N);
  constexpr int NG = N / P;
  extern __shared__ __align__(16) unsigned char smem[];

  const int tid = threadIdx.x;
  const int nthr = blockDim.x;
  const int ct = L.ct, gcnt = L.g, tc = L.tc;
  const int cl = tid % ct;
  const int g = tid / ct;
  const int64_t cblk = blockIdx.x % n_cblk;
  const int64_t b = blockIdx.x / n_cblk;
  const int64_t c0 = cblk * ct;
  const int64_t c = c0 + cl;
  const int64_t Di = a.Di, T = a.T;
  const bool active = c < Di;
  const int64_t cc = active ? c : Di - 1;
  const bool gate = a.z != nullptr;

  float a2[N];
#pragma unroll
  for (int n = 0; n < N; ++n) a2[n] = a2_from_alog(a.A_log[cc * N + n]);
  const float dtb = a.dt_bias ? a.dt_bias[cc] : 0.0f;
  const float Dc = a.D ? a.D[cc] : 0.0f;

  float* foldP = reinterpret_cast<float*>(smem + L.fold_offset());  // [g][ct][N]
  float* foldH = foldP + (int64_t)gcnt * ct * N;                    // [g][ct][N]
  float* carry = foldH + (int64_t)gcnt * ct * N;                    // [ct][N]

  float h[N];
  if (gcnt == 1) {
#pragma unroll
    for (int n = 0; n < N; ++n)
      h[n] = (active && a.state_in) ? a.state_in[(b * Di + c) * N + n] : 0.0f;
  } else if (g == 0) {
#pragma unroll
    for (int n = 0; n < N; ++n)
      carry[cl * N + n] = (active && a.state_in) ? a.state_in[(b * Di + c) * N + n] : 0.0f;
  }

  // ---- staging of chunk k (rows k*tc ..) into ring slot `stage` ----
  // source tensor `tens` of the activation tiles (0 u, 1 dt, 2 z) and of B/C
  auto act_src = [&](int tens) {
    return reinterpret_cast<const Tin*>(tens == 0 ? a.u : (tens == 1 ? a.dt : a.z));
  };
  auto act_ld = [&](int tens) { return tens == 0 ? a.ld_u : (tens == 1 ? a.ld_dt : a.ld_z); };
  auto bc_src = [&](int tens) { return reinterpret_cast<const Tin*>(tens == 0 ? a.Bm : a.Cm); };
  auto bc_ld = [&](int tens) { return tens == 0 ? a.ld_B : a.ld_C; };
  const int ntens = gate ? 3 : 2;
  const int es = (int)sizeof(Tin);

  auto issue = [&](int64_t k, int stage) {
    const int64_t row0 = k * tc;
    const int rows = (int)min((int64_t)tc, T - row0);
    unsigned char* sb = smem + stage * L.stage_bytes();
    const int64_t grow0 = b * T + row0;  // global row of the chunk's first token
    if (act_vec) {
      const int gA = ct * es / 16;  // 16-byte granules per tile row
      const int total = ntens * rows * gA;
      for (int i = tid; i < total; i += nthr) {
        const int q = i % gA;
        const int ra = i / gA;
        const int tens = ra / rows;
        const int r = ra - tens * rows;
        const int64_t ch = c0 + (int64_t)q * (16 / es);
        if (ch < Di) {
          const Tin* src = act_src(tens) + (grow0 + r) * act_ld(tens) + ch;
          Tin* dst = reinterpret_cast<Tin*>(sb + tens * L.act_tile()) + r * ct + q * (16 / es);
          cp_async16(dst, src);
        }
      }
    } else {
      const int total = ntens * rows * ct;
      for (int i = tid; i < total; i += nthr) {
        const int e = i % ct;
        const int ra = i / ct;
        const int tens = ra / rows;
        const int r = ra - tens * rows;
        if (c0 + e < Di) {
          Tin* dst = reinterpret_cast<Tin*>(sb + tens * L.act_tile()) + r * ct + e;
          *dst = act_src(tens)[(grow0 + r) * act_ld(tens) + c0 + e];
        }
      }
    }
    unsigned char* sbc = sb + 3 * L.act_tile();
    // granules per B/C row; bc_vec is only ever set when a row is >= 16 bytes
    constexpr int gB = (N * (int)sizeof(Tin)) / 16 > 0 ? (N * (int)sizeof(Tin)) / 16 : 1;
    if (bc_vec && N * (int)sizeof(Tin) >= 16) {
      const int total = 2 * rows * gB;
      for (int i = tid; i < total; i += nthr) {
        const int q = i % gB;
        const int ra = i / gB;
        const int tens = ra / rows;
        const int r = ra - tens * rows;
        const Tin* src = bc_src(tens) + (grow0 + r) * bc_ld(tens) + q * (16 / es);
        Tin* dst = reinterpret_cast<Tin*>(sbc + tens * L.bc_tile()) + r * L.npad + q * (16 / es);
        cp_async16(dst, src);
      }
    } else {
      const int total = 2 * rows * N;
      for (int i = tid; i < total; i += nthr) {
        const int n = i % N;
        const int ra = i / N;
        const int tens = ra / rows;
        const int r = ra - tens * rows;
        Tin* dst = reinterpret_cast<Tin*>(sbc + tens * L.bc_tile()) + r * L.npad + n;
        *dst = bc_src(tens)[(grow0 + r) * bc_ld(tens) + n];
      }
    }
  };

  const int64_t nchunks = (T + tc - 1) / tc;
#pragma unroll 1
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nchunks) issue(s, s);
    cp_async_commit();
  }

#pragma unroll 1
  for (int64_t k = 0; k < nchunks; ++k) {
    cp_async_wait<kStages - 2>();
    __syncthreads();  // chunk k is visible; every thread is done with chunk k-1
    if (k + kStages - 1 < nchunks) issue(k + kStages - 1, (int)((k + kStages - 1) % kStages));
    cp_async_commit();

    const unsigned char* sb = smem + (k % kStages) * L.stage_bytes();
    const Tin* su = reinterpret_cast<const Tin*>(sb);
    const Tin* sdt = reinterpret_cast<const Tin*>(sb + L.act_tile());
    const Tin* sz = reinterpret_cast<const Tin*>(sb + 2 * L.act_tile());
    const Tin* sB = reinterpret_cast<const Tin*>(sb + 3 * L.act_tile());
    const Tin* sC = reinterpret_cast<const Tin*>(sb + 3 * L.act_tile() + L.bc_tile());
    const int rows = (int)min((int64_t)tc, T - k * tc);
    const int r0 = g * ls;
    const int nr = max(0, min(ls, rows - r0));

    if (gcnt > 1) {
      // pass 1: end state and total decay of every segment but the last
      if (g < gcnt - 1) {
        float hl[N];
#pragma unroll
        for (int n = 0; n < N; ++n) hl[n] = 0.0f;
        float sd = 0.0f;
        const int nr1 = active ? nr : 0;
#pragma unroll 1
        for (int i = 0; i < nr1; ++i) {
          const int row = r0 + i;
          const float uv = to_f32(su[row * ct + cl]);
          const float delta = softplus_f(to_f32(sdt[row * ct + cl]) + dtb);
          sd += delta;
          const float du = delta * uv;
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            float Bv[P];
            load_group<P>(sB + row * L.npad + q * P, Bv);
            ssm_state_group<P>(hl + q * P, a2 + q * P, delta, du, Bv);
          }
        }
#pragma unroll
        for (int n = 0; n < N; ++n) {
          foldP[(g * ct + cl) * N + n] = ex2_approx(a2[n] * sd);
          foldH[(g * ct + cl) * N + n] = hl[n];
        }
      }
      __syncthreads();
      // fold: chain the carries through the segments, one (channel, state) per thread
      for (int w = tid; w < ct * N; w += nthr) {
        float H = carry[w];
#pragma unroll 4
        for (int gg = 0; gg < gcnt - 1; ++gg) {
          const int idx = gg * ct * N + w;
          const float hl = foldH[idx];
          foldH[idx] = H;
          H = fmaf(foldP[idx], H, hl);
        }
        foldH[(gcnt - 1) * ct * N + w] = H;
      }
      __syncthreads();
#pragma unroll
      for (int n = 0; n < N; ++n) h[n] = foldH[(g * ct + cl) * N + n];
    }

    // pass 2: scan the segment from its carry-in and write y
    if (active) {
      const int64_t grow = b * T + k * tc + r0;
#pragma unroll 2
      for (int i = 0; i < nr; ++i) {
        const int row = r0 + i;
        const float uv = to_f32(su[row * ct + cl]);
        const float delta = softplus_f(to_f32(sdt[row * ct + cl]) + dtb);
        const float du = delta * uv;
        float part[NG];
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          float Bv[P], Cv[P];
          load_group<P>(sB + row * L.npad + q * P, Bv);
          load_group<P>(sC + row * L.npad + q * P, Cv);
          part[q] = ssm_token_group<P>(h + q * P, a2 + q * P, delta, du, Bv, Cv);
        }
        const float zv = gate ? to_f32(sz[row * ct + cl]) : 0.0f;
        const float yv = ssm_output(tree_sum<NG>(part), Dc, uv, gate, zv);
        store_out(a.y, (grow + i) * a.ld_y + c, a.y_bf16, yv);
      }
    }
    if (gcnt > 1 && rows > 0 && g == (rows - 1) / ls) {
      // the segment holding the chunk's last row hands its state to the next chunk
#pragma unroll
      for (int n = 0; n < N; ++n) carry[cl * N + n] = h[n];
    }
  }
  cp_async_wait<0>();

  if (gcnt == 1) {
    if (active && a.state_out) {
#pragma unroll
      for (int n = 0; n < N; ++n) a.state_out[(b * Di + c) * N + n] = h[n];
    }
  } else {
    __syncthreads();
    if (g == 0 && active && a.state_out) {
#pragma unroll
      for (int n = 0; n < N; ++n) a.state_out[(b * Di + c) * N + n] = carry[cl * N + n];
    }
  }
}

ScanLayout layout_of(const ScanArgs& a, const ScanPlan& p) {
  ScanLayout L;
  L.tc = p.g * p.ls;
  L.ct = p.ct;
  L.es = a.in_bf16 ? 2 : 4;
  L.npad = p.bc_pad;
  L.g = p.g;
  L.n = a.N;
  return L;
}

template <int N, typename Tin>
cudaError_t launch_n(const ScanArgs& a, const ScanPlan& p, cudaStream_t stream) {
  const ScanLayout L = layout_of(a, p);
  const int64_t smem = L.total();
  auto kern = selective_scan_prefill_kernel<N, Tin>;
  static thread_local int opted_device = -1;
  static thread_local int64_t opted_bytes = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  if (smem > 48 * 1024 && (opted_device != dev || opted_bytes < smem)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    opted_device = dev;
    opted_bytes = smem;
  }
  const int64_t n_cblk = (a.Di + p.ct - 1) / p.ct;
  const int64_t blocks = n_cblk * a.B;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  kern<<<(unsigned)blocks, p.ct * p.g, (size_t)smem, stream>>>(a, L, p.ls, p.act_vec, p.bc_vec,
                                                               n_cblk);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const ScanArgs& a, const ScanPlan& p, cudaStream_t s) {
  switch (a.N) {
    case 1: return launch_n<1, Tin>(a, p, s);
    case 2: return launch_n<2, Tin>(a, p, s);
    case 4: return launch_n<4, Tin>(a, p, s);
    case 8: return launch_n<8, Tin>(a, p, s);
    case 16: return launch_n<16, Tin>(a, p, s);
    case 32: return launch_n<32, Tin>(a, p, s);
    case 64: return launch_n<64, Tin>(a, p, s);
  }
  return cudaErrorInvalidValue;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

ScanPlan plan_selective_scan(const ScanArgs& a, const DeviceInfo& dev) {
  ScanPlan p;
  const int es = a.in_bf16 ? 2 : 4;
  const int vw = 16 / es;
  p.stages = kStages;
  p.act_vec = al16(a.u) && al16(a.dt) && (!a.z || al16(a.z)) && (a.ld_u * es) % 16 == 0 &&
              (a.ld_dt * es) % 16 == 0 && (!a.z || (a.ld_z * es) % 16 == 0) && a.Di % vw == 0;
  p.bc_vec = al16(a.Bm) && al16(a.Cm) && (a.ld_B * es) % 16 == 0 && (a.ld_C * es) % 16 == 0 &&
             (a.N * es) % 16 == 0;

  const int64_t chans = a.B * a.Di;
  const int64_t want_warps = 8LL * dev.sm_count;  // two resident warps per scheduler
  int g = 1;
  if (a.T > 64) {
    while (g < 32 && chans * g < want_warps * 32) g *= 2;
  }
  if (g == 1) {
    p.ct = 32;
    p.g = 1;
    p.ls = es == 2 ? 32 : 16;
  } else {
    p.ct = 8;
    if (g < 4) g = 4;  // 8 channels x g segments >= one warp
    p.g = g;
    p.ls = 3;          // odd: segment rows of a warp fall in distinct banks
  }
  // B/C row stride in smem: whole 16-byte granules; with a T split (a warp
  // reads 32/ct different rows) an odd granule count keeps them conflict-free
  for (;;) {
    int gran = (a.N * es + 15) / 16;
    if (p.g > 1 && gran % 2 == 0) gran += 1;
    p.bc_pad = gran * 16 / es;
    p.smem_bytes = layout_of(a, p).total();
    if (p.smem_bytes <= dev.max_smem_optin || p.g <= 4) break;
    p.g /= 2;  // large d_state: fewer segments per chunk until the ring + fold fit
  }
  return p;
}

cudaError_t launch_selective_scan_prefill(const ScanArgs& a, const ScanPlan& p,
                                          const DeviceInfo& dev, cudaStream_t stream) {
  (void)dev;
  return a.in_bf16 ? launch_t<__nv_bfloat16>(a, p, stream) : launch_t<float>(a, p, stream);
}

}  // namespace mamba
