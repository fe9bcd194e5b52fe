// scan_prefill.cu - selective scan over T tokens with fused softplus, D skip
// and SiLU(z) gate, continuing from (and returning) the SSM state.
//
// mamba-rs prefill.rs `prefill_body` F4c/F4d computes, per (batch, channel),
//   delta_t = softplus(dt_t + dt_bias),  h_t = exp(delta_t A) h_{t-1} + delta_t B_t u_t,
//   y_t = (C_t . h_t + D u_t) SiLU(z_t),  starting from the persistent state
// ("do NOT zero, we build on top"), with A = -exp(A_log) (inference.rs
// `GpuMambaInference::new`).  The reference routes short prompts to a
// sequential kernel and long ones to a parallel one (`use_parallel(t, ds)`);
// here the route is picked from the shape (batch x channels vs SM count).
//
// Design (GB300):
//  * One warp per CTA; lane = channel, 32 consecutive channels of one batch
//    row, so every global access of u, dt, z and y is a coalesced row segment
//    and B_t / C_t (shared by all channels) are shared-memory broadcasts.  All
//    synchronisation is __syncwarp; 1-warp CTAs also give fine-grained load
//    balance over the 152 SMs.
//  * u, dt, z, B, C stream in chunks of TC rows through a 3-deep cp.async ring
//    (16-byte copies, L2-only): HBM sees one read of every input and one write
//    of y.  bf16 B/C rows are widened to f32 once per chunk in shared memory.
//  * A lane keeps all N states of its channel in registers (f32) and walks the
//    rows sequentially; two rows are issued together so the exps of the second
//    overlap the state FMAs of the first.  The state math is packed f32x2 plus
//    one MUFU ex2 per state and token; no tensor cores (no contraction).
//  * Route "sequential" (wide shapes: enough batch x channel rows to fill the
//    GPU): one launch, each CTA scans all T for its channels.
//  * Route "T-split" (narrow shapes, e.g. one 130m layer at batch 1): T is cut
//    into P parts.  Launch 1 scans parts 0..P-2 from a zero state and writes
//    each part's end state and total decay exp(A sum delta) to a workspace
//    (plus a snapshot of state_in).  Launch 2 folds the aggregates of the
//    preceding parts into each part's carry-in, then rescans the part from it
//    and writes y; the last part writes state_out.  Cost: the state-only
//    rescan of P-1 parts; no cross-CTA waiting.
#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace {

constexpr int kStages = 3;
constexpr int kLanes = 32;  // channels per CTA (one warp)

template <typename Tin>
struct Tile {
  static constexpr int TC = 16;                            // rows per staged chunk
  static constexpr int LOG_TC = 4;
  static constexpr int ES = sizeof(Tin);
  static constexpr int GA = kLanes * ES / 16;              // 16-byte granules per act row
  static constexpr int LOG_GA = GA == 8 ? 3 : (GA == 4 ? 2 : (GA == 2 ? 1 : 0));
};

template <int N, typename Tin>
struct Smem {
  Tin act[kStages][3][Tile<Tin>::TC][kLanes];  // u, dt, z
  Tin bc[kStages][2][Tile<Tin>::TC][N];        // B, C as staged (storage dtype)
  // bf16 only: this chunk's B, C widened to f32
  float bcf[sizeof(Tin) == 4 ? 1 : 2][sizeof(Tin) == 4 ? 1 : Tile<Tin>::TC][sizeof(Tin) == 4 ? 4 : N];
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

template <int P>
__device__ __forceinline__ void lds_f32(const float* p, float (&o)[P]) {
  if constexpr (P % 4 == 0) {
#pragma unroll
    for (int j = 0; j < P; j += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + j);
      o[j] = v.x; o[j + 1] = v.y; o[j + 2] = v.z; o[j + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < P; ++j) o[j] = p[j];
  }
}

// State-only update (pass 1 of the T split).
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

struct ScanWork {
  float* ws;           // T-split workspace (null for the sequential route)
  int parts;           // P
  int64_t part_len;    // rows per part (the last part may be shorter)
  int64_t n_tiles;     // channel tiles per batch row
  int64_t grid_parts;  // parts covered by this launch's grid
};

enum Mode { kSequential = 0, kPass1 = 1, kPass2 = 2 };

template <int N, typename Tin, int MODE>
__global__ void __launch_bounds__(kLanes) selective_scan_kernel(ScanArgs a, ScanWork w, int act_vec,
                                                                int bc_vec) {
  using TL = Tile<Tin>;
  constexpr int TC = TL::TC;
  constexpr int P = group_size(N);
  constexpr int NG = N / P;
  constexpr bool kBf16 = sizeof(Tin) == 2;
  __shared__ __align__(16) Smem<N, Tin> sm;

  const int lane = threadIdx.x;
  int64_t blk = blockIdx.x;
  const int64_t part = blk % w.grid_parts;
  blk /= w.grid_parts;
  const int64_t tile = blk % w.n_tiles;
  const int64_t b = blk / w.n_tiles;
  const int64_t c0 = tile * kLanes;
  const int64_t c = c0 + lane;
  const int64_t Di = a.Di, T = a.T;
  const bool active = c < Di;
  const int64_t cc = active ? c : Di - 1;
  const bool gate = (MODE != kPass1) && a.z != nullptr;
  const int64_t t_begin = part * w.part_len;
  const int64_t t_end = min(T, t_begin + w.part_len);
  const int64_t BDN = a.B * Di * N;
  const int64_t srow = (b * Di + cc) * N;  // this lane's state row

  float a2[N];
#pragma unroll
  for (int n = 0; n < N; ++n) a2[n] = a2_from_alog(a.A_log[cc * N + n]);
  const float dtb = a.dt_bias ? a.dt_bias[cc] : 0.0f;
  const float Dc = a.D ? a.D[cc] : 0.0f;

  // ---- carry-in ----
  float h[N];
  if (MODE == kSequential) {
#pragma unroll
    for (int n = 0; n < N; ++n) h[n] = (active && a.state_in) ? a.state_in[srow + n] : 0.0f;
  } else if (MODE == kPass1) {
#pragma unroll
    for (int n = 0; n < N; ++n) h[n] = 0.0f;
    if (part == 0 && active) {  // snapshot of the initial state for launch 2
#pragma unroll
      for (int n = 0; n < N; ++n) w.ws[srow + n] = a.state_in ? a.state_in[srow + n] : 0.0f;
    }
  } else {
    // fold the preceding parts, H <- P_j H + Hloc_j, starting from the snapshot
#pragma unroll
    for (int n = 0; n < N; ++n) h[n] = w.ws[srow + n];
    for (int64_t j = 0; j < part; ++j) {
      float pj[N], hj[N];
      lds_f32<N>(w.ws + BDN * (1 + 2 * j) + srow, pj);
      lds_f32<N>(w.ws + BDN * (2 + 2 * j) + srow, hj);
#pragma unroll
      for (int n = 0; n < N; ++n) h[n] = fmaf(pj[n], h[n], hj[n]);
    }
  }

  // ---- staging of chunk k (rows t_begin + k*TC ..) into ring slot `stage` ----
  const int ntens = gate ? 3 : 2;            // pass 1 needs u and dt only
  const int nbc = MODE == kPass1 ? 1 : 2;    // pass 1 needs B only
  auto act_src = [&](int tens) {
    return reinterpret_cast<const Tin*>(tens == 0 ? a.u : (tens == 1 ? a.dt : a.z));
  };
  auto act_ld = [&](int tens) { return tens == 0 ? a.ld_u : (tens == 1 ? a.ld_dt : a.ld_z); };

  auto issue = [&](int64_t k, int stage) {
    const int64_t row0 = t_begin + k * TC;
    const int rows = (int)min((int64_t)TC, t_end - row0);
    const int64_t grow0 = b * T + row0;
    if (act_vec) {
      // granule i: tensor i / (TC*GA), row (i / GA) % TC, granule-in-row i % GA
      const int total = ntens * TC * TL::GA;
      for (int i = lane; i < total; i += kLanes) {
        const int q = i & (TL::GA - 1);
        const int r = (i >> TL::LOG_GA) & (TC - 1);
        const int tens = i >> (TL::LOG_GA + TL::LOG_TC);
        const int64_t ch = c0 + q * (16 / TL::ES);
        if (r < rows && ch < Di)
          cp_async16(&sm.act[stage][tens][r][q * (16 / TL::ES)],
                     act_src(tens) + (grow0 + r) * act_ld(tens) + ch);
      }
    } else {
      for (int tens = 0; tens < ntens; ++tens)
        for (int r = 0; r < rows; ++r)
          if (active) sm.act[stage][tens][r][lane] = act_src(tens)[(grow0 + r) * act_ld(tens) + c];
    }
    constexpr int GB = (N * TL::ES) / 16 > 0 ? (N * TL::ES) / 16 : 1;  // granules per B/C row
    if (bc_vec && N * TL::ES >= 16) {
      const int total = nbc * TC * GB;
      for (int i = lane; i < total; i += kLanes) {
        const int q = i % GB;
        const int r = (i / GB) % TC;
        const int tens = i / (GB * TC);
        const Tin* src = reinterpret_cast<const Tin*>(tens == 0 ? a.Bm : a.Cm);
        const int64_t ld = tens == 0 ? a.ld_B : a.ld_C;
        if (r < rows)
          cp_async16(&sm.bc[stage][tens][r][q * (16 / TL::ES)], src + (grow0 + r) * ld + q * (16 / TL::ES));
      }
    } else {
      for (int i = lane; i < nbc * TC * N; i += kLanes) {
        const int n = i % N;
        const int r = (i / N) % TC;
        const int tens = i / (N * TC);
        const Tin* src = reinterpret_cast<const Tin*>(tens == 0 ? a.Bm : a.Cm);
        const int64_t ld = tens == 0 ? a.ld_B : a.ld_C;
        if (r < rows) sm.bc[stage][tens][r][n] = src[(grow0 + r) * ld + n];
      }
    }
  };

  const int64_t nrows = max((int64_t)0, t_end - t_begin);
  const int64_t nchunks = (nrows + TC - 1) / TC;
#pragma unroll 1
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nchunks) issue(s, s);
    cp_async_commit();
  }

  float sdelta = 0.0f;  // pass 1: sum of delta over the part
#pragma unroll 1
  for (int64_t k = 0; k < nchunks; ++k) {
    cp_async_wait<kStages - 2>();
    __syncwarp();  // chunk k visible to every lane; every lane is done with chunk k-1
    const int stage = (int)(k % kStages);
    const int rows = (int)min((int64_t)TC, nrows - k * TC);
    const float* sB;
    const float* sC;
    if constexpr (kBf16) {
      // widen this chunk's B (and C) rows to f32 once, shared by all lanes
      for (int i = lane; i < nbc * TC * N; i += kLanes) {
        const int n = i % N;
        const int r = (i / N) % TC;
        const int tens = i / (N * TC);
        if (r < rows) sm.bcf[tens][r][n] = to_f32(sm.bc[stage][tens][r][n]);
      }
      __syncwarp();
      sB = &sm.bcf[0][0][0];
      sC = &sm.bcf[nbc - 1][0][0];
    } else {
      sB = reinterpret_cast<const float*>(&sm.bc[stage][0][0][0]);
      sC = reinterpret_cast<const float*>(&sm.bc[stage][1][0][0]);
    }
    if (k + kStages - 1 < nchunks) issue(k + kStages - 1, (int)((k + kStages - 1) % kStages));
    cp_async_commit();

    const Tin* su = &sm.act[stage][0][0][0];
    const Tin* sdt = &sm.act[stage][1][0][0];
    const Tin* sz = &sm.act[stage][2][0][0];

    if (MODE == kPass1) {
      if (active) {
#pragma unroll 2
        for (int r = 0; r < rows; ++r) {
          const float uv = to_f32(su[r * kLanes + lane]);
          const float delta = softplus_f(to_f32(sdt[r * kLanes + lane]) + dtb);
          sdelta += delta;
          const float du = delta * uv;
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            float Bv[P];
            lds_f32<P>(sB + r * N + q * P, Bv);
            ssm_state_group<P>(h + q * P, a2 + q * P, delta, du, Bv);
          }
        }
      }
    } else if (active) {
      const int64_t grow = b * T + t_begin + k * TC;
      int r = 0;
      // two rows per iteration: the second row's exps do not depend on the
      // first row's state update and overlap it
#pragma unroll 1
      for (; r + 1 < rows; r += 2) {
        const float u0 = to_f32(su[r * kLanes + lane]);
        const float u1 = to_f32(su[(r + 1) * kLanes + lane]);
        const float d0 = softplus_f(to_f32(sdt[r * kLanes + lane]) + dtb);
        const float d1 = softplus_f(to_f32(sdt[(r + 1) * kLanes + lane]) + dtb);
        const float z0 = gate ? to_f32(sz[r * kLanes + lane]) : 0.0f;
        const float z1 = gate ? to_f32(sz[(r + 1) * kLanes + lane]) : 0.0f;
        const float du0 = d0 * u0, du1 = d1 * u1;
        float p0[NG], p1[NG];
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          float Bv[P], Cv[P];
          lds_f32<P>(sB + r * N + q * P, Bv);
          lds_f32<P>(sC + r * N + q * P, Cv);
          p0[q] = ssm_token_group<P>(h + q * P, a2 + q * P, d0, du0, Bv, Cv);
        }
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          float Bv[P], Cv[P];
          lds_f32<P>(sB + (r + 1) * N + q * P, Bv);
          lds_f32<P>(sC + (r + 1) * N + q * P, Cv);
          p1[q] = ssm_token_group<P>(h + q * P, a2 + q * P, d1, du1, Bv, Cv);
        }
        store_out(a.y, (grow + r) * a.ld_y + c, a.y_bf16, ssm_output(tree_sum<NG>(p0), Dc, u0, gate, z0));
        store_out(a.y, (grow + r + 1) * a.ld_y + c, a.y_bf16, ssm_output(tree_sum<NG>(p1), Dc, u1, gate, z1));
      }
      if (r < rows) {
        const float u0 = to_f32(su[r * kLanes + lane]);
        const float d0 = softplus_f(to_f32(sdt[r * kLanes + lane]) + dtb);
        const float z0 = gate ? to_f32(sz[r * kLanes + lane]) : 0.0f;
        const float du0 = d0 * u0;
        float p0[NG];
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          float Bv[P], Cv[P];
          lds_f32<P>(sB + r * N + q * P, Bv);
          lds_f32<P>(sC + r * N + q * P, Cv);
          p0[q] = ssm_token_group<P>(h + q * P, a2 + q * P, d0, du0, Bv, Cv);
        }
        store_out(a.y, (grow + r) * a.ld_y + c, a.y_bf16, ssm_output(tree_sum<NG>(p0), Dc, u0, gate, z0));
      }
    }
  }
  cp_async_wait<0>();

  if (!active) return;
  if (MODE == kPass1) {
    float* Pj = w.ws + BDN * (1 + 2 * part) + srow;
    float* Hj = w.ws + BDN * (2 + 2 * part) + srow;
#pragma unroll
    for (int n = 0; n < N; ++n) {
      Pj[n] = ex2_approx(a2[n] * sdelta);
      Hj[n] = h[n];
    }
  } else if (a.state_out && (MODE == kSequential || part == w.parts - 1)) {
#pragma unroll
    for (int n = 0; n < N; ++n) a.state_out[srow + n] = h[n];
  }
}

template <int N, typename Tin>
cudaError_t launch_n(const ScanArgs& a, const ScanPlan& p, float* ws, cudaStream_t stream) {
  ScanWork w;
  w.ws = ws;
  w.parts = p.parts;
  w.part_len = p.part_len;
  w.n_tiles = (a.Di + kLanes - 1) / kLanes;
  if (p.parts <= 1) {
    w.grid_parts = 1;
    const int64_t blocks = w.n_tiles * a.B;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    selective_scan_kernel<N, Tin, kSequential>
        <<<(unsigned)blocks, kLanes, 0, stream>>>(a, w, p.act_vec, p.bc_vec);
    return cudaGetLastError();
  }
  w.grid_parts = p.parts - 1;
  int64_t blocks = w.n_tiles * a.B * w.grid_parts;
  if (w.n_tiles * a.B * p.parts > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  selective_scan_kernel<N, Tin, kPass1><<<(unsigned)blocks, kLanes, 0, stream>>>(a, w, p.act_vec, p.bc_vec);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  w.grid_parts = p.parts;
  blocks = w.n_tiles * a.B * w.grid_parts;
  selective_scan_kernel<N, Tin, kPass2><<<(unsigned)blocks, kLanes, 0, stream>>>(a, w, p.act_vec, p.bc_vec);
  return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const ScanArgs& a, const ScanPlan& p, float* ws, cudaStream_t s) {
  switch (a.N) {
    case 1: return launch_n<1, Tin>(a, p, ws, s);
    case 2: return launch_n<2, Tin>(a, p, ws, s);
    case 4: return launch_n<4, Tin>(a, p, ws, s);
    case 8: return launch_n<8, Tin>(a, p, ws, s);
    case 16: return launch_n<16, Tin>(a, p, ws, s);
    case 32: return launch_n<32, Tin>(a, p, ws, s);
    case 64: return launch_n<64, Tin>(a, p, ws, s);
  }
  return cudaErrorInvalidValue;
}

inline bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

int64_t scan_workspace_bytes(int64_t B, int64_t Di, int64_t N, int parts) {
  if (parts <= 1) return 0;
  return (int64_t)(1 + 2 * (parts - 1)) * B * Di * N * (int64_t)sizeof(float);
}

int scan_parts(int64_t B, int64_t T, int64_t Di, const DeviceInfo& dev) {
  // Number of T parts P.  With w = ceil(tiles * P / SMs) one-warp CTAs per SM,
  // an SM needs about kWarpsSat warps to keep its pipes busy, and every part but
  // the last is scanned twice (the state-only pass costs ~3/4 of the full one),
  // so the time is ~ ceil(T / P) * (1 + 0.75 (P-1)/P) * max(w, kWarpsSat).
  constexpr double kWarpsSat = 6.0;
  const int64_t tiles = B * ((Di + kLanes - 1) / kLanes);
  double best = 0.0;
  int best_p = 1;
  for (int P = 1; P <= 64; ++P) {
    if (P > 1 && T / P < 64) break;  // parts of at least 64 rows
    const double len = (double)((T + P - 1) / P);
    const double wv = (double)((tiles * P + dev.sm_count - 1) / dev.sm_count);
    const double cost = len * (1.0 + 0.75 * (P - 1) / P) * (wv > kWarpsSat ? wv : kWarpsSat);
    if (P == 1 || cost < best * 0.97) {
      best = cost;
      best_p = P;
    }
  }
  return best_p;
}

ScanPlan plan_selective_scan(const ScanArgs& a, const DeviceInfo& dev, int64_t workspace_bytes) {
  ScanPlan p;
  const int es = a.in_bf16 ? 2 : 4;
  const int vw = 16 / es;
  p.act_vec = al16(a.u) && al16(a.dt) && (!a.z || al16(a.z)) && (a.ld_u * es) % 16 == 0 &&
              (a.ld_dt * es) % 16 == 0 && (!a.z || (a.ld_z * es) % 16 == 0) && a.Di % vw == 0;
  p.bc_vec = al16(a.Bm) && al16(a.Cm) && (a.ld_B * es) % 16 == 0 && (a.ld_C * es) % 16 == 0 &&
             (a.N * es) % 16 == 0;
  p.parts = scan_parts(a.B, a.T, a.Di, dev);
  p.workspace_bytes = scan_workspace_bytes(a.B, a.Di, a.N, p.parts);
  if (p.workspace_bytes > workspace_bytes) {  // not enough workspace: one sequential pass
    p.parts = 1;
    p.workspace_bytes = 0;
  }
  p.part_len = p.parts > 1 ? (a.T + p.parts - 1) / p.parts : a.T;
  return p;
}

cudaError_t launch_selective_scan_prefill(const ScanArgs& a, const ScanPlan& p, float* ws,
                                          const DeviceInfo& dev, cudaStream_t stream) {
  (void)dev;
  return a.in_bf16 ? launch_t<__nv_bfloat16>(a, p, ws, stream) : launch_t<float>(a, p, ws, stream);
}

}  // namespace mamba
