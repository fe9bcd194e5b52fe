// scan_kernel.cuh - kernels of the selective-scan prefill (see scan_prefill.cu
// for the design).  Included by scan_inst.cu, which the build compiles once per
// (storage dtype, d_state) so that the template set compiles in parallel.
#pragma once

#include <type_traits>

#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace scan {
namespace {  // internal linkage: each instantiation unit keeps its own copies

constexpr int kStages = 3;
constexpr int kLanes = 32;  // channels per CTA (one warp)
constexpr int kTC = 16;     // rows per staged chunk
constexpr int kLogTC = 4;

template <typename Tin>
struct Tile {
  static constexpr int ES = sizeof(Tin);
  static constexpr int GA = kLanes * ES / 16;  // 16-byte granules per activation row
  static constexpr int LOG_GA = GA == 8 ? 3 : (GA == 4 ? 2 : (GA == 2 ? 1 : 0));
};

template <int N, typename Tin>
struct Smem {
  Tin act[kStages][3][kTC][kLanes];  // u, dt, z
  Tin bc[kStages][2][kTC][N];        // B, C as staged (storage dtype)
  // bf16 only: this chunk's B, C widened to f32
  float bcf[sizeof(Tin) == 4 ? 1 : 2][sizeof(Tin) == 4 ? 1 : kTC][sizeof(Tin) == 4 ? 4 : N];
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
__device__ __forceinline__ void ld_f32(const float* p, float (&o)[P]) {
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

// State-only token update (pass 1 of the T split).
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

struct Work {
  float* ws;           // T-split workspace (null for the sequential route)
  int parts;           // P
  int64_t part_len;    // rows per part (the last part may be shorter)
  int64_t n_tiles;     // channel tiles per batch row
  int64_t grid_parts;  // parts covered by this launch's grid
};

enum Mode { kSequential = 0, kPass1 = 1, kPass2 = 2 };

// Workspace layout (f32, each slot B*Di*N): slot 0 = state snapshot; slot
// 1 + 2j = total decay of part j; slot 2 + 2j = end state of part j from zero,
// replaced by the fold with the carry-in of part j + 1.
__device__ __forceinline__ int64_t carry_slot(int64_t part) { return part == 0 ? 0 : 2 * part; }

// per-row scalars, computed one row pair ahead of the state update
struct RowS {
  float u, delta, du, g;
};

// KC > 0: the conv1d + SiLU of width KC is fused in; the staged "u" is x, and
// each lane carries the last KC-1 inputs of its channel from row to row.
// YB: the y dtype is bf16; VEC: u/dt/z and B/C stage as 16-byte copies.  Both
// are compile-time choices: a runtime flag in the unrolled row loop costs the
// scheduler's freedom across rows (measured 5-17% on GB300).
template <int N, typename Tin, int MODE, bool GATE, int KC, bool YB = false, bool VEC = false>
__global__ void __launch_bounds__(kLanes) scan_kernel(ScanArgs a, Work w, int act_vec_rt, int bc_vec_rt) {
  const bool act_vec = VEC || act_vec_rt;
  const bool bc_vec = VEC || bc_vec_rt;
  grid_dependency_wait();
  using TL = Tile<Tin>;
  constexpr int P = group_size(N);
  constexpr int NG = N / P;
  constexpr bool kBf16 = sizeof(Tin) == 2;
  constexpr int NTENS = MODE == kPass1 ? 2 : (GATE ? 3 : 2);  // u, dt (, z)
  constexpr int NBC = MODE == kPass1 ? 1 : 2;                 // B (, C)
  // rows unrolled together in a full chunk: all 16 for small states; large
  // states carry enough independent work per row with 4
  constexpr int kU = N <= 16 ? kTC : 4;
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
  const int64_t t_begin = part * w.part_len;
  const int64_t t_end = min(T, t_begin + w.part_len);
  const int64_t BDN = a.B * Di * N;
  const int64_t srow = (b * Di + cc) * N;  // this lane's state row

  // ---- staging of chunk k (rows t_begin + k*kTC ..) into ring slot `stage` ----
  auto act_src = [&](int tens) {
    return reinterpret_cast<const Tin*>(tens == 0 ? a.u : (tens == 1 ? a.dt : a.z));
  };
  auto act_ld = [&](int tens) { return tens == 0 ? a.ld_u : (tens == 1 ? a.ld_dt : a.ld_z); };
  auto issue = [&](int64_t k, int stage) {
    const int64_t row0 = t_begin + k * kTC;
    const int rows = (int)min((int64_t)kTC, t_end - row0);
    const int64_t grow0 = b * T + row0;
    if (act_vec) {
      // granule i: tensor i / (kTC*GA), row (i / GA) % kTC, granule-in-row i % GA
      constexpr int total = NTENS * kTC * TL::GA;
#pragma unroll
      for (int i = lane; i < total; i += kLanes) {
        const int q = i & (TL::GA - 1);
        const int r = (i >> TL::LOG_GA) & (kTC - 1);
        const int tens = i >> (TL::LOG_GA + kLogTC);
        const int64_t ch = c0 + q * (16 / TL::ES);
        if (r < rows && ch < Di)
          cp_async16(&sm.act[stage][tens][r][q * (16 / TL::ES)],
                     act_src(tens) + (grow0 + r) * act_ld(tens) + ch);
      }
    } else {
      for (int tens = 0; tens < NTENS; ++tens)
        for (int r = 0; r < rows; ++r)
          if (active) sm.act[stage][tens][r][lane] = act_src(tens)[(grow0 + r) * act_ld(tens) + c];
    }
    constexpr int GB = (N * TL::ES) / 16 > 0 ? (N * TL::ES) / 16 : 1;  // granules per B/C row
    if (bc_vec && N * TL::ES >= 16) {
      constexpr int total = NBC * kTC * GB;
#pragma unroll
      for (int i = lane; i < total; i += kLanes) {
        const int q = i % GB;
        const int r = (i / GB) % kTC;
        const int tens = i / (GB * kTC);
        const Tin* src = reinterpret_cast<const Tin*>(tens == 0 ? a.Bm : a.Cm);
        const int64_t ld = tens == 0 ? a.ld_B : a.ld_C;
        if (r < rows)
          cp_async16(&sm.bc[stage][tens][r][q * (16 / TL::ES)], src + (grow0 + r) * ld + q * (16 / TL::ES));
      }
    } else {
      for (int i = lane; i < NBC * kTC * N; i += kLanes) {
        const int n = i % N;
        const int r = (i / N) % kTC;
        const int tens = i / (N * kTC);
        const Tin* src = reinterpret_cast<const Tin*>(tens == 0 ? a.Bm : a.Cm);
        const int64_t ld = tens == 0 ? a.ld_B : a.ld_C;
        if (r < rows) sm.bc[stage][tens][r][n] = src[(grow0 + r) * ld + n];
      }
    }
  };

  const int64_t nrows = max((int64_t)0, t_end - t_begin);
  const int64_t nchunks = (nrows + kTC - 1) / kTC;
  auto prologue = [&]() {
#pragma unroll 1
    for (int s = 0; s < kStages - 1; ++s) {
      if (s < nchunks) issue(s, s);
      cp_async_commit();
    }
  };
  // Without the fused conv the first chunks are requested before the parameter
  // and carry-in loads (the 2.8b layer's scan: 943 -> 889 us on GB300); with it,
  // after them (that order measured up to 4% faster for the fused kernel).
  if constexpr (KC == 0) prologue();

  float a2[N];
#pragma unroll
  for (int n = 0; n < N; ++n) a2[n] = a2_from_alog(a.A_log[cc * N + n]);
  const float dtb = a.dt_bias ? a.dt_bias[cc] : 0.0f;
  const float Dc = a.D ? a.D[cc] : 0.0f;

  // ---- fused conv: taps, bias and the window of the KC-1 inputs before t_begin.
  // Input j of the extended sequence [conv_state_0..conv_state_{KC-1}, x_0, ...]
  // is conv state slot j for j < KC, else x_{j-KC}; token t sees j = t+1..t+KC.
  constexpr int KW = KC > 1 ? KC - 1 : 1;
  float cw[KC > 0 ? KC : 1], cwin[KW];
  float cbias = 0.0f;
  const Tin* xin = reinterpret_cast<const Tin*>(a.u);
  auto conv_input = [&](int64_t j) -> float {
    if (j < KC) return a.conv_state_in ? a.conv_state_in[(b * Di + cc) * KC + j] : 0.0f;
    return to_f32(xin[(b * T + j - KC) * a.ld_u + cc]);
  };
  if constexpr (KC > 0) {
#pragma unroll
    for (int k = 0; k < KC; ++k) cw[k] = a.conv_w[cc * KC + k];
    cbias = a.conv_b ? a.conv_b[cc] : 0.0f;
#pragma unroll
    for (int k = 0; k < KC - 1; ++k) cwin[k] = conv_input(t_begin + 1 + k);
  }

  // ---- carry-in ----
  float h[N];
  if (MODE == kSequential) {
    if (a.state_in) {
      // the caller's state may sit at any 4-byte offset: vector loads only when aligned
      if ((reinterpret_cast<uintptr_t>(a.state_in) & 15) == 0) {
        ld_f32<N>(a.state_in + srow, h);
      } else {
#pragma unroll
        for (int n = 0; n < N; ++n) h[n] = a.state_in[srow + n];
      }
    } else {
#pragma unroll
      for (int n = 0; n < N; ++n) h[n] = 0.0f;
    }
  } else if (MODE == kPass1) {
#pragma unroll
    for (int n = 0; n < N; ++n) h[n] = 0.0f;
    if (part == 0 && active) {  // snapshot of the initial state for the fold / pass 2
#pragma unroll
      for (int n = 0; n < N; ++n) w.ws[srow + n] = a.state_in ? a.state_in[srow + n] : 0.0f;
    }
  } else {
    ld_f32<N>(w.ws + BDN * carry_slot(part) + srow, h);
  }

  if constexpr (KC > 0) prologue();

  const int64_t yoff = (b * T + t_begin) * a.ld_y + c;  // this lane's first y element
  float sdelta = 0.0f;  // pass 1: sum of delta over the part
#pragma unroll 1
  for (int64_t k = 0; k < nchunks; ++k) {
    cp_async_wait<kStages - 2>();
    __syncwarp();  // chunk k visible to every lane; every lane is done with chunk k-1
    const int stage = (int)(k % kStages);
    const int rows = (int)min((int64_t)kTC, nrows - k * kTC);
    const float* sB;
    const float* sC;
    if constexpr (kBf16) {
      // widen this chunk's B (and C) rows to f32 once, shared by all lanes
#pragma unroll
      for (int i = lane; i < NBC * kTC * N; i += kLanes) {
        const int n = i % N;
        const int r = (i / N) % kTC;
        const int tens = i / (N * kTC);
        sm.bcf[tens][r][n] = to_f32(sm.bc[stage][tens][r][n]);
      }
      __syncwarp();
      sB = &sm.bcf[0][0][0];
      sC = &sm.bcf[NBC - 1][0][0];
    } else {
      sB = reinterpret_cast<const float*>(&sm.bc[stage][0][0][0]);
      sC = reinterpret_cast<const float*>(&sm.bc[stage][NBC - 1][0][0]);
    }
    if (k + kStages - 1 < nchunks) issue(k + kStages - 1, (int)((k + kStages - 1) % kStages));
    cp_async_commit();

    const Tin* su = &sm.act[stage][0][0][0];
    const Tin* sdt = &sm.act[stage][1][0][0];
    const Tin* sz = &sm.act[stage][GATE ? 2 : 0][0][0];
    auto prep = [&](int r) {
      RowS s;
      s.u = to_f32(su[r * kLanes + lane]);
      if constexpr (KC > 0) {  // rows are prepped in order: slide the window
        float sw[KC];
#pragma unroll
        for (int k = 0; k < KC - 1; ++k) sw[k] = cwin[k];
        sw[KC - 1] = s.u;
#pragma unroll
        for (int k = 0; k + 1 < KC - 1; ++k) cwin[k] = cwin[k + 1];
        if (KC > 1) cwin[KW - 1] = s.u;
        s.u = to_f32(from_f32<Tin>(silu_f(conv_taps<KC>(cw, sw, cbias))));
      }
      s.delta = softplus_f(to_f32(sdt[r * kLanes + lane]) + dtb);
      s.du = s.delta * s.u;
      s.g = (MODE != kPass1 && GATE) ? silu_f(to_f32(sz[r * kLanes + lane])) : 1.0f;
      return s;
    };
    if (!active) continue;

    if (MODE == kPass1) {
      auto row_state = [&](int r, const RowS& rs) {
        sdelta += rs.delta;
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          float Bv[P];
          ld_f32<P>(sB + r * N + q * P, Bv);
          ssm_state_group<P>(h + q * P, a2 + q * P, rs.delta, rs.du, Bv);
        }
      };
      if (rows == kTC) {
        // full chunk: unrolled by kU rows, every row's scalars first, so the
        // only serial chain left is the state update
#pragma unroll 1
        for (int r0 = 0; r0 < kTC; r0 += kU) {
          RowS rs[kU];
#pragma unroll
          for (int r = 0; r < kU; ++r) rs[r] = prep(r0 + r);
#pragma unroll
          for (int r = 0; r < kU; ++r) row_state(r0 + r, rs[r]);
        }
      } else {
#pragma unroll 1
        for (int r = 0; r < rows; ++r) row_state(r, prep(r));
      }
    } else {
      const int64_t yk = yoff + k * kTC * a.ld_y;
      auto row_out = [&](int r, const RowS& rs) {
        float part_[NG];
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          float Bv[P], Cv[P];
          ld_f32<P>(sB + r * N + q * P, Bv);
          ld_f32<P>(sC + r * N + q * P, Cv);
          part_[q] = ssm_token_group<P>(h + q * P, a2 + q * P, rs.delta, rs.du, Bv, Cv);
        }
        float y = fmaf(Dc, rs.u, tree_sum<NG>(part_));
        if (GATE) y *= rs.g;
        store_out(a.y, yk + r * a.ld_y, YB, y);
      };
      if (rows == kTC) {
#pragma unroll 1
        for (int r0 = 0; r0 < kTC; r0 += kU) {
          RowS rs[kU];
#pragma unroll
          for (int r = 0; r < kU; ++r) rs[r] = prep(r0 + r);
#pragma unroll
          for (int r = 0; r < kU; ++r) row_out(r0 + r, rs[r]);
        }
      } else {
#pragma unroll 1
        for (int r = 0; r < rows; ++r) row_out(r, prep(r));
      }
    }
  }
  cp_async_wait<0>();
  grid_dependents_launch();  // main loop done: the next grid may be scheduled

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
  if constexpr (KC > 0) {
    // new conv state = inputs T..T+KC-1 of the extended sequence; written by
    // part 0 of the final pass, the only reader of conv_state_in in that pass
    // (every read before any write: in-place safe)
    if (MODE != kPass1 && part == 0 && a.conv_state_out) {
      float fin[KC];
#pragma unroll
      for (int k = 0; k < KC; ++k) fin[k] = conv_input(T + k);
#pragma unroll
      for (int k = 0; k < KC; ++k) a.conv_state_out[(b * Di + cc) * KC + k] = fin[k];
    }
  }
}

// Chains the parts' aggregates: carry_{j+1} = decay_j * carry_j + end_j, with
// carry_0 = the state snapshot; carry_{j+1} overwrites end_j.  One thread per
// state element; the loads of up to kFoldBatch parts are issued before the
// batch's stores (the stores could alias later loads for the compiler, so
// without the batching every part would cost an L2 round trip).
constexpr int kFoldBatch = 32;
__global__ void __launch_bounds__(128) scan_fold_kernel(float* ws, int64_t BDN, int parts) {
  grid_dependency_begin();
  const int64_t i = (int64_t)blockIdx.x * 128 + threadIdx.x;
  if (i >= BDN) return;
  float acc = ws[i];
  for (int j0 = 0; j0 < parts - 1; j0 += kFoldBatch) {
    float p[kFoldBatch], e[kFoldBatch];
#pragma unroll
    for (int u = 0; u < kFoldBatch; ++u) {
      if (j0 + u < parts - 1) {
        p[u] = ws[BDN * (1 + 2 * (j0 + u)) + i];
        e[u] = ws[BDN * (2 + 2 * (j0 + u)) + i];
      }
    }
#pragma unroll
    for (int u = 0; u < kFoldBatch; ++u) {
      if (j0 + u < parts - 1) {
        acc = fmaf(p[u], acc, e[u]);
        ws[BDN * (2 + 2 * (j0 + u)) + i] = acc;
      }
    }
  }
}

template <int N, typename Tin, int MODE, bool GATE, bool YB, bool VEC>
cudaError_t launch_mode_v(const ScanArgs& a, const Work& w, const ScanPlan& p, cudaStream_t stream) {
  const int64_t blocks = w.n_tiles * a.B * w.grid_parts;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  if (a.K == 4)
    return launch_pdl(false, scan_kernel<N, Tin, MODE, GATE, 4, YB, VEC>, dim3((unsigned)blocks), dim3(kLanes), 0,
                      stream, a, w, p.act_vec, p.bc_vec);
  if (a.K != 0) return cudaErrorInvalidValue;
  return launch_pdl(false, scan_kernel<N, Tin, MODE, GATE, 0, YB, VEC>, dim3((unsigned)blocks), dim3(kLanes), 0,
                    stream, a, w, p.act_vec, p.bc_vec);
}

template <int N, typename Tin, int MODE, bool GATE, bool YB>
cudaError_t launch_mode_y(const ScanArgs& a, const Work& w, const ScanPlan& p, cudaStream_t stream) {
  // the 16-byte staging path exists only where every row can take it
  constexpr bool kCanVec = N * sizeof(Tin) >= 16;
  if constexpr (kCanVec) {
    if (p.act_vec && p.bc_vec) return launch_mode_v<N, Tin, MODE, GATE, YB, true>(a, w, p, stream);
  }
  return launch_mode_v<N, Tin, MODE, GATE, YB, false>(a, w, p, stream);
}

template <int N, typename Tin, int MODE, bool GATE>
cudaError_t launch_mode(const ScanArgs& a, const Work& w, const ScanPlan& p, cudaStream_t stream) {
  if constexpr (MODE == kPass1) return launch_mode_y<N, Tin, MODE, GATE, false>(a, w, p, stream);  // no y
  return a.y_bf16 ? launch_mode_y<N, Tin, MODE, GATE, true>(a, w, p, stream)
                  : launch_mode_y<N, Tin, MODE, GATE, false>(a, w, p, stream);
}

template <int N, typename Tin, int MODE>
cudaError_t launch_out(const ScanArgs& a, const Work& w, const ScanPlan& p, cudaStream_t s) {
  return a.z != nullptr ? launch_mode<N, Tin, MODE, true>(a, w, p, s)
                        : launch_mode<N, Tin, MODE, false>(a, w, p, s);
}

template <int N, typename Tin>
cudaError_t launch_n(const ScanArgs& a, const ScanPlan& p, float* ws, cudaStream_t stream) {
  Work w;
  w.ws = ws;
  w.parts = p.parts;
  w.part_len = p.part_len;
  w.n_tiles = (a.Di + kLanes - 1) / kLanes;
  if (p.parts <= 1) {
    w.grid_parts = 1;
    return launch_out<N, Tin, kSequential>(a, w, p, stream);
  }
  w.grid_parts = p.parts - 1;
  cudaError_t e = launch_mode<N, Tin, kPass1, false>(a, w, p, stream);
  if (e != cudaSuccess) return e;
  const int64_t BDN = a.B * a.Di * N;
  if ((BDN + 127) / 128 > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  e = launch_pdl(false, scan_fold_kernel, dim3((unsigned)((BDN + 127) / 128)), dim3(128), 0, stream, ws, BDN,
                 p.parts);
  if (e != cudaSuccess) return e;
  w.grid_parts = p.parts;
  return launch_out<N, Tin, kPass2>(a, w, p, stream);
}

}  // namespace
}  // namespace scan
}  // namespace mamba
