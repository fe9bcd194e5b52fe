// scan_kernel.cuh - the selective-scan prefill kernel (see scan_prefill.cu for
// the design and the route planner).  Included by scan_inst.cu, which the build
// compiles once per (storage dtype, d_state) so that the template set compiles
// in parallel.
#pragma once

#include <type_traits>

#include "device_math.cuh"
#include "launch.h"

namespace mamba {
namespace scan {
namespace {  // internal linkage: each instantiation unit keeps its own copies

// chunks in a warp's staging ring: two (the next chunk lands while this one is
// scanned; a 16-row chunk takes longer than a load).  Measured on the fused
// prefill: 2.8b layer 758 us with two, 785 with three, 775 with four; the 130m
// layer 39.4 / 39.6 / 65 us (four no longer fit eight warps of f32 staging)
constexpr int kStages = 2;
constexpr int kLanes = 32;  // channels per warp (one lane per channel)
constexpr int kTC = 16;     // rows per staged chunk
constexpr int kLogTC = 4;
constexpr long long kWaitLimit = 1ll << 31;  // SM cycles (about a second) before a wait gives up
constexpr int kFaultWait = 2;                 // MAMBA_FAULT_SCAN_WAIT

template <typename Tin>
struct Tile {
  static constexpr int ES = sizeof(Tin);
  static constexpr int GA = kLanes * ES / 16;  // 16-byte granules per activation row
  static constexpr int LOG_GA = GA == 8 ? 3 : (GA == 4 ? 2 : (GA == 2 ? 1 : 0));
};

template <int N, typename Tin>
struct Smem {
  Tin act[kStages][3][kTC][kLanes];  // u (or x), dt, z
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

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
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
template <int P>
__device__ __forceinline__ void st_f32(float* p, const float (&v)[P]) {
  if constexpr (P % 4 == 0) {
#pragma unroll
    for (int j = 0; j < P; j += 4) *reinterpret_cast<float4*>(p + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < P; ++j) p[j] = v[j];
  }
}

// State-only token update (the split route's first pass).
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

// The plan as the kernel sees it.  Workspace: a header of 32-bit words (the role
// queue head as a 64-bit word at 0, the abort flag at 2, a counter per tile from
// kHdrTiles and a second one after them; zeroed before every launch), then the
// state slots, [tile][slot][n][lane] f32 (one coalesced 128-byte row per state).
// Chained: slot 0 holds the state a tile's first role hands to the next.  Split:
// slot 0 = the initial state, slot 1 + 2j = part j's total decay exp(A sum
// delta), slot 2 + 2j = part j's end state from zero, which the fold replaces
// with the carry into part j + 1.
constexpr int kHdrTiles = 4;
struct Work {
  uint32_t* hdr;
  float* slots;
  int* faults;
  int mode;
  int parts;      // split: parts P (chained, plain: 1)
  int n_slots;    // slots per tile
  int wpc;        // warps per CTA
  int64_t seg;    // split: rows per part
  int64_t span;   // chained: tile-rows per role
  int64_t n_tiles;
  int64_t tiles_b;  // tiles per batch row
  int64_t n_roles;  // roles handed out by the queue (plain: one per tile, static)
};

__device__ __forceinline__ float* slot_ptr(const Work& w, int64_t tile, int s, int N) {
  return w.slots + (tile * w.n_slots + s) * (int64_t)N * kLanes;
}

// Bounded wait (all lanes) until *p >= v, polling with a growing sleep so that
// a waiting warp takes next to no issue slots from the warps it shares an SM
// sub-partition with; false if it ran out or another warp gave up first (the
// launch has then failed and this warp gives up at once).
__device__ __forceinline__ bool wait_at_least(const Work& w, const uint32_t* p, uint32_t v) {
  if (ld_acquire(p) >= v) return true;
  const long long t0 = clock64();
  unsigned ns = 64;
  while (true) {
    __nanosleep(ns);
    if (ns < 256) ns *= 2;
    if (ld_acquire(p) >= v) return true;
    if (ld_acquire(w.hdr + 2) != 0) return false;
    if (clock64() - t0 > kWaitLimit) {
      atomicOr(w.faults, kFaultWait);
      atomicExch(w.hdr + 2, 1u);
      return false;
    }
  }
}

// Stores this lane's N states (or loads them) at slot row `s` of a tile.
template <int N>
__device__ __forceinline__ void slot_store(const Work& w, int64_t tile, int s, int lane, const float (&v)[N]) {
  float* p = slot_ptr(w, tile, s, N) + lane;
#pragma unroll
  for (int n = 0; n < N; ++n) p[n * kLanes] = v[n];
}
template <int N>
__device__ __forceinline__ void slot_load(const Work& w, int64_t tile, int s, int lane, float (&v)[N]) {
  const float* p = slot_ptr(w, tile, s, N) + lane;
#pragma unroll
  for (int n = 0; n < N; ++n) v[n] = p[n * kLanes];
}

// per-row scalars, computed for a batch of rows before their state updates
struct RowS {
  float u, delta, du, g;
};

// Per-tile parameters, loaded when a warp moves to another tile.
template <int N, int KC>
struct TileParams {
  static constexpr int KW = KC > 1 ? KC - 1 : 1;
  float a2[N];
  float dtb, Dc;
  float cw[KC > 0 ? KC : 1];
  float cbias;
};

enum UnitKind { kFull = 0, kStateOnly = 1 };

// KC > 0: the conv1d + SiLU of width KC is fused in; the staged "u" is x, and
// each lane carries the last KC-1 inputs of its channel from row to row.
// YB: the y dtype is bf16; VEC: u/dt/z and B/C stage as 16-byte copies.  Both
// are compile-time choices: a runtime flag in the unrolled row loop costs the
// scheduler its freedom across rows (measured 5-17% on GB300).
//
// Scans rows [t_begin, t_end) of tile (b, c0) from state h (in/out).  kFull
// writes y; kStateOnly accumulates sum(delta) in sdelta instead.  The caller has
// already issued the first kStages-1 chunks (stage_prologue).
template <int KIND, int N, typename Tin, bool GATE, int KC, bool YB, bool VEC>
__device__ __forceinline__ void scan_rows(const ScanArgs& a, Smem<N, Tin>& sm, int lane, bool act_vec, bool bc_vec,
                                          int64_t b, int64_t c0, int64_t t_begin, int64_t t_end, float (&h)[N],
                                          const TileParams<N, KC>& tp, float (&cwin)[TileParams<N, KC>::KW],
                                          float& sdelta);

template <int KIND, int N, typename Tin, bool GATE>
__device__ __forceinline__ void issue_chunk(const ScanArgs& a, Smem<N, Tin>& sm, int lane, bool act_vec, bool bc_vec,
                                            int64_t b, int64_t c0, int64_t t_begin, int64_t t_end, int64_t k,
                                            int stage) {
  using TL = Tile<Tin>;
  constexpr int NTENS = KIND == kStateOnly ? 2 : (GATE ? 3 : 2);  // u, dt (, z)
  constexpr int NBC = KIND == kStateOnly ? 1 : 2;                 // B (, C)
  const int64_t Di = a.Di, T = a.T;
  const int64_t row0 = t_begin + k * kTC;
  const int rows = (int)min((int64_t)kTC, t_end - row0);
  const int64_t grow0 = b * T + row0;
  auto act_src = [&](int tens) {
    return reinterpret_cast<const Tin*>(tens == 0 ? a.u : (tens == 1 ? a.dt : a.z));
  };
  auto act_ld = [&](int tens) { return tens == 0 ? a.ld_u : (tens == 1 ? a.ld_dt : a.ld_z); };
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
        cp_async16(&sm.act[stage][tens][r][q * (16 / TL::ES)], act_src(tens) + (grow0 + r) * act_ld(tens) + ch);
    }
  } else {
    const int64_t c = c0 + lane;
    for (int tens = 0; tens < NTENS; ++tens)
      for (int r = 0; r < rows; ++r)
        if (c < Di) sm.act[stage][tens][r][lane] = act_src(tens)[(grow0 + r) * act_ld(tens) + c];
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
      if (r < rows) cp_async16(&sm.bc[stage][tens][r][q * (16 / TL::ES)], src + (grow0 + r) * ld + q * (16 / TL::ES));
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
}

// Requests the first kStages-1 chunks of rows [t_begin, t_end) (one commit group each).
template <int KIND, int N, typename Tin, bool GATE>
__device__ __forceinline__ void stage_prologue(const ScanArgs& a, Smem<N, Tin>& sm, int lane, bool act_vec,
                                               bool bc_vec, int64_t b, int64_t c0, int64_t t_begin, int64_t t_end) {
  const int64_t nchunks = (max((int64_t)0, t_end - t_begin) + kTC - 1) / kTC;
#pragma unroll 1
  for (int s = 0; s < kStages - 1; ++s) {
    if (s < nchunks) issue_chunk<KIND, N, Tin, GATE>(a, sm, lane, act_vec, bc_vec, b, c0, t_begin, t_end, s, s);
    cp_async_commit();
  }
}

template <int KIND, int N, typename Tin, bool GATE, int KC, bool YB, bool VEC>
__device__ __forceinline__ void scan_rows(const ScanArgs& a, Smem<N, Tin>& sm, int lane, bool act_vec, bool bc_vec,
                                          int64_t b, int64_t c0, int64_t t_begin, int64_t t_end, float (&h)[N],
                                          const TileParams<N, KC>& tp, float (&cwin)[TileParams<N, KC>::KW],
                                          float& sdelta) {
  constexpr int P = group_size(N);
  constexpr int NG = N / P;
  constexpr bool kBf16 = sizeof(Tin) == 2;
  constexpr int NBC = KIND == kStateOnly ? 1 : 2;
  constexpr int KW = TileParams<N, KC>::KW;
  // rows unrolled together in a full chunk: all 16 for small states; large
  // states carry enough independent work per row with 4
  constexpr int kU = N <= 16 ? kTC : 4;
  const int64_t c = c0 + lane;
  const bool active = c < a.Di;
  const int64_t nrows = max((int64_t)0, t_end - t_begin);
  const int64_t nchunks = (nrows + kTC - 1) / kTC;
  const int64_t yoff = (b * a.T + t_begin) * a.ld_y + c;  // this lane's first y element
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
    if (k + kStages - 1 < nchunks)
      issue_chunk<KIND, N, Tin, GATE>(a, sm, lane, act_vec, bc_vec, b, c0, t_begin, t_end, k + kStages - 1,
                                      (int)((k + kStages - 1) % kStages));
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
        for (int q = 0; q < KC - 1; ++q) sw[q] = cwin[q];
        sw[KC - 1] = s.u;
#pragma unroll
        for (int q = 0; q + 1 < KC - 1; ++q) cwin[q] = cwin[q + 1];
        if (KC > 1) cwin[KW - 1] = s.u;
        s.u = to_f32(from_f32<Tin>(silu_f(conv_taps<KC>(tp.cw, sw, tp.cbias))));
      }
      s.delta = softplus_f(to_f32(sdt[r * kLanes + lane]) + tp.dtb);
      s.du = s.delta * s.u;
      s.g = (KIND == kFull && GATE) ? silu_f(to_f32(sz[r * kLanes + lane])) : 1.0f;
      return s;
    };
    if (!active) continue;

    if constexpr (KIND == kStateOnly) {
      auto row_state = [&](int r, const RowS& rs) {
        sdelta += rs.delta;
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          float Bv[P];
          ld_f32<P>(sB + r * N + q * P, Bv);
          ssm_state_group<P>(h + q * P, tp.a2 + q * P, rs.delta, rs.du, Bv);
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
          part_[q] = ssm_token_group<P>(h + q * P, tp.a2 + q * P, rs.delta, rs.du, Bv, Cv);
        }
        float y = fmaf(tp.Dc, rs.u, tree_sum<NG>(part_));
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
  __syncwarp();  // the ring is free for the next unit
}

// The split route's fold: one thread per (tile, state n, lane) chains the
// parts' aggregates into carries: carry_0 = the initial state (kept in slot 0),
// carry_{j+1} = decay_j * carry_j + end_j, which overwrites end_j.  The loads of
// up to kFoldBatch parts are issued before the batch's stores (the stores could
// alias later loads for the compiler, so without the batching every part would
// cost an L2 round trip).  Slot rows are [n][lane]: consecutive threads touch
// consecutive floats.
constexpr int kFoldBatch = 32;
__global__ void __launch_bounds__(128) scan_fold_kernel(ScanArgs a, Work w, int N) {
  grid_dependency_wait();
  const int64_t i = (int64_t)blockIdx.x * 128 + threadIdx.x;
  const int64_t per_tile = (int64_t)N * kLanes;
  if (i >= w.n_tiles * per_tile) return;
  const int64_t tile = i / per_tile;
  const int n = (int)((i - tile * per_tile) / kLanes);
  const int lane = (int)(i % kLanes);
  const int64_t b = tile / w.tiles_b;
  const int64_t c = (tile - b * w.tiles_b) * kLanes + lane;
  float acc = (c < a.Di && a.state_in) ? a.state_in[(b * a.Di + c) * N + n] : 0.0f;
  float* base = w.slots + tile * w.n_slots * per_tile + (int64_t)n * kLanes + lane;
  base[0] = acc;
  const int parts = w.parts;
  for (int j0 = 0; j0 < parts - 1; j0 += kFoldBatch) {
    float dcy[kFoldBatch], end[kFoldBatch];
#pragma unroll
    for (int q = 0; q < kFoldBatch; ++q) {
      if (j0 + q < parts - 1) {
        dcy[q] = base[(1 + 2 * (j0 + q)) * per_tile];
        end[q] = base[(2 + 2 * (j0 + q)) * per_tile];
      }
    }
#pragma unroll
    for (int q = 0; q < kFoldBatch; ++q) {
      if (j0 + q < parts - 1) {
        acc = fmaf(dcy[q], acc, end[q]);
        base[(2 + 2 * (j0 + q)) * per_tile] = acc;
      }
    }
  }
}

// A stretch of rows of one tile that a warp scans in one go.
struct Segment {
  int64_t tile, t_begin, t_end;
};

// PASS kFull: the plain and chained routes and the split route's full pass;
// PASS kStateOnly: the split route's state-only pass.  Each kernel carries one
// row body only (both in one kernel measured slower: its warps stalled on
// instruction fetch).
template <int PASS, int N, typename Tin, bool GATE, int KC, bool YB, bool VEC>
__global__ void __launch_bounds__(256, 1) scan_kernel(ScanArgs a, Work w, int act_vec_rt, int bc_vec_rt) {
  const bool act_vec = VEC || act_vec_rt;
  const bool bc_vec = VEC || bc_vec_rt;
  grid_dependency_wait();
  using TP = TileParams<N, KC>;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & (kLanes - 1);
  const int warp = threadIdx.x / kLanes;
  Smem<N, Tin>& sm = reinterpret_cast<Smem<N, Tin>*>(smem_raw)[warp];
  const int64_t U = w.n_tiles, T = a.T, Di = a.Di;

  // roles: the chained route hands them out from the queue in index order, so
  // a role only ever waits on a role handed out before it, which a running warp
  // holds (progress needs no co-residency); the other routes have no waits and
  // give warp g role g
  auto grab = [&]() -> int64_t {
    unsigned long long v = 0;
    if (lane == 0) v = atomicAdd(reinterpret_cast<unsigned long long*>(w.hdr), 1ull);
    return (int64_t)__shfl_sync(0xffffffffu, v, 0);
  };
  const bool queued = PASS == kFull && w.mode == kScanChained;
  int64_t role = queued ? grab() : (int64_t)blockIdx.x * w.wpc + warp;
  int64_t cur_tile = -1;
  TP tp;

  // Scans one segment: first chunks, parameters (on a change of tile), carry-in
  // (after a bounded wait where it is handed over), the rows, then the final
  // state, the hand-off or the part's aggregate.
  //   carry: 0 = state_in (or zeros), 1 = zeros, 2 = chained slot after its
  //          flag, 3 = the split route's carry (folded by the previous launch)
  //   out:   0 = state_out, 1 = chained hand-off, 2 = split aggregate, 3 = none
  auto run = [&](const Segment& sg, int carry, int out, int part) {
    const int64_t tile = sg.tile;
    const int64_t b = tile / w.tiles_b;
    const int64_t c0 = (tile - b * w.tiles_b) * kLanes;
    const int64_t c = c0 + lane;
    const bool active = c < Di;
    const int64_t cc = active ? c : Di - 1;
    const int64_t srow = (b * Di + cc) * N;  // this lane's row of a [B][Di][N] state
    // first chunks: without the fused conv before the parameter loads, with it
    // after them (measured best for each on GB300); before any wait on a
    // hand-off either way (the rows do not depend on it)
    const bool early = KC == 0 || carry == 2;
    if (early) stage_prologue<PASS, N, Tin, GATE>(a, sm, lane, act_vec, bc_vec, b, c0, sg.t_begin, sg.t_end);
    if (tile != cur_tile) {
      cur_tile = tile;
#pragma unroll
      for (int n = 0; n < N; ++n) tp.a2[n] = a2_from_alog(a.A_log[cc * N + n]);
      tp.dtb = a.dt_bias ? a.dt_bias[cc] : 0.0f;
      tp.Dc = a.D ? a.D[cc] : 0.0f;
      if constexpr (KC > 0) {
#pragma unroll
        for (int q = 0; q < KC; ++q) tp.cw[q] = a.conv_w[cc * KC + q];
        tp.cbias = a.conv_b ? a.conv_b[cc] : 0.0f;
      }
    }
    // fused conv: the window of the KC-1 inputs before t_begin.  Input j of the
    // extended sequence [conv_state_0..conv_state_{KC-1}, x_0, ...] is conv
    // state slot j for j < KC, else x_{j-KC}; token t sees j = t+1..t+KC.
    const Tin* xin = reinterpret_cast<const Tin*>(a.u);
    auto conv_input = [&](int64_t j) -> float {
      if (j < KC) return a.conv_state_in ? a.conv_state_in[(b * Di + cc) * KC + j] : 0.0f;
      return to_f32(xin[(b * T + j - KC) * a.ld_u + cc]);
    };
    float cwin[TP::KW];
    if constexpr (KC > 1) {
#pragma unroll
      for (int q = 0; q < KC - 1; ++q) cwin[q] = conv_input(sg.t_begin + 1 + q);
    }
    float h[N];
    if (carry == 0 && a.state_in) {
      // the caller's state may sit at any 4-byte offset: vector loads only when aligned
      if ((reinterpret_cast<uintptr_t>(a.state_in) & 15) == 0) {
        ld_f32<N>(a.state_in + srow, h);
      } else {
#pragma unroll
        for (int n = 0; n < N; ++n) h[n] = a.state_in[srow + n];
      }
    } else if (carry <= 1) {
#pragma unroll
      for (int n = 0; n < N; ++n) h[n] = 0.0f;
    } else if (carry == 2) {
      // a wait that runs out has set the fault bit; the segment still runs, so
      // that nothing else waits on it
      wait_at_least(w, w.hdr + kHdrTiles + tile, 1u);
      slot_load<N>(w, tile, 0, lane, h);
    } else {
      slot_load<N>(w, tile, part == 0 ? 0 : 2 * part, lane, h);
    }
    if (!early) stage_prologue<PASS, N, Tin, GATE>(a, sm, lane, act_vec, bc_vec, b, c0, sg.t_begin, sg.t_end);
    float sdelta = 0.0f;
    scan_rows<PASS, N, Tin, GATE, KC, YB, VEC>(a, sm, lane, act_vec, bc_vec, b, c0, sg.t_begin, sg.t_end, h, tp,
                                               cwin, sdelta);
    if (out == 0) {
      if (active && a.state_out) {
#pragma unroll
        for (int n = 0; n < N; ++n) a.state_out[srow + n] = h[n];
      }
    } else if (out == 1) {
      slot_store<N>(w, tile, 0, lane, h);
      __threadfence();
      __syncwarp();
      if (lane == 0) st_release(w.hdr + kHdrTiles + tile, 1u);
    } else if (out == 2) {
      float dcy[N];
#pragma unroll
      for (int n = 0; n < N; ++n) dcy[n] = ex2_approx(tp.a2[n] * sdelta);
      slot_store<N>(w, tile, 1 + 2 * part, lane, dcy);
      slot_store<N>(w, tile, 2 + 2 * part, lane, h);
    }
    if constexpr (KC > 0 && PASS == kFull) {
      // new conv state = inputs T..T+KC-1 of the extended sequence, written by
      // the full-pass segment that reads conv_state_in last (in-place safe):
      // on the split route part 0's full pass (only a part that starts in the
      // first KC-1 rows reads the old state, and part 0's state-only pass ran in
      // an earlier launch); otherwise the segment that ends at T (a tail that
      // starts in the first KC-1 rows reads the old state, after the head it
      // waited for)
      const bool writer = w.mode == kScanSplit ? sg.t_begin == 0 : sg.t_end == T;
      if (writer && active && a.conv_state_out) {
        float fin[KC];
#pragma unroll
        for (int q = 0; q < KC; ++q) fin[q] = conv_input(T + q);
#pragma unroll
        for (int q = 0; q < KC; ++q) a.conv_state_out[(b * Di + cc) * KC + q] = fin[q];
      }
    }
  };

  // A role is a short list of segments, each scanned by the one call of run()
  // below (a single call site keeps the kernel small): the chained route's
  // head, whole tiles and tail, or one tile or one part.
#pragma unroll 1
  while (role < w.n_roles) {
    int64_t n_items = 1;
    int64_t k0 = 0, s0 = 0, k1 = 0, e1 = 0, kfull = 0;
    bool head = false;
    if (queued) {
      // tile-rows [role*span, (role+1)*span) of the tiles laid end to end; span
      // >= T, so the role ends in a tile it starts (its head, from row 0) and
      // may begin in the middle of a tile whose head the previous role scans:
      // head first (its end state goes to the next role), then whole tiles,
      // then the tail from the handed-over state
      const int64_t beg = role * w.span;
      const int64_t end = min(U * T, beg + w.span);
      k0 = beg / T;
      s0 = beg - k0 * T;
      k1 = (end - 1) / T;
      e1 = end - k1 * T;
      head = k1 > k0 || s0 == 0;
      kfull = s0 == 0 ? k0 : k0 + 1;
      n_items = beg >= end ? 0 : (head ? 1 : 0) + (k1 - kfull > 0 ? k1 - kfull : 0) + (s0 > 0 ? 1 : 0);
    }
#pragma unroll 1
    for (int64_t it = 0; it < n_items; ++it) {
      Segment sg;
      int carry = 0, out = 0, part = 0;
      if (queued) {
        const int64_t i = head ? it : it + 1;  // 0: head, 1..: whole tiles, last: tail
        const int64_t n_full = k1 - kfull > 0 ? k1 - kfull : 0;
        if (i == 0) {
          sg = Segment{k1, 0, e1};
          out = e1 == T ? 0 : 1;
        } else if (i <= n_full) {
          sg = Segment{kfull + i - 1, 0, T};
        } else {
          sg = Segment{k0, s0, k1 > k0 ? T : e1};
          carry = 2;
        }
      } else if (w.mode == kScanPlain) {
        sg = Segment{role, 0, T};
      } else {  // split: part j of a tile, j-major
        part = (int)(role / U);
        const int64_t tile = role - part * U;
        sg = Segment{tile, part * w.seg, min(T, (part + 1) * w.seg)};
        if (PASS == kStateOnly) {
          carry = 1;
          out = 2;
        } else {
          carry = 3;
          out = part == w.parts - 1 ? 0 : 3;
        }
      }
      run(sg, carry, out, part);
    }
    // the next role is taken only now: taken early, it could go to a warp that
    // is still busy while another warp, just started, finds the queue empty
    role = queued ? grab() : w.n_roles;
  }
  grid_dependents_launch();  // this warp is done: the next grid may be scheduled
}

// Warps per CTA for a persistent launch: up to 8 (two per SM sub-partition),
// as many as the shared memory and registers of one SM hold; worked out once
// per device and kernel (`cache` belongs to the kernel: each instantiation of
// launch_k passes its own).
template <typename K>
cudaError_t warps_per_cta(K kern, int warp_smem, int (&cache)[64], int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int wpc = __atomic_load_n(&cache[dev], __ATOMIC_RELAXED);
  if (wpc == 0) {
    int optin = 0;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin)) != cudaSuccess)
      return e;
    for (wpc = 8; wpc > 1; --wpc) {
      int occ = 0;
      if (wpc * warp_smem > optin) continue;
      if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kLanes * wpc, wpc * warp_smem)) !=
          cudaSuccess)
        return e;
      if (occ >= 1) break;
    }
    __atomic_store_n(&cache[dev], wpc, __ATOMIC_RELAXED);
  }
  *out = wpc;
  return cudaSuccess;
}

template <int PASS, int N, typename Tin, bool GATE, int KC, bool YB, bool VEC>
cudaError_t launch_k(const ScanArgs& a, Work w, const ScanPlan& p, cudaStream_t stream) {
  auto kern = scan_kernel<PASS, N, Tin, GATE, KC, YB, VEC>;
  constexpr int kWarpSmem = (int)sizeof(Smem<N, Tin>);
  static int wpc_cache[64];
  int wpc = 1;
  cudaError_t e = warps_per_cta(kern, kWarpSmem, wpc_cache, &wpc);
  if (e != cudaSuccess) return e;
  int64_t grid;
  if (w.mode == kScanPlain) {
    w.wpc = 1;  // one warp per tile: one-warp CTAs spread evenly over the SMs
    grid = w.n_roles;
  } else {
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (w.mode == kScanChained) {
      // one role per resident warp, one CTA per SM (at most one role per tile,
      // so a role spans at least T tile-rows and no tile is cut twice)
      const int64_t warps = (int64_t)wpc * sms;
      w.n_roles = w.n_tiles < warps ? w.n_tiles : warps;
      w.span = (w.n_tiles * a.T + w.n_roles - 1) / w.n_roles;
    } else {
      // a split pass with few roles spreads them over every SM rather than
      // packing 8 to an SM (a short prefill is latency-bound)
      const int64_t per_sm = (w.n_roles + sms - 1) / sms;
      if (per_sm < wpc) wpc = (int)(per_sm > 0 ? per_sm : 1);
    }
    w.wpc = wpc;
    grid = (w.n_roles + wpc - 1) / wpc;
  }
  if (grid > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  return launch_pdl(false, kern, dim3((unsigned)grid), dim3(kLanes * w.wpc), (size_t)w.wpc * kWarpSmem, stream, a, w,
                    p.act_vec, p.bc_vec);
}

template <int PASS, int N, typename Tin, bool GATE, int KC, bool YB>
cudaError_t launch_v(const ScanArgs& a, const Work& w, const ScanPlan& p, cudaStream_t stream) {
  // the 16-byte staging path exists only where every row can take it
  constexpr bool kCanVec = N * sizeof(Tin) >= 16;
  if constexpr (kCanVec) {
    if (p.act_vec && p.bc_vec) return launch_k<PASS, N, Tin, GATE, KC, YB, true>(a, w, p, stream);
  }
  return launch_k<PASS, N, Tin, GATE, KC, YB, false>(a, w, p, stream);
}

template <int PASS, int N, typename Tin, int KC>
cudaError_t launch_gy(const ScanArgs& a, const Work& w, const ScanPlan& p, cudaStream_t stream) {
  if constexpr (PASS == kStateOnly) {
    return launch_v<PASS, N, Tin, false, KC, false>(a, w, p, stream);  // no gate, no y
  } else {
    if (a.z != nullptr)
      return a.y_bf16 ? launch_v<PASS, N, Tin, true, KC, true>(a, w, p, stream)
                      : launch_v<PASS, N, Tin, true, KC, false>(a, w, p, stream);
    return a.y_bf16 ? launch_v<PASS, N, Tin, false, KC, true>(a, w, p, stream)
                    : launch_v<PASS, N, Tin, false, KC, false>(a, w, p, stream);
  }
}

template <int PASS, int N, typename Tin>
cudaError_t launch_kc(const ScanArgs& a, const Work& w, const ScanPlan& p, cudaStream_t stream) {
  switch (a.K) {
    case 0: return launch_gy<PASS, N, Tin, 0>(a, w, p, stream);
    case 1: return launch_gy<PASS, N, Tin, 1>(a, w, p, stream);
    case 2: return launch_gy<PASS, N, Tin, 2>(a, w, p, stream);
    case 3: return launch_gy<PASS, N, Tin, 3>(a, w, p, stream);
    case 4: return launch_gy<PASS, N, Tin, 4>(a, w, p, stream);
  }
  return cudaErrorInvalidValue;
}

inline int64_t header_bytes(int64_t tiles) {
  static_assert(kHdrTiles == 4, "scan_header_bytes counts 4 leading header words");
  return scan_header_bytes(tiles);
}

template <int N, typename Tin>
cudaError_t launch_n(const ScanArgs& a, const ScanPlan& p, float* ws, cudaStream_t stream) {
  Work w;
  w.mode = p.shape.mode;
  w.parts = w.mode == kScanSplit ? p.shape.parts : 1;
  w.seg = p.shape.seg;
  w.span = a.T;
  w.tiles_b = (a.Di + kLanes - 1) / kLanes;
  w.n_tiles = a.B * w.tiles_b;
  w.n_slots = w.mode == kScanSplit ? 2 * w.parts - 1 : 1;
  w.wpc = 1;
  w.hdr = nullptr;
  w.slots = nullptr;
  w.faults = scan_fault_word();
  if (!w.faults) return cudaErrorInvalidSymbol;
  if (w.mode != kScanPlain) {
    w.hdr = reinterpret_cast<uint32_t*>(ws);
    w.slots = reinterpret_cast<float*>(reinterpret_cast<char*>(ws) + header_bytes(w.n_tiles));
  }
  if (w.mode == kScanPlain) {
    w.n_roles = w.n_tiles;
    return launch_kc<kFull, N, Tin>(a, w, p, stream);
  }
  if (w.mode == kScanChained) {
    // the queue head, the abort flag and the per-tile hand-off flags start at zero
    cudaError_t e = cudaMemsetAsync(ws, 0, (size_t)header_bytes(w.n_tiles), stream);
    if (e != cudaSuccess) return e;
    w.n_roles = w.n_tiles;  // set from the resident warps at launch
    return launch_kc<kFull, N, Tin>(a, w, p, stream);
  }
  // split: state-only pass of parts 0..P-2, the fold, then the full pass of every part
  w.n_roles = w.n_tiles * (w.parts - 1);
  cudaError_t e = launch_kc<kStateOnly, N, Tin>(a, w, p, stream);
  if (e != cudaSuccess) return e;
  const int64_t threads = w.n_tiles * N * kLanes;
  if ((threads + 127) / 128 > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  e = launch_pdl(false, scan_fold_kernel, dim3((unsigned)((threads + 127) / 128)), dim3(128), 0, stream, a, w, N);
  if (e != cudaSuccess) return e;
  w.n_roles = w.n_tiles * w.parts;
  return launch_kc<kFull, N, Tin>(a, w, p, stream);
}

}  // namespace
}  // namespace scan
}  // namespace mamba
