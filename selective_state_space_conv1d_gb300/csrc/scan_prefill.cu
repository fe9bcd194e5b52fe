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
//    balance over the 152 SMs.  (Splitting a channel's states over several
//    lanes doubles the warps but costs more instructions per channel-row than
//    the extra occupancy returns; narrow shapes get occupancy from the T split.)
//  * u, dt, z, B, C stream in chunks of TC rows through a 2-deep cp.async ring
//    (16-byte copies, L2-only): HBM sees one read of every input and one write
//    of y.  bf16 B/C rows are widened to f32 once per chunk in shared memory.
//  * A lane keeps all N states of its channel in registers (f32) and walks the
//    rows sequentially.  Full 16-row chunks are unrolled with every row's
//    scalars (softplus, SiLU(z)) computed first, so the only serial chain is
//    the state FMA.  The state math is packed f32x2 plus one MUFU ex2 per state
//    and token: per token and channel at d_state 16 that is 16 ex2 + 64 FP32
//    lane-ops on two pipes that both saturate, which, not HBM, bounds the
//    prefill on GB300 (no tensor cores: there is no contraction).  The state math is packed f32x2 plus
//    one MUFU ex2 per state and token; no tensor cores (no contraction).
//  * One kernel serves every route.  Its warps scan "segments" (a 32-channel
//    tile of one batch row over a range of rows) and, on the persistent routes,
//    take "roles" from a queue in the workspace in index order: a role only
//    waits on roles handed out before it, which running warps hold, so the
//    order alone guarantees progress; every wait is bounded (about a second),
//    sleeps between polls, and reports MAMBA_FAULT_SCAN_WAIT if it runs out.
//  * Route "chained" (wide shapes: at least as many tiles as the GPU holds
//    warps, e.g. the 2.8b layer): one CTA of 8 warps per SM, two warps per SM
//    sub-partition, and one role per warp: role r is tile-rows [r*span,
//    (r+1)*span) of all tiles laid end to end, span = B*tiles*T / warps >= T.
//    A role scans the head of the tile it ends in first and hands that tile's
//    state to the next role through the workspace, then any whole tiles, then
//    the tail of the tile it starts in from the state the previous role handed
//    over (by then long done: the previous role's head is shorter).  Every
//    warp gets the same number of rows and no row is scanned twice.  (One
//    warp per tile left a third warp on some sub-partitions, which then ran
//    1.5x longer than the rest.)
//  * Route "plain" (half as many tiles as warps, up to as many; or no
//    workspace): one one-warp CTA per tile scans all T rows.
//  * Route "split" (narrow shapes, e.g. one 130m layer at batch 1): T is cut
//    into P parts.  A state-only role per part (all but the last) scans from a
//    zero state and leaves its end state and total decay exp(A sum delta) in
//    the workspace; fold roles (16 per tile, each a few states of every
//    channel) chain them into carries; a full role per part rescans from its
//    carry and writes y.  Cost: the state-only rescan of P-1 parts.
//  * The kernel lives in scan_kernel.cuh, instantiated per (storage dtype,
//    d_state) from scan_inst.cu; this file holds the route planner.
#include <atomic>
#include <cstdlib>

#include "launch.h"

namespace mamba {

// one per (storage dtype, d_state), compiled from scan_inst.cu
#define SCAN_DECL(n)                                                                          \
  cudaError_t launch_scan_f32_##n(const ScanArgs&, const ScanPlan&, float*, cudaStream_t);  \
  cudaError_t launch_scan_bf16_##n(const ScanArgs&, const ScanPlan&, float*, cudaStream_t);
SCAN_DECL(1)
SCAN_DECL(2)
SCAN_DECL(4)
SCAN_DECL(8)
SCAN_DECL(16)
SCAN_DECL(32)
SCAN_DECL(64)
#undef SCAN_DECL

namespace {
inline bool aligned(const void* p, int n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }
constexpr int64_t kLanes = 32;          // channels per warp (one lane per channel)
constexpr int64_t kMinPartRows = 64;    // split route: shortest part
constexpr int64_t kMaxParts = 64;       // split route: most parts
constexpr int kPlanWarpsPerSM = 8;      // warps per SM the planner assumes (two per sub-partition)

int64_t header_bytes(int64_t tiles) { return scan_header_bytes(tiles); }
int64_t slot_bytes(int64_t tiles, int64_t N) { return tiles * kLanes * N * (int64_t)sizeof(float); }
int64_t round_up(int64_t v, int64_t m) { return (v + m - 1) / m * m; }

// tuning knob read once: MAMBA_SCAN_PARTS (split part count); 0 or unset = the
// planner's choice
int64_t env_knob(const char* name) {
  const char* v = getenv(name);
  if (!v) return 0;
  const long long x = atoll(v);
  return x > 0 ? (int64_t)x : 0;
}
}  // namespace

// device-side word of MAMBA_FAULT_* bits set by the scan kernels' bounded waits
__device__ int g_scan_faults = 0;

int* scan_fault_word() {
  static std::atomic<int*> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  int* p = cache[dev].load(std::memory_order_acquire);
  if (!p) {
    void* q = nullptr;
    if (cudaGetSymbolAddress(&q, g_scan_faults) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    p = static_cast<int*>(q);
    cache[dev].store(p, std::memory_order_release);
  }
  return p;
}

int read_scan_faults(bool clear) {
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_scan_faults, sizeof(int)) != cudaSuccess) return -1;
  if (clear && v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_scan_faults, &zero, sizeof(int)) != cudaSuccess) return -1;
  }
  return v;
}

ScanShapePlan plan_scan_shape(int64_t B, int64_t T, int64_t Di, int64_t N, const DeviceInfo& dev,
                              int64_t workspace_bytes) {
  static const int64_t parts_knob = env_knob("MAMBA_SCAN_PARTS");
  ScanShapePlan p{kScanPlain, 1, T, 0};
  const int64_t tiles = B * ((Di + kLanes - 1) / kLanes);
  const int64_t warps = (int64_t)kPlanWarpsPerSM * dev.sm_count;
  if (tiles <= 0 || T <= 0) return p;
  if (tiles >= warps) {
    // wide: chained roles, one per resident warp
    const int64_t need = header_bytes(tiles) + slot_bytes(tiles, N);
    if (need > workspace_bytes) return p;
    p.mode = kScanChained;
    p.workspace_bytes = need;
    return p;
  }
  if (2 * tiles >= warps) return p;  // one warp per tile already keeps every SM busy
  // narrow: split into P parts.  A pass over a part of T/P rows takes
  // ceil(tiles P / warps) rounds of the resident warps, and the state-only pass
  // of the first P-1 parts costs about 0.88 of a full one:
  //   time ~ ceil(tiles P / warps) ceil(T / P) (1 + 0.88 (P - 1) / P)
  int64_t best_p = 1;
  double best = 0.0;
  for (int64_t P = 2; P <= kMaxParts && T / P >= kMinPartRows; ++P) {
    const double rounds = (double)((tiles * P + warps - 1) / warps);
    const double cost = rounds * (double)((T + P - 1) / P) * (1.0 + 0.88 * (double)(P - 1) / (double)P);
    if (best_p == 1 || cost < best * 0.999) {
      best = cost;
      best_p = P;
    }
  }
  int64_t P = parts_knob ? parts_knob : best_p;
  if (P > kMaxParts) P = kMaxParts;
  if (P > T / kMinPartRows) P = T / kMinPartRows;
  // the workspace holds 2P-1 slots: as many parts as it has room for
  if (workspace_bytes < header_bytes(tiles)) return p;
  const int64_t fit = (workspace_bytes - header_bytes(tiles)) / slot_bytes(tiles, N);
  if ((fit + 1) / 2 < P) P = (fit + 1) / 2;
  if (P < 2) return p;
  const int64_t seg = (T + P - 1) / P;
  P = (T + seg - 1) / seg;  // no empty part
  if (P < 2) return p;
  p.mode = kScanSplit;
  p.parts = (int)P;
  p.seg = seg;
  p.workspace_bytes = header_bytes(tiles) + (2 * P - 1) * slot_bytes(tiles, N);
  return p;
}

ScanPlan plan_selective_scan(const ScanArgs& a, const DeviceInfo& dev, int64_t workspace_bytes) {
  ScanPlan p;
  const int es = a.in_bf16 ? 2 : 4;
  // activation tiles move in granules of min(16, 32 channels * es) bytes
  const int64_t rowb = kLanes * es;
  const int g = (int)(rowb < 16 ? rowb : 16);
  p.act_vec = aligned(a.u, g) && aligned(a.dt, g) && (!a.z || aligned(a.z, g)) && (a.ld_u * es) % g == 0 &&
              (a.ld_dt * es) % g == 0 && (!a.z || (a.ld_z * es) % g == 0) && a.Di % (g / es) == 0;
  p.bc_vec = aligned(a.Bm, 16) && aligned(a.Cm, 16) && (a.ld_B * es) % 16 == 0 &&
             (a.ld_C * es) % 16 == 0 && (a.N * es) % 16 == 0;
  p.shape = plan_scan_shape(a.B, a.T, a.Di, a.N, dev, workspace_bytes);
  return p;
}

cudaError_t launch_selective_scan_prefill(const ScanArgs& a, const ScanPlan& p, float* ws,
                                          const DeviceInfo& dev, cudaStream_t stream) {
  (void)dev;
#define SCAN_CASE(n) \
  case n:            \
    return a.in_bf16 ? launch_scan_bf16_##n(a, p, ws, stream) : launch_scan_f32_##n(a, p, ws, stream);
  switch (a.N) {
    SCAN_CASE(1)
    SCAN_CASE(2)
    SCAN_CASE(4)
    SCAN_CASE(8)
    SCAN_CASE(16)
    SCAN_CASE(32)
    SCAN_CASE(64)
  }
#undef SCAN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace mamba
