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
//  * u, dt, z, B, C stream in chunks of TC rows through a 3-deep cp.async ring
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
//  * Route "sequential" (wide shapes: enough batch x channel rows to fill the
//    GPU): one launch, each CTA scans all T for its channels.
//  * Route "T-split" (narrow shapes, e.g. one 130m layer at batch 1): T is cut
//    into P parts.  Launch 1 scans parts 0..P-2 from a zero state and writes
//    each part's end state and total decay exp(A sum delta) to a workspace
//    (plus a snapshot of state_in).  Launch 2 folds the aggregates of the
//    preceding parts into each part's carry-in, then rescans the part from it
//    and writes y; the last part writes state_out.  A small fold kernel
//    between them chains the aggregates into each part's carry-in.  Cost: the
//    state-only rescan of P-1 parts; no cross-CTA waiting.
//  * The kernels live in scan_kernel.cuh, instantiated per (storage dtype,
//    d_state) from scan_inst.cu; this file holds the route planner.
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
// channels per one-warp CTA (one lane per channel)
inline int64_t channels_per_cta(int64_t) { return 32; }
}  // namespace

int64_t scan_workspace_bytes(int64_t B, int64_t Di, int64_t N, int parts) {
  if (parts <= 1) return 0;
  return (int64_t)(1 + 2 * (parts - 1)) * B * Di * N * (int64_t)sizeof(float);
}

int scan_parts(int64_t B, int64_t T, int64_t Di, int64_t N, const DeviceInfo& dev) {
  // Number of T parts P.  With w = ceil(tiles * P / SMs) one-warp CTAs per SM,
  // an SM needs about kWarpsSat warps to keep its pipes busy, and every part but
  // the last is scanned twice (the state-only pass costs ~3/4 of the full one),
  // so the time is ~ ceil(T / P) * (1 + 0.75 (P-1)/P) * max(w, kWarpsSat).
#ifndef MAMBA_SCAN_WARPS_SAT
#define MAMBA_SCAN_WARPS_SAT 8.0
#endif
  constexpr double kWarpsSat = MAMBA_SCAN_WARPS_SAT;
  const int64_t ct = channels_per_cta(N);
  const int64_t tiles = B * ((Di + ct - 1) / ct);
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
  // When one part per tile cannot fill the GPU, more parts keep paying well
  // past kWarpsSat while each stays long (measured on GB300: batch 4 x T 16384
  // x d_inner 2048 runs 1196 us at 5 parts, 1063 us at 32): split down to
  // parts of kLongPart rows.
  constexpr int64_t kLongPart = 512;
  if ((double)tiles < kWarpsSat * dev.sm_count) {
    const int64_t p_long = T / kLongPart < 64 ? T / kLongPart : 64;
    if (p_long > best_p) best_p = (int)p_long;
  }
  return best_p;
}

ScanPlan plan_selective_scan(const ScanArgs& a, const DeviceInfo& dev, int64_t workspace_bytes) {
  ScanPlan p;
  const int es = a.in_bf16 ? 2 : 4;
  // activation tiles move in granules of min(16, channels_per_cta * es) bytes
  const int64_t rowb = channels_per_cta(a.N) * es;
  const int g = (int)(rowb < 16 ? rowb : 16);
  p.act_vec = aligned(a.u, g) && aligned(a.dt, g) && (!a.z || aligned(a.z, g)) && (a.ld_u * es) % g == 0 &&
              (a.ld_dt * es) % g == 0 && (!a.z || (a.ld_z * es) % g == 0) && a.Di % (g / es) == 0;
  p.bc_vec = aligned(a.Bm, 16) && aligned(a.Cm, 16) && (a.ld_B * es) % 16 == 0 &&
             (a.ld_C * es) % 16 == 0 && (a.N * es) % 16 == 0;
  p.parts = scan_parts(a.B, a.T, a.Di, a.N, dev);
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
