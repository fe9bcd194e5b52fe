// launch.h - internal interface between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments have already been validated; every
// launcher only enqueues work on `stream` and returns cudaGetLastError().
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace mamba {

// Launches `kernel` on `stream`; with `pdl`, under programmatic stream
// serialisation: the kernel may be scheduled while the previous kernel on the
// stream finishes (every kernel here waits for it with griddepcontrol.wait
// before touching global memory).  The decode steps use it; the prefill
// kernels measured slower with it and launch plainly.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Sets the thread-local message returned by mamba_last_error(); returns code.
int set_last_error(int code, const char* msg);

// Synchronises the current device and returns its watchdog fault bits
// (MAMBA_FAULT_*), clearing them if asked; -1 and *err on a CUDA error.
// one CTA whose bounded mbarrier wait runs out unless `complete`, and its fault
// word (selftest.cu; read like the other watchdog words, -1 on a CUDA error)
cudaError_t launch_selftest_wait(long long limit, int complete, cudaStream_t stream);
int read_selftest_faults(bool clear);
int read_device_faults(bool clear, cudaError_t* err);

struct DeviceInfo {
  int sm_count;
  int max_smem_optin;  // bytes per block with opt-in
};

// ----------------------------------------------------------------- conv ----
struct ConvPrefillArgs {
  void* u;
  int64_t ld_u;
  const void* x;
  int64_t ld_x;
  const float* state_in;  // may be null
  float* state_out;       // may be null, may equal state_in
  const float* w;
  const float* bias;      // may be null
  int64_t B, T, Di;
  int K;
  int bf16;               // activation storage: 0 f32, 1 bf16
};
cudaError_t launch_conv1d_silu_prefill(const ConvPrefillArgs& a, const DeviceInfo& dev,
                                       cudaStream_t stream);

struct ConvStepArgs {
  void* u;
  const void* x;
  float* state;  // slab of the layer: [B][Di][K]
  const float* w;
  const float* bias;
  int64_t B, Di;
  int K;
  int bf16;
  int64_t ld_x = 0;  // row stride of x (elements); 0: dense (Di)
};
cudaError_t launch_conv1d_silu_step(const ConvStepArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream);

// ----------------------------------------------------------------- scan ----
struct ScanArgs {
  void* y;
  int64_t ld_y;
  int y_bf16;
  const void* u;
  int64_t ld_u;
  const void* dt;
  int64_t ld_dt;
  const void* z;  // may be null
  int64_t ld_z;
  const void* Bm;
  int64_t ld_B;
  const void* Cm;
  int64_t ld_C;
  int in_bf16;
  const float* A_log;
  const float* D;        // may be null
  const float* dt_bias;  // may be null
  const float* state_in;  // may be null
  float* state_out;       // may be null, may equal state_in
  int64_t B, T, Di;
  int N;
  // fused conv1d + SiLU (K > 0): u / ld_u then hold x, and u = SiLU(conv(x)) is
  // computed in the scan, rounded to the storage dtype as the conv kernel stores it
  int K = 0;
  const float* conv_w = nullptr;          // [Di][K]
  const float* conv_b = nullptr;          // [Di] or null
  const float* conv_state_in = nullptr;   // [B][Di][K] or null (zero)
  float* conv_state_out = nullptr;        // [B][Di][K] or null; may equal conv_state_in
};

// How a prefill is launched.  Every route is one launch of the scan kernel; its
// warps scan "segments": a 32-channel tile of one batch row over a range of rows.
//  * plain:   one warp per tile scans all T rows (no workspace)
//  * chained: one CTA per SM; its warps take "roles" from a queue in order, role
//             r being tile-rows [r*span, (r+1)*span) of the tiles laid end to
//             end, span >= T, so every warp gets the same share and a tile cut
//             between two roles is handed from one to the other through the
//             workspace: no row is scanned twice
//  * split:   T cut into `parts` parts of `seg` rows: a state-only pass per part
//             from a zero state, fold units that chain the parts' (decay, end
//             state) into carries, then a full pass per part from its carry
enum ScanMode { kScanPlain = 0, kScanChained = 1, kScanSplit = 2 };
struct ScanShapePlan {
  int mode;
  int parts;  // chained: levels; split: parts; plain: 1
  int64_t seg;  // rows per level / part
  int64_t workspace_bytes;
};
struct ScanPlan {
  ScanShapePlan shape;
  int act_vec;  // u/dt/z staged with 16-byte copies (else element loads)
  int bc_vec;   // B/C staged with 16-byte copies
};
// The route for a [B, T, Di] x N prefill given `workspace_bytes` of caller
// workspace (INT64_MAX: as much as the best route wants); it does not depend on
// the dtypes, strides or the fused conv, so the workspace query needs only sizes.
ScanShapePlan plan_scan_shape(int64_t B, int64_t T, int64_t Di, int64_t N, const DeviceInfo& dev,
                              int64_t workspace_bytes);
ScanPlan plan_selective_scan(const ScanArgs& a, const DeviceInfo& dev, int64_t workspace_bytes);
// Bytes of a chained / split workspace's header: 32-bit words (a 64-bit queue
// head, an abort flag, a counter and a flag per tile), rounded up to 256 bytes.
inline int64_t scan_header_bytes(int64_t tiles) { return ((4 * (4 + 2 * tiles)) + 255) / 256 * 256; }
// plan_scan_shape on the current device (api.cu); MAMBA_OK or an error status
int plan_scan_for_current_device(int64_t B, int64_t T, int64_t Di, int64_t N, int64_t workspace_bytes,
                                 ScanShapePlan* out);
cudaError_t launch_selective_scan_prefill(const ScanArgs& a, const ScanPlan& plan, float* ws,
                                          const DeviceInfo& dev, cudaStream_t stream);
// watchdog bits of the scan kernels' bounded waits (the device must be synchronised)
int read_scan_faults(bool clear);
// device address of the scan kernels' fault word on the current device (null on error)
int* scan_fault_word();

struct SsmStepArgs {
  void* y;
  int y_bf16;
  const void* u;
  const void* dt;
  const void* z;  // may be null
  const void* Bm;
  const void* Cm;
  int in_bf16;
  const float* A_log;
  const float* D;
  const float* dt_bias;
  float* state;  // slab of the layer: [B][Di][N]
  int64_t B, Di;
  int N;
  // row strides (elements) of u (x in the fused step), dt, z, B and C; 0: dense
  // (Di for the activations, N for B and C).  y and the states are dense.
  int64_t ld_ux = 0, ld_dt = 0, ld_z = 0, ld_B = 0, ld_C = 0;
};
cudaError_t launch_ssm_step_batched(const SsmStepArgs& a, const DeviceInfo& dev,
                                    cudaStream_t stream);

// Mamba-3 SISO T=1 step on one layer's slabs (pointers already offset).
struct M3StepArgs {
  void* y;              // [B][H][P], y_bf16 ? bf16 : f32
  int y_bf16;
  const void* x;        // [B][H][P]
  const void* k;        // [B][H][N] (B after RoPE)
  const void* q;        // [B][H][N] (C after RoPE)
  int in_bf16;
  const float* alpha;   // [B][H]
  const float* beta;    // [B][H]
  const float* gamma;   // [B][H]
  const float* D;       // [H] or null
  float* ssm_state;     // [B][H][P][N]
  float* k_state;       // [B][H][N]
  float* v_state;       // [B][H][P]
  int64_t B, H;
  int P, N;
  // the fused form (k_in non-null): k, q and alpha / beta / gamma are not
  // given but made in the step from these, as the preparation makes them
  const float* k_in;    // [B][H][N] f32 (B after norm and bias)
  const float* q_in;    // [B][H][N] f32 (C after norm and bias)
  const float* dt;      // [B][H]
  const float* A;       // [B][H]
  const float* lam;     // [B][H]
  const float* angles;  // [B][na]
  float* theta;         // this layer's angle state [B][H][na] (null when na == 0)
  int na;
};
// hd * ds / 8 must not exceed this
int m3_max_items();
cudaError_t launch_m3_step_batched(const M3StepArgs& a, const DeviceInfo& dev, cudaStream_t stream);

// The Mamba-3 step's inputs: angle state advanced, k and q rotated in pairs,
// alpha / beta / gamma (m3_prepare.cu).
struct M3PrepArgs {
  void* k;              // [B][H][N] out, kq_bf16 ? bf16 : f32
  void* q;              // [B][H][N] out
  int kq_bf16;
  float* alpha;         // [B][H] out
  float* beta;
  float* gamma;
  const float* k_in;    // [B][H][N] (B after norm and bias)
  const float* q_in;    // [B][H][N] (C after norm and bias)
  const float* dt;      // [B][H]
  const float* A;       // [B][H]
  const float* lam;     // [B][H]
  const float* angles;  // [B][na]
  float* theta;         // this layer's angle state [B][H][na] (null when na == 0)
  int64_t B, H;
  int N, na;
};
cudaError_t launch_m3_prepare(const M3PrepArgs& a, cudaStream_t stream);
// watchdog bits of the Mamba-3 ring kernel (the device must be synchronised)
int read_m3_faults(bool clear);

// ---------------------------------------------------------------- layer ----
// C[M][N] = A[M][K] . W[N][K]^T (+ R), bf16 operands, f32 accumulation on the
// tensor cores (gemm.cu).  ld_* in elements; A, W rows 16-byte aligned.
struct GemmArgs {
  void* c;
  int64_t ld_c;
  int c_bf16;
  const void* a;
  int64_t ld_a;
  const void* w;
  int64_t ld_w;
  const float* r;  // residual [M][N] at ld_r, or null
  int64_t ld_r;
  int64_t M, N, K;
};
cudaError_t launch_gemm_bf16(const GemmArgs& g, cudaStream_t stream);
int read_gemm_faults(bool clear);

// out[m][j] = x[m][j] / sqrt(mean_j x[m][j]^2 + eps) * w[j]   (rmsnorm.cu)
struct RmsNormArgs {
  void* out;
  int64_t ld_out;
  int out_bf16;
  const float* x;
  int64_t ld_x;
  const float* w;
  float eps;
  int64_t M, D;
};
cudaError_t launch_rmsnorm(const RmsNormArgs& a, cudaStream_t stream);

// Fused decode step: conv1d + SiLU step on x, then the SSM step on its u.
struct MixerStepArgs {
  SsmStepArgs ssm;         // ssm.u unused (u is produced in registers)
  const void* x;           // [B][Di], storage dtype ssm.in_bf16
  float* conv_state;       // slab of the layer: [B][Di][K]
  const float* conv_w;     // [Di][K]
  const float* conv_b;     // [Di] or null
  int K;
};
cudaError_t launch_mixer_step_batched(const MixerStepArgs& a, const DeviceInfo& dev,
                                      cudaStream_t stream);

}  // namespace mamba
