/*
 * mamba_ssm.h - C ABI of the GB300-native (sm_103a) Mamba-1 selective-SSM
 * mixer core: causal depthwise conv1d + SiLU, the selective scan with SiLU(z)
 * gate, and the batched T=1 decode steps on a persistent per-layer state.
 *
 * What is computed (Mamba-1, as the mamba-rs GPU inference engine runs it):
 *
 *   conv:  s = [conv_state[b][c][1..K-1], x[b][0..T-1][c]]
 *          pre_t = bias[c] + sum_{k<K} w[c][k] * s[t+k]     (w[c][K-1] meets x_t)
 *          u_t   = pre_t * sigmoid(pre_t)                    (SiLU)
 *          conv_state' = last K entries of [conv_state[b][c][0..K-1], x[b][..][c]]
 *   scan:  A = -exp(A_log),  delta_t = softplus(dt_t + dt_bias)
 *          h_t = exp(delta_t A) (.) h_{t-1} + delta_t B_t u_t
 *          y_t = C_t . h_t + D u_t,   out_t = y_t * SiLU(z_t)   (no gate if z == NULL)
 *
 * Sources (docs.rs source views of the `mamba-rs` crate):
 *   - mamba-rs 0.5.1 src/mamba_ssm/gpu/inference.rs: `GpuInferenceState` (state
 *     layout [n_layers][batch*d_inner*d_conv] / [n_layers][batch*d_inner*d_state],
 *     f32, full d_conv-slot shift register; `conv_offset` / `ssm_offset`),
 *     `GpuMambaInference::new` (A = -exp(A_log)), the f32 step chain F4-F10
 *     and the mixed step chain (conv1d step with fused SiLU; SSM step with fused
 *     gate; state stays f32 under bf16 activations; d_state <= 64 guard).
 *   - mamba-rs 0.6.4 src/mamba_ssm/gpu/prefill.rs: `gpu_forward_inference_prefill`
 *     (prefill builds on the persistent state, it does not zero it),
 *     `prefill_body` F4a (conv over all T with fused SiLU, strided x lane),
 *     F4c (softplus), F4d (scan, gate fused into the y store, strided gate and
 *     B/C reads).
 *
 * Conventions (every entry point):
 *   - Status: 0 (MAMBA_OK) or a negative MAMBA_ERR_* code.  On error nothing was
 *     launched and mamba_last_error() (thread-local) says why.
 *   - Arguments are checked on the host before any work: NULL required
 *     pointers, negative sizes, unsupported d_state / d_conv / dtypes, strides
 *     smaller than a row, 64-bit extent overflow and overlapping buffers.
 *   - Memory: every pointer is a DEVICE pointer owned by the caller.  The
 *     library allocates, frees and synchronises nothing; every call only
 *     enqueues kernels on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns.  Results are ready when the stream reaches them.
 *   - Layout: activations are row-major [batch][T][channels] with the channels
 *     contiguous; element (b, t, c) lives at base + (b*T + t)*ld + c, so `ld`
 *     (elements, >= channels) lets a caller pass a column slice of a wider
 *     buffer (e.g. the x or z half of an in_proj output, or the B / C columns
 *     of an x_proj output).  Parameters and states are f32.
 *   - Dtypes: MAMBA_F32 or MAMBA_BF16 storage; all arithmetic is f32; a bf16
 *     output is rounded once, to nearest even.
 *   - Optional pointers: bias, D, dt_bias may be NULL (treated as 0); z may be
 *     NULL (no gate); state_in may be NULL (zero state); state_out may be NULL
 *     (final state discarded).  state_out may equal state_in (in place); no
 *     other output may overlap any input or output.
 *   - Alignment: pointers need only their element's alignment (4 bytes for
 *     f32, 2 for bf16).  Bases and row strides that are multiples of 16
 *     bytes take the 16-byte vector and bulk-copy paths; any other layout
 *     runs an element-wise path with the same arithmetic and the same bits.
 *     Two buffers must be 16-byte aligned: a prefill workspace and the
 *     Mamba-3 step's ssm_state (both refused with MAMBA_ERR_INVALID_ARG).
 *   - The device must be compute capability 10.3 (GB300, sm_103a).
 *   - The first call of a kernel variant on a device configures it (shared
 *     memory opt-in, occupancy query); make that first call outside stream
 *     capture, or capture in relaxed mode (cudaStreamCaptureModeRelaxed).
 */
#ifndef MAMBA_SSM_H
#define MAMBA_SSM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MAMBA_API __attribute__((visibility("default")))
#else
#define MAMBA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define MAMBA_OK 0
#define MAMBA_ERR_INVALID_ARG (-1) /* bad pointer, size, stride, dtype or aliasing */
#define MAMBA_ERR_UNSUPPORTED (-2) /* valid but not built: d_state, d_conv, device */
#define MAMBA_ERR_CUDA (-3)        /* a CUDA runtime call or launch failed */

#define MAMBA_F32 0
#define MAMBA_BF16 1

#define MAMBA_MAX_D_CONV 8 /* d_conv in 1..8 */
#define MAMBA_MAX_FUSED_D_CONV 4 /* d_conv of the fused prefill: 1..4 */
/* d_state in {1, 2, 4, 8, 16, 32, 64} (mirrors the d_state <= 64 register
 * contract of the fused step kernel in inference.rs, mixed step F8+F9+F10). */
#define MAMBA_MAX_D_STATE 64

/*
 * Causal depthwise conv1d + SiLU over T tokens, continuing from a conv state.
 * (prefill.rs `prefill_body` F4a, the conv1d burn-in launch with fused SiLU;
 *  inference.rs `GpuInferenceState`: d_conv slots, slot 0 oldest.)
 *
 *   u              [B][T][Di] at ld_u (elements), dtype act_dtype      (out)
 *   x              [B][T][Di] at ld_x, dtype act_dtype                 (in)
 *   conv_state_in  [B][Di][K] f32, or NULL for a zero state            (in)
 *   conv_state_out [B][Di][K] f32, or NULL; may equal conv_state_in    (out)
 *   w              [Di][K] f32 taps; w[c][K-1] multiplies the newest x (in)
 *   bias           [Di] f32 or NULL                                   (in)
 * T == 0 copies conv_state_in to conv_state_out (zeros if in is NULL).
 * Errors: MAMBA_ERR_INVALID_ARG for NULL u/x/w (when T > 0), ld < Di,
 * u overlapping x; MAMBA_ERR_UNSUPPORTED for K outside 1..8.
 */
MAMBA_API int mamba_conv1d_silu_prefill(void* u, int64_t ld_u, const void* x, int64_t ld_x,
                              int act_dtype, const float* conv_state_in,
                              float* conv_state_out, const float* w, const float* bias,
                              int64_t B, int64_t T, int64_t Di, int64_t K, void* stream);

/*
 * One T=1 conv1d + SiLU step, in place on the `layer` slab of a persistent
 * conv state laid out [n_layers][B][Di][K] f32 (slab offset layer*B*Di*K).
 * (inference.rs step chain F4 + F4b, fused as in the mixed step's
 *  conv1d step with epilogue SiLU.)
 *
 *   u          [B][Di] dense, dtype act_dtype (out)
 *   x          [B][Di] dense, dtype act_dtype (in)
 *   conv_state base of [n_layers][B][Di][K] f32 (in/out, only slab `layer`)
 *   w, bias    as for the prefill
 * Errors: MAMBA_ERR_INVALID_ARG for layer outside [0, n_layers) or bad
 * pointers / overlap; MAMBA_ERR_UNSUPPORTED for K outside 1..8.
 */
MAMBA_API int mamba_conv1d_silu_step(void* u, const void* x, int act_dtype, float* conv_state,
                           int64_t layer, int64_t n_layers, const float* w,
                           const float* bias, int64_t B, int64_t Di, int64_t K,
                           void* stream);

/*
 * Selective scan over T tokens with SiLU(z) gate, continuing from a state and
 * returning the state after the last token, so prefill(T1) then prefill(T2)
 * equals prefill(T1 + T2) up to rounding.
 * (prefill.rs `gpu_forward_inference_prefill` "do NOT zero, we build on top";
 *  `prefill_body` F4c softplus and F4d scan with the gate fused into the y
 *  store; inference.rs `GpuMambaInference::new` exp_negate.)
 *
 *   y      [B][T][Di] at ld_y, dtype y_dtype                       (out)
 *   u      [B][T][Di] at ld_u, dtype in_dtype                      (in)
 *   dt     [B][T][Di] at ld_dt (pre-bias; delta = softplus(dt + dt_bias))
 *   z      [B][T][Di] at ld_z, or NULL for no gate
 *   Bm, Cm [B][T][N] at ld_B / ld_C (elements, >= N)
 *   A_log  [Di][N] f32;  D, dt_bias [Di] f32 or NULL
 *   ssm_state_in  [B][Di][N] f32 or NULL (zeros)
 *   ssm_state_out [B][Di][N] f32 or NULL; may equal ssm_state_in
 *   workspace     device scratch of workspace_bytes bytes (16-byte aligned),
 *                 or NULL / 0.  With mamba_selective_scan_workspace_bytes()
 *                 bytes the call balances the scan over all SMs: wide shapes
 *                 hand each tile's state from one stretch of rows to the next
 *                 through the workspace, and narrow shapes (few batch x channel
 *                 rows, e.g. batch 1) are split along T into parts scanned in
 *                 parallel and joined by their carries.  With less, a narrow
 *                 shape is split into as many parts as the workspace holds, and
 *                 anything else runs as one sequential pass per 32 channels
 *                 (same result up to rounding, slower).  Contents on entry are
 *                 ignored (the call clears what it needs); calls that share a
 *                 workspace must not overlap in time (same stream, or ordered
 *                 by events).
 * T == 0 copies the state.
 * Errors: MAMBA_ERR_INVALID_ARG for NULL required pointers, ld < row width,
 * y overlapping an input; MAMBA_ERR_UNSUPPORTED for N not in {1,2,4,...,64}.
 */
MAMBA_API int mamba_selective_scan_prefill(void* y, int64_t ld_y, int y_dtype, const void* u,
                                 int64_t ld_u, const void* dt, int64_t ld_dt,
                                 const void* z, int64_t ld_z, const void* Bm, int64_t ld_B,
                                 const void* Cm, int64_t ld_C, int in_dtype,
                                 const float* A_log, const float* D, const float* dt_bias,
                                 const float* ssm_state_in, float* ssm_state_out, int64_t B,
                                 int64_t T, int64_t Di, int64_t N, void* workspace,
                                 int64_t workspace_bytes, void* stream);

/*
 * Workspace (bytes) that mamba_selective_scan_prefill (and mamba_mixer_prefill)
 * uses to balance a [B, T, Di] x d_state N prefill over the SMs of the CURRENT
 * device (the plan depends on its SM count).  0 means the call runs as one
 * sequential pass per 32 channels and needs no workspace.  Negative MAMBA_ERR_*
 * on bad sizes or no usable device.
 */
MAMBA_API int64_t mamba_selective_scan_workspace_bytes(int64_t B, int64_t T, int64_t Di, int64_t N);

/*
 * Batched T=1 SSM step with fused gate, in place on the `layer` slab of a
 * persistent state laid out [n_layers][B][Di][N] f32 (offset layer*B*Di*N).
 * (inference.rs step chain F9 + F10, fused as in the mixed step's
 *  gather + SSM step + gate kernel; `GpuInferenceState::ssm_offset`.)
 *
 *   y      [B][Di] dense, dtype y_dtype (out)
 *   u, dt  [B][Di] dense, dtype in_dtype; z [B][Di] or NULL
 *   Bm, Cm [B][N] dense, dtype in_dtype
 *   A_log  [Di][N] f32; D, dt_bias [Di] f32 or NULL
 *   ssm_state base of [n_layers][B][Di][N] f32 (in/out, only slab `layer`)
 * The per-token arithmetic is the one the prefill uses, in the same order, so
 * one step equals a T=1 prefill bit for bit.
 * Errors: as for the prefill, plus layer outside [0, n_layers).
 */
MAMBA_API int mamba_ssm_step_batched(void* y, int y_dtype, const void* u, const void* dt,
                           const void* z, const void* Bm, const void* Cm, int in_dtype,
                           const float* A_log, const float* D, const float* dt_bias,
                           float* ssm_state, int64_t layer, int64_t n_layers, int64_t B,
                           int64_t Di, int64_t N, void* stream);

/*
 * Fused T=1 decode step of the whole mixer core: the conv1d + SiLU step on x
 * followed by the SSM step on its output u, in one kernel, in place on the
 * `layer` slabs of both persistent states ([n_layers][B][Di][K] and
 * [n_layers][B][Di][N], f32).  (inference.rs: the mixed step already fuses the
 * conv step with its SiLU and the gather + SSM step + gate; here both halves
 * share one launch and u stays in registers.)
 *
 *   y          [B][Di] dense, dtype y_dtype (out)
 *   x, dt      [B][Di] dense, dtype act_dtype; z [B][Di] or NULL
 *   Bm, Cm     [B][N] dense, dtype act_dtype
 *   conv_w [Di][K], conv_b [Di] or NULL, A_log [Di][N], D / dt_bias [Di] or NULL: f32
 * The result equals mamba_conv1d_silu_step then mamba_ssm_step_batched bit for
 * bit (u is rounded to act_dtype in between, as the separate calls store it).
 * Errors: as for the two separate steps.
 */
MAMBA_API int mamba_mixer_step_batched(void* y, int y_dtype, const void* x, const void* dt,
                                       const void* z, const void* Bm, const void* Cm,
                                       int act_dtype, const float* conv_w, const float* conv_b,
                                       const float* A_log, const float* D, const float* dt_bias,
                                       float* conv_state, float* ssm_state, int64_t layer,
                                       int64_t n_layers, int64_t B, int64_t Di, int64_t K,
                                       int64_t N, void* stream);

/*
 * Fused prefill of the whole mixer core: the conv1d + SiLU prefill and the
 * selective-scan prefill in one pass, so u is never stored.  (prefill.rs
 * `prefill_body` runs F4a, conv over all T with fused SiLU, and then F4c/F4d,
 * softplus and the scan with the gate fused into the y store; here the scan
 * computes each token's u from x itself.)  The result equals
 * mamba_conv1d_silu_prefill followed by mamba_selective_scan_prefill on its u
 * bit for bit: u is rounded to act_dtype in between, as the separate conv
 * stores it.
 *
 *   y [B][T] rows of ld_y, dtype y_dtype (out)
 *   x, dt, z (or NULL): [B][T] rows of ld_x / ld_dt / ld_z, dtype act_dtype
 *   Bm, Cm [B][T][N] rows of ld_B / ld_C, dtype act_dtype
 *   conv_w [Di][K], conv_b [Di] or NULL, A_log [Di][N], D / dt_bias [Di] or NULL: f32
 *   conv_state_in / _out [B][Di][K], ssm_state_in / _out [B][Di][N]: f32; an _in
 *   may be NULL (zero state), an _out NULL (discarded), and each _out may equal
 *   its _in (in place).
 *   workspace: as for mamba_selective_scan_prefill (same size query).
 * d_conv must be in 1..MAMBA_MAX_FUSED_D_CONV (MAMBA_ERR_UNSUPPORTED otherwise:
 * use the two calls).
 * Errors: as for the two separate prefills.
 */
MAMBA_API int mamba_mixer_prefill(void* y, int64_t ld_y, int y_dtype, const void* x, int64_t ld_x,
                                  const void* dt, int64_t ld_dt, const void* z, int64_t ld_z,
                                  const void* Bm, int64_t ld_B, const void* Cm, int64_t ld_C,
                                  int act_dtype, const float* conv_w, const float* conv_b,
                                  const float* conv_state_in, float* conv_state_out,
                                  const float* A_log, const float* D, const float* dt_bias,
                                  const float* ssm_state_in, float* ssm_state_out, int64_t B,
                                  int64_t T, int64_t Di, int64_t K, int64_t N, void* workspace,
                                  int64_t workspace_bytes, void* stream);

/*
 * mamba3_siso_step_batched - batched T=1 step of the Mamba-3 SISO mixer (the
 * trapezoidal SSM recurrence), in place on the `layer` slabs of its three
 * persistent states.  (mamba-rs 0.2.1 mamba3_siso/gpu/inference.rs:
 * `Mamba3GpuInferenceState` -- SSM [n_layers][batch*nh*hd*ds], k = previous B
 * after RoPE [n_layers][batch*nh*ds], v = previous x [n_layers][batch*nh*hd] --
 * and step F6 `m3_step_fwd` on the current x, k, q and the alpha / beta /
 * gamma of F5.  The page prints the launch, not the kernel; the update read off
 * its arguments is, per (batch b, head h, row p, state n):
 *   h = alpha h + beta k_prev[n] v_prev[p] + gamma k[n] x[p]
 *   y[p] = sum_n q[n] h[p][n] + D[h] x[p]
 * after which the k state holds k and the v state holds x.)
 *
 *   y          [B][H][P] dense, dtype y_dtype (out)
 *   x          [B][H][P] dense, dtype act_dtype
 *   k, q       [B][H][N] dense, dtype act_dtype (B and C after norm, bias, RoPE)
 *   alpha, beta, gamma [B][H] f32; D [H] f32 or NULL
 *   ssm_state  base of [n_layers][B][H][P][N] f32 (16-byte aligned)
 *   k_state    base of [n_layers][B][H][N] f32; v_state base of [n_layers][B][H][P] f32
 * N (d_state) in {16, 32, 64, 128}; P * N / 8 <= 2048.
 * Errors: as for mamba_ssm_step_batched.
 */
MAMBA_API int mamba3_siso_step_batched(void* y, int y_dtype, const void* x, const void* k, const void* q,
                                       int act_dtype, const float* alpha, const float* beta,
                                       const float* gamma, const float* D, float* ssm_state, float* k_state,
                                       float* v_state, int64_t layer, int64_t n_layers, int64_t B, int64_t H,
                                       int64_t P, int64_t N, void* stream);

/*
 * mamba3_siso_step_prepare - the inputs of one Mamba-3 SISO step from the
 * token's projections, and the fourth persistent state advanced by one token.
 * (mamba-rs 0.2.1 mamba3_siso/gpu/inference.rs: `Mamba3GpuInferenceState`
 * keeps an angle state [n_layers][batch*nh*n_angles]; step F4c launches
 * `m3_angle_dt_fwd_batch` (angle_cumsum out, angle_state in/out, angles_raw
 * [batch][n_angles], dt [batch][nh]) and `rope_fwd` (B and C rotated in pairs
 * by angle_cumsum into the step's k and q), and step F5 `m3_compute_abg`
 * (alpha, beta, gamma from dt, a_val and trap).  The page prints the launches,
 * not the kernel bodies; read plainly, with the exponential-trapezoidal rule
 * of the Mamba-3 paper the page cites, per (batch b, head h):
 *   theta[i] += dt angles[b][i]                        (i < n_angles)
 *   (k[2i], k[2i+1]) = R(theta[i]) (k_in[2i], k_in[2i+1]), q likewise,
 *       R(t) = [[cos t, -sin t], [sin t, cos t]]; components 2 n_angles.. copied
 *   alpha = exp(dt A), beta = (1 - lam) dt alpha, gamma = lam dt
 * One launch does F4c and F5; its k, q, alpha, beta and gamma are the inputs
 * of mamba3_siso_step_batched.)
 *
 *   k, q         [B][H][N] dense, dtype kq_dtype (out)
 *   alpha, beta, gamma [B][H] f32 (out)
 *   k_in, q_in   [B][H][N] f32 (B and C after the norm and the bias)
 *   dt, A, lam   [B][H] f32 (step size after softplus, the decay rate A < 0 as
 *                the split produces it, the trapezoid weight in [0, 1])
 *   angles       [B][n_angles] f32 (the token's raw angles; NULL when n_angles = 0)
 *   angle_state  base of [n_layers][B][H][n_angles] f32, slab `layer` updated in
 *                place (NULL when n_angles = 0; layer and n_layers are then
 *                not used)
 * N (d_state) even; 2 n_angles <= N.  The outputs may not overlap each other or
 * the inputs.  Errors: as for mamba_ssm_step_batched.
 */
MAMBA_API int mamba3_siso_step_prepare(void* k, void* q, int kq_dtype, float* alpha, float* beta, float* gamma,
                                       const float* k_in, const float* q_in, const float* dt, const float* A,
                                       const float* lam, const float* angles, float* angle_state, int64_t layer,
                                       int64_t n_layers, int64_t B, int64_t H, int64_t N, int64_t n_angles,
                                       void* stream);

/*
 * mamba3_siso_step_fused_batched - one Mamba-3 SISO token in one launch: the
 * step's inputs made exactly as mamba3_siso_step_prepare makes them (the angle
 * state advanced, k_in and q_in turned in pairs into k and q, alpha / beta /
 * gamma), then the step of mamba3_siso_step_batched on them, on the `layer`
 * slabs of the four persistent states.  (inference.rs steps F4c, F5 and F6 of
 * `step_layer_kernels`; the page launches them separately.)  k and q stay in
 * f32 registers and shared memory and never reach global memory, so the result
 * equals the two calls with f32 k and q bit for bit.
 *
 *   y          [B][H][P] dense, dtype y_dtype (out)
 *   x          [B][H][P] dense, dtype x_dtype
 *   k_in, q_in [B][H][N] f32; dt, A, lam [B][H] f32; angles [B][n_angles] f32
 *              (NULL when n_angles = 0); D [H] f32 or NULL
 *   ssm_state, k_state, v_state as for mamba3_siso_step_batched (the k state
 *              receives the turned k)
 *   angle_state base of [n_layers][B][H][n_angles] f32 (NULL when n_angles = 0)
 * N (d_state) in {16, 32, 64, 128}; 2 n_angles <= N; P * N / 8 <= 2048.
 * Errors: as for mamba_ssm_step_batched.
 */
MAMBA_API int mamba3_siso_step_fused_batched(void* y, int y_dtype, const void* x, int x_dtype, const float* k_in,
                                             const float* q_in, const float* dt, const float* A, const float* lam,
                                             const float* angles, const float* D, float* ssm_state, float* k_state,
                                             float* v_state, float* angle_state, int64_t layer, int64_t n_layers,
                                             int64_t B, int64_t H, int64_t P, int64_t N, int64_t n_angles,
                                             void* stream);

/*
 * Graph-captured decode driver.  (inference.rs `capture_graph` / `step`: after
 * a warm-up step the engine records its whole T=1 step chain into a CUDA graph
 * once and replays it every token, cutting the launch overhead from ~50 us to
 * ~5 us per step; the device pointers are fixed at capture, and the state and
 * scratch buffers must be the ones the graph was captured with.)
 *
 * mamba_decode_graph_create records n_steps x n_layers fused mixer steps
 * (mamba_mixer_step_batched), step-major: entry io[s * n_layers + l] is step s
 * of layer l, with the parameters params[l] and slab l of both states.  Every
 * step is validated exactly as mamba_mixer_step_batched validates it, before
 * the graph is instantiated; on an error nothing is created and *out is NULL.
 * mamba_decode_graph_launch replays the whole recording on `stream`: it reads
 * and writes the buffers named at creation (write new inputs into the same
 * buffers between launches), and the states advance by n_steps tokens.
 *
 *   params  [n_layers] per-layer parameters (shapes as mamba_mixer_step_batched)
 *   io      [n_steps * n_layers] per-step buffers: y (out), x, dt, z (or NULL), Bm, Cm
 *   conv_state [n_layers][B][Di][K] f32, ssm_state [n_layers][B][Di][N] f32
 * Ownership: the graph objects are the library's (host side and driver
 * resources; no device memory is allocated) until mamba_decode_graph_destroy;
 * every buffer stays the caller's and must outlive the graph.  Launches of one
 * graph on two streams at once race on the states.
 */
typedef struct MambaMixerLayerParams {
  const float* conv_w;  /* [Di][K] */
  const float* conv_b;  /* [Di] or NULL */
  const float* A_log;   /* [Di][N] */
  const float* D;       /* [Di] or NULL */
  const float* dt_bias; /* [Di] or NULL */
} MambaMixerLayerParams;

typedef struct MambaMixerStepIO {
  void* y;        /* [B][Di], y_dtype (out) */
  const void* x;  /* [B][Di], act_dtype */
  const void* dt; /* [B][Di], act_dtype */
  const void* z;  /* [B][Di], act_dtype, or NULL (no gate) */
  const void* Bm; /* [B][N], act_dtype */
  const void* Cm; /* [B][N], act_dtype */
} MambaMixerStepIO;

typedef struct MambaDecodeGraph MambaDecodeGraph;

MAMBA_API int mamba_decode_graph_create(MambaDecodeGraph** out, const MambaMixerLayerParams* params,
                                        const MambaMixerStepIO* io, int64_t n_steps, int64_t n_layers,
                                        int y_dtype, int act_dtype, float* conv_state, float* ssm_state,
                                        int64_t B, int64_t Di, int64_t K, int64_t N);
MAMBA_API int mamba_decode_graph_launch(MambaDecodeGraph* graph, void* stream);
/* Kernel launches one replay makes (n_steps * n_layers), or a negative error code. */
MAMBA_API int64_t mamba_decode_graph_kernels(const MambaDecodeGraph* graph);
/* Releases the graph; NULL is accepted.  Not while a launch of it is still running. */
MAMBA_API int mamba_decode_graph_destroy(MambaDecodeGraph* graph);

/*
 * mamba3_decode_graph_create - the Mamba-3 decode recorded once as a CUDA graph
 * (the Mamba-3 page's engine, "T=1 step + CUDA Graph": its step chain per layer
 * captured once and replayed per token; device pointers fixed at capture).
 * Records n_steps x n_layers one-launch tokens (mamba3_siso_step_fused_batched),
 * step-major: entry io[s * n_layers + l] is token s of layer l, on slab l of
 * the four states, with D[l] (D may be NULL, or hold NULL entries).  Every
 * token is validated exactly as the direct call validates it, before the graph
 * is instantiated; on an error nothing is created and *out is NULL.  Launched,
 * counted and freed with mamba_decode_graph_launch / _kernels / _destroy; the
 * buffers stay the caller's and must outlive the graph (write the next
 * tokens' inputs into the same buffers between launches).
 *
 *   io       [n_steps * n_layers] per-token buffers, shapes and dtypes as for
 *            mamba3_siso_step_fused_batched (angles NULL when n_angles = 0)
 *   ssm_state [n_layers][B][H][P][N], k_state [n_layers][B][H][N],
 *   v_state  [n_layers][B][H][P], angle_state [n_layers][B][H][n_angles] (f32)
 */
typedef struct Mamba3TokenIO {
  void* y;             /* [B][H][P], y_dtype (out) */
  const void* x;       /* [B][H][P], x_dtype */
  const float* k_in;   /* [B][H][N] */
  const float* q_in;   /* [B][H][N] */
  const float* dt;     /* [B][H] */
  const float* A;      /* [B][H] */
  const float* lam;    /* [B][H] */
  const float* angles; /* [B][n_angles] or NULL */
} Mamba3TokenIO;

MAMBA_API int mamba3_decode_graph_create(MambaDecodeGraph** out, const Mamba3TokenIO* io, const float* const* D,
                                         int64_t n_steps, int64_t n_layers, int y_dtype, int x_dtype,
                                         float* ssm_state, float* k_state, float* v_state, float* angle_state,
                                         int64_t B, int64_t H, int64_t P, int64_t N, int64_t n_angles);

/*
 * One linear layer of the Mamba-1 block on the tensor cores (bf16 operands,
 * f32 accumulation):  C[M][N] = A[M][K] . W[N][K]^T (+ R[M][N]).
 * (inference.rs step chain F2 in_proj, F5 x_proj, F6 dt_proj and F11
 *  out_proj with the residual add; prefill.rs `prefill_body` runs the same
 *  projections over all T rows.)
 *
 *   c         [M] rows of N at ld_c, dtype c_dtype (MAMBA_F32 or MAMBA_BF16)
 *   a         [M] rows of K bf16 at ld_a (activations)
 *   w         [N] rows of K bf16 at ld_w (the weight, [out_features][in_features])
 *   residual  [M] rows of N f32 at ld_r, added before the store, or NULL; it
 *             may be c itself (f32, same stride) for an in-place residual add
 * a and w must be 16-byte aligned with ld_a, ld_w multiples of 8 (the tiles
 * are moved by the tensor memory accelerator); K >= 1 of any size (the tiles
 * past K read as zero).  M, N, K below 2^31.  A shape with few output tiles
 * and a long K splits K over a cluster of CTAs that sum their parts in a fixed
 * order; the split depends on (M, N, K) only, so results are deterministic.
 * Errors: MAMBA_ERR_INVALID_ARG for NULL pointers, strides smaller than a row,
 * misaligned a / w, overlap of c with an input (other than the residual as
 * above), extent overflow.
 */
MAMBA_API int mamba_linear_bf16(void* c, int64_t ld_c, int c_dtype, const void* a, int64_t ld_a, const void* w,
                                int64_t ld_w, const float* residual, int64_t ld_r, int64_t M, int64_t N, int64_t K,
                                void* stream);

/*
 * RMSNorm of the residual stream, row by row:
 *     out[m][j] = x[m][j] / sqrt(mean_j x[m][j]^2 + eps) * weight[j]
 * (inference.rs step chain F1 "Save residual + RmsNorm" with rms_norm_eps;
 *  the mixed-precision chain and prefill.rs `prefill_body` F1 read the f32
 *  residual and write bf16 activations.)
 *
 *   out     [M] rows of D at ld_out, dtype out_dtype (rounded once)     (out)
 *   x       [M] rows of D f32 at ld_x                                   (in)
 *   weight  [D] f32                                                     (in)
 * Errors: MAMBA_ERR_INVALID_ARG for NULL pointers, eps outside [0, 1],
 * strides smaller than D, out overlapping x or weight.
 */
MAMBA_API int mamba_rmsnorm(void* out, int64_t ld_out, int out_dtype, const float* x, int64_t ld_x,
                            const float* weight, float eps, int64_t M, int64_t D, void* stream);

/*
 * One whole Mamba-1 block (residual block around the mixer), as the mamba-rs
 * engine runs a layer (inference.rs step chain F1-F12; prefill.rs
 * `prefill_body`, mixed-precision path with the residual stream in f32):
 *
 *   h  = RMSNorm(x) * norm_w                       -> bf16
 *   xz = h in_proj^T                               -> bf16 [2 d_inner]: x | z
 *   u  = SiLU(conv1d(x half) + conv_b)             -> bf16   (conv state in / out)
 *   xd = u x_proj^T                                -> bf16 [dt_rank | B | C]
 *   dt = xd[:, :dt_rank] dt_proj^T                 -> bf16   (pre-bias)
 *   y  = scan(u, softplus(dt + dt_proj_b), B, C, A_log, D) * SiLU(z)  -> bf16
 *   x  = x + y out_proj^T                          (f32, in place)
 *
 * The projections are mamba_linear_bf16 calls, the norm mamba_rmsnorm, the
 * conv and scan mamba_conv1d_silu_prefill and mamba_selective_scan_prefill
 * on strided views of the workspace (x and z at row stride 2 d_inner, B and C
 * at the x_proj output's stride): the block is exactly that sequence of calls.
 * Weights are [out_features][in_features], bf16 for the projections, f32
 * otherwise.  d_model, d_inner and dt_rank must be multiples of 8 (the
 * projections' rows are moved in 16-byte granules) and the bf16 weights
 * 16-byte aligned.
 */
typedef struct MambaLayer {
  int64_t d_model, d_inner, d_state, d_conv, dt_rank;
  float eps;              /* RMSNorm epsilon (1e-5 in the mamba-rs configs) */
  const float* norm_w;    /* [d_model] */
  const void* in_proj_w;  /* [2 d_inner][d_model] bf16 */
  const float* conv_w;    /* [d_inner][d_conv] */
  const float* conv_b;    /* [d_inner] or NULL */
  const void* x_proj_w;   /* [dt_rank + 2 d_state][d_inner] bf16 */
  const void* dt_proj_w;  /* [d_inner][dt_rank] bf16 */
  const float* dt_proj_b; /* [d_inner] or NULL (the scan's dt_bias) */
  const float* A_log;     /* [d_inner][d_state] */
  const float* D;         /* [d_inner] or NULL */
  const void* out_proj_w; /* [d_model][d_inner] bf16 */
} MambaLayer;

/* Workspace bytes a block over B x T tokens uses: the bf16 activations
 * (h, xz, u, xd, dt, y) plus, for a prefill, what the scan's fastest route
 * wants.  A step (T = 1) needs no more than mamba_layer_workspace_bytes(l, B, 1).
 * Negative MAMBA_ERR_* on invalid dims. */
MAMBA_API int64_t mamba_layer_workspace_bytes(const MambaLayer* layer, int64_t B, int64_t T);

/*
 *   hidden           [B][T][d_model] f32 residual stream, updated in place
 *   conv_state_in/out, ssm_state_in/out  as for mamba_mixer_prefill ([B][d_inner][d_conv]
 *                    and [B][d_inner][d_state] f32; in may equal out; NULL in = zeros)
 *   workspace        16-byte aligned device scratch of workspace_bytes (contents
 *                    on entry ignored); a smaller scan share than the query's
 *                    picks a slower scan route with the same results
 * Errors: MAMBA_ERR_INVALID_ARG (NULL, misaligned, overlap, workspace smaller
 * than the activations), MAMBA_ERR_UNSUPPORTED (dims); everything is checked
 * before the first launch.
 */
MAMBA_API int mamba_layer_prefill(float* hidden, const MambaLayer* layer, const float* conv_state_in,
                                  float* conv_state_out, const float* ssm_state_in, float* ssm_state_out, int64_t B,
                                  int64_t T, void* workspace, int64_t workspace_bytes, void* stream);

/*
 * One T = 1 block step for B sequences on slab `layer_index` of the
 * persistent layer-major states (conv [n_layers][B][d_inner][d_conv], ssm
 * [n_layers][B][d_inner][d_state], both updated in place): the prefill's
 * sequence with T = 1 (inference.rs `step_kernels`), the conv and the scan
 * being the T = 1 step kernels of mamba_conv1d_silu_step and
 * mamba_ssm_step_batched on the same strided views (equal to a T = 1 prefill
 * bit for bit).  hidden [B][d_model] f32 in place; workspace as for
 * mamba_layer_prefill with T = 1.
 */
MAMBA_API int mamba_layer_step(float* hidden, const MambaLayer* layer, float* conv_state, float* ssm_state,
                               int64_t layer_index, int64_t n_layers, int64_t B, void* workspace,
                               int64_t workspace_bytes, void* stream);

/*
 * One decode token through n_layers whole blocks, recorded once as a CUDA
 * graph (inference.rs `capture_graph` / `step`: the full step chain F1-F12 of
 * every layer captured after a warm-up and replayed per token): the graph
 * holds mamba_layer_step(hidden, &layers[l], conv_state, ssm_state, l,
 * n_layers, B, workspace, ...) for l = 0 .. n_layers-1, each validated as the
 * direct call validates it; on an error nothing is created.  Every layer must
 * have layer 0's dims.  Launch with mamba_decode_graph_launch (write the next
 * token's f32 hidden state [B][d_model] into `hidden` before each launch; it
 * holds the last block's output after it); mamba_decode_graph_kernels gives
 * the graph's node count; mamba_decode_graph_destroy frees it.  The buffers
 * and the weights stay the caller's and must outlive the graph.
 */
MAMBA_API int mamba_layer_decode_graph_create(MambaDecodeGraph** out, const MambaLayer* layers, int64_t n_layers,
                                              float* hidden, float* conv_state, float* ssm_state, int64_t B,
                                              void* workspace, int64_t workspace_bytes);

/*
 * mamba_selective_scan_prefill_noalloc - the selective-scan prefill for callers
 * that cannot allocate device memory.  (No counterpart in the mamba-rs pages:
 * it is an addition of this library.)
 *
 * Some callers cannot call cudaMalloc or any allocating routine when they run
 * the prefill -- an engine whose device memory is fixed at start-up, or a
 * plugin inside a framework that owns the allocator -- so they cannot supply
 * the workspace mamba_selective_scan_prefill uses to split narrow prefills
 * along T.  This variant takes that scratch from a static device array of
 * MAMBA_NOALLOC_SCRATCH_BYTES inside the library (held on every GPU that loads
 * the library, until the process exits) and otherwise behaves exactly like
 * mamba_selective_scan_prefill given a workspace of the smaller of the size
 * mamba_selective_scan_workspace_bytes reports and the array: same arguments
 * minus the workspace, same plan, same result bit for bit.  It allocates and
 * frees nothing.
 *   - A shape whose plan needs more scratch than the array holds runs as the
 *     regular entry point runs it with a workspace of MAMBA_NOALLOC_SCRATCH_BYTES
 *     (a narrow shape split into as many parts as the array holds).  A narrow
 *     shape for which not even two parts fit is rejected with
 *     MAMBA_ERR_UNSUPPORTED before anything is launched: run as one sequential
 *     pass it would be many times slower than its split.
 *   - The first call on each device looks up the array's device address with
 *     that device current; make that first call before any stream capture.
 *   - All calls share the array and it keeps the last call's contents (none of
 *     which is read before being rewritten); calls that overlap on the GPU,
 *     from two streams or two threads, race on it and must be serialised by
 *     the caller.
 */
#define MAMBA_NOALLOC_SCRATCH_BYTES (16LL * 1024 * 1024)
MAMBA_API int mamba_selective_scan_prefill_noalloc(
    void* y, int64_t ld_y, int y_dtype, const void* u, int64_t ld_u, const void* dt,
    int64_t ld_dt, const void* z, int64_t ld_z, const void* Bm, int64_t ld_B, const void* Cm,
    int64_t ld_C, int in_dtype, const float* A_log, const float* D, const float* dt_bias,
    const float* ssm_state_in, float* ssm_state_out, int64_t B, int64_t T, int64_t Di, int64_t N,
    void* stream);

/*
 * mamba_device_faults - device-side watchdog events since the last clear.
 * (No counterpart in the mamba-rs pages: an addition of this library.)
 *
 * The decode-step kernels stream their tiles through a ring of shared-memory
 * stages filled by bulk asynchronous copies and handed over with mbarriers.
 * Every wait on such a barrier is bounded (about a second of SM clock); a wait
 * that runs out sets MAMBA_FAULT_RING_WAIT here and the kernel leaves its loop
 * instead of hanging, so that launch's outputs are incomplete.  In correct
 * operation no wait runs out and the value stays 0 (mamba_selftest_bounded_wait
 * sets the bit on purpose, through the same bounded wait).
 *   - Synchronises the current device (so it cannot be called during stream
 *     capture), then returns the fault bits (>= 0) of that device, or
 *     MAMBA_ERR_CUDA.  `clear` != 0 resets the bits after reading them.
 */
#define MAMBA_FAULT_RING_WAIT 1
#define MAMBA_FAULT_SCAN_WAIT 2 /* a prefill unit waited too long for the state it continues */
#define MAMBA_FAULT_GEMM_WAIT 4 /* a projection GEMM waited too long for a tile or its MMAs */
MAMBA_API int mamba_device_faults(int clear);

/*
 * mamba_selftest_bounded_wait - exercises the watchdog path of
 * mamba_device_faults without a fault.  (No counterpart in the mamba-rs pages:
 * an addition of this library.)  It enqueues on `stream` one CTA that waits,
 * with the same bounded wait as the decode kernels' copy rings, on a fresh
 * mbarrier that needs one arrival.  With complete != 0 the CTA arrives first
 * and the wait succeeds at once.  With complete == 0 nothing arrives: after
 * limit_cycles SM clock cycles (1 .. 2^31; 2e6 is about 1 ms at 2 GHz) the wait
 * gives up, sets MAMBA_FAULT_RING_WAIT, and the kernel returns.  The device
 * stays usable.  Errors: MAMBA_ERR_INVALID_ARG for a limit out of range,
 * MAMBA_ERR_UNSUPPORTED / MAMBA_ERR_CUDA as for the other calls.
 */
MAMBA_API int mamba_selftest_bounded_wait(int64_t limit_cycles, int complete, void* stream);

/* Thread-local description of the last error returned on this thread
 * (empty string after a successful call).  Never NULL; owned by the library. */
MAMBA_API const char* mamba_last_error(void);

/* Library version string, e.g. "0.1.0". */
MAMBA_API const char* mamba_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SSM_H */
