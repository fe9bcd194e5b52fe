/*
 * mamba_oracle.c - plain, slow, sequential f64 CPU oracle for the Mamba-1
 * selective-SSM mixer core (causal depthwise conv1d + SiLU, selective scan
 * with SiLU(z) gate, and the T=1 decode steps on a per-layer state slab).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness oracle that the CUDA
 * path is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load it.  The product library
 * never links, loads or calls it, and it shares no code with the CUDA kernels.
 *
 * Everything is computed in IEEE double precision, one (batch, channel) row at
 * a time, in the order the recurrence is written.  Threads are used only to
 * run independent rows side by side; each row is computed by one thread with
 * no reordering.  Inputs arrive as dense f64 arrays (f32 and bf16 upcast to f64
 * exactly by the caller).
 *
 * Sources (the docs.rs source views of the `mamba-rs` crate):
 *   - mamba-rs 0.5.1 src/mamba_ssm/gpu/inference.rs, `GpuInferenceState`
 *     doc comment: per-layer state layout conv [n_layers][batch*d_inner*d_conv]
 *     and ssm [n_layers][batch*d_inner*d_state]; the GPU conv keeps all d_conv
 *     slots as a shift register.
 *   - same page, `GpuMambaInference::new`: A = -exp(A_log) ("exp_negate").
 *   - same page, step chain F7 (dt_proj GEMM with bias, then softplus), F4/F4b
 *     (conv1d step, then SiLU), F9/F10 (SSM step, then y * SiLU(gate)), and the
 *     mixed-precision step F4+F4b comment, which writes SiLU as x / (1 + exp(-x)).
 *   - mamba-rs 0.6.4 src/mamba_ssm/gpu/prefill.rs, `gpu_forward_inference_prefill`:
 *     the prefill builds on top of the persistent state rather than zeroing it;
 *     `prefill_body` F4a (conv over all T with fused SiLU) and F4d (scan with the
 *     gate fused into the y store).
 *   - The recurrence itself is not printed on the pages (the kernels are only
 *     named at their launch sites); it is the Mamba-1 selective scan
 *         h_t = exp(delta_t * A) (.) h_{t-1} + delta_t * B_t * u_t
 *         y_t = C_t . h_t + D * u_t,      out_t = y_t * SiLU(z_t)
 *     with delta = softplus(dt + dt_bias), whose argument list matches the
 *     launch sites of `ssm_step_fwd` and `ssm_parallel_fwd_nosave`.
 *
 * Readings where the pages are silent:
 *   - conv tap orientation: w[c][K-1] multiplies the newest input x_t (causal
 *     Conv1d with K-1 left padding); state slot 0 is the oldest, slot K-1 the
 *     newest; each token shifts the window left by one and appends x_t, so the
 *     slot that drops out (slot 0 before the shift) never feeds an output.
 *   - the conv prefill also takes and returns the conv state (continuation).
 *   - NULL bias / D / dt_bias mean 0; NULL z means no gate; NULL state_in means
 *     a zero state; NULL state_out discards the final state.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#include "mamba_oracle.h"

#define ORACLE_MAX_K 64
#define ORACLE_MAX_N 256

/* softplus(v) = log(1 + exp(v)), written in the overflow-free form
 * max(v, 0) + log1p(exp(-|v|)).  (inference.rs step chain F7 "softplus".) */
double oracle_softplus(double v)
{
    double a = fabs(v);
    return (v > 0.0 ? v : 0.0) + log1p(exp(-a));
}

/* SiLU(x) = x / (1 + exp(-x))  (inference.rs, mixed step F4+F4b comment). */
double oracle_silu(double x)
{
    return x / (1.0 + exp(-x));
}

/* ------------------------------------------------------------------------ */
/* Row-parallel driver: runs fn(ctx, row) for row in [0, rows) on nthreads.  */
/* ------------------------------------------------------------------------ */

typedef void (*row_fn)(const void* ctx, long row);

typedef struct {
    row_fn fn;
    const void* ctx;
    long r0, r1;
} row_task;

static void* run_rows(void* arg)
{
    row_task* t = (row_task*)arg;
    for (long r = t->r0; r < t->r1; ++r) t->fn(t->ctx, r);
    return NULL;
}

static int for_each_row(row_fn fn, const void* ctx, long rows, int nthreads)
{
    if (rows <= 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if ((long)nthreads > rows) nthreads = (int)rows;
    pthread_t th[512];
    int started[512];
    row_task tasks[512];
    long per = rows / nthreads, extra = rows % nthreads, start = 0;
    for (int i = 0; i < nthreads; ++i) {
        long cnt = per + (i < extra ? 1 : 0);
        tasks[i].fn = fn;
        tasks[i].ctx = ctx;
        tasks[i].r0 = start;
        tasks[i].r1 = start + cnt;
        start += cnt;
        started[i] = 0;
        if (i > 0 && pthread_create(&th[i], NULL, run_rows, &tasks[i]) == 0) started[i] = 1;
    }
    /* slice 0, and any slice whose thread could not start, run here */
    for (int i = 0; i < nthreads; ++i)
        if (!started[i]) run_rows(&tasks[i]);
    for (int i = 0; i < nthreads; ++i)
        if (started[i]) pthread_join(th[i], NULL);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Causal depthwise conv1d + SiLU (prefill over T tokens, state in/out).     */
/* prefill.rs `prefill_body` F4a; inference.rs `GpuInferenceState` layout.   */
/* ------------------------------------------------------------------------ */

typedef struct {
    double* u;
    double* state_out;
    const double* x;
    const double* state_in;
    const double* w;
    const double* bias;
    long B, T, Di, K;
} conv_ctx;

static void conv_row(const void* vctx, long row)
{
    const conv_ctx* p = (const conv_ctx*)vctx;
    long b = row / p->Di, c = row % p->Di, K = p->K;
    double win[ORACLE_MAX_K];
    /* the K-slot window, oldest first, starts as the stored conv state */
    for (long k = 0; k < K; ++k)
        win[k] = p->state_in ? p->state_in[(b * p->Di + c) * K + k] : 0.0;
    double bias = p->bias ? p->bias[c] : 0.0;
    for (long t = 0; t < p->T; ++t) {
        long idx = (b * p->T + t) * p->Di + c;
        /* shift register: drop the oldest slot, append the new input */
        for (long k = 0; k + 1 < K; ++k) win[k] = win[k + 1];
        win[K - 1] = p->x[idx];
        double pre = bias;
        for (long k = 0; k < K; ++k) pre += p->w[c * K + k] * win[k];
        p->u[idx] = oracle_silu(pre);
    }
    if (p->state_out)
        for (long k = 0; k < K; ++k) p->state_out[(b * p->Di + c) * K + k] = win[k];
}

int oracle_conv1d_silu_prefill(double* u, double* state_out, const double* x,
                               const double* state_in, const double* w,
                               const double* bias, long B, long T, long Di, long K,
                               int nthreads)
{
    if (B < 0 || T < 0 || Di < 0 || K < 1 || K > ORACLE_MAX_K) return -1;
    if (!w || (T > 0 && (!u || !x))) return -1;
    conv_ctx c = {u, state_out, x, state_in, w, bias, B, T, Di, K};
    return for_each_row(conv_row, &c, B * Di, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Selective scan with SiLU(z) gate (prefill over T tokens, state in/out).   */
/* prefill.rs `prefill_body` F4c-F4d; inference.rs `GpuMambaInference::new`. */
/* ------------------------------------------------------------------------ */

typedef struct {
    double* y;
    double* state_out;
    const double *u, *dt, *z, *Bm, *Cm, *A_log, *D, *dt_bias, *state_in;
    long B, T, Di, N;
} scan_ctx;

static void scan_row(const void* vctx, long row)
{
    const scan_ctx* p = (const scan_ctx*)vctx;
    long b = row / p->Di, c = row % p->Di, N = p->N;
    double A[ORACLE_MAX_N], h[ORACLE_MAX_N];
    for (long n = 0; n < N; ++n) {
        A[n] = -exp(p->A_log[c * N + n]);                        /* A = -exp(A_log) */
        h[n] = p->state_in ? p->state_in[(b * p->Di + c) * N + n] : 0.0;
    }
    double Dc = p->D ? p->D[c] : 0.0;
    double bias = p->dt_bias ? p->dt_bias[c] : 0.0;
    for (long t = 0; t < p->T; ++t) {
        long idx = (b * p->T + t) * p->Di + c;
        long bc = (b * p->T + t) * N;
        double ut = p->u[idx];
        double delta = oracle_softplus(p->dt[idx] + bias);      /* delta = softplus(dt + dt_bias) */
        for (long n = 0; n < N; ++n)                             /* h = exp(delta A) h + delta B u */
            h[n] = exp(delta * A[n]) * h[n] + delta * p->Bm[bc + n] * ut;
        double yt = 0.0;
        for (long n = 0; n < N; ++n) yt += p->Cm[bc + n] * h[n]; /* y = C . h + D u */
        yt += Dc * ut;
        if (p->z) yt *= oracle_silu(p->z[idx]);                  /* out = y * SiLU(z) */
        p->y[idx] = yt;
    }
    if (p->state_out)
        for (long n = 0; n < N; ++n) p->state_out[(b * p->Di + c) * N + n] = h[n];
}

int oracle_selective_scan_prefill(double* y, double* state_out, const double* u,
                                  const double* dt, const double* z, const double* Bm,
                                  const double* Cm, const double* A_log, const double* D,
                                  const double* dt_bias, const double* state_in, long B,
                                  long T, long Di, long N, int nthreads)
{
    if (B < 0 || T < 0 || Di < 0 || N < 1 || N > ORACLE_MAX_N) return -1;
    if (!A_log || (T > 0 && (!y || !u || !dt || !Bm || !Cm))) return -1;
    scan_ctx s = {y, state_out, u, dt, z, Bm, Cm, A_log, D, dt_bias, state_in, B, T, Di, N};
    return for_each_row(scan_row, &s, B * Di, nthreads);
}

/* ------------------------------------------------------------------------ */
/* T=1 decode steps on the layer slab of a [n_layers][B*Di*S] state buffer.  */
/* inference.rs `GpuInferenceState::conv_offset` / `ssm_offset`, step chain  */
/* F4/F4b and F9/F10.  Each is the prefill above with T = 1, in place.       */
/* ------------------------------------------------------------------------ */

int oracle_conv1d_silu_step(double* u, double* conv_state, long layer, const double* x,
                            const double* w, const double* bias, long B, long Di, long K,
                            int nthreads)
{
    if (layer < 0 || !conv_state) return -1;
    double* slab = conv_state + layer * B * Di * K;
    return oracle_conv1d_silu_prefill(u, slab, x, slab, w, bias, B, 1, Di, K, nthreads);
}

int oracle_ssm_step(double* y, double* ssm_state, long layer, const double* u,
                    const double* dt, const double* z, const double* Bm, const double* Cm,
                    const double* A_log, const double* D, const double* dt_bias, long B,
                    long Di, long N, int nthreads)
{
    if (layer < 0 || !ssm_state) return -1;
    double* slab = ssm_state + layer * B * Di * N;
    return oracle_selective_scan_prefill(y, slab, u, dt, z, Bm, Cm, A_log, D, dt_bias, slab,
                                         B, 1, Di, N, nthreads);
}

/*
 * Mamba-3 SISO T=1 step (docs.rs source view of mamba-rs 0.2.1
 * src/mamba3_siso/gpu/inference.rs: `Mamba3GpuInferenceState` and the F6
 * `m3_step_fwd` launch in `step_layer_kernels`).  The page shows the state
 * buffers -- ssm [n_layers][batch*nh*hd*ds], k (the previous B after RoPE)
 * [n_layers][batch*nh*ds], v (the previous x) [n_layers][batch*nh*hd] -- and
 * the step's arguments (state, k state, v state, y, x, current k and q,
 * alpha, beta, gamma per (batch, head), D), but not the kernel body.  Read
 * plainly, the trapezoidal update mixes the previous token's input (k_prev,
 * v_prev) with weight beta and the current one with weight gamma:
 *   h[p][n] = alpha h[p][n] + beta k_prev[n] v_prev[p] + gamma k[n] x[p]
 *   y[p]    = sum_n q[n] h[p][n] + D x[p]
 * after which the k state holds k and the v state holds x.
 */
int oracle_m3_step(double* y, double* ssm_state, double* k_state, double* v_state, long layer,
                   const double* x, const double* k, const double* q, const double* alpha,
                   const double* beta, const double* gamma, const double* D, long B, long H,
                   long P, long N)
{
    if (layer < 0 || !ssm_state || !k_state || !v_state || B < 0 || H < 0 || P < 0 || N < 0)
        return -1;
    double* hs = ssm_state + layer * B * H * P * N;
    double* ks = k_state + layer * B * H * N;
    double* vs = v_state + layer * B * H * P;
    for (long b = 0; b < B; ++b) {
        for (long hd = 0; hd < H; ++hd) {
            const long bh = b * H + hd;
            const double a = alpha[bh], be = beta[bh], g = gamma[bh];
            for (long p = 0; p < P; ++p) {
                double* hrow = hs + (bh * P + p) * N;
                const double xp = x[bh * P + p];
                const double vp = vs[bh * P + p];
                double acc = 0.0;
                for (long n = 0; n < N; ++n) {
                    const double kp = ks[bh * N + n];
                    hrow[n] = a * hrow[n] + be * kp * vp + g * k[bh * N + n] * xp;
                    acc += q[bh * N + n] * hrow[n];
                }
                y[bh * P + p] = acc + (D ? D[hd] : 0.0) * xp;
            }
            for (long n = 0; n < N; ++n) ks[bh * N + n] = k[bh * N + n];
            for (long p = 0; p < P; ++p) vs[bh * P + p] = x[bh * P + p];
        }
    }
    return 0;
}

/*
 * Mamba-3 SISO step inputs from one token's projections (docs.rs source view
 * of mamba-rs 0.2.1 src/mamba3_siso/gpu/inference.rs, `step_layer_kernels`:
 * step F4c "Angle accumulation + RoPE" -- the `m3_angle_dt_fwd_batch` launch
 * (angle_cumsum out, the layer's angle_state in/out, angles_raw
 * [batch][n_angles], dt [batch][nh]) and the `rope_fwd` launch (B and C
 * rotated in pairs by angle_cumsum into the step's k and q) -- and step F5
 * `m3_compute_abg` (alpha, beta, gamma from dt, a_val and trap); the page
 * header cites the Mamba-3 paper for the method).  The page prints the
 * launches, not the kernel bodies.  Read plainly, with the paper's
 * exponential-trapezoidal rule and its data-dependent rotation:
 *   theta[b][h][i] += dt[b][h] * angles[b][i]                  (i < n_angles)
 *   (k[2i], k[2i+1]) = R(theta[b][h][i]) (k_in[2i], k_in[2i+1]),
 *       R(t) = [[cos t, -sin t], [sin t, cos t]]; q likewise from q_in;
 *       the components from 2 n_angles on are copied
 *   alpha = exp(dt A), beta = (1 - lam) dt alpha, gamma = lam dt
 * (beta weighs the previous token's input, decayed over the step; gamma the
 * current one).  Layouts: k_in, q_in, k, q [B][H][N]; dt, A, lam, alpha,
 * beta, gamma [B][H]; angles [B][n_angles]; angle_state the base of
 * [n_layers][B][H][n_angles] (NULL allowed when n_angles == 0).
 */
int oracle_m3_prepare(double* k, double* q, double* alpha, double* beta, double* gamma,
                      double* angle_state, long layer, const double* k_in, const double* q_in,
                      const double* dt, const double* A, const double* lam,
                      const double* angles, long B, long H, long N, long n_angles)
{
    if (layer < 0 || B < 0 || H < 0 || N < 0 || n_angles < 0 || 2 * n_angles > N)
        return -1;
    if (n_angles > 0 && (!angle_state || !angles))
        return -1;
    double* th = n_angles > 0 ? angle_state + layer * B * H * n_angles : NULL;
    for (long b = 0; b < B; ++b) {
        for (long hd = 0; hd < H; ++hd) {
            const long bh = b * H + hd;
            const double d = dt[bh];
            for (long n = 0; n < N; ++n) {
                k[bh * N + n] = k_in[bh * N + n];
                q[bh * N + n] = q_in[bh * N + n];
            }
            for (long i = 0; i < n_angles; ++i) {
                th[bh * n_angles + i] += d * angles[b * n_angles + i];
                const double t = th[bh * n_angles + i];
                const double c = cos(t), s = sin(t);
                const long e = bh * N + 2 * i, o = e + 1;
                k[e] = c * k_in[e] - s * k_in[o];
                k[o] = s * k_in[e] + c * k_in[o];
                q[e] = c * q_in[e] - s * q_in[o];
                q[o] = s * q_in[e] + c * q_in[o];
            }
            const double a = exp(d * A[bh]);
            alpha[bh] = a;
            beta[bh] = (1.0 - lam[bh]) * d * a;
            gamma[bh] = lam[bh] * d;
        }
    }
    return 0;
}
