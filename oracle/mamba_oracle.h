/*
 * mamba_oracle.h - declarations of the f64 CPU oracle (test infrastructure
 * only; see mamba_oracle.c).  All arrays are dense, row-major, f64:
 *   activations x, u, dt, z, y : [B][T][Di]
 *   B, C                       : [B][T][N]
 *   A_log                      : [Di][N]
 *   w                          : [Di][K]
 *   bias, D, dt_bias           : [Di]           (NULL = 0)
 *   conv state                 : [B][Di][K]     (slot 0 oldest)
 *   ssm state                  : [B][Di][N]
 * The *_step functions take the base of a [n_layers][B*Di*S] state buffer and
 * update the slab of `layer` in place.  Return 0 on success, -1 on a bad
 * argument.  `nthreads` only spreads independent (b, c) rows over threads.
 */
#ifndef MAMBA_ORACLE_H
#define MAMBA_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

double oracle_softplus(double v);
double oracle_silu(double x);

int oracle_conv1d_silu_prefill(double* u, double* state_out, const double* x,
                               const double* state_in, const double* w,
                               const double* bias, long B, long T, long Di, long K,
                               int nthreads);

int oracle_selective_scan_prefill(double* y, double* state_out, const double* u,
                                  const double* dt, const double* z, const double* Bm,
                                  const double* Cm, const double* A_log, const double* D,
                                  const double* dt_bias, const double* state_in, long B,
                                  long T, long Di, long N, int nthreads);

int oracle_conv1d_silu_step(double* u, double* conv_state, long layer, const double* x,
                            const double* w, const double* bias, long B, long Di, long K,
                            int nthreads);

int oracle_ssm_step(double* y, double* ssm_state, long layer, const double* u,
                    const double* dt, const double* z, const double* Bm, const double* Cm,
                    const double* A_log, const double* D, const double* dt_bias, long B,
                    long Di, long N, int nthreads);

/* Mamba-3 SISO step on the `layer` slabs (in place): x [B][H][P]; k, q
 * [B][H][N]; alpha, beta, gamma [B][H]; D [H] or NULL; ssm state
 * [n_layers][B][H][P][N], k state [n_layers][B][H][N], v state
 * [n_layers][B][H][P]; y [B][H][P]. */
int oracle_m3_step(double* y, double* ssm_state, double* k_state, double* v_state, long layer,
                   const double* x, const double* k, const double* q, const double* alpha,
                   const double* beta, const double* gamma, const double* D, long B, long H,
                   long P, long N);

/* Mamba-3 SISO step inputs (angle accumulation, rotation of k and q in pairs,
 * alpha / beta / gamma) on the `layer` slab of the angle state (in place):
 * k_in, q_in, k, q [B][H][N]; dt, A, lam, alpha, beta, gamma [B][H]; angles
 * [B][n_angles]; angle state [n_layers][B][H][n_angles]; 2 n_angles <= N. */
int oracle_m3_prepare(double* k, double* q, double* alpha, double* beta, double* gamma,
                      double* angle_state, long layer, const double* k_in, const double* q_in,
                      const double* dt, const double* A, const double* lam,
                      const double* angles, long B, long H, long N, long n_angles);

#ifdef __cplusplus
}
#endif

#endif
