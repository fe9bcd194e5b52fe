// m3_prepare.cu - the inputs of one Mamba-3 SISO step from the token's
// projections, with the layer's angle state advanced by one token.
//
// mamba-rs 0.2.1 mamba3_siso/gpu/inference.rs: `Mamba3GpuInferenceState` keeps
// per layer an angle state [batch][nh][n_angles] besides the SSM, k and v
// states; step F4c launches `m3_angle_dt_fwd_batch` (angle_cumsum out, the
// angle state in/out, angles_raw [batch][n_angles], dt [batch][nh]) and
// `rope_fwd` (B and C rotated in pairs by angle_cumsum into the step's k and
// q), and step F5 `m3_compute_abg` (alpha, beta, gamma from dt, a_val and
// trap).  The page prints the launches only; read plainly, with the
// exponential-trapezoidal rule of the Mamba-3 paper the page cites:
//   theta[j] += dt * angles[b][j]                        (j < n_angles)
//   (k[2j], k[2j+1]) = R(theta[j]) (k_in[2j], k_in[2j+1]),  R(t) the rotation by +t;
//   q likewise; the pairs from n_angles on are copied
//   alpha = exp(dt A), beta = (1 - lam) dt alpha, gamma = lam dt
// (beta weighs the previous token's input, decayed over the step; gamma the
// current one).
//
// Design (GB300): the three launches of the page are one here.  One thread per
// (batch, head, pair j of the d_state components) reads its pair of k_in and
// q_in (consecutive threads, consecutive pairs), advances and stores its angle,
// rotates and stores both pairs; the thread of pair 0 writes alpha, beta and
// gamma.  The accumulated angle grows without bound over a stream of tokens,
// so its sine and cosine come from an explicit range reduction and the MUFU
// sine and cosine (m3_math.cuh), the same arithmetic as the fused step's.  The
// kernel signals its dependents at entry, so the step that
// reads its outputs is scheduled while it runs (the step waits for it to
// complete before its first global access).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_math.cuh"
#include "launch.h"
#include "m3_math.cuh"

namespace mamba {
namespace {

template <typename Tkq>
__global__ void __launch_bounds__(256) m3_prepare_kernel(M3PrepArgs a) {
  grid_dependency_begin();
  const int half = a.N / 2;
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (i >= a.B * a.H * half) return;
  const int64_t bh = i / half;
  const int j = (int)(i - bh * half);
  const int64_t e = bh * a.N + 2 * j;
  const float d = a.dt[bh];
  float ke = a.k_in[e], ko = a.k_in[e + 1], qe = a.q_in[e], qo = a.q_in[e + 1];
  if (j < a.na) {
    const int64_t b = bh / a.H;
    const float t = m3_advance_angle(a.theta[bh * a.na + j], d, a.angles[b * a.na + j]);
    a.theta[bh * a.na + j] = t;
    float sn, cs;
    m3_sincos(t, &sn, &cs);
    m3_rotate(sn, cs, ke, ko);
    m3_rotate(sn, cs, qe, qo);
  }
  Tkq* K = reinterpret_cast<Tkq*>(a.k);
  Tkq* Q = reinterpret_cast<Tkq*>(a.q);
  K[e] = from_f32<Tkq>(ke);
  K[e + 1] = from_f32<Tkq>(ko);
  Q[e] = from_f32<Tkq>(qe);
  Q[e + 1] = from_f32<Tkq>(qo);
  if (j == 0) {
    const M3Weights w = m3_weights(d, a.A[bh], a.lam[bh]);
    a.alpha[bh] = w.alpha;
    a.beta[bh] = w.beta;
    a.gamma[bh] = w.gamma;
  }
}

}  // namespace

cudaError_t launch_m3_prepare(const M3PrepArgs& a, cudaStream_t stream) {
  const int64_t threads = a.B * a.H * (a.N / 2);
  if (threads == 0) return cudaSuccess;
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
  if (a.kq_bf16)
    return launch_pdl(true, m3_prepare_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0, stream, a);
  return launch_pdl(true, m3_prepare_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, stream, a);
}

}  // namespace mamba
