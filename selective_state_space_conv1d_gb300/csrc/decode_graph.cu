// decode_graph.cu - the graph-captured decode driver (mamba_decode_graph_*).
//
// inference.rs `capture_graph` records the engine's whole T=1 step chain into
// a CUDA graph once, after a warm-up step, and `step` replays it for every
// token (the launch overhead of a step drops from ~50 us to ~5 us); the device
// pointers are fixed at capture.  Here the recorded chain is n_steps x n_layers
// fused mixer steps, each one the public mamba_mixer_step_batched call, so the
// recording validates every step with the same host checks and launches the
// same kernels (with their programmatic-launch edges) as the direct calls.
//
// mamba_layer_decode_graph_create records the same way one token through whole
// Mamba-1 blocks (the pages' full F1-F12 chain per layer): n_layers
// mamba_layer_step calls; the graph handle is the same type.
//
// mamba3_decode_graph_create records n_steps x n_layers Mamba-3 SISO tokens,
// each the public mamba3_siso_step_fused_batched call (the Mamba-3 page's
// "T=1 step + CUDA Graph": steps F4c-F6 per layer, captured once).
//
// Capture runs on a private stream in relaxed mode: the first call of a kernel
// instance configures it (shared-memory opt-in, occupancy query), which is not
// a stream operation and must not be refused inside the capture.  Nothing runs
// on the GPU until mamba_decode_graph_launch.
#include <cuda_runtime.h>

#include <cstdio>
#include <new>
#include <string>

#include "../../include/mamba_ssm.h"
#include "launch.h"

struct MambaDecodeGraph {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  int device = 0;
  int64_t kernels = 0;
};

namespace {

int cuda_error(const char* what, cudaError_t e) {
  char msg[256];
  snprintf(msg, sizeof(msg), "%s: %s", what, cudaGetErrorString(e));
  return mamba::set_last_error(MAMBA_ERR_CUDA, msg);
}

}  // namespace

extern "C" int mamba_decode_graph_create(MambaDecodeGraph** out, const MambaMixerLayerParams* params,
                                         const MambaMixerStepIO* io, int64_t n_steps, int64_t n_layers,
                                         int y_dtype, int act_dtype, float* conv_state, float* ssm_state,
                                         int64_t B, int64_t Di, int64_t K, int64_t N) {
  if (!out) return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, "mamba_decode_graph_create: out is NULL");
  *out = nullptr;
  if (!params || !io)
    return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, "mamba_decode_graph_create: params and io must not be NULL");
  if (n_steps < 1 || n_layers < 1 || n_steps > (int64_t(1) << 20) || n_layers > (int64_t(1) << 20) ||
      n_steps * n_layers > (int64_t(1) << 24))
    return mamba::set_last_error(MAMBA_ERR_INVALID_ARG,
                                 "mamba_decode_graph_create: n_steps and n_layers must be >= 1 (at most 2^24 steps "
                                 "in one graph)");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error("cudaGetDevice", e);
  cudaStream_t s = nullptr;
  if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess)
    return cuda_error("cudaStreamCreateWithFlags", e);
  if ((e = cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed)) != cudaSuccess) {
    cudaStreamDestroy(s);
    return cuda_error("cudaStreamBeginCapture", e);
  }
  int rc = MAMBA_OK;
  std::string msg;
  int64_t kernels = 0;
  for (int64_t st = 0; st < n_steps && rc == MAMBA_OK; ++st) {
    for (int64_t l = 0; l < n_layers; ++l) {
      const MambaMixerLayerParams& p = params[l];
      const MambaMixerStepIO& q = io[st * n_layers + l];
      rc = mamba_mixer_step_batched(q.y, y_dtype, q.x, q.dt, q.z, q.Bm, q.Cm, act_dtype, p.conv_w, p.conv_b,
                                    p.A_log, p.D, p.dt_bias, conv_state, ssm_state, l, n_layers, B, Di, K, N, s);
      if (rc != MAMBA_OK) {
        char head[96];
        snprintf(head, sizeof(head), "mamba_decode_graph_create: step %lld, layer %lld: ", (long long)st,
                 (long long)l);
        msg = std::string(head) + mamba_last_error();
        break;
      }
      if (B > 0 && Di > 0) ++kernels;
    }
  }
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(s, &graph);  // ends the capture on every path
  cudaStreamDestroy(s);
  if (rc != MAMBA_OK || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    if (rc != MAMBA_OK) return mamba::set_last_error(rc, msg.c_str());
    return cuda_error("cudaStreamEndCapture", e);
  }
  cudaGraphExec_t exec = nullptr;
  if ((e = cudaGraphInstantiate(&exec, graph, 0)) != cudaSuccess) {
    cudaGraphDestroy(graph);
    return cuda_error("cudaGraphInstantiate", e);
  }
  MambaDecodeGraph* g = new (std::nothrow) MambaDecodeGraph;
  if (!g) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return mamba::set_last_error(MAMBA_ERR_CUDA, "mamba_decode_graph_create: out of host memory");
  }
  g->graph = graph;
  g->exec = exec;
  g->device = dev;
  g->kernels = kernels;
  *out = g;
  return mamba::set_last_error(MAMBA_OK, "");
}

extern "C" int mamba3_decode_graph_create(MambaDecodeGraph** out, const Mamba3TokenIO* io, const float* const* D,
                                          int64_t n_steps, int64_t n_layers, int y_dtype, int x_dtype,
                                          float* ssm_state, float* k_state, float* v_state, float* angle_state,
                                          int64_t B, int64_t H, int64_t P, int64_t N, int64_t n_angles) {
  if (!out) return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, "mamba3_decode_graph_create: out is NULL");
  *out = nullptr;
  if (!io) return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, "mamba3_decode_graph_create: io must not be NULL");
  if (n_steps < 1 || n_layers < 1 || n_steps > (int64_t(1) << 20) || n_layers > (int64_t(1) << 20) ||
      n_steps * n_layers > (int64_t(1) << 24))
    return mamba::set_last_error(MAMBA_ERR_INVALID_ARG,
                                 "mamba3_decode_graph_create: n_steps and n_layers must be >= 1 (at most 2^24 "
                                 "tokens x layers in one graph)");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error("cudaGetDevice", e);
  cudaStream_t s = nullptr;
  if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess)
    return cuda_error("cudaStreamCreateWithFlags", e);
  if ((e = cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed)) != cudaSuccess) {
    cudaStreamDestroy(s);
    return cuda_error("cudaStreamBeginCapture", e);
  }
  int rc = MAMBA_OK;
  std::string msg;
  int64_t kernels = 0;
  for (int64_t st = 0; st < n_steps && rc == MAMBA_OK; ++st) {
    for (int64_t l = 0; l < n_layers; ++l) {
      const Mamba3TokenIO& q = io[st * n_layers + l];
      rc = mamba3_siso_step_fused_batched(q.y, y_dtype, q.x, x_dtype, q.k_in, q.q_in, q.dt, q.A, q.lam, q.angles,
                                          D ? D[l] : nullptr, ssm_state, k_state, v_state, angle_state, l,
                                          n_layers, B, H, P, N, n_angles, s);
      if (rc != MAMBA_OK) {
        char head[96];
        snprintf(head, sizeof(head), "mamba3_decode_graph_create: step %lld, layer %lld: ", (long long)st,
                 (long long)l);
        msg = std::string(head) + mamba_last_error();
        break;
      }
      if (B > 0 && H > 0 && P > 0) ++kernels;
    }
  }
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(s, &graph);  // ends the capture on every path
  cudaStreamDestroy(s);
  if (rc != MAMBA_OK || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    if (rc != MAMBA_OK) return mamba::set_last_error(rc, msg.c_str());
    return cuda_error("cudaStreamEndCapture", e);
  }
  cudaGraphExec_t exec = nullptr;
  if ((e = cudaGraphInstantiate(&exec, graph, 0)) != cudaSuccess) {
    cudaGraphDestroy(graph);
    return cuda_error("cudaGraphInstantiate", e);
  }
  MambaDecodeGraph* g = new (std::nothrow) MambaDecodeGraph;
  if (!g) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return mamba::set_last_error(MAMBA_ERR_CUDA, "mamba3_decode_graph_create: out of host memory");
  }
  g->graph = graph;
  g->exec = exec;
  g->device = dev;
  g->kernels = kernels;
  *out = g;
  return mamba::set_last_error(MAMBA_OK, "");
}

// The whole-block form: one token through n_layers Mamba-1 blocks, each the
// public mamba_layer_step call on slab l of the states, recorded once.
extern "C" int mamba_layer_decode_graph_create(MambaDecodeGraph** out, const MambaLayer* layers, int64_t n_layers,
                                               float* hidden, float* conv_state, float* ssm_state, int64_t B,
                                               void* workspace, int64_t workspace_bytes) {
  if (!out) return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, "mamba_layer_decode_graph_create: out is NULL");
  *out = nullptr;
  if (!layers) return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, "mamba_layer_decode_graph_create: layers is NULL");
  if (n_layers < 1 || n_layers > (int64_t(1) << 16))
    return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, "mamba_layer_decode_graph_create: n_layers not in 1..2^16");
  for (int64_t l = 1; l < n_layers; ++l) {
    const MambaLayer& a = layers[0];
    const MambaLayer& b = layers[l];
    if (a.d_model != b.d_model || a.d_inner != b.d_inner || a.d_state != b.d_state || a.d_conv != b.d_conv ||
        a.dt_rank != b.dt_rank)
      return mamba::set_last_error(MAMBA_ERR_INVALID_ARG,
                                   "mamba_layer_decode_graph_create: every layer must have the dims of layer 0 "
                                   "(the states are one [n_layers][B][d_inner][.] slab array)");
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error("cudaGetDevice", e);
  cudaStream_t s = nullptr;
  if ((e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking)) != cudaSuccess)
    return cuda_error("cudaStreamCreateWithFlags", e);
  if ((e = cudaStreamBeginCapture(s, cudaStreamCaptureModeRelaxed)) != cudaSuccess) {
    cudaStreamDestroy(s);
    return cuda_error("cudaStreamBeginCapture", e);
  }
  int rc = MAMBA_OK;
  std::string msg;
  for (int64_t l = 0; l < n_layers; ++l) {
    rc = mamba_layer_step(hidden, &layers[l], conv_state, ssm_state, l, n_layers, B, workspace, workspace_bytes, s);
    if (rc != MAMBA_OK) {
      char head[80];
      snprintf(head, sizeof(head), "mamba_layer_decode_graph_create: layer %lld: ", (long long)l);
      msg = std::string(head) + mamba_last_error();
      break;
    }
  }
  cudaGraph_t graph = nullptr;
  e = cudaStreamEndCapture(s, &graph);  // ends the capture on every path
  cudaStreamDestroy(s);
  if (rc != MAMBA_OK || e != cudaSuccess) {
    if (graph) cudaGraphDestroy(graph);
    if (rc != MAMBA_OK) return mamba::set_last_error(rc, msg.c_str());
    return cuda_error("cudaStreamEndCapture", e);
  }
  size_t nodes = 0;
  if ((e = cudaGraphGetNodes(graph, nullptr, &nodes)) != cudaSuccess) {
    cudaGraphDestroy(graph);
    return cuda_error("cudaGraphGetNodes", e);
  }
  cudaGraphExec_t exec = nullptr;
  if ((e = cudaGraphInstantiate(&exec, graph, 0)) != cudaSuccess) {
    cudaGraphDestroy(graph);
    return cuda_error("cudaGraphInstantiate", e);
  }
  MambaDecodeGraph* g = new (std::nothrow) MambaDecodeGraph;
  if (!g) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return mamba::set_last_error(MAMBA_ERR_CUDA, "mamba_layer_decode_graph_create: out of host memory");
  }
  g->graph = graph;
  g->exec = exec;
  g->device = dev;
  g->kernels = (int64_t)nodes;
  *out = g;
  return mamba::set_last_error(MAMBA_OK, "");
}

extern "C" int mamba_decode_graph_launch(MambaDecodeGraph* g, void* stream) {
  if (!g || !g->exec) return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, "mamba_decode_graph_launch: graph is NULL");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error("cudaGetDevice", e);
  if (dev != g->device) {
    char m[128];
    snprintf(m, sizeof(m), "mamba_decode_graph_launch: graph was created on device %d, current device is %d",
             g->device, dev);
    return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, m);
  }
  if ((e = cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream))) != cudaSuccess)
    return cuda_error("cudaGraphLaunch", e);
  return mamba::set_last_error(MAMBA_OK, "");
}

extern "C" int64_t mamba_decode_graph_kernels(const MambaDecodeGraph* g) {
  if (!g) return mamba::set_last_error(MAMBA_ERR_INVALID_ARG, "mamba_decode_graph_kernels: graph is NULL");
  return g->kernels;
}

extern "C" int mamba_decode_graph_destroy(MambaDecodeGraph* g) {
  if (!g) return MAMBA_OK;
  cudaError_t e1 = g->exec ? cudaGraphExecDestroy(g->exec) : cudaSuccess;
  cudaError_t e2 = g->graph ? cudaGraphDestroy(g->graph) : cudaSuccess;
  delete g;
  if (e1 != cudaSuccess) return cuda_error("cudaGraphExecDestroy", e1);
  if (e2 != cudaSuccess) return cuda_error("cudaGraphDestroy", e2);
  return MAMBA_OK;
}
