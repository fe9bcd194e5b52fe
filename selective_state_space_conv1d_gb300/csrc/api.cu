// api.cu - the extern "C" entry points declared in include/mamba_ssm.h.
//
// Every entry point validates its arguments on the host (sizes, dtypes,
// strides, 64-bit extents, pointer kinds, overlap), picks a kernel variant from
// the shape, and enqueues it on the caller's stream.  Nothing is allocated,
// freed or synchronised, so the calls are usable inside CUDA graph capture.
// Errors follow the pages' Result<_, String> convention (mamba-rs prefill.rs
// length checks before any work) as a status code plus a thread-local message.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "../../include/mamba_ssm.h"
#include "launch.h"

namespace {

thread_local char g_err[512] = {0};

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_err[0] = 0;
  return MAMBA_OK;
}

// ---- device checks (cached per device ordinal) ------------------------------
constexpr int kMaxDevices = 64;
std::atomic<int> g_dev_state[kMaxDevices];  // 0 unknown, 1 ok, 2 unsupported
mamba::DeviceInfo g_dev_info[kMaxDevices];
int g_dev_cc[kMaxDevices];

int current_device(mamba::DeviceInfo* info) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(MAMBA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(MAMBA_ERR_UNSUPPORTED, "device ordinal %d", dev);
  int st = g_dev_state[dev].load(std::memory_order_acquire);
  if (st == 0) {
    int major = 0, minor = 0, sms = 0, smem = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return fail(MAMBA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
    g_dev_info[dev].sm_count = sms;
    g_dev_info[dev].max_smem_optin = smem;
    g_dev_cc[dev] = major * 10 + minor;
    st = (major == 10 && minor == 3) ? 1 : 2;
    g_dev_state[dev].store(st, std::memory_order_release);
  }
  if (st != 1)
    return fail(MAMBA_ERR_UNSUPPORTED,
                "this library is built for sm_103a (GB300); device %d is sm_%d", dev, g_dev_cc[dev]);
  *info = g_dev_info[dev];
  return MAMBA_OK;
}

// ---- argument checks --------------------------------------------------------
constexpr int64_t kMaxExtent = int64_t(1) << 46;  // elements per dimension product

struct Range {
  const char* name;
  uintptr_t lo, hi;  // [lo, hi) bytes; empty if lo == hi
};

// bytes spanned by rows*[cols] at stride ld (elements of es bytes)
bool span_bytes(int64_t rows, int64_t cols, int64_t ld, int es, int64_t* out) {
  if (rows <= 0 || cols <= 0) {
    *out = 0;
    return true;
  }
  if (rows > kMaxExtent || ld > kMaxExtent || cols > ld) return false;
  const __int128 span = (__int128)(rows - 1) * ld + cols;
  const __int128 bytes = span * es;
  if (bytes > (__int128)(int64_t(1) << 60)) return false;
  *out = (int64_t)bytes;
  return true;
}

Range range_of(const char* name, const void* p, int64_t bytes) {
  Range r{name, reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p)};
  if (p && bytes > 0) r.hi = r.lo + (uintptr_t)bytes;
  return r;
}

bool overlaps(const Range& a, const Range& b) {
  if (a.lo == a.hi || b.lo == b.hi) return false;
  return a.lo < b.hi && b.lo < a.hi;
}

// outputs must not overlap any other listed range
int check_overlaps(const Range* outs, int n_out, const Range* ins, int n_in) {
  for (int i = 0; i < n_out; ++i) {
    for (int j = 0; j < n_in; ++j)
      if (overlaps(outs[i], ins[j]))
        return fail(MAMBA_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, ins[j].name);
    for (int j = i + 1; j < n_out; ++j)
      if (overlaps(outs[i], outs[j]))
        return fail(MAMBA_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, outs[j].name);
  }
  return MAMBA_OK;
}

// the kernels dereference these: they must be memory this device can reach
int check_pointer(const char* name, const void* p, int dev) {
  if (!p) return MAMBA_OK;
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(MAMBA_ERR_INVALID_ARG, "%s: cudaPointerGetAttributes: %s", name, cudaGetErrorString(e));
  }
  if (at.type == cudaMemoryTypeUnregistered)
    return fail(MAMBA_ERR_INVALID_ARG, "%s is not device-accessible memory (plain host pointer)", name);
  if (at.type == cudaMemoryTypeDevice && at.device != dev)
    return fail(MAMBA_ERR_INVALID_ARG, "%s lives on device %d, current device is %d", name, at.device, dev);
  return MAMBA_OK;
}

int check_pointers(const Range* rs, int n, int dev) {
  for (int i = 0; i < n; ++i) {
    if (rs[i].lo == rs[i].hi) continue;
    int rc = check_pointer(rs[i].name, reinterpret_cast<const void*>(rs[i].lo), dev);
    if (rc) return rc;
  }
  return MAMBA_OK;
}

int check_dtype(const char* name, int dt) {
  if (dt != MAMBA_F32 && dt != MAMBA_BF16)
    return fail(MAMBA_ERR_INVALID_ARG, "%s: unknown dtype %d (expected MAMBA_F32=0 or MAMBA_BF16=1)", name, dt);
  return MAMBA_OK;
}

int es_of(int dt) { return dt == MAMBA_BF16 ? 2 : 4; }

// every size and every product of sizes used below stays under 2^46
bool sizes_ok(int64_t a, int64_t b, int64_t c = 1) {
  if (a > kMaxExtent || b > kMaxExtent || c > kMaxExtent) return false;
  return (__int128)a * b * c <= (__int128)kMaxExtent;
}

bool valid_n(int64_t n) {
  return n == 1 || n == 2 || n == 4 || n == 8 || n == 16 || n == 32 || n == 64;
}

int cuda_fail(const char* what, cudaError_t e) {
  return fail(MAMBA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// T == 0: state_out <- state_in (or zeros)
int copy_state(float* out, const float* in, int64_t count, cudaStream_t s) {
  if (!out || count <= 0 || out == in) return ok();
  cudaError_t e = in ? cudaMemcpyAsync(out, in, (size_t)count * 4, cudaMemcpyDeviceToDevice, s)
                     : cudaMemsetAsync(out, 0, (size_t)count * 4, s);
  if (e != cudaSuccess) return cuda_fail("state copy", e);
  return ok();
}

// ---- the whole Mamba-1 block ---------------------------------------------------
// Workspace layout of a block over rows = B*T tokens: six bf16 activation
// buffers, each starting on a 256-byte boundary, then the scan's share.
struct LayerPlan {
  int64_t rows, ldx;  // ldx: row stride of the x_proj output (dt_rank + 2 d_state, rounded up to 8)
  int64_t off_h, off_xz, off_u, off_xd, off_dt, off_y, act_bytes;
};

int64_t round256(int64_t b) { return (b + 255) / 256 * 256; }

int layer_plan(const MambaLayer* L, int64_t B, int64_t T, LayerPlan* p) {
  if (!L) return fail(MAMBA_ERR_INVALID_ARG, "layer is NULL");
  if (B < 0 || T < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld T=%lld)", (long long)B, (long long)T);
  const int64_t dm = L->d_model, Di = L->d_inner, N = L->d_state, K = L->d_conv, R = L->dt_rank;
  if (dm < 1 || Di < 1 || R < 1)
    return fail(MAMBA_ERR_INVALID_ARG, "d_model, d_inner and dt_rank must be >= 1");
  if (!valid_n(N)) return fail(MAMBA_ERR_UNSUPPORTED, "d_state=%lld not in {1,2,4,8,16,32,64}", (long long)N);
  if (K < 1 || K > MAMBA_MAX_D_CONV)
    return fail(MAMBA_ERR_UNSUPPORTED, "d_conv=%lld not in 1..%d", (long long)K, MAMBA_MAX_D_CONV);
  if (dm % 8 || Di % 8 || R % 8)
    return fail(MAMBA_ERR_UNSUPPORTED, "d_model=%lld, d_inner=%lld and dt_rank=%lld must be multiples of 8",
                (long long)dm, (long long)Di, (long long)R);
  if (!(L->eps >= 0.0f) || L->eps > 1.0f) return fail(MAMBA_ERR_INVALID_ARG, "eps must be in [0, 1]");
  if (dm > INT32_MAX || Di > INT32_MAX / 2 || R > INT32_MAX || !sizes_ok(B, T) || !sizes_ok(B * T, 2 * Di) ||
      !sizes_ok(B * T, dm) || !sizes_ok(B * T, R + 2 * N + 8) || !sizes_ok(2 * Di, dm) || !sizes_ok(B, Di, N) ||
      !sizes_ok(B, Di, K))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  p->rows = B * T;
  p->ldx = (R + 2 * N + 7) / 8 * 8;
  p->off_h = 0;
  p->off_xz = p->off_h + round256(p->rows * dm * 2);
  p->off_u = p->off_xz + round256(p->rows * 2 * Di * 2);
  p->off_xd = p->off_u + round256(p->rows * Di * 2);
  p->off_dt = p->off_xd + round256(p->rows * p->ldx * 2);
  p->off_y = p->off_dt + round256(p->rows * Di * 2);
  p->act_bytes = p->off_y + round256(p->rows * Di * 2);
  return MAMBA_OK;
}

// the block over B x T tokens.  A prefill gives the scan the workspace past
// the activations; a step (T = 1, states updated in place on their slab) runs
// the conv and SSM step kernels on the same strided views instead of the
// prefill kernels -- the same arithmetic, bit for bit
int run_layer(float* hidden, const MambaLayer* L, const float* conv_in, float* conv_out, const float* ssm_in,
              float* ssm_out, int64_t B, int64_t T, void* workspace, int64_t workspace_bytes, bool step,
              void* stream) {
  int rc;
  LayerPlan p;
  if ((rc = layer_plan(L, B, T, &p))) return rc;
  const int64_t dm = L->d_model, Di = L->d_inner, N = L->d_state, K = L->d_conv, R = L->dt_rank;
  if (B == 0) return ok();
  if (T == 0) {  // the states pass through
    if ((rc = mamba_conv1d_silu_prefill(nullptr, Di, nullptr, Di, MAMBA_BF16, conv_in, conv_out, L->conv_w,
                                        L->conv_b, B, 0, Di, K, stream)))
      return rc;
    return mamba_selective_scan_prefill(nullptr, Di, MAMBA_BF16, nullptr, Di, nullptr, Di, nullptr, Di, nullptr, N,
                                        nullptr, N, MAMBA_BF16, L->A_log, L->D, L->dt_proj_b, ssm_in, ssm_out, B, 0,
                                        Di, N, nullptr, 0, stream);
  }
  if (!hidden || !workspace) return fail(MAMBA_ERR_INVALID_ARG, "hidden and workspace must not be NULL");
  if (!L->norm_w || !L->in_proj_w || !L->conv_w || !L->x_proj_w || !L->dt_proj_w || !L->A_log || !L->out_proj_w)
    return fail(MAMBA_ERR_INVALID_ARG, "a required weight of the layer is NULL");
  if (reinterpret_cast<uintptr_t>(workspace) & 15) return fail(MAMBA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (workspace_bytes < p.act_bytes)
    return fail(MAMBA_ERR_INVALID_ARG, "workspace_bytes=%lld below the %lld bytes of the block's activations",
                (long long)workspace_bytes, (long long)p.act_bytes);
  for (const void* w : {L->in_proj_w, L->x_proj_w, L->dt_proj_w, L->out_proj_w})
    if (reinterpret_cast<uintptr_t>(w) & 15) return fail(MAMBA_ERR_INVALID_ARG, "the bf16 weights must be 16-byte aligned");
  // every range the sequence touches, checked together before the first launch
  const int64_t xdim = R + 2 * N;
  Range ins[] = {range_of("norm_w", L->norm_w, dm * 4), range_of("in_proj_w", L->in_proj_w, 2 * Di * dm * 2),
                 range_of("conv_w", L->conv_w, Di * K * 4), range_of("conv_b", L->conv_b, Di * 4),
                 range_of("x_proj_w", L->x_proj_w, xdim * Di * 2), range_of("dt_proj_w", L->dt_proj_w, Di * R * 2),
                 range_of("dt_proj_b", L->dt_proj_b, Di * 4), range_of("A_log", L->A_log, Di * N * 4),
                 range_of("D", L->D, Di * 4), range_of("out_proj_w", L->out_proj_w, dm * Di * 2),
                 range_of("conv_state_in", conv_in, B * Di * K * 4), range_of("ssm_state_in", ssm_in, B * Di * N * 4)};
  Range outs[] = {range_of("hidden", hidden, p.rows * dm * 4), range_of("workspace", workspace, workspace_bytes),
                  range_of("conv_state_out", conv_out, B * Di * K * 4),
                  range_of("ssm_state_out", ssm_out, B * Di * N * 4)};
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  if ((rc = check_pointers(ins, 12, dev_id)) || (rc = check_pointers(outs, 4, dev_id))) return rc;
  // a state may be updated in place: then its input range is its output range
  Range ins_x[12];
  int n_in = 0;
  for (int i = 0; i < 12; ++i) {
    if ((i == 10 && conv_in && conv_in == conv_out) || (i == 11 && ssm_in && ssm_in == ssm_out)) continue;
    ins_x[n_in++] = ins[i];
  }
  if ((rc = check_overlaps(outs, 4, ins_x, n_in))) return rc;

  char* ws = static_cast<char*>(workspace);
  auto* h = ws + p.off_h;
  auto* xz = ws + p.off_xz;
  auto* u = ws + p.off_u;
  auto* xd = ws + p.off_xd;
  auto* dt = ws + p.off_dt;
  auto* y = ws + p.off_y;
  void* scan_ws = !step && workspace_bytes > p.act_bytes ? ws + p.act_bytes : nullptr;
  const int64_t scan_bytes = scan_ws ? workspace_bytes - p.act_bytes : 0;
  const int64_t rows = p.rows, ldx = p.ldx;
  // F1 RMSNorm (f32 residual in, bf16 out); F2 in_proj
  if ((rc = mamba_rmsnorm(h, dm, MAMBA_BF16, hidden, dm, L->norm_w, L->eps, rows, dm, stream))) return rc;
  if ((rc = mamba_linear_bf16(xz, 2 * Di, MAMBA_BF16, h, dm, L->in_proj_w, dm, nullptr, 0, rows, 2 * Di, dm, stream)))
    return rc;
  // F3-F4: the conv reads the x half of xz in place (row stride 2 d_inner)
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (step) {
    mamba::ConvStepArgs ca{u, xz, conv_out, L->conv_w, L->conv_b, B, Di, (int)K, 1};
    ca.ld_x = 2 * Di;
    const cudaError_t e = mamba::launch_conv1d_silu_step(ca, dev, cs);
    if (e != cudaSuccess) return cuda_fail("layer step: conv1d_silu_step launch", e);
  } else if ((rc = mamba_conv1d_silu_prefill(u, Di, xz, 2 * Di, MAMBA_BF16, conv_in, conv_out, L->conv_w, L->conv_b,
                                             B, T, Di, K, stream))) {
    return rc;
  }
  // F5 x_proj -> [dt_rank | B | C]; F6 dt_proj on the first dt_rank columns
  if ((rc = mamba_linear_bf16(xd, ldx, MAMBA_BF16, u, Di, L->x_proj_w, Di, nullptr, 0, rows, xdim, Di, stream)))
    return rc;
  if ((rc = mamba_linear_bf16(dt, Di, MAMBA_BF16, xd, ldx, L->dt_proj_w, R, nullptr, 0, rows, Di, R, stream)))
    return rc;
  // F7-F10: softplus(dt + dt_proj_b), the scan and the SiLU(z) gate in one call
  char* xz_z = xz + Di * 2;
  char* xd_b = xd + R * 2;
  char* xd_c = xd + (R + N) * 2;
  if (step) {
    mamba::SsmStepArgs sa{y, 1, u, dt, xz_z, xd_b, xd_c, 1, L->A_log, L->D, L->dt_proj_b, ssm_out, B, Di, (int)N};
    sa.ld_ux = Di;
    sa.ld_dt = Di;
    sa.ld_z = 2 * Di;
    sa.ld_B = ldx;
    sa.ld_C = ldx;
    const cudaError_t e = mamba::launch_ssm_step_batched(sa, dev, cs);
    if (e != cudaSuccess) return cuda_fail("layer step: ssm_step_batched launch", e);
  } else if ((rc = mamba_selective_scan_prefill(y, Di, MAMBA_BF16, u, Di, dt, Di, xz_z, 2 * Di, xd_b, ldx, xd_c,
                                                ldx, MAMBA_BF16, L->A_log, L->D, L->dt_proj_b, ssm_in, ssm_out, B, T,
                                                Di, N, scan_ws, scan_bytes, stream))) {
    return rc;
  }
  // F11-F12: out_proj with the residual added in its epilogue, in place
  return mamba_linear_bf16(hidden, dm, MAMBA_F32, y, Di, L->out_proj_w, Di, hidden, dm, rows, dm, Di, stream);
}

}  // namespace

int mamba::plan_scan_for_current_device(int64_t B, int64_t T, int64_t Di, int64_t N, int64_t workspace_bytes,
                                        ScanShapePlan* out) {
  mamba::DeviceInfo dev;
  const int rc = current_device(&dev);
  if (rc) return rc;
  *out = mamba::plan_scan_shape(B, T, Di, N, dev, workspace_bytes);
  return MAMBA_OK;
}

int mamba::set_last_error(int code, const char* msg) {
  snprintf(g_err, sizeof(g_err), "%s", msg ? msg : "");
  return code;
}

extern "C" {

const char* mamba_last_error(void) { return g_err; }

const char* mamba_version(void) { return "0.1.0"; }

int mamba_device_faults(int clear) {
  cudaError_t e = cudaSuccess;
  const int v = mamba::read_device_faults(clear != 0, &e);
  if (v < 0) return fail(MAMBA_ERR_CUDA, "mamba_device_faults: %s", cudaGetErrorString(e));
  const int v3 = mamba::read_m3_faults(clear != 0);
  const int v2 = mamba::read_scan_faults(clear != 0);
  if (v2 < 0) return fail(MAMBA_ERR_CUDA, "mamba_device_faults: reading the scan watchdog failed");
  const int vg = mamba::read_gemm_faults(clear != 0);
  if (vg < 0) return fail(MAMBA_ERR_CUDA, "mamba_device_faults: reading the GEMM watchdog failed");
  if (v3 < 0) return fail(MAMBA_ERR_CUDA, "mamba_device_faults: reading the Mamba-3 watchdog failed");
  const int vs = mamba::read_selftest_faults(clear != 0);
  if (vs < 0) return fail(MAMBA_ERR_CUDA, "mamba_device_faults: reading the self-test watchdog failed");
  return ok(), v | v2 | v3 | vs | vg;
}

int mamba_selftest_bounded_wait(int64_t limit_cycles, int complete, void* stream) {
  if (limit_cycles < 1 || limit_cycles > (int64_t(1) << 31))
    return fail(MAMBA_ERR_INVALID_ARG, "limit_cycles=%lld not in 1..2^31", (long long)limit_cycles);
  mamba::DeviceInfo dev;
  int rc;
  if ((rc = current_device(&dev))) return rc;
  cudaError_t e = mamba::launch_selftest_wait(limit_cycles, complete != 0, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("mamba_selftest_bounded_wait launch", e);
  return ok();
}

int mamba_conv1d_silu_prefill(void* u, int64_t ld_u, const void* x, int64_t ld_x, int act_dtype,
                              const float* conv_state_in, float* conv_state_out, const float* w,
                              const float* bias, int64_t B, int64_t T, int64_t Di, int64_t K,
                              void* stream) {
  int rc;
  if ((rc = check_dtype("act_dtype", act_dtype))) return rc;
  if (B < 0 || T < 0 || Di < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld T=%lld Di=%lld)", (long long)B, (long long)T, (long long)Di);
  if (K < 1 || K > MAMBA_MAX_D_CONV) return fail(MAMBA_ERR_UNSUPPORTED, "d_conv=%lld not in 1..%d", (long long)K, MAMBA_MAX_D_CONV);
  if (B == 0 || Di == 0) return ok();
  if (!sizes_ok(B, T, Di) || !sizes_ok(B, Di, K)) return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!w) return fail(MAMBA_ERR_INVALID_ARG, "w is NULL");
  if (T > 0 && (!u || !x)) return fail(MAMBA_ERR_INVALID_ARG, "u and x must not be NULL");
  if (T > 0 && (ld_u < Di || ld_x < Di)) return fail(MAMBA_ERR_INVALID_ARG, "ld_u=%lld / ld_x=%lld smaller than Di=%lld", (long long)ld_u, (long long)ld_x, (long long)Di);
  const int es = es_of(act_dtype);
  int64_t bu = 0, bx = 0, bst = 0, bw = 0, bb = 0;
  if (!span_bytes(B * T, Di, ld_u, es, &bu) || !span_bytes(B * T, Di, ld_x, es, &bx) ||
      !span_bytes(B * Di, K, K, 4, &bst) || !span_bytes(Di, K, K, 4, &bw) || !span_bytes(1, Di, Di, 4, &bb))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (T == 0) bu = bx = 0;
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  Range ins[] = {range_of("x", x, bx), range_of("w", w, bw), range_of("bias", bias, bb),
                 range_of("conv_state_in", conv_state_in, bst)};
  const bool inplace = conv_state_out && conv_state_out == conv_state_in;
  Range outs[] = {range_of("u", u, bu), range_of("conv_state_out", conv_state_out, bst)};
  if ((rc = check_pointers(ins, 4, dev_id)) || (rc = check_pointers(outs, 2, dev_id))) return rc;
  if ((rc = check_overlaps(outs, 2, ins, inplace ? 3 : 4))) return rc;
  if (inplace && overlaps(outs[0], ins[3])) return fail(MAMBA_ERR_INVALID_ARG, "u overlaps conv_state_in");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) return copy_state(conv_state_out, conv_state_in, B * Di * K, s);
  mamba::ConvPrefillArgs a{u, ld_u, x, ld_x, conv_state_in, conv_state_out, w, bias, B, T, Di, (int)K, act_dtype == MAMBA_BF16};
  cudaError_t e = mamba::launch_conv1d_silu_prefill(a, dev, s);
  if (e != cudaSuccess) return cuda_fail("conv1d_silu_prefill launch", e);
  return ok();
}

int mamba_conv1d_silu_step(void* u, const void* x, int act_dtype, float* conv_state, int64_t layer,
                           int64_t n_layers, const float* w, const float* bias, int64_t B, int64_t Di,
                           int64_t K, void* stream) {
  int rc;
  if ((rc = check_dtype("act_dtype", act_dtype))) return rc;
  if (B < 0 || Di < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld Di=%lld)", (long long)B, (long long)Di);
  if (K < 1 || K > MAMBA_MAX_D_CONV) return fail(MAMBA_ERR_UNSUPPORTED, "d_conv=%lld not in 1..%d", (long long)K, MAMBA_MAX_D_CONV);
  if (n_layers < 1 || layer < 0 || layer >= n_layers) return fail(MAMBA_ERR_INVALID_ARG, "layer=%lld outside [0, n_layers=%lld)", (long long)layer, (long long)n_layers);
  if (B == 0 || Di == 0) return ok();
  if (!sizes_ok(B, Di, K) || !sizes_ok(n_layers, B * Di * K)) return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!u || !x || !conv_state || !w) return fail(MAMBA_ERR_INVALID_ARG, "u, x, conv_state and w must not be NULL");
  const int es = es_of(act_dtype);
  int64_t bact = 0, bst = 0, bw = 0, bb = 0, ball = 0;
  if (!span_bytes(1, B * Di, B * Di, es, &bact) || !span_bytes(B * Di, K, K, 4, &bst) ||
      !span_bytes(n_layers, B * Di * K, B * Di * K, 4, &ball) || !span_bytes(Di, K, K, 4, &bw) ||
      !span_bytes(1, Di, Di, 4, &bb))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  float* slab = conv_state + layer * B * Di * K;
  Range ins[] = {range_of("x", x, bact), range_of("w", w, bw), range_of("bias", bias, bb)};
  Range outs[] = {range_of("u", u, bact), range_of("conv_state", slab, bst)};
  if ((rc = check_pointers(ins, 3, dev_id)) || (rc = check_pointers(outs, 2, dev_id))) return rc;
  if ((rc = check_overlaps(outs, 2, ins, 3))) return rc;
  mamba::ConvStepArgs a{u, x, slab, w, bias, B, Di, (int)K, act_dtype == MAMBA_BF16};
  cudaError_t e = mamba::launch_conv1d_silu_step(a, dev, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("conv1d_silu_step launch", e);
  return ok();
}

int mamba_selective_scan_prefill(void* y, int64_t ld_y, int y_dtype, const void* u, int64_t ld_u,
                                 const void* dt, int64_t ld_dt, const void* z, int64_t ld_z,
                                 const void* Bm, int64_t ld_B, const void* Cm, int64_t ld_C,
                                 int in_dtype, const float* A_log, const float* D,
                                 const float* dt_bias, const float* ssm_state_in,
                                 float* ssm_state_out, int64_t B, int64_t T, int64_t Di, int64_t N,
                                 void* workspace, int64_t workspace_bytes, void* stream) {
  int rc;
  if ((rc = check_dtype("y_dtype", y_dtype)) || (rc = check_dtype("in_dtype", in_dtype))) return rc;
  if (B < 0 || T < 0 || Di < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld T=%lld Di=%lld)", (long long)B, (long long)T, (long long)Di);
  if (!valid_n(N)) return fail(MAMBA_ERR_UNSUPPORTED, "d_state=%lld not in {1,2,4,8,16,32,64}", (long long)N);
  if (workspace_bytes < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative workspace_bytes");
  if (!workspace) workspace_bytes = 0;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15))
    return fail(MAMBA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (B == 0 || Di == 0) return ok();
  if (!sizes_ok(B, T, Di) || !sizes_ok(B, T, N) || !sizes_ok(B, Di, N)) return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!A_log) return fail(MAMBA_ERR_INVALID_ARG, "A_log is NULL");
  if (T > 0) {
    if (!y || !u || !dt || !Bm || !Cm) return fail(MAMBA_ERR_INVALID_ARG, "y, u, dt, Bm and Cm must not be NULL");
    if (ld_y < Di || ld_u < Di || ld_dt < Di || (z && ld_z < Di))
      return fail(MAMBA_ERR_INVALID_ARG, "an activation stride is smaller than Di=%lld", (long long)Di);
    if (ld_B < N || ld_C < N) return fail(MAMBA_ERR_INVALID_ARG, "ld_B / ld_C smaller than d_state=%lld", (long long)N);
  }
  const int es = es_of(in_dtype), esy = es_of(y_dtype);
  int64_t by = 0, bu = 0, bdt = 0, bz = 0, bB = 0, bC = 0, bA = 0, bv = 0, bst = 0;
  if (!span_bytes(B * Di, N, N, 4, &bst) || !span_bytes(Di, N, N, 4, &bA) || !span_bytes(1, Di, Di, 4, &bv))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (T > 0 &&
      (!span_bytes(B * T, Di, ld_y, esy, &by) || !span_bytes(B * T, Di, ld_u, es, &bu) ||
       !span_bytes(B * T, Di, ld_dt, es, &bdt) || (z && !span_bytes(B * T, Di, ld_z, es, &bz)) ||
       !span_bytes(B * T, N, ld_B, es, &bB) || !span_bytes(B * T, N, ld_C, es, &bC)))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  const bool inplace = ssm_state_out && ssm_state_out == ssm_state_in;
  Range ins[] = {range_of("u", u, bu), range_of("dt", dt, bdt), range_of("z", z, bz),
                 range_of("Bm", Bm, bB), range_of("Cm", Cm, bC), range_of("A_log", A_log, bA),
                 range_of("D", D, bv), range_of("dt_bias", dt_bias, bv),
                 range_of("ssm_state_in", ssm_state_in, bst)};
  Range outs[] = {range_of("y", y, by), range_of("ssm_state_out", ssm_state_out, bst),
                  range_of("workspace", workspace, workspace_bytes)};
  if ((rc = check_pointers(ins, 9, dev_id)) || (rc = check_pointers(outs, 3, dev_id))) return rc;
  if ((rc = check_overlaps(outs, 3, ins, inplace ? 8 : 9))) return rc;
  if (inplace && (overlaps(outs[0], ins[8]) || overlaps(outs[2], ins[8])))
    return fail(MAMBA_ERR_INVALID_ARG, "y or workspace overlaps ssm_state_in");
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) return copy_state(ssm_state_out, ssm_state_in, B * Di * N, s);
  mamba::ScanArgs a{y, ld_y, y_dtype == MAMBA_BF16, u, ld_u, dt, ld_dt, z, ld_z, Bm, ld_B, Cm, ld_C,
                    in_dtype == MAMBA_BF16, A_log, D, dt_bias, ssm_state_in, ssm_state_out,
                    B, T, Di, (int)N};
  const mamba::ScanPlan plan = mamba::plan_selective_scan(a, dev, workspace_bytes);
  cudaError_t e = mamba::launch_selective_scan_prefill(a, plan, static_cast<float*>(workspace), dev, s);
  if (e != cudaSuccess) return cuda_fail("selective_scan_prefill launch", e);
  return ok();
}

int mamba_mixer_prefill(void* y, int64_t ld_y, int y_dtype, const void* x, int64_t ld_x, const void* dt,
                        int64_t ld_dt, const void* z, int64_t ld_z, const void* Bm, int64_t ld_B, const void* Cm,
                        int64_t ld_C, int act_dtype, const float* conv_w, const float* conv_b,
                        const float* conv_state_in, float* conv_state_out, const float* A_log, const float* D,
                        const float* dt_bias, const float* ssm_state_in, float* ssm_state_out, int64_t B,
                        int64_t T, int64_t Di, int64_t K, int64_t N, void* workspace, int64_t workspace_bytes,
                        void* stream) {
  int rc;
  if ((rc = check_dtype("y_dtype", y_dtype)) || (rc = check_dtype("act_dtype", act_dtype))) return rc;
  if (B < 0 || T < 0 || Di < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld T=%lld Di=%lld)", (long long)B, (long long)T, (long long)Di);
  if (!valid_n(N)) return fail(MAMBA_ERR_UNSUPPORTED, "d_state=%lld not in {1,2,4,8,16,32,64}", (long long)N);
  if (K < 1 || K > MAMBA_MAX_FUSED_D_CONV)
    return fail(MAMBA_ERR_UNSUPPORTED, "the fused prefill supports d_conv 1..%d (got %lld); call "
                "mamba_conv1d_silu_prefill and mamba_selective_scan_prefill instead", MAMBA_MAX_FUSED_D_CONV,
                (long long)K);
  if (workspace_bytes < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative workspace_bytes");
  if (!workspace) workspace_bytes = 0;
  if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15))
    return fail(MAMBA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (B == 0 || Di == 0) return ok();
  if (!sizes_ok(B, T, Di) || !sizes_ok(B, T, N) || !sizes_ok(B, Di, N) || !sizes_ok(B, Di, K))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!A_log || !conv_w) return fail(MAMBA_ERR_INVALID_ARG, "A_log and conv_w must not be NULL");
  if (T > 0) {
    if (!y || !x || !dt || !Bm || !Cm) return fail(MAMBA_ERR_INVALID_ARG, "y, x, dt, Bm and Cm must not be NULL");
    if (ld_y < Di || ld_x < Di || ld_dt < Di || (z && ld_z < Di))
      return fail(MAMBA_ERR_INVALID_ARG, "an activation stride is smaller than Di=%lld", (long long)Di);
    if (ld_B < N || ld_C < N) return fail(MAMBA_ERR_INVALID_ARG, "ld_B / ld_C smaller than d_state=%lld", (long long)N);
  }
  const int es = es_of(act_dtype), esy = es_of(y_dtype);
  int64_t by = 0, bx = 0, bdt = 0, bz = 0, bB = 0, bC = 0, bA = 0, bv = 0, bst = 0, bcs = 0, bw = 0;
  if (!span_bytes(B * Di, N, N, 4, &bst) || !span_bytes(Di, N, N, 4, &bA) || !span_bytes(1, Di, Di, 4, &bv) ||
      !span_bytes(B * Di, K, K, 4, &bcs) || !span_bytes(Di, K, K, 4, &bw))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (T > 0 &&
      (!span_bytes(B * T, Di, ld_y, esy, &by) || !span_bytes(B * T, Di, ld_x, es, &bx) ||
       !span_bytes(B * T, Di, ld_dt, es, &bdt) || (z && !span_bytes(B * T, Di, ld_z, es, &bz)) ||
       !span_bytes(B * T, N, ld_B, es, &bB) || !span_bytes(B * T, N, ld_C, es, &bC)))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  const bool ssm_inplace = ssm_state_out && ssm_state_out == ssm_state_in;
  const bool conv_inplace = conv_state_out && conv_state_out == conv_state_in;
  const Range sin = range_of("ssm_state_in", ssm_state_in, bst);
  const Range cin = range_of("conv_state_in", conv_state_in, bcs);
  const Range none = range_of("", nullptr, 0);
  Range ins[] = {range_of("x", x, bx), range_of("dt", dt, bdt), range_of("z", z, bz),
                 range_of("Bm", Bm, bB), range_of("Cm", Cm, bC), range_of("A_log", A_log, bA),
                 range_of("D", D, bv), range_of("dt_bias", dt_bias, bv), range_of("conv_w", conv_w, bw),
                 range_of("conv_b", conv_b, bv), sin, cin};
  Range outs[] = {range_of("y", y, by), range_of("ssm_state_out", ssm_state_out, bst),
                  range_of("conv_state_out", conv_state_out, bcs), range_of("workspace", workspace, workspace_bytes)};
  if ((rc = check_pointers(ins, 12, dev_id)) || (rc = check_pointers(outs, 4, dev_id))) return rc;
  // a state may be updated in place; nothing else may touch it
  if (ssm_inplace) ins[10] = none;
  if (conv_inplace) ins[11] = none;
  if ((rc = check_overlaps(outs, 4, ins, 12))) return rc;
  for (int o = 0; o < 4; ++o) {
    if (ssm_inplace && o != 1 && overlaps(outs[o], sin))
      return fail(MAMBA_ERR_INVALID_ARG, "%s overlaps ssm_state_in", outs[o].name);
    if (conv_inplace && o != 2 && overlaps(outs[o], cin))
      return fail(MAMBA_ERR_INVALID_ARG, "%s overlaps conv_state_in", outs[o].name);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {
    if ((rc = copy_state(ssm_state_out, ssm_state_in, B * Di * N, s))) return rc;
    return copy_state(conv_state_out, conv_state_in, B * Di * K, s);
  }
  mamba::ScanArgs a{y, ld_y, y_dtype == MAMBA_BF16, x, ld_x, dt, ld_dt, z, ld_z, Bm, ld_B, Cm, ld_C,
                    act_dtype == MAMBA_BF16, A_log, D, dt_bias, ssm_state_in, ssm_state_out,
                    B, T, Di, (int)N};
  a.K = (int)K;
  a.conv_w = conv_w;
  a.conv_b = conv_b;
  a.conv_state_in = conv_state_in;
  a.conv_state_out = conv_state_out;
  const mamba::ScanPlan plan = mamba::plan_selective_scan(a, dev, workspace_bytes);
  cudaError_t e = mamba::launch_selective_scan_prefill(a, plan, static_cast<float*>(workspace), dev, s);
  if (e != cudaSuccess) return cuda_fail("mixer_prefill launch", e);
  return ok();
}

int mamba3_siso_step_batched(void* y, int y_dtype, const void* x, const void* k, const void* q, int act_dtype,
                             const float* alpha, const float* beta, const float* gamma, const float* D,
                             float* ssm_state, float* k_state, float* v_state, int64_t layer, int64_t n_layers,
                             int64_t B, int64_t H, int64_t P, int64_t N, void* stream) {
  int rc;
  if ((rc = check_dtype("y_dtype", y_dtype)) || (rc = check_dtype("act_dtype", act_dtype))) return rc;
  if (B < 0 || H < 0 || P < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld H=%lld P=%lld)", (long long)B, (long long)H, (long long)P);
  if (N != 16 && N != 32 && N != 64 && N != 128)
    return fail(MAMBA_ERR_UNSUPPORTED, "d_state=%lld not in {16,32,64,128}", (long long)N);
  if (P * (N / 8) > mamba::m3_max_items())
    return fail(MAMBA_ERR_UNSUPPORTED, "headdim * d_state / 8 = %lld exceeds %d", (long long)(P * (N / 8)),
                mamba::m3_max_items());
  if (n_layers < 1 || layer < 0 || layer >= n_layers) return fail(MAMBA_ERR_INVALID_ARG, "layer=%lld outside [0, n_layers=%lld)", (long long)layer, (long long)n_layers);
  if (B == 0 || H == 0 || P == 0) return ok();
  if (!sizes_ok(B, H, P * N) || !sizes_ok(n_layers, B * H, P * N)) return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!y || !x || !k || !q || !alpha || !beta || !gamma || !ssm_state || !k_state || !v_state)
    return fail(MAMBA_ERR_INVALID_ARG, "y, x, k, q, alpha, beta, gamma and the three states must not be NULL");
  if (reinterpret_cast<uintptr_t>(ssm_state) & 15) return fail(MAMBA_ERR_INVALID_ARG, "ssm_state must be 16-byte aligned");
  const int es = es_of(act_dtype), esy = es_of(y_dtype);
  const int64_t BH = B * H;
  int64_t by = 0, bx = 0, bk = 0, bs = 0, bh = 0, bss = 0, bks = 0, bvs = 0;
  if (!span_bytes(1, BH * P, BH * P, esy, &by) || !span_bytes(1, BH * P, BH * P, es, &bx) ||
      !span_bytes(1, BH * N, BH * N, es, &bk) || !span_bytes(1, BH, BH, 4, &bs) || !span_bytes(1, H, H, 4, &bh) ||
      !span_bytes(BH * P, N, N, 4, &bss) || !span_bytes(1, BH * N, BH * N, 4, &bks) ||
      !span_bytes(1, BH * P, BH * P, 4, &bvs))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  float* sslab = ssm_state + layer * BH * P * N;
  float* kslab = k_state + layer * BH * N;
  float* vslab = v_state + layer * BH * P;
  Range ins[] = {range_of("x", x, bx), range_of("k", k, bk), range_of("q", q, bk), range_of("alpha", alpha, bs),
                 range_of("beta", beta, bs), range_of("gamma", gamma, bs), range_of("D", D, bh)};
  Range outs[] = {range_of("y", y, by), range_of("ssm_state", sslab, bss), range_of("k_state", kslab, bks),
                  range_of("v_state", vslab, bvs)};
  if ((rc = check_pointers(ins, 7, dev_id)) || (rc = check_pointers(outs, 4, dev_id))) return rc;
  if ((rc = check_overlaps(outs, 4, ins, 7))) return rc;
  mamba::M3StepArgs a{y, y_dtype == MAMBA_BF16, x, k, q, act_dtype == MAMBA_BF16, alpha, beta, gamma, D,
                      sslab, kslab, vslab, B, H, (int)P, (int)N};
  cudaError_t e = mamba::launch_m3_step_batched(a, dev, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("mamba3_siso_step_batched launch", e);
  return ok();
}

int mamba3_siso_step_prepare(void* k, void* q, int kq_dtype, float* alpha, float* beta, float* gamma,
                             const float* k_in, const float* q_in, const float* dt, const float* A, const float* lam,
                             const float* angles, float* angle_state, int64_t layer, int64_t n_layers, int64_t B,
                             int64_t H, int64_t N, int64_t n_angles, void* stream) {
  int rc;
  if ((rc = check_dtype("kq_dtype", kq_dtype))) return rc;
  if (B < 0 || H < 0 || N < 0 || n_angles < 0)
    return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld H=%lld N=%lld n_angles=%lld)", (long long)B,
                (long long)H, (long long)N, (long long)n_angles);
  if (N % 2 || N > INT32_MAX) return fail(MAMBA_ERR_UNSUPPORTED, "d_state=%lld must be even", (long long)N);
  if (2 * n_angles > N)
    return fail(MAMBA_ERR_INVALID_ARG, "n_angles=%lld rotates more than the d_state=%lld components",
                (long long)n_angles, (long long)N);
  // layer selects the slab of the angle state, the only per-layer buffer here
  if (n_angles > 0 && (n_layers < 1 || layer < 0 || layer >= n_layers))
    return fail(MAMBA_ERR_INVALID_ARG, "layer=%lld outside [0, n_layers=%lld)", (long long)layer, (long long)n_layers);
  if (B == 0 || H == 0 || N == 0) return ok();
  if (!sizes_ok(B, H, N) || (n_angles > 0 && !sizes_ok(n_layers, B * H, n_angles)))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!k || !q || !alpha || !beta || !gamma || !k_in || !q_in || !dt || !A || !lam)
    return fail(MAMBA_ERR_INVALID_ARG, "k, q, alpha, beta, gamma, k_in, q_in, dt, A and lam must not be NULL");
  if (n_angles > 0 && (!angles || !angle_state))
    return fail(MAMBA_ERR_INVALID_ARG, "angles and angle_state must not be NULL when n_angles > 0");
  const int64_t BH = B * H;
  int64_t bkq = 0, bkin = 0, bs = 0, ban = 0, bth = 0;
  if (!span_bytes(1, BH * N, BH * N, es_of(kq_dtype), &bkq) || !span_bytes(1, BH * N, BH * N, 4, &bkin) ||
      !span_bytes(1, BH, BH, 4, &bs) || !span_bytes(1, B * n_angles, B * n_angles, 4, &ban) ||
      !span_bytes(1, BH * n_angles, BH * n_angles, 4, &bth))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  float* th = n_angles > 0 ? angle_state + layer * BH * n_angles : nullptr;
  const float* an = n_angles > 0 ? angles : nullptr;
  Range ins[] = {range_of("k_in", k_in, bkin), range_of("q_in", q_in, bkin), range_of("dt", dt, bs),
                 range_of("A", A, bs), range_of("lam", lam, bs), range_of("angles", an, ban)};
  Range outs[] = {range_of("k", k, bkq), range_of("q", q, bkq), range_of("alpha", alpha, bs),
                  range_of("beta", beta, bs), range_of("gamma", gamma, bs), range_of("angle_state", th, bth)};
  if ((rc = check_pointers(ins, 6, dev_id)) || (rc = check_pointers(outs, 6, dev_id))) return rc;
  if ((rc = check_overlaps(outs, 6, ins, 6))) return rc;
  mamba::M3PrepArgs a{k, q, kq_dtype == MAMBA_BF16, alpha, beta, gamma, k_in, q_in, dt, A, lam, an, th, B, H,
                      (int)N, (int)n_angles};
  cudaError_t e = mamba::launch_m3_prepare(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("mamba3_siso_step_prepare launch", e);
  return ok();
}

int mamba3_siso_step_fused_batched(void* y, int y_dtype, const void* x, int x_dtype, const float* k_in,
                                   const float* q_in, const float* dt, const float* A, const float* lam,
                                   const float* angles, const float* D, float* ssm_state, float* k_state,
                                   float* v_state, float* angle_state, int64_t layer, int64_t n_layers, int64_t B,
                                   int64_t H, int64_t P, int64_t N, int64_t n_angles, void* stream) {
  int rc;
  if ((rc = check_dtype("y_dtype", y_dtype)) || (rc = check_dtype("x_dtype", x_dtype))) return rc;
  if (B < 0 || H < 0 || P < 0 || n_angles < 0)
    return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld H=%lld P=%lld n_angles=%lld)", (long long)B,
                (long long)H, (long long)P, (long long)n_angles);
  if (N != 16 && N != 32 && N != 64 && N != 128)
    return fail(MAMBA_ERR_UNSUPPORTED, "d_state=%lld not in {16,32,64,128}", (long long)N);
  if (2 * n_angles > N)
    return fail(MAMBA_ERR_INVALID_ARG, "n_angles=%lld rotates more than the d_state=%lld components",
                (long long)n_angles, (long long)N);
  if (P * (N / 8) > mamba::m3_max_items())
    return fail(MAMBA_ERR_UNSUPPORTED, "headdim * d_state / 8 = %lld exceeds %d", (long long)(P * (N / 8)),
                mamba::m3_max_items());
  if (n_layers < 1 || layer < 0 || layer >= n_layers)
    return fail(MAMBA_ERR_INVALID_ARG, "layer=%lld outside [0, n_layers=%lld)", (long long)layer, (long long)n_layers);
  if (B == 0 || H == 0 || P == 0) return ok();
  if (!sizes_ok(B, H, P * N) || !sizes_ok(n_layers, B * H, P * N) ||
      (n_angles > 0 && !sizes_ok(n_layers, B * H, n_angles)))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!y || !x || !k_in || !q_in || !dt || !A || !lam || !ssm_state || !k_state || !v_state)
    return fail(MAMBA_ERR_INVALID_ARG, "y, x, k_in, q_in, dt, A, lam and the three step states must not be NULL");
  if (n_angles > 0 && (!angles || !angle_state))
    return fail(MAMBA_ERR_INVALID_ARG, "angles and angle_state must not be NULL when n_angles > 0");
  if (reinterpret_cast<uintptr_t>(ssm_state) & 15) return fail(MAMBA_ERR_INVALID_ARG, "ssm_state must be 16-byte aligned");
  const int es = es_of(x_dtype), esy = es_of(y_dtype);
  const int64_t BH = B * H;
  int64_t by = 0, bx = 0, bk = 0, bs = 0, bh = 0, bss = 0, bks = 0, bvs = 0, ban = 0, bth = 0;
  if (!span_bytes(1, BH * P, BH * P, esy, &by) || !span_bytes(1, BH * P, BH * P, es, &bx) ||
      !span_bytes(1, BH * N, BH * N, 4, &bk) || !span_bytes(1, BH, BH, 4, &bs) || !span_bytes(1, H, H, 4, &bh) ||
      !span_bytes(BH * P, N, N, 4, &bss) || !span_bytes(1, BH * N, BH * N, 4, &bks) ||
      !span_bytes(1, BH * P, BH * P, 4, &bvs) || !span_bytes(1, B * n_angles, B * n_angles, 4, &ban) ||
      !span_bytes(1, BH * n_angles, BH * n_angles, 4, &bth))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  float* sslab = ssm_state + layer * BH * P * N;
  float* kslab = k_state + layer * BH * N;
  float* vslab = v_state + layer * BH * P;
  float* th = n_angles > 0 ? angle_state + layer * BH * n_angles : nullptr;
  const float* an = n_angles > 0 ? angles : nullptr;
  Range ins[] = {range_of("x", x, bx),        range_of("k_in", k_in, bk), range_of("q_in", q_in, bk),
                 range_of("dt", dt, bs),      range_of("A", A, bs),       range_of("lam", lam, bs),
                 range_of("angles", an, ban), range_of("D", D, bh)};
  Range outs[] = {range_of("y", y, by), range_of("ssm_state", sslab, bss), range_of("k_state", kslab, bks),
                  range_of("v_state", vslab, bvs), range_of("angle_state", th, bth)};
  if ((rc = check_pointers(ins, 8, dev_id)) || (rc = check_pointers(outs, 5, dev_id))) return rc;
  if ((rc = check_overlaps(outs, 5, ins, 8))) return rc;
  mamba::M3StepArgs a{y, y_dtype == MAMBA_BF16, x, nullptr, nullptr, x_dtype == MAMBA_BF16, nullptr, nullptr, nullptr,
                      D, sslab, kslab, vslab, B, H, (int)P, (int)N, k_in, q_in, dt, A, lam, an, th,
                      (int)n_angles};
  cudaError_t e = mamba::launch_m3_step_batched(a, dev, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("mamba3_siso_step_fused_batched launch", e);
  return ok();
}

int mamba_linear_bf16(void* c, int64_t ld_c, int c_dtype, const void* a, int64_t ld_a, const void* w, int64_t ld_w,
                      const float* residual, int64_t ld_r, int64_t M, int64_t N, int64_t K, void* stream) {
  int rc;
  if ((rc = check_dtype("c_dtype", c_dtype))) return rc;
  if (M < 0 || N < 0 || K < 1) return fail(MAMBA_ERR_INVALID_ARG, "sizes must be M >= 0, N >= 0, K >= 1 (M=%lld N=%lld K=%lld)", (long long)M, (long long)N, (long long)K);
  if (M == 0 || N == 0) return ok();
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX || !sizes_ok(M, K) || !sizes_ok(N, K) || !sizes_ok(M, N) ||
      ((M + 127) / 128) * ((N + 63) / 64) > INT32_MAX)  // output tiles are counted in 32 bits
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!c || !a || !w) return fail(MAMBA_ERR_INVALID_ARG, "c, a and w must not be NULL");
  if (ld_c < N || (residual && ld_r < N) || ld_a < K || ld_w < K)
    return fail(MAMBA_ERR_INVALID_ARG, "a row stride is smaller than its row");
  // the tensor-memory copies read whole 16-byte granules of A and W rows
  if ((reinterpret_cast<uintptr_t>(a) & 15) || (reinterpret_cast<uintptr_t>(w) & 15) || (ld_a * 2) % 16 ||
      (ld_w * 2) % 16)
    return fail(MAMBA_ERR_INVALID_ARG, "a and w must be 16-byte aligned with row strides of a multiple of 8 elements");
  const int esc = es_of(c_dtype);
  int64_t bc = 0, ba = 0, bw = 0, br = 0;
  if (!span_bytes(M, N, ld_c, esc, &bc) || !span_bytes(M, K, ld_a, 2, &ba) || !span_bytes(N, K, ld_w, 2, &bw) ||
      (residual && !span_bytes(M, N, ld_r, 4, &br)))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  Range ins[] = {range_of("a", a, ba), range_of("w", w, bw), range_of("residual", residual, br)};
  Range outs[] = {range_of("c", c, bc)};
  if ((rc = check_pointers(ins, 3, dev_id)) || (rc = check_pointers(outs, 1, dev_id))) return rc;
  // the residual may be the output itself (x += out_proj(y)); nothing else may overlap c
  const bool inplace_r = residual && reinterpret_cast<const void*>(residual) == c && ld_r == ld_c && c_dtype == MAMBA_F32;
  if ((rc = check_overlaps(outs, 1, ins, inplace_r ? 2 : 3))) return rc;
  mamba::GemmArgs g{c, ld_c, c_dtype == MAMBA_BF16, a, ld_a, w, ld_w, residual, ld_r, M, N, K};
  cudaError_t e = mamba::launch_gemm_bf16(g, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("linear_bf16 launch", e);
  return ok();
}

int mamba_rmsnorm(void* out, int64_t ld_out, int out_dtype, const float* x, int64_t ld_x, const float* weight,
                  float eps, int64_t M, int64_t D, void* stream) {
  int rc;
  if ((rc = check_dtype("out_dtype", out_dtype))) return rc;
  if (M < 0 || D < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (M=%lld D=%lld)", (long long)M, (long long)D);
  if (!(eps >= 0.0f) || eps > 1.0f) return fail(MAMBA_ERR_INVALID_ARG, "eps must be in [0, 1]");
  if (M == 0 || D == 0) return ok();
  if (D > INT32_MAX || !sizes_ok(M, D)) return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!out || !x || !weight) return fail(MAMBA_ERR_INVALID_ARG, "out, x and weight must not be NULL");
  if (ld_out < D || ld_x < D) return fail(MAMBA_ERR_INVALID_ARG, "a row stride is smaller than D=%lld", (long long)D);
  int64_t bo = 0, bx = 0, bw = 0;
  if (!span_bytes(M, D, ld_out, es_of(out_dtype), &bo) || !span_bytes(M, D, ld_x, 4, &bx) ||
      !span_bytes(1, D, D, 4, &bw))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  Range ins[] = {range_of("x", x, bx), range_of("weight", weight, bw)};
  Range outs[] = {range_of("out", out, bo)};
  if ((rc = check_pointers(ins, 2, dev_id)) || (rc = check_pointers(outs, 1, dev_id))) return rc;
  if ((rc = check_overlaps(outs, 1, ins, 2))) return rc;
  mamba::RmsNormArgs a{out, ld_out, out_dtype == MAMBA_BF16, x, ld_x, weight, eps, M, D};
  cudaError_t e = mamba::launch_rmsnorm(a, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("rmsnorm launch", e);
  return ok();
}

int64_t mamba_selective_scan_workspace_bytes(int64_t B, int64_t T, int64_t Di, int64_t N) {
  if (B < 0 || T < 0 || Di < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size");
  if (!valid_n(N)) return fail(MAMBA_ERR_UNSUPPORTED, "d_state=%lld not in {1,2,4,8,16,32,64}", (long long)N);
  if (!sizes_ok(B, T, Di) || !sizes_ok(B, Di, N)) return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (B == 0 || Di == 0 || T == 0) {
    ok();
    return 0;
  }
  mamba::ScanShapePlan p;
  const int rc = mamba::plan_scan_for_current_device(B, T, Di, N, INT64_MAX, &p);
  if (rc) return rc;
  ok();
  return p.workspace_bytes;
}

int mamba_ssm_step_batched(void* y, int y_dtype, const void* u, const void* dt, const void* z,
                           const void* Bm, const void* Cm, int in_dtype, const float* A_log,
                           const float* D, const float* dt_bias, float* ssm_state, int64_t layer,
                           int64_t n_layers, int64_t B, int64_t Di, int64_t N, void* stream) {
  int rc;
  if ((rc = check_dtype("y_dtype", y_dtype)) || (rc = check_dtype("in_dtype", in_dtype))) return rc;
  if (B < 0 || Di < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld Di=%lld)", (long long)B, (long long)Di);
  if (!valid_n(N)) return fail(MAMBA_ERR_UNSUPPORTED, "d_state=%lld not in {1,2,4,8,16,32,64}", (long long)N);
  if (n_layers < 1 || layer < 0 || layer >= n_layers) return fail(MAMBA_ERR_INVALID_ARG, "layer=%lld outside [0, n_layers=%lld)", (long long)layer, (long long)n_layers);
  if (B == 0 || Di == 0) return ok();
  if (!sizes_ok(B, Di, N) || !sizes_ok(n_layers, B * Di * N)) return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!y || !u || !dt || !Bm || !Cm || !A_log || !ssm_state)
    return fail(MAMBA_ERR_INVALID_ARG, "y, u, dt, Bm, Cm, A_log and ssm_state must not be NULL");
  const int es = es_of(in_dtype), esy = es_of(y_dtype);
  int64_t by = 0, bact = 0, bbc = 0, bA = 0, bv = 0, bst = 0, ball = 0;
  if (!span_bytes(1, B * Di, B * Di, esy, &by) || !span_bytes(1, B * Di, B * Di, es, &bact) ||
      !span_bytes(1, B * N, B * N, es, &bbc) || !span_bytes(Di, N, N, 4, &bA) ||
      !span_bytes(1, Di, Di, 4, &bv) || !span_bytes(B * Di, N, N, 4, &bst) ||
      !span_bytes(n_layers, B * Di * N, B * Di * N, 4, &ball))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  float* slab = ssm_state + layer * B * Di * N;
  Range ins[] = {range_of("u", u, bact), range_of("dt", dt, bact), range_of("z", z, z ? bact : 0),
                 range_of("Bm", Bm, bbc), range_of("Cm", Cm, bbc), range_of("A_log", A_log, bA),
                 range_of("D", D, bv), range_of("dt_bias", dt_bias, bv)};
  Range outs[] = {range_of("y", y, by), range_of("ssm_state", slab, bst)};
  if ((rc = check_pointers(ins, 8, dev_id)) || (rc = check_pointers(outs, 2, dev_id))) return rc;
  if ((rc = check_overlaps(outs, 2, ins, 8))) return rc;
  mamba::SsmStepArgs a{y, y_dtype == MAMBA_BF16, u, dt, z, Bm, Cm, in_dtype == MAMBA_BF16,
                       A_log, D, dt_bias, slab, B, Di, (int)N};
  cudaError_t e = mamba::launch_ssm_step_batched(a, dev, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("ssm_step_batched launch", e);
  return ok();
}

int mamba_mixer_step_batched(void* y, int y_dtype, const void* x, const void* dt, const void* z,
                             const void* Bm, const void* Cm, int act_dtype, const float* conv_w,
                             const float* conv_b, const float* A_log, const float* D,
                             const float* dt_bias, float* conv_state, float* ssm_state, int64_t layer,
                             int64_t n_layers, int64_t B, int64_t Di, int64_t K, int64_t N,
                             void* stream) {
  int rc;
  if ((rc = check_dtype("y_dtype", y_dtype)) || (rc = check_dtype("act_dtype", act_dtype))) return rc;
  if (B < 0 || Di < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative size (B=%lld Di=%lld)", (long long)B, (long long)Di);
  if (!valid_n(N)) return fail(MAMBA_ERR_UNSUPPORTED, "d_state=%lld not in {1,2,4,8,16,32,64}", (long long)N);
  if (K < 1 || K > MAMBA_MAX_D_CONV) return fail(MAMBA_ERR_UNSUPPORTED, "d_conv=%lld not in 1..%d", (long long)K, MAMBA_MAX_D_CONV);
  if (n_layers < 1 || layer < 0 || layer >= n_layers) return fail(MAMBA_ERR_INVALID_ARG, "layer=%lld outside [0, n_layers=%lld)", (long long)layer, (long long)n_layers);
  if (B == 0 || Di == 0) return ok();
  if (!sizes_ok(B, Di, N) || !sizes_ok(B, Di, K) || !sizes_ok(n_layers, B * Di * N) || !sizes_ok(n_layers, B * Di * K))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  if (!y || !x || !dt || !Bm || !Cm || !A_log || !conv_w || !conv_state || !ssm_state)
    return fail(MAMBA_ERR_INVALID_ARG, "y, x, dt, Bm, Cm, A_log, conv_w, conv_state and ssm_state must not be NULL");
  const int es = es_of(act_dtype), esy = es_of(y_dtype);
  int64_t by = 0, bact = 0, bbc = 0, bA = 0, bv = 0, bss = 0, bcs = 0, bw = 0;
  if (!span_bytes(1, B * Di, B * Di, esy, &by) || !span_bytes(1, B * Di, B * Di, es, &bact) ||
      !span_bytes(1, B * N, B * N, es, &bbc) || !span_bytes(Di, N, N, 4, &bA) ||
      !span_bytes(1, Di, Di, 4, &bv) || !span_bytes(B * Di, N, N, 4, &bss) ||
      !span_bytes(B * Di, K, K, 4, &bcs) || !span_bytes(Di, K, K, 4, &bw))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow");
  mamba::DeviceInfo dev;
  if ((rc = current_device(&dev))) return rc;
  int dev_id = 0;
  cudaGetDevice(&dev_id);
  float* sslab = ssm_state + layer * B * Di * N;
  float* cslab = conv_state + layer * B * Di * K;
  Range ins[] = {range_of("x", x, bact), range_of("dt", dt, bact), range_of("z", z, z ? bact : 0),
                 range_of("Bm", Bm, bbc), range_of("Cm", Cm, bbc), range_of("A_log", A_log, bA),
                 range_of("D", D, bv), range_of("dt_bias", dt_bias, bv), range_of("conv_w", conv_w, bw),
                 range_of("conv_b", conv_b, bv)};
  Range outs[] = {range_of("y", y, by), range_of("ssm_state", sslab, bss),
                  range_of("conv_state", cslab, bcs)};
  if ((rc = check_pointers(ins, 10, dev_id)) || (rc = check_pointers(outs, 3, dev_id))) return rc;
  if ((rc = check_overlaps(outs, 3, ins, 10))) return rc;
  mamba::MixerStepArgs a{{y, y_dtype == MAMBA_BF16, nullptr, dt, z, Bm, Cm, act_dtype == MAMBA_BF16, A_log,
                          D, dt_bias, sslab, B, Di, (int)N},
                         x, cslab, conv_w, conv_b, (int)K};
  cudaError_t e = mamba::launch_mixer_step_batched(a, dev, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail("mixer_step_batched launch", e);
  return ok();
}

int64_t mamba_layer_workspace_bytes(const MambaLayer* layer, int64_t B, int64_t T) {
  LayerPlan p;
  int rc;
  if ((rc = layer_plan(layer, B, T, &p))) return rc;
  if (B == 0 || T == 0) return ok(), 0;
  mamba::ScanShapePlan sp;
  if ((rc = mamba::plan_scan_for_current_device(B, T, layer->d_inner, layer->d_state, INT64_MAX, &sp))) return rc;
  ok();
  return p.act_bytes + sp.workspace_bytes;
}

int mamba_layer_prefill(float* hidden, const MambaLayer* layer, const float* conv_state_in, float* conv_state_out,
                        const float* ssm_state_in, float* ssm_state_out, int64_t B, int64_t T, void* workspace,
                        int64_t workspace_bytes, void* stream) {
  if (workspace_bytes < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative workspace_bytes");
  return run_layer(hidden, layer, conv_state_in, conv_state_out, ssm_state_in, ssm_state_out, B, T, workspace,
                   workspace_bytes, false, stream);
}

int mamba_layer_step(float* hidden, const MambaLayer* layer, float* conv_state, float* ssm_state,
                     int64_t layer_index, int64_t n_layers, int64_t B, void* workspace, int64_t workspace_bytes,
                     void* stream) {
  if (workspace_bytes < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative workspace_bytes");
  if (!layer) return fail(MAMBA_ERR_INVALID_ARG, "layer is NULL");
  if (n_layers < 1 || layer_index < 0 || layer_index >= n_layers)
    return fail(MAMBA_ERR_INVALID_ARG, "layer_index=%lld outside [0, n_layers=%lld)", (long long)layer_index,
                (long long)n_layers);
  if (B < 0) return fail(MAMBA_ERR_INVALID_ARG, "negative B");
  if (B == 0) return ok();
  if (!conv_state || !ssm_state) return fail(MAMBA_ERR_INVALID_ARG, "conv_state and ssm_state must not be NULL");
  const int64_t Di = layer->d_inner, N = layer->d_state, K = layer->d_conv;
  if (Di < 1 || N < 1 || K < 1 || !sizes_ok(B, Di, N > K ? N : K) || !sizes_ok(n_layers, B * Di * (N > K ? N : K)))
    return fail(MAMBA_ERR_INVALID_ARG, "extent overflow or invalid dims");
  float* cslab = conv_state + layer_index * B * Di * K;
  float* sslab = ssm_state + layer_index * B * Di * N;
  return run_layer(hidden, layer, cslab, cslab, sslab, sslab, B, 1, workspace, workspace_bytes, true, stream);
}

}  // extern "C"
