"""ctypes binding of libmamba_ssm.so (the C ABI in include/mamba_ssm.h).

Argument marshalling only: shapes and strides are read off torch tensors and
passed as plain pointers and sizes; every step of the computation runs in the
library's CUDA kernels on the caller's current torch stream.  There is no CPU
or PyTorch fallback: if the library is missing or the device is not a GB300,
the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

MAMBA_OK = 0
MAMBA_ERR_INVALID_ARG = -1
MAMBA_ERR_UNSUPPORTED = -2
MAMBA_ERR_CUDA = -3
MAMBA_F32 = 0
MAMBA_BF16 = 1
MAMBA_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024
MAMBA_MAX_FUSED_D_CONV = 4
MAMBA_FAULT_SCAN_WAIT = 2
MAMBA_FAULT_GEMM_WAIT = 4

LIB_PATH = _build.LIB_PATH

# every exported entry point of include/mamba_ssm.h
ABI_SYMBOLS = (
    "mamba_conv1d_silu_prefill",
    "mamba_conv1d_silu_step",
    "mamba_selective_scan_prefill",
    "mamba_selective_scan_workspace_bytes",
    "mamba_selective_scan_prefill_noalloc",
    "mamba_ssm_step_batched",
    "mamba_mixer_step_batched",
    "mamba_mixer_prefill",
    "mamba3_siso_step_batched",
    "mamba3_siso_step_prepare",
    "mamba3_siso_step_fused_batched",
    "mamba3_decode_graph_create",
    "mamba_linear_bf16",
    "mamba_rmsnorm",
    "mamba_layer_workspace_bytes",
    "mamba_layer_prefill",
    "mamba_layer_step",
    "mamba_layer_decode_graph_create",
    "mamba_decode_graph_create",
    "mamba_decode_graph_launch",
    "mamba_decode_graph_kernels",
    "mamba_decode_graph_destroy",
    "mamba_device_faults",
    "mamba_selftest_bounded_wait",
    "mamba_last_error",
    "mamba_version",
)

_lock = threading.Lock()
_lib = None


class MambaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"[{status}] {message}")
        self.status = status


class _MambaLayer(ctypes.Structure):
    """struct MambaLayer of the C ABI (dims, RMSNorm eps, weight pointers)."""
    _fields_ = [("d_model", ctypes.c_int64), ("d_inner", ctypes.c_int64), ("d_state", ctypes.c_int64),
                ("d_conv", ctypes.c_int64), ("dt_rank", ctypes.c_int64), ("eps", ctypes.c_float),
                ("norm_w", ctypes.c_void_p), ("in_proj_w", ctypes.c_void_p), ("conv_w", ctypes.c_void_p),
                ("conv_b", ctypes.c_void_p), ("x_proj_w", ctypes.c_void_p), ("dt_proj_w", ctypes.c_void_p),
                ("dt_proj_b", ctypes.c_void_p), ("A_log", ctypes.c_void_p), ("D", ctypes.c_void_p),
                ("out_proj_w", ctypes.c_void_p)]


def load(path: str | None = None):
    """Load libmamba_ssm.so (built in-tree by build.py) and declare its ABI."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build the CUDA library first "
                "(python -m selective_state_space_conv1d_gb300.build, or __graft_entry__.build())")
        lib = ctypes.CDLL(p)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        lib.mamba_conv1d_silu_prefill.argtypes = [vp, i64, vp, i64, i32, vp, vp, vp, vp, i64, i64, i64, i64, vp]
        lib.mamba_conv1d_silu_step.argtypes = [vp, vp, i32, vp, i64, i64, vp, vp, i64, i64, i64, vp]
        lib.mamba_selective_scan_prefill.argtypes = (
            [vp, i64, i32, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32]
            + [vp] * 5 + [i64, i64, i64, i64, vp, i64, vp])
        lib.mamba_selective_scan_prefill_noalloc.argtypes = (
            [vp, i64, i32, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32]
            + [vp] * 5 + [i64, i64, i64, i64, vp])
        lib.mamba_selective_scan_prefill_noalloc.restype = ctypes.c_int
        lib.mamba_selective_scan_workspace_bytes.argtypes = [i64, i64, i64, i64]
        lib.mamba_selective_scan_workspace_bytes.restype = i64
        lib.mamba_ssm_step_batched.argtypes = [vp, i32, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp]
        lib.mamba_mixer_step_batched.argtypes = ([vp, i32, vp, vp, vp, vp, vp, i32] + [vp] * 7
                                                 + [i64, i64, i64, i64, i64, i64, vp])
        for f in ("mamba_mixer_step_batched", "mamba_conv1d_silu_prefill", "mamba_conv1d_silu_step",
                  "mamba_selective_scan_prefill", "mamba_ssm_step_batched"):
            getattr(lib, f).restype = ctypes.c_int
        lib.mamba_mixer_prefill.argtypes = ([vp, i64, i32, vp, i64, vp, i64, vp, i64, vp, i64, vp, i64, i32]
                                            + [vp] * 9 + [i64, i64, i64, i64, i64, vp, i64, vp])
        lib.mamba_mixer_prefill.restype = ctypes.c_int
        lib.mamba3_siso_step_batched.argtypes = [vp, i32, vp, vp, vp, i32] + [vp] * 7 + [i64] * 6 + [vp]
        lib.mamba3_siso_step_batched.restype = ctypes.c_int
        lib.mamba3_siso_step_prepare.argtypes = [vp, vp, i32] + [vp] * 10 + [i64] * 6 + [vp]
        lib.mamba3_siso_step_prepare.restype = ctypes.c_int
        lib.mamba3_siso_step_fused_batched.argtypes = [vp, i32, vp, i32] + [vp] * 11 + [i64] * 7 + [vp]
        lib.mamba3_siso_step_fused_batched.restype = ctypes.c_int
        lib.mamba_linear_bf16.argtypes = [vp, i64, i32, vp, i64, vp, i64, vp, i64, i64, i64, i64, vp]
        lib.mamba_linear_bf16.restype = ctypes.c_int
        lib.mamba_rmsnorm.argtypes = [vp, i64, i32, vp, i64, vp, ctypes.c_float, i64, i64, vp]
        lib.mamba_rmsnorm.restype = ctypes.c_int
        lp = ctypes.POINTER(_MambaLayer)
        lib.mamba_layer_workspace_bytes.argtypes = [lp, i64, i64]
        lib.mamba_layer_workspace_bytes.restype = i64
        lib.mamba_layer_prefill.argtypes = [vp, lp, vp, vp, vp, vp, i64, i64, vp, i64, vp]
        lib.mamba_layer_prefill.restype = ctypes.c_int
        lib.mamba_layer_step.argtypes = [vp, lp, vp, vp, i64, i64, i64, vp, i64, vp]
        lib.mamba_layer_step.restype = ctypes.c_int
        lib.mamba_layer_decode_graph_create.argtypes = [ctypes.POINTER(vp), lp, i64, vp, vp, vp, i64, vp, i64]
        lib.mamba_layer_decode_graph_create.restype = ctypes.c_int
        lib.mamba_decode_graph_create.argtypes = [ctypes.POINTER(vp), vp, vp, i64, i64, i32, i32, vp, vp,
                                                  i64, i64, i64, i64]
        lib.mamba_decode_graph_create.restype = ctypes.c_int
        lib.mamba3_decode_graph_create.argtypes = [ctypes.POINTER(vp), vp, vp, i64, i64, i32, i32, vp, vp, vp, vp,
                                                   i64, i64, i64, i64, i64]
        lib.mamba3_decode_graph_create.restype = ctypes.c_int
        lib.mamba_decode_graph_launch.argtypes = [vp, vp]
        lib.mamba_decode_graph_launch.restype = ctypes.c_int
        lib.mamba_decode_graph_kernels.argtypes = [vp]
        lib.mamba_decode_graph_kernels.restype = i64
        lib.mamba_decode_graph_destroy.argtypes = [vp]
        lib.mamba_decode_graph_destroy.restype = ctypes.c_int
        lib.mamba_device_faults.argtypes = [i32]
        lib.mamba_device_faults.restype = ctypes.c_int
        lib.mamba_selftest_bounded_wait.argtypes = [i64, i32, vp]
        lib.mamba_selftest_bounded_wait.restype = ctypes.c_int
        lib.mamba_last_error.argtypes = []
        lib.mamba_last_error.restype = ctypes.c_char_p
        lib.mamba_version.argtypes = []
        lib.mamba_version.restype = ctypes.c_char_p
        _lib = lib
        return lib


def mamba_last_error() -> str:
    return load().mamba_last_error().decode()


def mamba_version() -> str:
    return load().mamba_version().decode()


MAMBA_FAULT_RING_WAIT = 1


def mamba_device_faults(clear: bool = False) -> int:
    """Watchdog bits of the current device (MAMBA_FAULT_RING_WAIT: a bounded
    wait of the decode-step copy ring ran out); synchronises the device."""
    v = load().mamba_device_faults(1 if clear else 0)
    if v < 0:
        raise MambaError(int(v), mamba_last_error())
    return int(v)


def mamba_selftest_bounded_wait(limit_cycles: int, complete: bool, stream=None):
    """One CTA waits, with the decode rings' bounded wait, on an mbarrier that is
    completed first (complete=True) or never (False: the wait runs out after
    limit_cycles and sets MAMBA_FAULT_RING_WAIT).  Enqueued on `stream` (default:
    the current stream)."""
    import torch

    st = torch.cuda.current_stream().cuda_stream if stream is None else (
        stream if isinstance(stream, int) else stream.cuda_stream)
    _check(load().mamba_selftest_bounded_wait(int(limit_cycles), 1 if complete else 0, st))


def _check(status: int):
    if status != MAMBA_OK:
        raise MambaError(status, mamba_last_error())


# ------------------------------------------------------------------ helpers --

def _dtype_code(t):
    import torch

    if t.dtype == torch.float32:
        return MAMBA_F32
    if t.dtype == torch.bfloat16:
        return MAMBA_BF16
    raise TypeError(f"unsupported storage dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream, like):
    import torch

    if stream is None:
        return torch.cuda.current_stream(like.device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _rows_ld(t, name):
    """Row stride `ld` of a [B, T, C] tensor laid out as (b*T + t)*ld + c."""
    if t.dim() != 3:
        raise ValueError(f"{name} must be 3-D [batch, T, channels], got {tuple(t.shape)}")
    Bsz, T, C = t.shape
    if C > 1 and t.stride(2) != 1:
        raise ValueError(f"{name}: channels must be contiguous (stride {t.stride(2)})")
    if T > 1:
        ld = t.stride(1)
        if Bsz > 1 and t.stride(0) != T * ld:
            raise ValueError(f"{name}: batch stride {t.stride(0)} != T * row stride {T * ld}")
    elif Bsz > 1:
        ld = t.stride(0)
    else:
        ld = C
    return ld


def _f32_param(t, name, shape=None):
    import torch

    if t is None:
        return None
    if t.dtype != torch.float32 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


# ---------------------------------------------------------------- entry points --

def mamba_conv1d_silu_prefill(u, x, w, bias=None, conv_state_in=None, conv_state_out=None,
                              *, stream=None):
    """Causal depthwise conv1d + SiLU over T tokens (u, x: [B, T, Di]; w: [Di, K])."""
    Bsz, T, Di = x.shape
    K = w.shape[1]
    _f32_param(w, "w", (Di, K))
    _f32_param(bias, "bias", (Di,))
    _f32_param(conv_state_in, "conv_state_in", (Bsz, Di, K))
    _f32_param(conv_state_out, "conv_state_out", (Bsz, Di, K))
    if tuple(u.shape) != (Bsz, T, Di) or u.dtype != x.dtype:
        raise ValueError("u must match x in shape and dtype")
    _check(load().mamba_conv1d_silu_prefill(
        _ptr(u), _rows_ld(u, "u"), _ptr(x), _rows_ld(x, "x"), _dtype_code(x),
        _ptr(conv_state_in), _ptr(conv_state_out), _ptr(w), _ptr(bias),
        Bsz, T, Di, K, _stream(stream, x)))


def mamba_conv1d_silu_step(u, x, conv_state, layer, w, bias=None, *, stream=None):
    """One T=1 conv step on slab `layer` of conv_state [L, B, Di, K] (u, x: [B, Di])."""
    Bsz, Di = x.shape
    K = w.shape[1]
    if conv_state.dim() != 4 or tuple(conv_state.shape[1:]) != (Bsz, Di, K) or not conv_state.is_contiguous():
        raise ValueError("conv_state must be a contiguous [n_layers, B, Di, K] tensor")
    _f32_param(conv_state, "conv_state")
    _f32_param(w, "w", (Di, K))
    _f32_param(bias, "bias", (Di,))
    if not (x.is_contiguous() and u.is_contiguous()) or tuple(u.shape) != (Bsz, Di) or u.dtype != x.dtype:
        raise ValueError("u and x must be contiguous [B, Di] tensors of one dtype")
    _check(load().mamba_conv1d_silu_step(
        _ptr(u), _ptr(x), _dtype_code(x), _ptr(conv_state), int(layer), conv_state.shape[0],
        _ptr(w), _ptr(bias), Bsz, Di, K, _stream(stream, x)))


def mamba_selective_scan_workspace_bytes(Bsz, T, Di, N) -> int:
    """Workspace bytes the T-split route needs on the current device (0: none)."""
    v = load().mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
    if v < 0:
        raise MambaError(int(v), mamba_last_error())
    return int(v)


_ws_cache = {}    # (device index, stream handle) -> uint8 scratch tensor
_ws_retired = []  # outgrown scratch tensors, kept alive (see _workspace)


def _workspace(device, nbytes, stream_handle):
    """A scratch buffer per (device, stream), reused across calls and grown on
    demand (at least doubling).  Calls on different streams never share one, so
    concurrent streams cannot overwrite each other's carries.  An outgrown
    buffer is kept alive rather than freed: a CUDA graph captured earlier may
    still hold its address."""
    import torch

    dev = device.index if device.index is not None else torch.cuda.current_device()
    key = (dev, int(stream_handle))
    with _lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            size = max(nbytes, 1 << 20, 2 * buf.numel() if buf is not None else 0)
            if buf is not None:
                _ws_retired.append(buf)
            buf = torch.empty(size, dtype=torch.uint8, device=torch.device("cuda", dev))
            _ws_cache[key] = buf
    return buf


def _check_scan_args(y, u, dt, Bm, Cm, A_log, D, dt_bias, z, ssm_state_in, ssm_state_out):
    """Shapes and dtypes of a selective-scan prefill call, checked before any
    launch: the C ABI sees only pointers and sizes, so a tensor that is shorter
    than the sizes say, or holds another dtype, must be refused here.
    Returns (B, T, Di, N)."""
    if u.dim() != 3:
        raise ValueError(f"u must be 3-D [B, T, Di], got {tuple(u.shape)}")
    if A_log.dim() != 2:
        raise ValueError(f"A_log must be 2-D [Di, N], got {tuple(A_log.shape)}")
    Bsz, T, Di = u.shape
    N = A_log.shape[1]
    _f32_param(A_log, "A_log", (Di, N))
    _f32_param(D, "D", (Di,))
    _f32_param(dt_bias, "dt_bias", (Di,))
    _f32_param(ssm_state_in, "ssm_state_in", (Bsz, Di, N))
    _f32_param(ssm_state_out, "ssm_state_out", (Bsz, Di, N))
    for t, nm in ((y, "y"), (dt, "dt"), (Bm, "Bm"), (Cm, "Cm")):
        if t is None:
            raise ValueError(f"{nm} must not be None")
    for t, nm in ((dt, "dt"), (z, "z"), (Bm, "Bm"), (Cm, "Cm")):
        if t is not None and t.dtype != u.dtype:
            raise ValueError(f"{nm} must have the dtype of u")
    for t, nm in ((y, "y"), (dt, "dt"), (z, "z")):
        if t is not None and tuple(t.shape) != (Bsz, T, Di):
            raise ValueError(f"{nm} must be [B, T, Di] = {(Bsz, T, Di)}, got {tuple(t.shape)}")
    for t, nm in ((Bm, "Bm"), (Cm, "Cm")):
        if tuple(t.shape) != (Bsz, T, N):
            raise ValueError(f"{nm} must be [B, T, N] = {(Bsz, T, N)}, got {tuple(t.shape)}")
    return Bsz, T, Di, N


def mamba_selective_scan_prefill(y, u, dt, Bm, Cm, A_log, D=None, dt_bias=None, z=None,
                                 ssm_state_in=None, ssm_state_out=None, *, workspace=None,
                                 stream=None):
    """Selective scan with SiLU(z) gate over T tokens, state in / state out.

    y, u, dt, z: [B, T, Di] (row-strided views allowed); Bm, Cm: [B, T, N];
    A_log: [Di, N]; D, dt_bias: [Di]; states: [B, Di, N] f32.
    workspace: None = a cached buffer per (device, stream) sized by
    mamba_selective_scan_workspace_bytes; False = none (one sequential pass);
    or a uint8 cuda tensor (16-byte aligned), which the caller must not reuse
    on another stream while this call may still be running."""
    Bsz, T, Di, N = _check_scan_args(y, u, dt, Bm, Cm, A_log, D, dt_bias, z, ssm_state_in, ssm_state_out)
    st = _stream(stream, u)
    if workspace is None:
        need = mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
        ws = _workspace(u.device, need, st) if need > 0 else None
    elif workspace is False:
        ws = None
    else:
        ws = workspace
    ws_ptr = ws.data_ptr() if ws is not None else None
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().mamba_selective_scan_prefill(
        _ptr(y), _rows_ld(y, "y"), _dtype_code(y), _ptr(u), _rows_ld(u, "u"),
        _ptr(dt), _rows_ld(dt, "dt"), _ptr(z), _rows_ld(z, "z") if z is not None else 0,
        _ptr(Bm), _rows_ld(Bm, "Bm"), _ptr(Cm), _rows_ld(Cm, "Cm"), _dtype_code(u),
        _ptr(A_log), _ptr(D), _ptr(dt_bias), _ptr(ssm_state_in), _ptr(ssm_state_out),
        Bsz, T, Di, N, ws_ptr, ws_bytes, st))


def mamba_mixer_prefill(y, x, dt, Bm, Cm, conv_w, A_log, conv_b=None, D=None, dt_bias=None, z=None,
                        conv_state_in=None, conv_state_out=None, ssm_state_in=None, ssm_state_out=None, *,
                        workspace=None, stream=None):
    """Fused conv1d + SiLU and selective-scan prefill (u never stored).

    y, x, dt, z: [B, T, Di] (row-strided views allowed); Bm, Cm: [B, T, N];
    conv_w: [Di, K] with K in 1..4; A_log: [Di, N]; conv_b, D, dt_bias: [Di];
    conv states [B, Di, K] and ssm states [B, Di, N], f32.  workspace: as for
    mamba_selective_scan_prefill.  Equals mamba_conv1d_silu_prefill followed by
    mamba_selective_scan_prefill, bit for bit."""
    Bsz, T, Di = x.shape
    N = A_log.shape[1]
    K = conv_w.shape[1]
    _f32_param(conv_w, "conv_w", (Di, K))
    _f32_param(conv_b, "conv_b", (Di,))
    _f32_param(A_log, "A_log", (Di, N))
    _f32_param(D, "D", (Di,))
    _f32_param(dt_bias, "dt_bias", (Di,))
    for t, nm in ((conv_state_in, "conv_state_in"), (conv_state_out, "conv_state_out")):
        _f32_param(t, nm, (Bsz, Di, K))
    for t, nm in ((ssm_state_in, "ssm_state_in"), (ssm_state_out, "ssm_state_out")):
        _f32_param(t, nm, (Bsz, Di, N))
    for t, nm in ((dt, "dt"), (z, "z"), (Bm, "Bm"), (Cm, "Cm")):
        if t is not None and t.dtype != x.dtype:
            raise ValueError(f"{nm} must have the dtype of x")
    for t, nm in ((y, "y"), (dt, "dt"), (z, "z")):
        if t is not None and tuple(t.shape) != (Bsz, T, Di):
            raise ValueError(f"{nm} must be [B, T, Di]")
    for t, nm in ((Bm, "Bm"), (Cm, "Cm")):
        if tuple(t.shape) != (Bsz, T, N):
            raise ValueError(f"{nm} must be [B, T, N]")
    st = _stream(stream, x)
    if workspace is None:
        need = mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
        ws = _workspace(x.device, need, st) if need > 0 else None
    elif workspace is False:
        ws = None
    else:
        ws = workspace
    ws_ptr = ws.data_ptr() if ws is not None else None
    ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
    _check(load().mamba_mixer_prefill(
        _ptr(y), _rows_ld(y, "y"), _dtype_code(y), _ptr(x), _rows_ld(x, "x"),
        _ptr(dt), _rows_ld(dt, "dt"), _ptr(z), _rows_ld(z, "z") if z is not None else 0,
        _ptr(Bm), _rows_ld(Bm, "Bm"), _ptr(Cm), _rows_ld(Cm, "Cm"), _dtype_code(x),
        _ptr(conv_w), _ptr(conv_b), _ptr(conv_state_in), _ptr(conv_state_out),
        _ptr(A_log), _ptr(D), _ptr(dt_bias), _ptr(ssm_state_in), _ptr(ssm_state_out),
        Bsz, T, Di, K, N, ws_ptr, ws_bytes, st))


def mamba3_siso_step_batched(y, x, k, q, alpha, beta, gamma, ssm_state, k_state, v_state, layer, D=None, *,
                             stream=None):
    """Mamba-3 SISO T=1 step on slab `layer` of ssm_state [L, B, H, P, N],
    k_state [L, B, H, N] and v_state [L, B, H, P] (all updated in place).

    y, x: contiguous [B, H, P]; k, q: contiguous [B, H, N]; alpha, beta, gamma:
    f32 [B, H]; D: f32 [H]."""
    Bsz, H, P = x.shape
    N = k.shape[2]
    L = ssm_state.shape[0]
    for st, nm, shp in ((ssm_state, "ssm_state", (L, Bsz, H, P, N)), (k_state, "k_state", (L, Bsz, H, N)),
                        (v_state, "v_state", (L, Bsz, H, P))):
        _f32_param(st, nm, shp)
    for t, nm in ((alpha, "alpha"), (beta, "beta"), (gamma, "gamma")):
        _f32_param(t, nm, (Bsz, H))
    _f32_param(D, "D", (H,))
    for t, nm, shp in ((y, "y", (Bsz, H, P)), (x, "x", (Bsz, H, P)), (k, "k", (Bsz, H, N)), (q, "q", (Bsz, H, N))):
        if tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous {shp} tensor")
        if nm in ("k", "q") and t.dtype != x.dtype:
            raise ValueError(f"{nm} must have the dtype of x")
    _check(load().mamba3_siso_step_batched(
        _ptr(y), _dtype_code(y), _ptr(x), _ptr(k), _ptr(q), _dtype_code(x), _ptr(alpha), _ptr(beta), _ptr(gamma),
        _ptr(D), _ptr(ssm_state), _ptr(k_state), _ptr(v_state), int(layer), L, Bsz, H, P, N, _stream(stream, x)))


def mamba3_siso_step_prepare(k, q, alpha, beta, gamma, k_in, q_in, dt, A, lam, angles, angle_state, layer, *,
                             stream=None):
    """The Mamba-3 SISO step's inputs from one token's projections: slab
    `layer` of angle_state [L, B, H, n_angles] advanced by dt * angles, k_in and
    q_in rotated in pairs by it into k and q, and alpha / beta / gamma.

    k, q: contiguous [B, H, N] (f32 or bf16, one dtype); alpha, beta, gamma,
    dt, A, lam: f32 [B, H]; k_in, q_in: f32 [B, H, N]; angles: f32 [B,
    n_angles], or None (with angle_state None) for no rotation."""
    Bsz, H, N = k_in.shape
    for t, nm in ((k_in, "k_in"), (q_in, "q_in")):
        _f32_param(t, nm, (Bsz, H, N))
    for t, nm in ((alpha, "alpha"), (beta, "beta"), (gamma, "gamma"), (dt, "dt"), (A, "A"), (lam, "lam")):
        _f32_param(t, nm, (Bsz, H))
    for t, nm in ((k, "k"), (q, "q")):
        if tuple(t.shape) != (Bsz, H, N) or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous {(Bsz, H, N)} tensor")
    if q.dtype != k.dtype:
        raise ValueError("q must have the dtype of k")
    if (angles is None) != (angle_state is None):
        raise ValueError("angles and angle_state go together")
    na, L = 0, 1
    if angles is not None:
        na = angles.shape[1] if angles.dim() == 2 else -1
        _f32_param(angles, "angles", (Bsz, na))
        L = angle_state.shape[0]
        _f32_param(angle_state, "angle_state", (L, Bsz, H, na))
    _check(load().mamba3_siso_step_prepare(
        _ptr(k), _ptr(q), _dtype_code(k), _ptr(alpha), _ptr(beta), _ptr(gamma), _ptr(k_in), _ptr(q_in), _ptr(dt),
        _ptr(A), _ptr(lam), _ptr(angles), _ptr(angle_state), int(layer), L, Bsz, H, N, na, _stream(stream, k_in)))


def mamba3_siso_step_fused_batched(y, x, k_in, q_in, dt, A, lam, angles, ssm_state, k_state, v_state, angle_state,
                                   layer, D=None, *, stream=None):
    """One Mamba-3 SISO token in one launch: the step's inputs made as
    mamba3_siso_step_prepare makes them, then the step, on slab `layer` of
    ssm_state [L, B, H, P, N], k_state [L, B, H, N], v_state [L, B, H, P] and
    angle_state [L, B, H, n_angles] (all updated in place).

    y, x: contiguous [B, H, P]; k_in, q_in: f32 [B, H, N]; dt, A, lam: f32
    [B, H]; angles: f32 [B, n_angles], or None (with angle_state None) for no
    rotation; D: f32 [H]."""
    Bsz, H, P = x.shape
    N = k_in.shape[2]
    L = ssm_state.shape[0]
    for st, nm, shp in ((ssm_state, "ssm_state", (L, Bsz, H, P, N)), (k_state, "k_state", (L, Bsz, H, N)),
                        (v_state, "v_state", (L, Bsz, H, P))):
        _f32_param(st, nm, shp)
    for t, nm in ((k_in, "k_in"), (q_in, "q_in")):
        _f32_param(t, nm, (Bsz, H, N))
    for t, nm in ((dt, "dt"), (A, "A"), (lam, "lam")):
        _f32_param(t, nm, (Bsz, H))
    _f32_param(D, "D", (H,))
    for t, nm in ((y, "y"), (x, "x")):
        if tuple(t.shape) != (Bsz, H, P) or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous {(Bsz, H, P)} tensor")
    if (angles is None) != (angle_state is None):
        raise ValueError("angles and angle_state go together")
    na = 0
    if angles is not None:
        na = angles.shape[1] if angles.dim() == 2 else -1
        _f32_param(angles, "angles", (Bsz, na))
        _f32_param(angle_state, "angle_state", (L, Bsz, H, na))
    _check(load().mamba3_siso_step_fused_batched(
        _ptr(y), _dtype_code(y), _ptr(x), _dtype_code(x), _ptr(k_in), _ptr(q_in), _ptr(dt), _ptr(A), _ptr(lam),
        _ptr(angles), _ptr(D), _ptr(ssm_state), _ptr(k_state), _ptr(v_state), _ptr(angle_state), int(layer), L, Bsz,
        H, P, N, na, _stream(stream, x)))


def mamba_ssm_step_batched(y, u, dt, Bm, Cm, ssm_state, layer, A_log, D=None, dt_bias=None,
                           z=None, *, stream=None):
    """One T=1 SSM step on slab `layer` of ssm_state [L, B, Di, N].

    y, u, dt, z: contiguous [B, Di]; Bm, Cm: contiguous [B, N]."""
    Bsz, Di = u.shape
    N = A_log.shape[1]
    if ssm_state.dim() != 4 or tuple(ssm_state.shape[1:]) != (Bsz, Di, N) or not ssm_state.is_contiguous():
        raise ValueError("ssm_state must be a contiguous [n_layers, B, Di, N] tensor")
    _f32_param(ssm_state, "ssm_state")
    _f32_param(A_log, "A_log", (Di, N))
    _f32_param(D, "D", (Di,))
    _f32_param(dt_bias, "dt_bias", (Di,))
    for t, nm, shp in ((y, "y", (Bsz, Di)), (dt, "dt", (Bsz, Di)), (z, "z", (Bsz, Di)),
                       (Bm, "Bm", (Bsz, N)), (Cm, "Cm", (Bsz, N))):
        if t is None:
            continue
        if tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous {shp} tensor")
        if nm != "y" and t.dtype != u.dtype:
            raise ValueError(f"{nm} must have the dtype of u")
    _check(load().mamba_ssm_step_batched(
        _ptr(y), _dtype_code(y), _ptr(u), _ptr(dt), _ptr(z), _ptr(Bm), _ptr(Cm), _dtype_code(u),
        _ptr(A_log), _ptr(D), _ptr(dt_bias), _ptr(ssm_state), int(layer), ssm_state.shape[0],
        Bsz, Di, N, _stream(stream, u)))


def _rows2d(t, name):
    """Row stride of a 2-D [rows, cols] tensor with contiguous columns."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D [rows, cols], got {tuple(t.shape)}")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name}: columns must be contiguous (stride {t.stride(1)})")
    return t.stride(0) if t.shape[0] > 1 else t.shape[1]


def mamba_linear_bf16(c, a, w, residual=None, *, stream=None):
    """c[M, N] = a[M, K] @ w[N, K]^T (+ residual[M, N]) on the tensor cores.

    a, w: bf16 (row-strided views allowed, rows 16-byte aligned); c: f32 or
    bf16 [M, N]; residual: f32 [M, N], may be c itself."""
    import torch

    M, K = a.shape
    N = w.shape[0]
    if a.dtype != torch.bfloat16 or w.dtype != torch.bfloat16:
        raise ValueError("a and w must be bfloat16")
    if w.dim() != 2 or w.shape[1] != K:
        raise ValueError(f"w must be [N, K={K}], got {tuple(w.shape)}")
    if tuple(c.shape) != (M, N):
        raise ValueError(f"c must be [M, N] = {(M, N)}, got {tuple(c.shape)}")
    if residual is not None and (residual.dtype != torch.float32 or tuple(residual.shape) != (M, N)):
        raise ValueError("residual must be a float32 [M, N] tensor")
    _check(load().mamba_linear_bf16(
        _ptr(c), _rows2d(c, "c"), _dtype_code(c), _ptr(a), _rows2d(a, "a"), _ptr(w), _rows2d(w, "w"),
        _ptr(residual), _rows2d(residual, "residual") if residual is not None else 0, M, N, K,
        _stream(stream, a)))


def mamba_rmsnorm(out, x, weight, eps=1e-5, *, stream=None):
    """out[m] = x[m] / sqrt(mean(x[m]^2) + eps) * weight; x f32 [M, D], out f32
    or bf16 [M, D] (row-strided views allowed), weight f32 [D]."""
    import torch

    if x.dtype != torch.float32 or x.dim() != 2:
        raise ValueError("x must be a 2-D float32 tensor [M, D]")
    M, Dm = x.shape
    _f32_param(weight, "weight", (Dm,))
    if tuple(out.shape) != (M, Dm):
        raise ValueError(f"out must be [M, D] = {(M, Dm)}, got {tuple(out.shape)}")
    _check(load().mamba_rmsnorm(_ptr(out), _rows2d(out, "out"), _dtype_code(out), _ptr(x), _rows2d(x, "x"),
                                _ptr(weight), float(eps), M, Dm, _stream(stream, x)))


LAYER_WEIGHTS = ("norm_w", "in_proj_w", "conv_w", "conv_b", "x_proj_w", "dt_proj_w", "dt_bias", "A_log", "D",
                 "out_proj_w")


def layer_struct(w, eps=1e-5):
    """The C struct MambaLayer for a dict of block weights: norm_w [dm],
    in_proj_w [2 Di, dm] bf16, conv_w [Di, K], conv_b [Di] or None, x_proj_w
    [R + 2N, Di] bf16, dt_proj_w [Di, R] bf16, dt_bias (dt_proj's bias) [Di] or
    None, A_log [Di, N], D [Di] or None, out_proj_w [dm, Di] bf16.  Shapes and
    dtypes are checked here; the tensors must outlive every call that uses
    the struct."""
    import torch

    for k in ("norm_w", "in_proj_w", "conv_w", "x_proj_w", "dt_proj_w", "A_log", "out_proj_w"):
        if w.get(k) is None:
            raise ValueError(f"layer weight {k} is missing")
    Di, K = w["conv_w"].shape
    N = w["A_log"].shape[1]
    dm = w["norm_w"].shape[0]
    R = w["dt_proj_w"].shape[1]
    for k, shp in (("in_proj_w", (2 * Di, dm)), ("x_proj_w", (R + 2 * N, Di)), ("dt_proj_w", (Di, R)),
                   ("out_proj_w", (dm, Di))):
        t = w[k]
        if t.dtype != torch.bfloat16 or tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError(f"{k} must be a contiguous bfloat16 {shp} tensor")
    _f32_param(w["norm_w"], "norm_w", (dm,))
    _f32_param(w["conv_w"], "conv_w", (Di, K))
    _f32_param(w["A_log"], "A_log", (Di, N))
    for k in ("conv_b", "dt_bias", "D"):
        _f32_param(w.get(k), k, (Di,))
    return _MambaLayer(dm, Di, N, K, R, float(eps), _ptr(w["norm_w"]), _ptr(w["in_proj_w"]), _ptr(w["conv_w"]),
                       _ptr(w.get("conv_b")), _ptr(w["x_proj_w"]), _ptr(w["dt_proj_w"]), _ptr(w.get("dt_bias")),
                       _ptr(w["A_log"]), _ptr(w.get("D")), _ptr(w["out_proj_w"]))


def mamba_layer_workspace_bytes(w, Bsz, T, eps=1e-5) -> int:
    """Workspace bytes of a block over Bsz x T tokens (activations + the scan's share)."""
    v = load().mamba_layer_workspace_bytes(ctypes.byref(layer_struct(w, eps)), Bsz, T)
    if v < 0:
        raise MambaError(int(v), mamba_last_error())
    return int(v)


def _layer_workspace(workspace, w, Bsz, T, eps, device, st):
    if workspace is None:
        return _workspace(device, mamba_layer_workspace_bytes(w, Bsz, T, eps), st)
    return workspace


def mamba_layer_prefill(hidden, w, conv_state_in=None, conv_state_out=None, ssm_state_in=None,
                        ssm_state_out=None, *, eps=1e-5, workspace=None, stream=None):
    """One Mamba-1 block over T tokens: hidden [B, T, d_model] f32 (contiguous)
    is updated in place, hidden += out_proj(mixer(RMSNorm(hidden))).  States
    [B, Di, K] / [B, Di, N] f32 (in may be out; None in = zeros).  workspace:
    None = a cached buffer per (device, stream), or a uint8 cuda tensor."""
    import torch

    if hidden.dtype != torch.float32 or hidden.dim() != 3 or not hidden.is_contiguous():
        raise ValueError("hidden must be a contiguous float32 [B, T, d_model] tensor")
    Bsz, T, dm = hidden.shape
    S = layer_struct(w, eps)
    if dm != S.d_model:
        raise ValueError(f"hidden has d_model {dm}, the weights {S.d_model}")
    for t, nm, last in ((conv_state_in, "conv_state_in", S.d_conv), (conv_state_out, "conv_state_out", S.d_conv),
                        (ssm_state_in, "ssm_state_in", S.d_state), (ssm_state_out, "ssm_state_out", S.d_state)):
        _f32_param(t, nm, (Bsz, S.d_inner, last))
    st = _stream(stream, hidden)
    ws = _layer_workspace(workspace, w, Bsz, T, eps, hidden.device, st)
    _check(load().mamba_layer_prefill(_ptr(hidden), ctypes.byref(S), _ptr(conv_state_in), _ptr(conv_state_out),
                                      _ptr(ssm_state_in), _ptr(ssm_state_out), Bsz, T, _ptr(ws),
                                      ws.numel() * ws.element_size(), st))


def mamba_layer_step(hidden, w, conv_state, ssm_state, layer, *, eps=1e-5, workspace=None, stream=None):
    """One T=1 block step: hidden [B, d_model] f32 (contiguous, in place) on slab
    `layer` of conv_state [L, B, Di, K] and ssm_state [L, B, Di, N] (in place)."""
    import torch

    if hidden.dtype != torch.float32 or hidden.dim() != 2 or not hidden.is_contiguous():
        raise ValueError("hidden must be a contiguous float32 [B, d_model] tensor")
    Bsz, dm = hidden.shape
    S = layer_struct(w, eps)
    if dm != S.d_model:
        raise ValueError(f"hidden has d_model {dm}, the weights {S.d_model}")
    for t, nm, last in ((conv_state, "conv_state", S.d_conv), (ssm_state, "ssm_state", S.d_state)):
        if t.dim() != 4 or tuple(t.shape[1:]) != (Bsz, S.d_inner, last):
            raise ValueError(f"{nm} must be [n_layers, B, Di, {last}]")
        _f32_param(t, nm)
    if conv_state.shape[0] != ssm_state.shape[0]:
        raise ValueError("conv_state and ssm_state must have the same number of layers")
    st = _stream(stream, hidden)
    ws = _layer_workspace(workspace, w, Bsz, 1, eps, hidden.device, st)
    _check(load().mamba_layer_step(_ptr(hidden), ctypes.byref(S), _ptr(conv_state), _ptr(ssm_state), int(layer),
                                   conv_state.shape[0], Bsz, _ptr(ws), ws.numel() * ws.element_size(), st))


def mamba_selective_scan_prefill_noalloc(y, u, dt, Bm, Cm, A_log, D=None, dt_bias=None, z=None,
                                         ssm_state_in=None, ssm_state_out=None, *, stream=None):
    """The selective-scan prefill for callers that cannot allocate device memory:
    its T-split scratch is a static array inside the library (see the C header).
    Same arguments and result as mamba_selective_scan_prefill, minus the workspace."""
    Bsz, T, Di, N = _check_scan_args(y, u, dt, Bm, Cm, A_log, D, dt_bias, z, ssm_state_in, ssm_state_out)
    _check(load().mamba_selective_scan_prefill_noalloc(
        _ptr(y), _rows_ld(y, "y"), _dtype_code(y), _ptr(u), _rows_ld(u, "u"),
        _ptr(dt), _rows_ld(dt, "dt"), _ptr(z), _rows_ld(z, "z") if z is not None else 0,
        _ptr(Bm), _rows_ld(Bm, "Bm"), _ptr(Cm), _rows_ld(Cm, "Cm"), _dtype_code(u),
        _ptr(A_log), _ptr(D), _ptr(dt_bias), _ptr(ssm_state_in), _ptr(ssm_state_out),
        Bsz, T, Di, N, _stream(stream, u)))


def mamba_mixer_step_batched(y, x, dt, Bm, Cm, conv_state, ssm_state, layer, conv_w, A_log,
                             conv_b=None, D=None, dt_bias=None, z=None, *, stream=None):
    """Fused T=1 step: conv1d + SiLU step on x, then the SSM step, on slab `layer`
    of conv_state [L, B, Di, K] and ssm_state [L, B, Di, N] (both updated in place).

    y, x, dt, z: contiguous [B, Di]; Bm, Cm: contiguous [B, N]."""
    Bsz, Di = x.shape
    N = A_log.shape[1]
    K = conv_w.shape[1]
    for st, nm, last in ((conv_state, "conv_state", K), (ssm_state, "ssm_state", N)):
        if st.dim() != 4 or tuple(st.shape[1:]) != (Bsz, Di, last) or not st.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous [n_layers, B, Di, {last}] tensor")
        _f32_param(st, nm)
    if conv_state.shape[0] != ssm_state.shape[0]:
        raise ValueError("conv_state and ssm_state must have the same n_layers")
    _f32_param(conv_w, "conv_w", (Di, K))
    _f32_param(conv_b, "conv_b", (Di,))
    _f32_param(A_log, "A_log", (Di, N))
    _f32_param(D, "D", (Di,))
    _f32_param(dt_bias, "dt_bias", (Di,))
    for t, nm, shp in ((y, "y", (Bsz, Di)), (dt, "dt", (Bsz, Di)), (z, "z", (Bsz, Di)),
                       (Bm, "Bm", (Bsz, N)), (Cm, "Cm", (Bsz, N))):
        if t is None:
            continue
        if tuple(t.shape) != shp or not t.is_contiguous():
            raise ValueError(f"{nm} must be a contiguous {shp} tensor")
        if nm != "y" and t.dtype != x.dtype:
            raise ValueError(f"{nm} must have the dtype of x")
    _check(load().mamba_mixer_step_batched(
        _ptr(y), _dtype_code(y), _ptr(x), _ptr(dt), _ptr(z), _ptr(Bm), _ptr(Cm), _dtype_code(x),
        _ptr(conv_w), _ptr(conv_b), _ptr(A_log), _ptr(D), _ptr(dt_bias), _ptr(conv_state),
        _ptr(ssm_state), int(layer), ssm_state.shape[0], Bsz, Di, K, N, _stream(stream, x)))


class LayerDecodeGraph:
    """One decode token through whole Mamba-1 blocks, recorded once as a CUDA
    graph (mamba_layer_decode_graph_create): weights is a list of n_layers
    block weight dicts (see layer_struct), hidden a contiguous f32 [B,
    d_model] tensor updated in place by every launch (write the next token's
    hidden state into it first), conv_state / ssm_state [n_layers, B, Di, K|N].
    The tensors must outlive the graph; close() (or `with`) frees it."""

    def __init__(self, weights, hidden, conv_state, ssm_state, *, eps=1e-5, workspace=None):
        import torch

        lib = load()
        L = len(weights)
        if L == 0:
            raise ValueError("weights must hold at least one layer")
        if hidden.dtype != torch.float32 or hidden.dim() != 2 or not hidden.is_contiguous():
            raise ValueError("hidden must be a contiguous float32 [B, d_model] tensor")
        Bsz, dm = hidden.shape
        structs = (_MambaLayer * L)(*[layer_struct(w, eps) for w in weights])
        S0 = structs[0]
        if dm != S0.d_model:
            raise ValueError(f"hidden has d_model {dm}, the weights {S0.d_model}")
        for t, nm, last in ((conv_state, "conv_state", S0.d_conv), (ssm_state, "ssm_state", S0.d_state)):
            if t.dim() != 4 or tuple(t.shape) != (L, Bsz, S0.d_inner, last):
                raise ValueError(f"{nm} must be [{L}, B, Di, {last}]")
            _f32_param(t, nm)
        self._keep = (weights, hidden, conv_state, ssm_state, structs)
        if workspace is None:
            v = lib.mamba_layer_workspace_bytes(ctypes.byref(S0), Bsz, 1)
            if v < 0:
                raise MambaError(int(v), mamba_last_error())
            workspace = torch.empty(max(int(v), 16), dtype=torch.uint8, device=hidden.device)
        self._ws = workspace
        h = ctypes.c_void_p()
        _check(lib.mamba_layer_decode_graph_create(ctypes.byref(h), structs, L, _ptr(hidden), _ptr(conv_state),
                                                   _ptr(ssm_state), Bsz, _ptr(workspace),
                                                   workspace.numel() * workspace.element_size()))
        self._h = h
        self._device = hidden.device
        self.n_layers = L

    @property
    def kernels(self) -> int:
        v = load().mamba_decode_graph_kernels(self._h)
        if v < 0:
            raise MambaError(int(v), mamba_last_error())
        return int(v)

    def launch(self, stream=None):
        if self._h is None:
            raise ValueError("graph is closed")
        import torch

        s = torch.cuda.current_stream(self._device).cuda_stream if stream is None else (
            stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
        _check(load().mamba_decode_graph_launch(self._h, s))

    def close(self):
        if getattr(self, "_h", None) is not None:
            _check(load().mamba_decode_graph_destroy(self._h))
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _LayerParams(ctypes.Structure):
    _fields_ = [("conv_w", ctypes.c_void_p), ("conv_b", ctypes.c_void_p), ("A_log", ctypes.c_void_p),
                ("D", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p)]


class _StepIO(ctypes.Structure):
    _fields_ = [("y", ctypes.c_void_p), ("x", ctypes.c_void_p), ("dt", ctypes.c_void_p),
                ("z", ctypes.c_void_p), ("Bm", ctypes.c_void_p), ("Cm", ctypes.c_void_p)]


class DecodeGraph:
    """Graph-captured decode driver over the C ABI (mamba_decode_graph_*).

    params: n_layers dicts with conv_w, A_log and optional conv_b, D, dt_bias.
    io: n_steps lists of n_layers dicts with y, x, dt, Bm, Cm and optional z
    (contiguous [B, Di] / [B, N] tensors).  One launch() replays all
    n_steps x n_layers fused mixer steps on the given (or current) stream,
    reading and writing exactly these tensors; keep them alive, and write new
    inputs into them between launches.  Call close() (or use `with`) to free
    the graph."""

    def __init__(self, params, io, conv_state, ssm_state):
        lib = load()
        n_layers, n_steps = len(params), len(io)
        if n_layers == 0 or n_steps == 0 or any(len(row) != n_layers for row in io):
            raise ValueError("io must be n_steps lists of n_layers entries, params n_layers entries")
        x0 = io[0][0]["x"]
        Bsz, Di = x0.shape
        N = params[0]["A_log"].shape[1]
        K = params[0]["conv_w"].shape[1]
        for st, nm, last in ((conv_state, "conv_state", K), (ssm_state, "ssm_state", N)):
            if st.dim() != 4 or tuple(st.shape) != (n_layers, Bsz, Di, last) or not st.is_contiguous():
                raise ValueError(f"{nm} must be a contiguous [{n_layers}, B, Di, {last}] tensor")
            _f32_param(st, nm)
        P = (_LayerParams * n_layers)()
        for l, p in enumerate(params):
            _f32_param(p["conv_w"], "conv_w", (Di, K))
            _f32_param(p["A_log"], "A_log", (Di, N))
            for k in ("conv_b", "D", "dt_bias"):
                _f32_param(p.get(k), k, (Di,))
            P[l] = _LayerParams(_ptr(p["conv_w"]), _ptr(p.get("conv_b")), _ptr(p["A_log"]), _ptr(p.get("D")),
                                _ptr(p.get("dt_bias")))
        Q = (_StepIO * (n_steps * n_layers))()
        y_code = _dtype_code(io[0][0]["y"])
        for s_, row in enumerate(io):
            for l, q in enumerate(row):
                for k, shp in (("y", (Bsz, Di)), ("x", (Bsz, Di)), ("dt", (Bsz, Di)), ("z", (Bsz, Di)),
                               ("Bm", (Bsz, N)), ("Cm", (Bsz, N))):
                    t = q.get(k)
                    if t is None:
                        continue
                    if tuple(t.shape) != shp or not t.is_contiguous():
                        raise ValueError(f"io[{s_}][{l}]['{k}'] must be a contiguous {shp} tensor")
                    if k == "y" and _dtype_code(t) != y_code:
                        raise ValueError("every y must have the same dtype")
                    if k != "y" and t.dtype != x0.dtype:
                        raise ValueError(f"io[{s_}][{l}]['{k}'] must have the dtype of x")
                Q[s_ * n_layers + l] = _StepIO(_ptr(q["y"]), _ptr(q["x"]), _ptr(q["dt"]), _ptr(q.get("z")),
                                               _ptr(q["Bm"]), _ptr(q["Cm"]))
        h = ctypes.c_void_p()
        _check(lib.mamba_decode_graph_create(ctypes.byref(h), P, Q, n_steps, n_layers, y_code, _dtype_code(x0),
                                             _ptr(conv_state), _ptr(ssm_state), Bsz, Di, K, N))
        self._h = h
        self._device = x0.device
        self.n_steps, self.n_layers = n_steps, n_layers

    @property
    def kernels(self) -> int:
        """Kernel launches one replay makes."""
        v = load().mamba_decode_graph_kernels(self._h)
        if v < 0:
            raise MambaError(int(v), mamba_last_error())
        return int(v)

    def launch(self, stream=None):
        if self._h is None:
            raise ValueError("graph is closed")
        import torch

        s = torch.cuda.current_stream(self._device).cuda_stream if stream is None else (
            stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
        _check(load().mamba_decode_graph_launch(self._h, s))

    def close(self):
        if getattr(self, "_h", None) is not None:
            _check(load().mamba_decode_graph_destroy(self._h))
            self._h = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _M3TokenIO(ctypes.Structure):
    _fields_ = [("y", ctypes.c_void_p), ("x", ctypes.c_void_p), ("k_in", ctypes.c_void_p),
                ("q_in", ctypes.c_void_p), ("dt", ctypes.c_void_p), ("A", ctypes.c_void_p),
                ("lam", ctypes.c_void_p), ("angles", ctypes.c_void_p)]


class Mamba3DecodeGraph(DecodeGraph):
    """The Mamba-3 SISO decode recorded once as a CUDA graph
    (mamba3_decode_graph_create): io is n_steps lists of n_layers dicts with y,
    x, k_in, q_in, dt, A, lam and angles (or None) -- the tensors of
    mamba3_siso_step_fused_batched -- and D a list of n_layers [H] tensors (or
    None).  One launch() replays the n_steps x n_layers one-launch tokens on
    the given (or current) stream over slab l of the four states; write the
    next tokens' inputs into the same tensors between launches."""

    def __init__(self, io, ssm_state, k_state, v_state, angle_state=None, D=None):
        lib = load()
        n_steps = len(io)
        n_layers = len(io[0]) if n_steps else 0
        if n_layers == 0 or any(len(row) != n_layers for row in io):
            raise ValueError("io must be n_steps lists of n_layers entries")
        x0, k0 = io[0][0]["x"], io[0][0]["k_in"]
        Bsz, H, P = x0.shape
        N = k0.shape[2]
        a0 = io[0][0].get("angles")
        na = 0 if a0 is None else a0.shape[1]
        if (na > 0) != (angle_state is not None):
            raise ValueError("angles and angle_state go together")
        for st, nm, shp in ((ssm_state, "ssm_state", (n_layers, Bsz, H, P, N)),
                            (k_state, "k_state", (n_layers, Bsz, H, N)), (v_state, "v_state", (n_layers, Bsz, H, P)),
                            (angle_state, "angle_state", (n_layers, Bsz, H, na))):
            _f32_param(st, nm, shp)
        Dp = None
        if D is not None:
            if len(D) != n_layers:
                raise ValueError("D must hold one entry per layer")
            for d in D:
                _f32_param(d, "D", (H,))
            Dp = (ctypes.c_void_p * n_layers)(*[_ptr(d) for d in D])
        Q = (_M3TokenIO * (n_steps * n_layers))()
        y_code = _dtype_code(io[0][0]["y"])
        for s_, row in enumerate(io):
            for l, q in enumerate(row):
                for k, shp in (("y", (Bsz, H, P)), ("x", (Bsz, H, P))):
                    t = q[k]
                    if tuple(t.shape) != shp or not t.is_contiguous():
                        raise ValueError(f"io[{s_}][{l}]['{k}'] must be a contiguous {shp} tensor")
                if _dtype_code(q["y"]) != y_code or q["x"].dtype != x0.dtype:
                    raise ValueError("every y, and every x, must have one dtype")
                for k in ("k_in", "q_in"):
                    _f32_param(q[k], k, (Bsz, H, N))
                for k in ("dt", "A", "lam"):
                    _f32_param(q[k], k, (Bsz, H))
                if na:
                    _f32_param(q["angles"], "angles", (Bsz, na))
                elif q.get("angles") is not None:
                    raise ValueError("angles given for one token and not for another")
                Q[s_ * n_layers + l] = _M3TokenIO(_ptr(q["y"]), _ptr(q["x"]), _ptr(q["k_in"]), _ptr(q["q_in"]),
                                                  _ptr(q["dt"]), _ptr(q["A"]), _ptr(q["lam"]), _ptr(q.get("angles")))
        h = ctypes.c_void_p()
        _check(lib.mamba3_decode_graph_create(ctypes.byref(h), Q, Dp, n_steps, n_layers, y_code, _dtype_code(x0),
                                              _ptr(ssm_state), _ptr(k_state), _ptr(v_state), _ptr(angle_state), Bsz,
                                              H, P, N, na))
        self._keep = (io, D, Q, Dp)
        self._h = h
        self._device = x0.device
        self.n_steps, self.n_layers = n_steps, n_layers
