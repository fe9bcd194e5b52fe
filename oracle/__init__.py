"""f64 CPU oracle for the Mamba-1 mixer core -- TEST INFRASTRUCTURE ONLY.

Thin ctypes wrapper around ``mamba_oracle.c`` (plain sequential f64 C).  Only
the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference arm may import this package.  The product library and its Python
binding never import it; the oracle shares no code with the CUDA path.

Every function takes numpy arrays of any float dtype, upcasts them to f64
(exact for f32 and for bf16 already widened to f32), and returns f64 arrays.
Layouts: activations [B, T, Di]; B/C [B, T, N]; A_log [Di, N]; w [Di, K];
conv state [B, Di, K]; ssm state [B, Di, N].  ``None`` for bias / D / dt_bias
means 0, for z means "no gate", for a state means zeros.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mamba_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (strict IEEE: no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)
    ):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = [
            "gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
            "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm",
        ]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            L = ctypes.c_long
            lib.oracle_softplus.argtypes = [ctypes.c_double]
            lib.oracle_softplus.restype = ctypes.c_double
            lib.oracle_silu.argtypes = [ctypes.c_double]
            lib.oracle_silu.restype = ctypes.c_double
            lib.oracle_conv1d_silu_prefill.argtypes = [dp, dp, dp, dp, dp, dp, L, L, L, L, ctypes.c_int]
            lib.oracle_conv1d_silu_prefill.restype = ctypes.c_int
            lib.oracle_selective_scan_prefill.argtypes = [dp] * 11 + [L, L, L, L, ctypes.c_int]
            lib.oracle_selective_scan_prefill.restype = ctypes.c_int
            lib.oracle_conv1d_silu_step.argtypes = [dp, dp, L, dp, dp, dp, L, L, L, ctypes.c_int]
            lib.oracle_conv1d_silu_step.restype = ctypes.c_int
            lib.oracle_ssm_step.argtypes = [dp, dp, L] + [dp] * 8 + [L, L, L, ctypes.c_int]
            lib.oracle_m3_step.argtypes = [dp, dp, dp, dp, L] + [dp] * 7 + [L, L, L, L]
            lib.oracle_ssm_step.restype = ctypes.c_int
            lib.oracle_m3_prepare.argtypes = [dp] * 6 + [L] + [dp] * 6 + [L, L, L, L]
            lib.oracle_m3_prepare.restype = ctypes.c_int
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def softplus(v: float) -> float:
    return _load().oracle_softplus(float(v))


def silu(x: float) -> float:
    return _load().oracle_silu(float(x))


def conv1d_silu_prefill(x, w, bias=None, state_in=None, nthreads=None):
    """Causal depthwise conv1d + SiLU over T tokens.  Returns (u, state_out)."""
    x, w, bias, state_in = _f64(x), _f64(w), _f64(bias), _f64(state_in)
    Bsz, T, Di = x.shape
    K = w.shape[1]
    assert w.shape == (Di, K)
    if bias is not None:
        assert bias.shape == (Di,)
    if state_in is not None:
        assert state_in.shape == (Bsz, Di, K)
    u = np.empty((Bsz, T, Di))
    st = np.empty((Bsz, Di, K))
    rc = _load().oracle_conv1d_silu_prefill(
        _ptr(u), _ptr(st), _ptr(x), _ptr(state_in), _ptr(w), _ptr(bias),
        Bsz, T, Di, K, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_conv1d_silu_prefill rejected its arguments")
    return u, st


def selective_scan_prefill(u, dt, Bm, Cm, A_log, D=None, dt_bias=None, z=None,
                           state_in=None, nthreads=None):
    """Selective scan with SiLU(z) gate over T tokens.  Returns (y, state_out)."""
    u, dt, Bm, Cm, A_log = _f64(u), _f64(dt), _f64(Bm), _f64(Cm), _f64(A_log)
    D, dt_bias, z, state_in = _f64(D), _f64(dt_bias), _f64(z), _f64(state_in)
    Bsz, T, Di = u.shape
    N = A_log.shape[1]
    assert dt.shape == u.shape and Bm.shape == (Bsz, T, N) and Cm.shape == (Bsz, T, N)
    assert A_log.shape == (Di, N)
    if z is not None:
        assert z.shape == u.shape
    if state_in is not None:
        assert state_in.shape == (Bsz, Di, N)
    y = np.empty((Bsz, T, Di))
    st = np.empty((Bsz, Di, N))
    rc = _load().oracle_selective_scan_prefill(
        _ptr(y), _ptr(st), _ptr(u), _ptr(dt), _ptr(z), _ptr(Bm), _ptr(Cm),
        _ptr(A_log), _ptr(D), _ptr(dt_bias), _ptr(state_in),
        Bsz, T, Di, N, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_selective_scan_prefill rejected its arguments")
    return y, st


def conv1d_silu_step(x, conv_state, layer, w, bias=None, nthreads=None):
    """One T=1 conv step on the `layer` slab of conv_state [L, B, Di, K].

    conv_state is updated in place (it must be a C-contiguous f64 array);
    returns u [B, Di]."""
    assert conv_state.dtype == np.float64 and conv_state.flags.c_contiguous
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    Bsz, Di = x.shape
    K = w.shape[1]
    assert conv_state.shape[1:] == (Bsz, Di, K)
    u = np.empty((Bsz, Di))
    rc = _load().oracle_conv1d_silu_step(
        _ptr(u), _ptr(conv_state), layer, _ptr(x), _ptr(w), _ptr(bias),
        Bsz, Di, K, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_conv1d_silu_step rejected its arguments")
    return u


def ssm_step(u, dt, Bm, Cm, ssm_state, layer, A_log, D=None, dt_bias=None, z=None,
             nthreads=None):
    """One T=1 SSM step on the `layer` slab of ssm_state [L, B, Di, N] (in place).

    u, dt, z: [B, Di]; Bm, Cm: [B, N].  Returns y [B, Di]."""
    assert ssm_state.dtype == np.float64 and ssm_state.flags.c_contiguous
    u, dt, Bm, Cm, A_log = _f64(u), _f64(dt), _f64(Bm), _f64(Cm), _f64(A_log)
    D, dt_bias, z = _f64(D), _f64(dt_bias), _f64(z)
    Bsz, Di = u.shape
    N = A_log.shape[1]
    assert ssm_state.shape[1:] == (Bsz, Di, N)
    y = np.empty((Bsz, Di))
    rc = _load().oracle_ssm_step(
        _ptr(y), _ptr(ssm_state), layer, _ptr(u), _ptr(dt), _ptr(z), _ptr(Bm), _ptr(Cm),
        _ptr(A_log), _ptr(D), _ptr(dt_bias), Bsz, Di, N, nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_ssm_step rejected its arguments")
    return y


def m3_prepare(k_in, q_in, dt, A, lam, angles, angle_state, layer):
    """The Mamba-3 SISO step's inputs from one token's projections: the layer's
    angle state advanced by dt * angles, k_in and q_in rotated in pairs by it,
    and alpha / beta / gamma (the exponential-trapezoidal weights).

    k_in, q_in: [B, H, N]; dt, A, lam: [B, H]; angles: [B, n_angles] (None or
    n_angles = 0: no rotation); angle_state [L, B, H, n_angles] (f64,
    C-contiguous, updated in place).  Returns (k, q, alpha, beta, gamma)."""
    k_in, q_in, dt, A, lam = _f64(k_in), _f64(q_in), _f64(dt), _f64(A), _f64(lam)
    Bsz, H, N = k_in.shape
    assert q_in.shape == k_in.shape and dt.shape == (Bsz, H) and A.shape == (Bsz, H) and lam.shape == (Bsz, H)
    na = 0 if angles is None else np.asarray(angles).shape[1]
    if na:
        angles = _f64(angles)
        assert angles.shape == (Bsz, na)
        assert angle_state.dtype == np.float64 and angle_state.flags.c_contiguous
        assert angle_state.shape[1:] == (Bsz, H, na)
    else:
        angles, angle_state = None, None
    k, q = np.empty_like(k_in), np.empty_like(q_in)
    alpha, beta, gamma = np.empty((Bsz, H)), np.empty((Bsz, H)), np.empty((Bsz, H))
    rc = _load().oracle_m3_prepare(_ptr(k), _ptr(q), _ptr(alpha), _ptr(beta), _ptr(gamma), _ptr(angle_state),
                                   layer, _ptr(k_in), _ptr(q_in), _ptr(dt), _ptr(A), _ptr(lam), _ptr(angles),
                                   Bsz, H, N, na)
    if rc != 0:
        raise ValueError("oracle_m3_prepare rejected its arguments")
    return k, q, alpha, beta, gamma


def m3_step(x, k, q, alpha, beta, gamma, ssm_state, k_state, v_state, layer, D=None):
    """One Mamba-3 SISO T=1 step on the `layer` slabs (states updated in place).

    x: [B, H, P]; k, q: [B, H, N]; alpha, beta, gamma: [B, H]; D: [H];
    ssm_state [L, B, H, P, N], k_state [L, B, H, N], v_state [L, B, H, P] (f64,
    C-contiguous).  Returns y [B, H, P]."""
    for s_ in (ssm_state, k_state, v_state):
        assert s_.dtype == np.float64 and s_.flags.c_contiguous
    x, k, q = _f64(x), _f64(k), _f64(q)
    alpha, beta, gamma, D = _f64(alpha), _f64(beta), _f64(gamma), _f64(D)
    Bsz, H, P = x.shape
    N = k.shape[2]
    assert ssm_state.shape[1:] == (Bsz, H, P, N) and k_state.shape[1:] == (Bsz, H, N)
    assert v_state.shape[1:] == (Bsz, H, P)
    y = np.empty((Bsz, H, P))
    rc = _load().oracle_m3_step(_ptr(y), _ptr(ssm_state), _ptr(k_state), _ptr(v_state), layer, _ptr(x), _ptr(k),
                                _ptr(q), _ptr(alpha), _ptr(beta), _ptr(gamma), _ptr(D), Bsz, H, P, N)
    if rc != 0:
        raise ValueError("oracle_m3_step rejected its arguments")
    return y
