"""f64 CPU oracle of the rest of the Mamba-1 block -- TEST INFRASTRUCTURE ONLY.

Only the test suite and the benchmark's CPU baseline may import this module;
the product library never does, and it shares no code with the CUDA path.

What a Mamba-1 block computes around its mixer core, in the order of the
mamba-rs inference.rs step chain (`step_kernels`, steps F1-F12) and of the
prefill.rs prefill body, with the residual stream kept in f32 (the pages'
`residual_in_fp32`):

  F1   h      = x / sqrt(mean(x^2) + eps) * norm_w            RMSNorm per token row
  F2   xz     = h W_in^T                                       in_proj, [2 d_inner]
  F3   x, z   = xz[:, :d_inner], xz[:, d_inner:]              split: x branch, gate
  F4   u      = SiLU(causal depthwise conv1d(x) + conv_b)      (the C oracle)
  F5   x_dbl  = u W_x^T                                        x_proj, [dt_rank + 2 d_state]
  F6-F7 dt    = x_dbl[:, :dt_rank] W_dt^T                      dt_proj; its bias and the
                                                               softplus are the scan's
  F8-F10 y    = scan(u, dt, B = x_dbl[:, dt_rank:dt_rank+N],
                     C = x_dbl[:, dt_rank+N:], z)              (the C oracle, gate included)
  F11-F12 x'  = x + y W_out^T                                  out_proj + residual add

The pages print no body for the RMSNorm kernel; the plain definition above
(mean over d_model, eps inside the square root, then the per-feature weight)
is the reading taken.

Every matrix product is numpy's f64 matmul (a library primitive standing for
the plain sum over k); nothing is fused or reordered.  ``store`` says how an
activation is stored between steps: None keeps f64; a function (for example
a bf16 rounding) is applied where the GPU path stores an activation, so a
caller can mirror the GPU path's storage.  Layouts: x [rows, d_model] with
rows = B*T in (b, t) order; weights [out_features, in_features].
"""
from __future__ import annotations

import numpy as np

from . import conv1d_silu_prefill, conv1d_silu_step, selective_scan_prefill, ssm_step

RMS_NORM_EPS = 1e-5  # mamba-rs MambaConfig rms_norm_eps


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


def rmsnorm(x, weight, eps=RMS_NORM_EPS):
    """F1: each row scaled by 1/sqrt(mean of its squares + eps), then by weight."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * _f64(weight)


def linear(a, w, residual=None):
    """a [M, K] times w [N, K] transposed, plus an optional residual [M, N]."""
    out = _f64(a) @ _f64(w).T
    if residual is not None:
        out = out + _f64(residual)
    return out


def _keep(v, store):
    return v if store is None else store(v)


def layer_prefill(x, p, B, T, conv_state=None, ssm_state=None, eps=RMS_NORM_EPS, store=None):
    """One Mamba-1 block over T tokens of B sequences.

    x: [B*T, d_model] residual stream (f32 values); p: dict with norm_w
    [d_model], in_proj_w [2 Di, d_model], conv_w [Di, K], conv_b [Di],
    x_proj_w [R + 2N, Di], dt_proj_w [Di, R], dt_bias [Di], A_log [Di, N],
    D [Di], out_proj_w [d_model, Di].  States [B, Di, K] / [B, Di, N] or
    None (zeros).  Returns (x', conv_state', ssm_state', stages) where stages
    holds every intermediate (h, xz, u, x_dbl, dt, y) as stored."""
    x = _f64(x)
    Di = p["conv_w"].shape[0]
    N = p["A_log"].shape[1]
    R = p["dt_proj_w"].shape[1]
    h = _keep(rmsnorm(x, p["norm_w"], eps), store)
    xz = _keep(linear(h, p["in_proj_w"]), store)
    xin = xz[:, :Di].reshape(B, T, Di)
    z = xz[:, Di:].reshape(B, T, Di)
    u, conv_out = conv1d_silu_prefill(xin, p["conv_w"], p.get("conv_b"), conv_state)
    u = _keep(u, store)
    x_dbl = _keep(linear(u.reshape(B * T, Di), p["x_proj_w"]), store)
    dt = _keep(linear(x_dbl[:, :R], p["dt_proj_w"]), store)
    Bm = x_dbl[:, R:R + N].reshape(B, T, N)
    Cm = x_dbl[:, R + N:R + 2 * N].reshape(B, T, N)
    y, ssm_out = selective_scan_prefill(u, dt.reshape(B, T, Di), Bm, Cm, p["A_log"], p.get("D"), p.get("dt_bias"),
                                        z, ssm_state)
    y = _keep(y, store)
    x_new = linear(y.reshape(B * T, Di), p["out_proj_w"], x)
    stages = {"h": h, "xz": xz, "u": u.reshape(B * T, Di), "x_dbl": x_dbl, "dt": dt, "y": y.reshape(B * T, Di)}
    return x_new, conv_out, ssm_out, stages


def layer_step(x, p, conv_state, ssm_state, layer, eps=RMS_NORM_EPS, store=None):
    """One T=1 step of the block for B sequences: x [B, d_model]; states
    [L, B, Di, K] / [L, B, Di, N] (f64, C-contiguous) updated in place on slab
    `layer`.  Returns (x', stages)."""
    x = _f64(x)
    Di = p["conv_w"].shape[0]
    N = p["A_log"].shape[1]
    R = p["dt_proj_w"].shape[1]
    h = _keep(rmsnorm(x, p["norm_w"], eps), store)
    xz = _keep(linear(h, p["in_proj_w"]), store)
    u = _keep(conv1d_silu_step(np.ascontiguousarray(xz[:, :Di]), conv_state, layer, p["conv_w"], p.get("conv_b")),
              store)
    x_dbl = _keep(linear(u, p["x_proj_w"]), store)
    dt = _keep(linear(x_dbl[:, :R], p["dt_proj_w"]), store)
    y = ssm_step(u, dt, np.ascontiguousarray(x_dbl[:, R:R + N]), np.ascontiguousarray(x_dbl[:, R + N:R + 2 * N]),
                 ssm_state, layer, p["A_log"], p.get("D"), p.get("dt_bias"), np.ascontiguousarray(xz[:, Di:]))
    y = _keep(y, store)
    x_new = linear(y, p["out_proj_w"], x)
    stages = {"h": h, "xz": xz, "u": u, "x_dbl": x_dbl, "dt": dt, "y": y}
    return x_new, stages
