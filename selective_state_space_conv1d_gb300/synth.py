"""Seeded synthetic inputs for the Mamba-1 mixer core.

This module only draws random numbers and rounds them to the storage dtype; it
holds none of the mixer's arithmetic.  Both the CUDA path (tests, bench) and the
CPU oracle read the arrays it returns, so the two sides always see identical
inputs.

Streams are counter-based: every tensor is drawn from ``numpy.random.Philox``
keyed by ``(seed, tensor id)``, so a tensor never depends on what was drawn
before it.  ``seed = 0x5EED0000 + workload index``.

Distributions (the tiny-mixer recipe, reused by every workload):
  x, z, u  ~ N(0, 1)
  dt       ~ N(0, 1) * 0.1
  dt_bias  = softplus^-1(y),  y = exp(U(ln 1e-3, ln 0.1))   (log-uniform)
  A_log[c, n] = log(n + 1)          (n counted from 0, so A = -1 .. -N)
  B, C     ~ N(0, 1)  [batch, T, d_state]
  D = 1;   conv_w ~ U(-0.5, 0.5) [d_inner, d_conv];   conv_b = 0
  states   zero, or N(0, 0.5^2) where a workload asks for a seeded state
           (the long-context workload draws the conv state from N(0, 1)).
bf16 storage rounds the f32 draw to nearest-even; the returned f32 array then
holds exactly the bf16 values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

SEED_BASE = 0x5EED0000

_TENSOR_IDS = {
    "x": 1, "z": 2, "dt": 3, "u": 4, "B": 5, "C": 6,
    "conv_w": 10, "conv_b": 11, "dt_bias": 12, "D": 13, "A_log": 14,
    "conv_state": 20, "ssm_state": 21,
    # Mamba-3 SISO step
    "m3_x": 30, "m3_k": 31, "m3_q": 32, "m3_alpha": 33, "m3_beta": 34, "m3_gamma": 35, "m3_D": 36,
    "m3_ssm_state": 37, "m3_k_state": 38, "m3_v_state": 39,
    # the rest of the Mamba-1 block
    "norm_w": 40, "in_proj_w": 41, "x_proj_w": 42, "dt_proj_w": 43, "out_proj_w": 44, "hidden": 45,
    # inputs of the Mamba-3 step's preparation (angle state, rotation, trapezoid weights)
    "m3p_k": 50, "m3p_q": 51, "m3p_dt": 52, "m3p_A": 53, "m3p_lam": 54, "m3p_angles": 55, "m3_angle_state": 56,
}


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, storage dtype and initial-state recipe."""
    index: int
    name: str
    batch: int
    seqlen: int
    d_inner: int
    d_state: int
    d_conv: int
    dtype: str            # storage dtype of u, dt, B, C, z (and x): "f32" | "bf16"
    n_layers: int = 1
    steps: int = 0        # decode steps after the prefill (decode / long-context)
    state: str = "zero"   # "zero" | "seeded"

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index


WORKLOADS = {
    0: Workload(0, "tiny-mixer-f32", 1, 64, 128, 16, 4, "f32"),
    1: Workload(1, "mamba130m-layer-prefill-f32", 1, 2048, 1536, 16, 4, "f32"),
    2: Workload(2, "mamba130m-decode-b128-l24", 128, 1, 1536, 16, 4, "f32",
                n_layers=24, steps=256, state="seeded"),
    3: Workload(3, "mamba2.8b-layer-prefill-bf16", 8, 4096, 5120, 16, 4, "bf16"),
    4: Workload(4, "long-context-continuation-f32", 4, 16384, 2048, 16, 4, "f32",
                steps=64, state="seeded"),
}


def _key(seed: int, name: str, layer: int = 0, step: int = 0, part: int = 0) -> np.ndarray:
    tid = (_TENSOR_IDS[name] << 48) | ((layer & 0xFFFF) << 32) | ((step & 0xFFFF) << 16) | (part & 0xFFFF)
    return np.array([seed & 0xFFFFFFFFFFFFFFFF, tid], dtype=np.uint64)


def generator(seed: int, name: str, layer: int = 0, step: int = 0, part: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=_key(seed, name, layer, step, part)))


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """Round f32 values to the nearest bf16 (ties to even); returns f32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    bits = a.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    nan = np.isnan(a)
    out = rounded.astype(np.uint32).view(np.float32).copy()
    out[nan] = np.nan
    return out


def store(a: np.ndarray, dtype: str) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=np.float32)
    if dtype == "f32":
        return a
    if dtype == "bf16":
        return round_to_bf16(a)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def normal(seed, name, shape, std=1.0, dtype="f32", layer=0, step=0, part=0) -> np.ndarray:
    g = generator(seed, name, layer, step, part)
    a = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return store(a, dtype)


def uniform(seed, name, shape, lo, hi, layer=0) -> np.ndarray:
    g = generator(seed, name, layer)
    return g.uniform(lo, hi, size=shape).astype(np.float32)


def inverse_softplus_of_log_uniform(seed, name, shape, lo=1e-3, hi=0.1, layer=0) -> np.ndarray:
    """dt_bias recipe: y log-uniform in [lo, hi], returned as softplus^-1(y)."""
    g = generator(seed, name, layer)
    y = np.exp(g.uniform(math.log(lo), math.log(hi), size=shape))
    return (y + np.log(-np.expm1(-y))).astype(np.float32)


def mixer_params(seed: int, d_inner: int, d_state: int, d_conv: int, layer: int = 0) -> dict:
    """Per-layer parameters (all f32): conv_w, conv_b, A_log, D, dt_bias."""
    A_log = np.log(np.arange(1, d_state + 1, dtype=np.float64))[None, :].repeat(d_inner, 0)
    return {
        "conv_w": uniform(seed, "conv_w", (d_inner, d_conv), -0.5, 0.5, layer),
        "conv_b": np.zeros(d_inner, np.float32),
        "A_log": A_log.astype(np.float32),
        "D": np.ones(d_inner, np.float32),
        "dt_bias": inverse_softplus_of_log_uniform(seed, "dt_bias", (d_inner,), layer=layer),
    }


def parity_params(seed: int, d_inner: int, d_state: int, d_conv: int, layer: int = 0) -> dict:
    """Per-layer parameters for parity cases, varied per channel and per state
    so that a kernel reading a parameter at the wrong channel or state fails:
      A_log[c, n] = log(U(0.5, 16))  (A from -0.5 to -16, independent per (c, n))
      D[c] ~ N(1, 0.5^2),  conv_b[c] ~ N(0, 0.2^2),  dt_bias and conv_w as in
      the workload recipe.  The workloads keep mixer_params."""
    g = generator(seed, "A_log", layer)
    A_log = np.log(g.uniform(0.5, 16.0, size=(d_inner, d_state)))
    p = mixer_params(seed, d_inner, d_state, d_conv, layer)
    p["A_log"] = A_log.astype(np.float32)
    p["D"] = (1.0 + 0.5 * generator(seed, "D", layer).standard_normal(d_inner)).astype(np.float32)
    p["conv_b"] = normal(seed, "conv_b", (d_inner,), 0.2, layer=layer)
    return p


def layer_params(seed: int, d_model: int, d_inner: int, d_state: int, d_conv: int, dt_rank: int,
                 layer: int = 0, parity: bool = False) -> dict:
    """Weights of one Mamba-1 block (random init, no trained weights):
      in_proj_w [2 Di, dm], x_proj_w [R + 2N, Di], out_proj_w [dm, Di]
                ~ N(0, 1/fan_in), stored bf16
      dt_proj_w [Di, R] ~ U(-R^-1/2, R^-1/2), stored bf16
      norm_w [dm] = 1 (U(0.5, 1.5) for parity cases)
      the mixer's conv_w, conv_b, A_log, D and dt_bias (dt_proj's bias) from
      mixer_params, or parity_params for parity cases.
    Every array is f32; the bf16 weights hold exactly their bf16 values."""
    p = (parity_params if parity else mixer_params)(seed, d_inner, d_state, d_conv, layer)
    p["in_proj_w"] = normal(seed, "in_proj_w", (2 * d_inner, d_model), d_model ** -0.5, "bf16", layer)
    p["x_proj_w"] = normal(seed, "x_proj_w", (dt_rank + 2 * d_state, d_inner), d_inner ** -0.5, "bf16", layer)
    p["out_proj_w"] = normal(seed, "out_proj_w", (d_model, d_inner), d_inner ** -0.5, "bf16", layer)
    r = dt_rank ** -0.5
    p["dt_proj_w"] = store(uniform(seed, "dt_proj_w", (d_inner, dt_rank), -r, r, layer), "bf16")
    p["norm_w"] = (uniform(seed, "norm_w", (d_model,), 0.5, 1.5, layer) if parity
                   else np.ones(d_model, np.float32))
    return p


def prefill_inputs(seed: int, batch: int, seqlen: int, d_inner: int, d_state: int,
                   dtype: str = "f32", names=("x", "u", "dt", "z", "B", "C"),
                   t_offset_part: int = 0) -> dict:
    """Activations for one prefill call: x, u, z, dt [B, T, Di]; B, C [B, T, N]."""
    out = {}
    act = (batch, seqlen, d_inner)
    bc = (batch, seqlen, d_state)
    for name in names:
        if name in ("x", "u", "z"):
            out[name] = normal(seed, name, act, 1.0, dtype, part=t_offset_part)
        elif name == "dt":
            out[name] = normal(seed, name, act, 0.1, dtype, part=t_offset_part)
        elif name in ("B", "C"):
            out[name] = normal(seed, name, bc, 1.0, dtype, part=t_offset_part)
        else:
            raise KeyError(name)
    return out


def seeded_states(seed: int, n_layers: int, batch: int, d_inner: int, d_state: int,
                  d_conv: int, ssm_std: float = 0.5, conv_std: float = 0.5):
    """f32 states [n_layers, batch, d_inner, d_conv] and [n_layers, batch, d_inner, d_state]."""
    conv = normal(seed, "conv_state", (n_layers, batch, d_inner, d_conv), conv_std)
    ssm = normal(seed, "ssm_state", (n_layers, batch, d_inner, d_state), ssm_std)
    return conv, ssm


def decode_step_inputs(seed: int, layer: int, step: int, batch: int, d_inner: int,
                       d_state: int, dtype: str = "f32") -> dict:
    """Fresh per-(layer, step) activations for one T=1 decode step."""
    act = (batch, d_inner)
    bc = (batch, d_state)
    return {
        "x": normal(seed, "x", act, 1.0, dtype, layer, step),
        "z": normal(seed, "z", act, 1.0, dtype, layer, step),
        "dt": normal(seed, "dt", act, 0.1, dtype, layer, step),
        "B": normal(seed, "B", bc, 1.0, dtype, layer, step),
        "C": normal(seed, "C", bc, 1.0, dtype, layer, step),
    }


def m3_step_inputs(seed: int, layer: int, step: int, batch: int, nheads: int, headdim: int,
                   d_state: int, dtype: str = "f32") -> dict:
    """Per-(layer, step) inputs of one Mamba-3 SISO step: x [B, H, P]; k, q
    [B, H, N] (standing for B and C after norm, bias and RoPE); alpha, beta,
    gamma [B, H] f32 in the ranges exp(dt A), (1 - lambda) dt alpha and
    lambda dt take for dt ~ 1e-3..0.1 and A of order -1."""
    bh = (batch, nheads)
    g = generator(seed, "m3_alpha", layer, step)
    return {
        "x": normal(seed, "m3_x", (batch, nheads, headdim), 1.0, dtype, layer, step),
        "k": normal(seed, "m3_k", (batch, nheads, d_state), 1.0, dtype, layer, step),
        "q": normal(seed, "m3_q", (batch, nheads, d_state), 1.0, dtype, layer, step),
        "alpha": np.exp(-g.uniform(1e-3, 0.2, size=bh)).astype(np.float32),
        "beta": generator(seed, "m3_beta", layer, step).uniform(0.0, 0.1, size=bh).astype(np.float32),
        "gamma": generator(seed, "m3_gamma", layer, step).uniform(0.0, 0.1, size=bh).astype(np.float32),
    }


def m3_states(seed: int, n_layers: int, batch: int, nheads: int, headdim: int, d_state: int, std: float = 0.5):
    """f32 Mamba-3 states: ssm [L, B, H, P, N], k [L, B, H, N], v [L, B, H, P]."""
    return (normal(seed, "m3_ssm_state", (n_layers, batch, nheads, headdim, d_state), std),
            normal(seed, "m3_k_state", (n_layers, batch, nheads, d_state), 1.0),
            normal(seed, "m3_v_state", (n_layers, batch, nheads, headdim), 1.0))


def m3_prepare_inputs(seed: int, layer: int, step: int, batch: int, nheads: int, d_state: int,
                      n_angles: int) -> dict:
    """Per-(layer, step) inputs of the preparation of one Mamba-3 SISO step, all
    f32: k_in, q_in [B, H, N] N(0, 1) (B and C after norm and bias); dt [B, H]
    log-uniform in [1e-3, 0.1] (a softplus output); A [B, H] = -U(0.05, 4) (the
    decay rate); lam [B, H] U(0, 1) (the trapezoid weight, a sigmoid output);
    angles [B, n_angles] U(-pi, pi) (the token's raw angles)."""
    bh = (batch, nheads)
    dt = np.exp(generator(seed, "m3p_dt", layer, step).uniform(math.log(1e-3), math.log(0.1), size=bh))
    return {
        "k_in": normal(seed, "m3p_k", (batch, nheads, d_state), 1.0, "f32", layer, step),
        "q_in": normal(seed, "m3p_q", (batch, nheads, d_state), 1.0, "f32", layer, step),
        "dt": dt.astype(np.float32),
        "A": (-generator(seed, "m3p_A", layer, step).uniform(0.05, 4.0, size=bh)).astype(np.float32),
        "lam": generator(seed, "m3p_lam", layer, step).uniform(0.0, 1.0, size=bh).astype(np.float32),
        "angles": generator(seed, "m3p_angles", layer, step).uniform(-math.pi, math.pi,
                                                                     size=(batch, n_angles)).astype(np.float32),
    }


def m3_angle_state(seed: int, n_layers: int, batch: int, nheads: int, n_angles: int, span: float = 50.0):
    """f32 angle state [L, B, H, n_angles], U(-span, span): the angles a stretch
    of earlier tokens has accumulated."""
    g = generator(seed, "m3_angle_state")
    return g.uniform(-span, span, size=(n_layers, batch, nheads, n_angles)).astype(np.float32)


def torch_normal(shape, std, seed, device, dtype=None):
    """Same distribution drawn with torch's generator on `device` (used for
    decode workloads too large to draw on the host; the oracle gets copies)."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if dtype is not None and dtype != torch.float32:
        t = t.to(dtype)
    return t
