"""GPU parity: the CUDA path (through the C ABI) against the f64 CPU oracle.

Element-by-element on seeded synthetic inputs, at sizes the oracle finishes in
seconds that still span several chunks / tiles and a ragged tail, for both
storage dtypes, strided (column-slice) inputs, every supported d_state and
several d_conv, with and without gate / state, in place, and on the edge cases
(T = 0, T = 1, delta -> 0, NaN containment, guard bands).
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_conv1d_gb300 import synth
from _helpers import Guarded, assert_within, strided_copy, to_dev, to_host

pytestmark = pytest.mark.gpu

SEED = 0x5EED1000


def _params(seed, Di, N, K, layer=0, bias=True):
    """Parameters drawn per channel (and per state for A_log), so that a kernel
    that reads one at the wrong channel or state cannot pass."""
    p = synth.parity_params(seed, Di, N, K, layer)
    if not bias:
        p["conv_b"] = np.zeros(Di, np.float32)
    return p


# ------------------------------------------------------------------ conv ----

CONV_CASES = [
    # B, T, Di, K, dtype, state, strided
    (1, 64, 128, 4, "f32", False, False),
    (2, 257, 136, 4, "f32", True, False),
    (3, 5, 130, 3, "f32", True, False),       # Di not a multiple of 4: scalar path
    (2, 1000, 256, 2, "f32", True, True),     # x / u are column slices (ld = 2 Di)
    (2, 300, 512, 4, "bf16", True, False),
    (1, 77, 136, 4, "bf16", True, True),
    (2, 33, 64, 1, "f32", True, False),
    (1, 19, 64, 8, "bf16", True, False),
    (4, 2, 96, 4, "f32", True, False),        # T < K: the new state mixes old state and x
]


@pytest.mark.parametrize("Bsz,T,Di,K,dtype,state,strided", CONV_CASES)
def test_conv_prefill_matches_oracle(cuda_lib, Bsz, T, Di, K, dtype, state, strided):
    m = cuda_lib
    p = _params(SEED + K, Di, 16, K)
    x = synth.normal(SEED, "x", (Bsz, T, Di), 1.0, dtype)
    s0 = synth.normal(SEED, "conv_state", (Bsz, Di, K), 1.0) if state else None
    if strided:
        xd = strided_copy(x, dtype, 2 * Di, offset=Di)
        ud = strided_copy(np.zeros_like(x), dtype, 2 * Di)
    else:
        xd = to_dev(x, dtype)
        ud = torch.empty_like(xd)
    sd_in = to_dev(s0) if state else None
    sd_out = torch.empty((Bsz, Di, K), device="cuda")
    m.mamba_conv1d_silu_prefill(ud, xd, to_dev(p["conv_w"]), to_dev(p["conv_b"]), sd_in, sd_out)
    torch.cuda.synchronize()
    u_ref, s_ref = oracle.conv1d_silu_prefill(x, p["conv_w"], p["conv_b"], s0)
    assert_within(to_host(ud), u_ref, "u", bf16_out=dtype == "bf16")
    assert np.array_equal(to_host(sd_out), s_ref), "conv state is a copy of inputs: must be exact"


def test_conv_prefill_in_place_state_and_guard_bands(cuda_lib):
    m = cuda_lib
    Bsz, T, Di, K = 2, 123, 264, 4
    p = _params(SEED, Di, 16, K)
    x = synth.normal(SEED, "x", (Bsz, T, Di))
    s0 = synth.normal(SEED, "conv_state", (Bsz, Di, K))
    st = to_dev(s0)
    u = Guarded((Bsz, T, Di))
    m.mamba_conv1d_silu_prefill(u.view, to_dev(x), to_dev(p["conv_w"]), to_dev(p["conv_b"]), st, st)
    torch.cuda.synchronize()
    u.check()
    u_ref, s_ref = oracle.conv1d_silu_prefill(x, p["conv_w"], p["conv_b"], s0)
    assert_within(to_host(u.view), u_ref, "u")
    assert np.array_equal(to_host(st), s_ref)


def test_conv_T0_copies_state(cuda_lib):
    m = cuda_lib
    Bsz, Di, K = 2, 64, 4
    s0 = synth.normal(SEED, "conv_state", (Bsz, Di, K))
    out = torch.full((Bsz, Di, K), 3.0, device="cuda")
    x = torch.empty((Bsz, 0, Di), device="cuda")
    m.mamba_conv1d_silu_prefill(torch.empty_like(x), x, torch.zeros(Di, K, device="cuda"), None,
                                to_dev(s0), out)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(out), s0)


@pytest.mark.parametrize("dtype,K", [("f32", 4), ("bf16", 4), ("f32", 3), ("f32", 2)])
def test_conv_step_matches_oracle_and_prefill_bitwise(cuda_lib, dtype, K):
    m = cuda_lib
    L, Bsz, Di = 3, 5, 200
    p = _params(SEED + 1, Di, 16, K)
    conv = synth.normal(SEED, "conv_state", (L, Bsz, Di, K), 0.5)
    st = to_dev(conv)
    ref_state = conv.astype(np.float64).copy()
    w, b = to_dev(p["conv_w"]), to_dev(p["conv_b"])
    for step in range(4):
        x = synth.normal(SEED, "x", (Bsz, Di), 1.0, dtype, layer=1, step=step)
        xd = to_dev(x, dtype)
        # T=1 prefill on the same slab, for the bitwise comparison
        u_pf = torch.empty((Bsz, 1, Di), device="cuda", dtype=xd.dtype)
        s_pf = torch.empty((Bsz, Di, K), device="cuda")
        m.mamba_conv1d_silu_prefill(u_pf, xd.view(Bsz, 1, Di), w, b, st[1].clone(), s_pf)
        u = torch.empty_like(xd)
        m.mamba_conv1d_silu_step(u, xd, st, 1, w, b)
        torch.cuda.synchronize()
        u_ref = oracle.conv1d_silu_step(x, ref_state, 1, p["conv_w"], p["conv_b"])
        assert_within(to_host(u), u_ref, f"u step {step}", bf16_out=dtype == "bf16")
        assert torch.equal(u, u_pf[:, 0]), "conv step != T=1 conv prefill"
        assert torch.equal(st[1], s_pf)
    assert np.array_equal(to_host(st), ref_state)


# ------------------------------------------------------------------ scan ----

SCAN_CASES = [
    # B, T, Di, N, in, y, gate, state, strided
    (1, 64, 128, 16, "f32", "f32", True, False, False),     # tiny-mixer shape
    (1, 300, 128, 16, "f32", "f32", True, True, False),     # T split inside the CTA
    (1, 1000, 136, 16, "f32", "f32", True, True, True),     # T split, strided, ragged tail
    (2, 777, 130, 16, "f32", "f32", True, True, False),     # Di % 4 != 0: element staging
    (24, 70, 1024, 16, "f32", "f32", True, True, False),    # wide: one sequential pass
    (2, 513, 256, 16, "bf16", "f32", True, True, False),
    (3, 129, 136, 16, "bf16", "bf16", True, True, True),
    (1, 200, 64, 1, "f32", "f32", True, True, False),
    (1, 200, 64, 2, "f32", "f32", False, True, False),
    (1, 200, 64, 4, "bf16", "f32", True, True, False),
    (1, 200, 64, 8, "f32", "bf16", True, False, False),
    (2, 150, 64, 32, "f32", "f32", True, True, False),
    (2, 150, 64, 64, "f32", "f32", True, True, False),
    (1, 90, 64, 64, "bf16", "f32", True, True, True),
    (2, 1, 96, 16, "f32", "f32", True, True, False),        # T = 1
    (1, 2, 64, 16, "bf16", "f32", True, True, False),
]


def _scan_inputs(Bsz, T, Di, N, dtype, seed=SEED):
    a = synth.prefill_inputs(seed, Bsz, T, Di, N, dtype, names=("u", "dt", "z", "B", "C"))
    p = _params(seed, Di, N, 4)
    return a, p


def _run_scan(m, a, p, dtype, y_dtype, gate, state_in, strided, inplace=False, workspace=None):
    Bsz, T, Di = a["u"].shape
    N = a["B"].shape[2]
    if strided:
        # u / z as the two halves of one buffer, B / C as columns of an x_proj-like row
        u = strided_copy(a["u"], dtype, 2 * Di)
        z = strided_copy(a["z"], dtype, 2 * Di, offset=Di) if gate else None
        dt = strided_copy(a["dt"], dtype, Di + 8, offset=8)
        xdbl = Di // 4 + 2 * N  # dt_rank + 2 N
        Bm = strided_copy(a["B"], dtype, xdbl, offset=Di // 4)
        Cm = strided_copy(a["C"], dtype, xdbl, offset=Di // 4 + N)
        y = strided_copy(np.zeros((Bsz, T, Di), np.float32), y_dtype, Di + 4)
    else:
        u, dt = to_dev(a["u"], dtype), to_dev(a["dt"], dtype)
        z = to_dev(a["z"], dtype) if gate else None
        Bm, Cm = to_dev(a["B"], dtype), to_dev(a["C"], dtype)
        y = to_dev(np.zeros((Bsz, T, Di), np.float32), y_dtype)
    s_in = to_dev(state_in) if state_in is not None else None
    s_out = s_in if (inplace and s_in is not None) else torch.empty((Bsz, Di, N), device="cuda")
    m.mamba_selective_scan_prefill(y, u, dt, Bm, Cm, to_dev(p["A_log"]), to_dev(p["D"]),
                                   to_dev(p["dt_bias"]), z, s_in, s_out, workspace=workspace)
    torch.cuda.synchronize()
    return to_host(y), to_host(s_out)


@pytest.mark.parametrize("Bsz,T,Di,N,dtype,y_dtype,gate,state,strided", SCAN_CASES)
def test_scan_prefill_matches_oracle(cuda_lib, Bsz, T, Di, N, dtype, y_dtype, gate, state, strided):
    m = cuda_lib
    a, p = _scan_inputs(Bsz, T, Di, N, dtype)
    s0 = synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5) if state else None
    y, s = _run_scan(m, a, p, dtype, y_dtype, gate, s0, strided)
    y_ref, s_ref = oracle.selective_scan_prefill(a["u"], a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                 p["dt_bias"], a["z"] if gate else None, s0)
    assert_within(y, y_ref, "y", bf16_out=y_dtype == "bf16")
    assert_within(s, s_ref, "state")


SPLIT_CASES = [
    # narrow shapes that the plan splits along T; checked on both routes
    (1, 2048, 256, 16, "f32", "f32", True, True, False),
    (1, 3001, 96, 16, "bf16", "f32", True, True, False),
    (2, 999, 64, 64, "f32", "f32", True, True, False),
    (1, 1500, 64, 1, "f32", "f32", False, True, False),
    (1, 700, 160, 8, "bf16", "bf16", True, False, True),
]


@pytest.mark.parametrize("route", ["auto", "sequential"])
@pytest.mark.parametrize("Bsz,T,Di,N,dtype,y_dtype,gate,state,strided", SPLIT_CASES)
def test_scan_routes_match_oracle(cuda_lib, route, Bsz, T, Di, N, dtype, y_dtype, gate, state, strided):
    m = cuda_lib
    need = m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
    assert need > 0, "expected a T-split plan for this narrow shape"
    a, p = _scan_inputs(Bsz, T, Di, N, dtype)
    s0 = synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5) if state else None
    ws = None if route == "auto" else False
    y, s = _run_scan(m, a, p, dtype, y_dtype, gate, s0, strided, workspace=ws)
    y_ref, s_ref = oracle.selective_scan_prefill(a["u"], a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                 p["dt_bias"], a["z"] if gate else None, s0)
    assert_within(y, y_ref, "y", bf16_out=y_dtype == "bf16")
    assert_within(s, s_ref, "state")


def test_scan_workspace_smaller_than_asked_splits_less_or_runs_one_pass(cuda_lib):
    """With half the workspace the narrow shape is split into fewer parts (still
    within the bound of the oracle); with less than two parts' worth it runs as
    one sequential pass, bit for bit the no-workspace result."""
    m = cuda_lib
    Bsz, T, Di, N = 1, 1024, 128, 16
    a, p = _scan_inputs(Bsz, T, Di, N, "f32")
    need = m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
    y_ref, s_ref = oracle.selective_scan_prefill(a["u"], a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                 p["dt_bias"], a["z"], None)
    half = torch.empty(need // 2, dtype=torch.uint8, device="cuda")
    y1, s1 = _run_scan(m, a, p, "f32", "f32", True, None, False, workspace=half)
    assert_within(y1, y_ref, "y (half workspace)")
    assert_within(s1, s_ref, "state (half workspace)")
    tiny = torch.empty(4096, dtype=torch.uint8, device="cuda")
    y2, s2 = _run_scan(m, a, p, "f32", "f32", True, None, False, workspace=tiny)
    y3, s3 = _run_scan(m, a, p, "f32", "f32", True, None, False, workspace=False)
    assert np.array_equal(y2, y3) and np.array_equal(s2, s3)
    assert_within(y3, y_ref, "y (one pass)")


@pytest.mark.parametrize("Bsz,T,Di", [(1, 2000, 128), (8, 64, 512)])
def test_scan_ssm_part_without_D_and_gate(cuda_lib, Bsz, T, Di):
    """Tighter diagnostic: y - D u (the pure SSM part, ~1e-2) at the same bound."""
    m = cuda_lib
    a, p = _scan_inputs(Bsz, T, Di, 16, "f32", seed=SEED + 5)
    s0 = synth.normal(SEED, "ssm_state", (Bsz, Di, 16), 0.5)
    p = dict(p, D=np.zeros(Di, np.float32))
    y, s = _run_scan(m, a, p, "f32", "f32", False, s0, False)
    y_ref, s_ref = oracle.selective_scan_prefill(a["u"], a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                 p["dt_bias"], None, s0)
    assert_within(y, y_ref, "C.h")
    assert_within(s, s_ref, "state")


def test_scan_in_place_state_and_guard_bands(cuda_lib):
    m = cuda_lib
    Bsz, T, Di, N = 1, 700, 192, 16
    a, p = _scan_inputs(Bsz, T, Di, N, "f32")
    s0 = synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5)
    st = to_dev(s0)
    y = Guarded((Bsz, T, Di))
    m.mamba_selective_scan_prefill(y.view, to_dev(a["u"]), to_dev(a["dt"]), to_dev(a["B"]), to_dev(a["C"]),
                                   to_dev(p["A_log"]), to_dev(p["D"]), to_dev(p["dt_bias"]),
                                   to_dev(a["z"]), st, st)
    torch.cuda.synchronize()
    y.check()
    y_ref, s_ref = oracle.selective_scan_prefill(a["u"], a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                 p["dt_bias"], a["z"], s0)
    assert_within(to_host(y.view), y_ref, "y")
    assert_within(to_host(st), s_ref, "state")


def test_scan_strided_y_leaves_gap_columns_untouched(cuda_lib):
    m = cuda_lib
    Bsz, T, Di, N = 2, 300, 64, 16
    a, p = _scan_inputs(Bsz, T, Di, N, "f32")
    ybuf = torch.full((Bsz, T, Di + 16), -3.5, device="cuda")
    y = ybuf[:, :, 8:8 + Di]
    m.mamba_selective_scan_prefill(y, to_dev(a["u"]), to_dev(a["dt"]), to_dev(a["B"]), to_dev(a["C"]),
                                   to_dev(p["A_log"]), to_dev(p["D"]), to_dev(p["dt_bias"]), to_dev(a["z"]))
    torch.cuda.synchronize()
    assert bool((ybuf[:, :, :8] == -3.5).all()) and bool((ybuf[:, :, 8 + Di:] == -3.5).all())


@pytest.mark.parametrize("T1,T2,Di", [(100, 157, 128), (1, 63, 256), (2048, 333, 128)])
def test_scan_continuation(cuda_lib, T1, T2, Di):
    """prefill(T1) then prefill(T2) from the returned state == prefill(T1 + T2)."""
    m = cuda_lib
    Bsz, N = 2, 16
    a, p = _scan_inputs(Bsz, T1 + T2, Di, N, "f32")
    s0 = synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5)
    y, s = _run_scan(m, a, p, "f32", "f32", True, s0, False)
    a1 = {k: v[:, :T1].copy() for k, v in a.items()}
    a2 = {k: v[:, T1:].copy() for k, v in a.items()}
    y1, s1 = _run_scan(m, a1, p, "f32", "f32", True, s0, False)
    y2, s2 = _run_scan(m, a2, p, "f32", "f32", True, s1.astype(np.float32), False)
    y_ref, s_ref = oracle.selective_scan_prefill(a["u"], a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                 p["dt_bias"], a["z"], s0)
    assert_within(np.concatenate([y1, y2], 1), y_ref, "y (two calls)")
    assert_within(s2, s_ref, "state (two calls)")
    assert_within(y, y_ref, "y (one call)")
    assert_within(s, s_ref, "state (one call)")


def test_scan_T0_copies_or_zeroes_state(cuda_lib):
    m = cuda_lib
    Bsz, Di, N = 2, 64, 16
    s0 = synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5)
    e = torch.empty((Bsz, 0, Di), device="cuda")
    eb = torch.empty((Bsz, 0, N), device="cuda")
    A = torch.zeros(Di, N, device="cuda")
    out = torch.full((Bsz, Di, N), 9.0, device="cuda")
    m.mamba_selective_scan_prefill(e, e, e, eb, eb, A, None, None, None, to_dev(s0), out)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(out), s0)
    m.mamba_selective_scan_prefill(e, e, e, eb, eb, A, None, None, None, None, out)
    torch.cuda.synchronize()
    assert not bool(out.any())


@pytest.mark.parametrize("T,Di", [(40, 128), (500, 128)])
def test_scan_delta_to_zero_keeps_state(cuda_lib, T, Di):
    """dt + dt_bias = -200: delta underflows to 0, the state is unchanged bit for bit
    and y = C . h0 + D u (gate off)."""
    m = cuda_lib
    Bsz, N = 1, 16
    a, p = _scan_inputs(Bsz, T, Di, N, "f32")
    a["dt"] = np.zeros_like(a["dt"])
    p = dict(p, dt_bias=np.full(Di, -200.0, np.float32))
    s0 = synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5)
    y, s = _run_scan(m, a, p, "f32", "f32", False, s0, False)
    assert np.array_equal(s, s0.astype(np.float64))
    expect = (np.einsum("btn,bcn->btc", a["C"].astype(np.float64), s0.astype(np.float64))
              + p["D"].astype(np.float64) * a["u"])
    assert_within(y, expect, "y = C.h0 + D u")


@pytest.mark.parametrize("case", ["memoryless", "wide_dt", "mixed"])
@pytest.mark.parametrize("route", ["auto", "sequential"])
def test_scan_extreme_parameters_match_oracle(cuda_lib, case, route):
    """Parameters at the edges of the recurrence, against the oracle:
    - memoryless: A_log = 80 makes exp(delta A) = 0, so h_t = delta_t B_t u_t;
    - wide_dt: dt + dt_bias spread over about -60..60, across the softplus
      threshold, so delta runs from ~0 to ~60 and the decay from 1 to 0;
    - mixed: half the channels memoryless, the other half with delta ~ 0."""
    m = cuda_lib
    Bsz, T, Di, N = 2, 700, 96, 16
    a, p = _scan_inputs(Bsz, T, Di, N, "f32", seed=SEED + 21)
    p = dict(p)
    if case == "memoryless":
        p["A_log"] = np.full((Di, N), 80.0, np.float32)
    elif case == "wide_dt":
        a["dt"] = synth.normal(SEED + 21, "dt", a["dt"].shape, 20.0, part=7)
        p["dt_bias"] = np.zeros(Di, np.float32)
    else:
        p["A_log"] = p["A_log"].copy()
        p["A_log"][::2] = 80.0
        p["dt_bias"] = p["dt_bias"].copy()
        p["dt_bias"][1::2] = -200.0
    s0 = synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5)
    ws = None if route == "auto" else False
    y, s = _run_scan(m, a, p, "f32", "f32", True, s0, False, workspace=ws)
    y_ref, s_ref = oracle.selective_scan_prefill(a["u"], a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                 p["dt_bias"], a["z"], s0)
    assert_within(y, y_ref, f"{case} y")
    assert_within(s, s_ref, f"{case} state")
    if case == "memoryless":
        # h_T = delta_{T-1} B_{T-1} u_{T-1}, with delta = softplus(dt + dt_bias)
        v = a["dt"][:, -1, :].astype(np.float64) + p["dt_bias"].astype(np.float64)
        delta = np.maximum(v, 0) + np.log1p(np.exp(-np.abs(v)))
        h_last = (delta * a["u"][:, -1, :])[:, :, None] * a["B"][:, -1, None, :].astype(np.float64)
        assert_within(s, h_last, "memoryless state")


def test_scan_nan_stays_in_its_channel(cuda_lib):
    m = cuda_lib
    Bsz, T, Di, N = 2, 600, 128, 16
    a, p = _scan_inputs(Bsz, T, Di, N, "f32")
    t0, c0 = 250, 37
    a["u"][1, t0, c0] = np.nan
    y, s = _run_scan(m, a, p, "f32", "f32", True, None, False)
    nan = np.isnan(y)
    assert not nan[:, :t0].any() and not nan[0].any()
    assert nan[1, t0:, c0].all()
    other = np.ones(Di, bool)
    other[c0] = False
    assert not nan[1][:, other].any()
    assert np.isnan(s[1, c0]).all() and not np.isnan(s[1, other]).any() and not np.isnan(s[0]).any()


def test_scan_is_deterministic_and_batch_rows_are_independent(cuda_lib):
    m = cuda_lib
    Bsz, T, Di, N = 4, 48, 256, 16  # T <= 64: one sequential pass for any batch
    a, p = _scan_inputs(Bsz, T, Di, N, "f32")
    s0 = synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5)
    y, s = _run_scan(m, a, p, "f32", "f32", True, s0, False)
    y2, s2 = _run_scan(m, a, p, "f32", "f32", True, s0, False)
    assert np.array_equal(y, y2) and np.array_equal(s, s2)
    a2 = {k: v[2:3].copy() for k, v in a.items()}
    y1, s1 = _run_scan(m, a2, p, "f32", "f32", True, s0[2:3].copy(), False)
    assert np.array_equal(y1[0], y[2]) and np.array_equal(s1[0], s[2])


# ------------------------------------------------------------------ step ----

@pytest.mark.parametrize("N,dtype,y_dtype,gate", [
    (16, "f32", "f32", True), (16, "bf16", "f32", True), (16, "bf16", "bf16", True),
    (1, "f32", "f32", True), (2, "f32", "f32", False), (4, "f32", "f32", True),
    (8, "f32", "f32", True), (32, "f32", "f32", True), (64, "f32", "f32", True),
    (64, "bf16", "f32", False),
])
def test_ssm_step_matches_oracle_and_T1_prefill_bitwise(cuda_lib, N, dtype, y_dtype, gate):
    m = cuda_lib
    L, Bsz, Di = 3, 9, 160
    p = _params(SEED + N, Di, N, 4, layer=2)
    st_h = synth.normal(SEED, "ssm_state", (L, Bsz, Di, N), 0.5)
    st = to_dev(st_h)
    ref_state = st_h.astype(np.float64).copy()
    A, D, dtb = to_dev(p["A_log"]), to_dev(p["D"]), to_dev(p["dt_bias"])
    for step in range(3):
        inp = synth.decode_step_inputs(SEED, 2, step, Bsz, Di, N, dtype)
        u_h = synth.normal(SEED, "u", (Bsz, Di), 1.0, dtype, layer=2, step=step)
        u, dt = to_dev(u_h, dtype), to_dev(inp["dt"], dtype)
        z = to_dev(inp["z"], dtype) if gate else None
        Bm, Cm = to_dev(inp["B"], dtype), to_dev(inp["C"], dtype)
        # T=1 prefill of the same slab (one sequential pass)
        y_pf = torch.empty((Bsz, 1, Di), device="cuda", dtype=torch.bfloat16 if y_dtype == "bf16" else torch.float32)
        s_pf = torch.empty((Bsz, Di, N), device="cuda")
        m.mamba_selective_scan_prefill(y_pf, u.view(Bsz, 1, Di), dt.view(Bsz, 1, Di), Bm.view(Bsz, 1, N),
                                       Cm.view(Bsz, 1, N), A, D, dtb,
                                       z.view(Bsz, 1, Di) if gate else None, st[2].clone(), s_pf)
        y = torch.empty((Bsz, Di), device="cuda", dtype=y_pf.dtype)
        m.mamba_ssm_step_batched(y, u, dt, Bm, Cm, st, 2, A, D, dtb, z)
        torch.cuda.synchronize()
        y_ref = oracle.ssm_step(u_h, inp["dt"], inp["B"], inp["C"], ref_state, 2, p["A_log"], p["D"],
                                p["dt_bias"], inp["z"] if gate else None)
        assert_within(to_host(y), y_ref, f"y step {step}", bf16_out=y_dtype == "bf16")
        assert_within(to_host(st[2]), ref_state[2], f"state step {step}")
        assert torch.equal(y, y_pf[:, 0]), "ssm step != T=1 prefill"
        assert torch.equal(st[2], s_pf), "ssm step state != T=1 prefill state"
    assert np.array_equal(to_host(st[0]), st_h[0]) and np.array_equal(to_host(st[1]), st_h[1])


# ------------------------------------------------------------- fused step ----

@pytest.mark.parametrize("N,K,dtype,gate", [(16, 4, "f32", True), (16, 4, "bf16", True), (16, 3, "f32", False),
                                            (64, 4, "f32", True), (4, 2, "bf16", True), (1, 4, "f32", True)])
def test_mixer_step_equals_conv_step_then_ssm_step_bitwise(cuda_lib, N, K, dtype, gate):
    m = cuda_lib
    L, Bsz, Di = 3, 11, 200
    p = _params(SEED + 3, Di, N, K, layer=1)
    conv_h = synth.normal(SEED, "conv_state", (L, Bsz, Di, K), 0.5)
    ssm_h = synth.normal(SEED, "ssm_state", (L, Bsz, Di, N), 0.5)
    c1, s1 = to_dev(conv_h), to_dev(ssm_h)
    c2, s2 = to_dev(conv_h), to_dev(ssm_h)
    pd = {k: to_dev(v) for k, v in p.items()}
    conv_ref, ssm_ref = conv_h.astype(np.float64), ssm_h.astype(np.float64)
    for step in range(3):
        inp = synth.decode_step_inputs(SEED, 1, step, Bsz, Di, N, dtype)
        x, dt = to_dev(inp["x"], dtype), to_dev(inp["dt"], dtype)
        z = to_dev(inp["z"], dtype) if gate else None
        Bm, Cm = to_dev(inp["B"], dtype), to_dev(inp["C"], dtype)
        u = torch.empty_like(x)
        ya = torch.empty((Bsz, Di), device="cuda")
        m.mamba_conv1d_silu_step(u, x, c1, 1, pd["conv_w"], pd["conv_b"])
        m.mamba_ssm_step_batched(ya, u, dt, Bm, Cm, s1, 1, pd["A_log"], pd["D"], pd["dt_bias"], z)
        yb = torch.empty((Bsz, Di), device="cuda")
        m.mamba_mixer_step_batched(yb, x, dt, Bm, Cm, c2, s2, 1, pd["conv_w"], pd["A_log"], pd["conv_b"],
                                   pd["D"], pd["dt_bias"], z)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), "fused step != conv step + ssm step"
        assert torch.equal(c1, c2) and torch.equal(s1, s2)
        u_ref = oracle.conv1d_silu_step(inp["x"], conv_ref, 1, p["conv_w"], p["conv_b"])
        if dtype == "f32":
            # (bf16: u is rounded to bf16 between the halves; the fused step is held
            # to the separate steps bit for bit above, and those are oracle-checked)
            y_ref = oracle.ssm_step(u_ref, inp["dt"], inp["B"], inp["C"], ssm_ref, 1, p["A_log"], p["D"],
                                    p["dt_bias"], inp["z"] if gate else None)
            assert_within(to_host(yb), y_ref, f"fused y step {step}")
    assert np.array_equal(to_host(c2), conv_ref)
    if dtype == "f32":
        assert_within(to_host(s2), ssm_ref, "ssm state")


# ------------------------------------------------- ring vs direct step path ----

def _offset_like(t, elems=1):
    """A copy of t whose data starts `elems` elements past a 16-byte boundary
    (so the decode steps take their any-alignment kernel)."""
    flat = torch.empty(t.numel() + elems, device=t.device, dtype=t.dtype)
    v = flat[elems:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("N,K,dtype,fused", [(16, 4, "f32", True), (16, 4, "bf16", False), (64, 4, "f32", True),
                                             (8, 3, "bf16", True), (4, 4, "f32", False), (32, 2, "f32", True)])
def test_step_ring_and_direct_paths_agree_bitwise(cuda_lib, N, K, dtype, fused):
    """The copy-ring kernel (aligned buffers, d_inner % 8 == 0) and the
    any-alignment kernel give identical y and states."""
    m = cuda_lib
    L, Bsz, Di = 2, 37, 264
    p = _params(SEED + 5, Di, N, K, layer=0)
    pd = {k: to_dev(v) for k, v in p.items()}
    conv_a = to_dev(synth.normal(SEED, "conv_state", (L, Bsz, Di, K), 0.5))
    ssm_a = to_dev(synth.normal(SEED, "ssm_state", (L, Bsz, Di, N), 0.5))
    conv_b, ssm_b = _offset_like(conv_a), _offset_like(ssm_a)
    for step in range(4):
        inp = synth.decode_step_inputs(SEED, 0, step, Bsz, Di, N, dtype)
        x, dt, z = (to_dev(inp[k], dtype) for k in ("x", "dt", "z"))
        Bm, Cm = to_dev(inp["B"], dtype), to_dev(inp["C"], dtype)
        ya = torch.empty((Bsz, Di), device="cuda")
        yb = torch.empty((Bsz, Di), device="cuda")
        if fused:
            m.mamba_mixer_step_batched(ya, x, dt, Bm, Cm, conv_a, ssm_a, 1, pd["conv_w"], pd["A_log"],
                                       pd["conv_b"], pd["D"], pd["dt_bias"], z)
            m.mamba_mixer_step_batched(yb, x, dt, Bm, Cm, conv_b, ssm_b, 1, pd["conv_w"], pd["A_log"],
                                       pd["conv_b"], pd["D"], pd["dt_bias"], z)
        else:
            m.mamba_ssm_step_batched(ya, x, dt, Bm, Cm, ssm_a, 1, pd["A_log"], pd["D"], pd["dt_bias"], z)
            m.mamba_ssm_step_batched(yb, x, dt, Bm, Cm, ssm_b, 1, pd["A_log"], pd["D"], pd["dt_bias"], z)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), f"y differs at step {step}"
        assert torch.equal(ssm_a, ssm_b) and torch.equal(conv_a, conv_b)
    assert m.mamba_device_faults(clear=True) == 0


@pytest.mark.parametrize("fused", [True, False])
def test_ring_step_with_per_channel_parameters_across_channel_blocks_matches_oracle(cuda_lib, fused):
    """The copy-ring decode kernel keeps a channel block's parameters in
    registers while its CTA walks consecutive (channel block, batch row)
    tiles.  With batch 3 and 200 channel blocks every CTA crosses block
    boundaries, and per-channel A_log, D, dt_bias and conv weights make a
    stale or shifted parameter fail against the oracle."""
    m = cuda_lib
    L, Bsz, Di, N, K = 2, 3, 64 * 200, 16, 4
    p = _params(SEED + 21, Di, N, K, layer=1)
    pd = {k: to_dev(v) for k, v in p.items()}
    conv_h = synth.normal(SEED, "conv_state", (L, Bsz, Di, K), 0.5)
    ssm_h = synth.normal(SEED, "ssm_state", (L, Bsz, Di, N), 0.5)
    conv, ssm = to_dev(conv_h), to_dev(ssm_h)
    conv_ref, ssm_ref = conv_h.astype(np.float64), ssm_h.astype(np.float64)
    for step in range(2):
        inp = synth.decode_step_inputs(SEED + 21, 1, step, Bsz, Di, N, "f32")
        x, dt, z, Bm, Cm = (to_dev(inp[k]) for k in ("x", "dt", "z", "B", "C"))
        y = torch.empty((Bsz, Di), device="cuda")
        if fused:
            m.mamba_mixer_step_batched(y, x, dt, Bm, Cm, conv, ssm, 1, pd["conv_w"], pd["A_log"], pd["conv_b"],
                                       pd["D"], pd["dt_bias"], z)
            u_ref = oracle.conv1d_silu_step(inp["x"], conv_ref, 1, p["conv_w"], p["conv_b"])
        else:
            u_ref = inp["x"]
            m.mamba_ssm_step_batched(y, x, dt, Bm, Cm, ssm, 1, pd["A_log"], pd["D"], pd["dt_bias"], z)
        torch.cuda.synchronize()
        y_ref = oracle.ssm_step(u_ref, inp["dt"], inp["B"], inp["C"], ssm_ref, 1, p["A_log"], p["D"],
                                p["dt_bias"], inp["z"])
        assert_within(to_host(y), y_ref, f"y step {step}")
        assert_within(to_host(ssm[1]), ssm_ref[1], f"ssm state step {step}")
        if fused:
            assert np.array_equal(to_host(conv[1]), conv_ref[1])
    assert np.array_equal(to_host(ssm[0]), ssm_h[0])
    assert m.mamba_device_faults(clear=True) == 0


def test_a_bounded_wait_that_runs_out_sets_the_fault_bit_and_the_device_stays_usable(cuda_lib):
    """The watchdog path without a fault: a CTA waits, with the copy rings'
    bounded wait, on an mbarrier that nothing completes.  The wait gives up
    after its limit (about 1 ms here), the kernel returns, the host reads
    MAMBA_FAULT_RING_WAIT, and a ring-kernel decode step run afterwards still
    matches the oracle.  With the barrier completed first, no bit is set."""
    m = cuda_lib
    assert m.mamba_device_faults(clear=True) == 0
    try:
        m.mamba_selftest_bounded_wait(2_000_000, complete=True)
        assert m.mamba_device_faults() == 0
        m.mamba_selftest_bounded_wait(2_000_000, complete=False)
        assert m.mamba_device_faults() & m.MAMBA_FAULT_RING_WAIT
    finally:
        m.mamba_device_faults(clear=True)
    assert m.mamba_device_faults() == 0
    with pytest.raises(m.MambaError) as ei:
        m.mamba_selftest_bounded_wait(0, complete=False)
    assert ei.value.status == m.MAMBA_ERR_INVALID_ARG
    # the context is intact: a ring-path mixer step against the oracle
    L, Bsz, Di, N, K = 1, 8, 256, 16, 4
    p = _params(SEED + 13, Di, N, K)
    conv0 = synth.normal(SEED, "conv_state", (L, Bsz, Di, K), 0.5)
    ssm0 = synth.normal(SEED, "ssm_state", (L, Bsz, Di, N), 0.5)
    inp = synth.decode_step_inputs(SEED, 0, 0, Bsz, Di, N, "f32")
    conv, ssm = to_dev(conv0), to_dev(ssm0)
    y = torch.empty((Bsz, Di), device="cuda")
    pd = {k: to_dev(v) for k, v in p.items()}
    m.mamba_mixer_step_batched(y, to_dev(inp["x"]), to_dev(inp["dt"]), to_dev(inp["B"]), to_dev(inp["C"]), conv,
                               ssm, 0, pd["conv_w"], pd["A_log"], pd["conv_b"], pd["D"], pd["dt_bias"],
                               to_dev(inp["z"]))
    torch.cuda.synchronize()
    cs, ss = conv0.astype(np.float64), ssm0.astype(np.float64)
    u = oracle.conv1d_silu_step(inp["x"], cs, 0, p["conv_w"], p["conv_b"])
    y_ref = oracle.ssm_step(u, inp["dt"], inp["B"], inp["C"], ss, 0, p["A_log"], D=p["D"], dt_bias=p["dt_bias"],
                            z=inp["z"])
    assert_within(to_host(y), y_ref, "y after the watchdog self-test")
    assert_within(to_host(ssm), ss, "ssm state after the watchdog self-test")
    assert np.array_equal(to_host(conv), cs)
    assert m.mamba_device_faults(clear=True) == 0


# ------------------------------------------------------ decode graph driver ----

@pytest.mark.parametrize("dtype,gate,Di", [("f32", True, 200), ("bf16", True, 160), ("f32", False, 100)])
def test_decode_graph_replays_the_direct_calls_bitwise(cuda_lib, dtype, gate, Di):
    """A recorded n_steps x n_layers decode graph, launched twice, gives the same
    y and states, bit for bit, as the same fused mixer steps called directly."""
    m = cuda_lib
    L, S, Bsz, N, K = 3, 2, 9, 16, 4
    ps = [_params(SEED + 7, Di, N, K, layer=l) for l in range(L)]
    pd = [{k: to_dev(v) for k, v in p.items()} for p in ps]
    conv_h = synth.normal(SEED, "conv_state", (L, Bsz, Di, K), 0.5)
    ssm_h = synth.normal(SEED, "ssm_state", (L, Bsz, Di, N), 0.5)
    cg, sg, cd, sd = to_dev(conv_h), to_dev(ssm_h), to_dev(conv_h), to_dev(ssm_h)
    io = []
    for s in range(S):
        row = []
        for l in range(L):
            inp = synth.decode_step_inputs(SEED, l, s, Bsz, Di, N, dtype)
            q = {k: to_dev(inp[k], dtype) for k in ("x", "dt", "B", "C")}
            row.append({"y": torch.empty((Bsz, Di), device="cuda"), "x": q["x"], "dt": q["dt"],
                        "z": to_dev(inp["z"], dtype) if gate else None, "Bm": q["B"], "Cm": q["C"]})
        io.append(row)
    with m.DecodeGraph(pd, io, cg, sg) as g:
        assert g.kernels == S * L
        for rep in range(2):
            g.launch()
            torch.cuda.synchronize()
            ys = {}
            for s in range(S):
                for l in range(L):
                    q = io[s][l]
                    ys[s, l] = torch.empty((Bsz, Di), device="cuda")
                    m.mamba_mixer_step_batched(ys[s, l], q["x"], q["dt"], q["Bm"], q["Cm"], cd, sd, l,
                                               pd[l]["conv_w"], pd[l]["A_log"], pd[l]["conv_b"], pd[l]["D"],
                                               pd[l]["dt_bias"], q["z"])
            torch.cuda.synchronize()
            for (s, l), y in ys.items():
                assert torch.equal(y, io[s][l]["y"]), f"y differs (launch {rep}, step {s}, layer {l})"
            assert torch.equal(cg, cd) and torch.equal(sg, sd), f"states differ after launch {rep}"
    assert m.mamba_device_faults(clear=True) == 0


def test_decode_graph_reports_the_failing_step(cuda_lib):
    m = cuda_lib
    L, Bsz, Di, N, K = 2, 4, 64, 16, 4
    pd = [{k: to_dev(v) for k, v in _params(SEED, Di, N, K, layer=l).items()} for l in range(L)]
    conv, ssm = torch.zeros((L, Bsz, Di, K), device="cuda"), torch.zeros((L, Bsz, Di, N), device="cuda")
    mk = lambda: {"y": torch.empty((Bsz, Di), device="cuda"), "x": torch.zeros((Bsz, Di), device="cuda"),
                  "dt": torch.zeros((Bsz, Di), device="cuda"), "Bm": torch.zeros((Bsz, N), device="cuda"),
                  "Cm": torch.zeros((Bsz, N), device="cuda")}
    io = [[mk(), mk()]]
    io[0][1]["y"] = io[0][1]["x"]  # output overlapping an input: refused by the step's host checks
    with pytest.raises(m.MambaError) as ei:
        m.DecodeGraph(pd, io, conv, ssm)
    assert ei.value.status == m.MAMBA_ERR_INVALID_ARG and "layer 1" in str(ei.value)


# ------------------------------------------------------- fused mixer prefill ----

MIXER_PREFILL_CASES = [
    # (B, T, Di, N, K, dtype, y_dtype, gate, states, strided x) -- T-split and sequential shapes
    (1, 2048, 256, 16, 4, "f32", "f32", True, True, False),
    (1, 1500, 96, 16, 4, "bf16", "f32", True, True, True),
    (6, 333, 200, 16, 4, "f32", "bf16", False, True, False),
    (3, 77, 64, 64, 4, "bf16", "f32", True, False, False),
    (2, 2, 40, 8, 4, "f32", "f32", True, True, False),  # T < K: the new conv state mixes state and x
    (1, 999, 130, 4, 4, "f32", "f32", True, True, True),
    # every fused d_conv below 4, on both routes and both dtypes
    (1, 1700, 96, 16, 3, "f32", "f32", True, True, False),
    (2, 300, 72, 16, 3, "bf16", "f32", True, True, True),
    (1, 1300, 64, 8, 2, "bf16", "bf16", False, True, False),
    (3, 200, 136, 16, 2, "f32", "f32", True, True, False),
    (1, 900, 64, 32, 1, "f32", "f32", True, True, False),
    (2, 1, 48, 16, 1, "bf16", "f32", True, True, False),
    (2, 1, 48, 16, 3, "f32", "f32", True, True, False),   # T < K - 1
]


@pytest.mark.parametrize("inplace", [False, True])
@pytest.mark.parametrize("Bsz,T,Di,N,K,dtype,y_dtype,gate,states,strided", MIXER_PREFILL_CASES)
def test_mixer_prefill_equals_conv_then_scan_bitwise(cuda_lib, inplace, Bsz, T, Di, N, K, dtype, y_dtype, gate,
                                                      states, strided):
    m = cuda_lib
    p = _params(SEED + 11, Di, N, K)
    pd = {k: to_dev(v) for k, v in p.items()}
    a = synth.prefill_inputs(SEED + 11, Bsz, T, Di, N, dtype, names=("x", "dt", "z", "B", "C"))
    if strided:  # x as the first half of an in_proj-like row, z as the second
        x = strided_copy(a["x"], dtype, 2 * Di)
        z = strided_copy(a["z"], dtype, 2 * Di, offset=Di) if gate else None
    else:
        x = to_dev(a["x"], dtype)
        z = to_dev(a["z"], dtype) if gate else None
    dt, Bm, Cm = (to_dev(a[k], dtype) for k in ("dt", "B", "C"))
    c0 = to_dev(synth.normal(SEED, "conv_state", (Bsz, Di, K), 0.5)) if states else None
    s0 = to_dev(synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5)) if states else None
    ytd = torch.bfloat16 if y_dtype == "bf16" else torch.float32
    # separate calls
    u = torch.empty((Bsz, T, Di), device="cuda", dtype=x.dtype)
    c1, s1 = torch.empty((Bsz, Di, K), device="cuda"), torch.empty((Bsz, Di, N), device="cuda")
    y1 = torch.empty((Bsz, T, Di), device="cuda", dtype=ytd)
    m.mamba_conv1d_silu_prefill(u, x, pd["conv_w"], pd["conv_b"], c0, c1)
    m.mamba_selective_scan_prefill(y1, u, dt, Bm, Cm, pd["A_log"], pd["D"], pd["dt_bias"], z, s0, s1)
    # fused
    y2 = torch.empty((Bsz, T, Di), device="cuda", dtype=ytd)
    if inplace and states:
        c2, s2 = c0.clone(), s0.clone()
        m.mamba_mixer_prefill(y2, x, dt, Bm, Cm, pd["conv_w"], pd["A_log"], pd["conv_b"], pd["D"], pd["dt_bias"],
                              z, c2, c2, s2, s2)
    else:
        c2, s2 = torch.empty_like(c1), torch.empty_like(s1)
        m.mamba_mixer_prefill(y2, x, dt, Bm, Cm, pd["conv_w"], pd["A_log"], pd["conv_b"], pd["D"], pd["dt_bias"],
                              z, c0, c2, s0, s2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2), "fused prefill y != conv prefill + scan prefill"
    assert torch.equal(c1, c2) and torch.equal(s1, s2), "fused prefill states differ"
    if dtype == "f32" and y_dtype == "f32" and not inplace:
        # (bf16: u is rounded to bf16 between the halves; the separate calls are oracle-checked)
        ch = synth.normal(SEED, "conv_state", (Bsz, Di, K), 0.5) if states else None
        sh = synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5) if states else None
        u_ref, c_ref = oracle.conv1d_silu_prefill(a["x"], p["conv_w"], p["conv_b"], ch)
        y_ref, s_ref = oracle.selective_scan_prefill(u_ref, a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                     p["dt_bias"], a["z"] if gate else None, sh)
        assert_within(to_host(y2), y_ref, "fused y vs oracle")
        assert_within(to_host(s2), s_ref, "fused ssm state vs oracle")
        assert np.array_equal(to_host(c2), c_ref)


def test_mixer_prefill_T0_copies_both_states(cuda_lib):
    m = cuda_lib
    Bsz, Di, N, K = 2, 32, 16, 4
    p = {k: to_dev(v) for k, v in _params(SEED, Di, N, K).items()}
    e = torch.empty((Bsz, 0, Di), device="cuda")
    eb = torch.empty((Bsz, 0, N), device="cuda")
    c0, s0 = torch.randn((Bsz, Di, K), device="cuda"), torch.randn((Bsz, Di, N), device="cuda")
    c1, s1 = torch.full_like(c0, 7.0), torch.full_like(s0, 7.0)
    m.mamba_mixer_prefill(e, e, e, eb, eb, p["conv_w"], p["A_log"], conv_state_in=c0, conv_state_out=c1,
                          ssm_state_in=s0, ssm_state_out=s1)
    torch.cuda.synchronize()
    assert torch.equal(c0, c1) and torch.equal(s0, s1)


@pytest.mark.parametrize("route", ["auto", "sequential"])
@pytest.mark.parametrize("Bsz,T,Di,N", [(1, 1200, 96, 16), (2, 300, 64, 4), (1, 500, 40, 64)])
def test_prefill_states_at_a_4_byte_offset_match_aligned_states(cuda_lib, route, Bsz, T, Di, N):
    """States passed as views one float past a 16-byte boundary (in, out and in
    place) give the same bits as aligned ones, for the scan and the fused
    prefill, on the T-split and the one-pass route."""
    m = cuda_lib
    K = 4
    assert m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N) > 0
    ws = None if route == "auto" else False
    p = {k: to_dev(v) for k, v in _params(SEED + 5, Di, N, K).items()}
    a = synth.prefill_inputs(SEED + 5, Bsz, T, Di, N, "f32", names=("x", "dt", "z", "B", "C"))
    x, dt, z, Bm, Cm = (to_dev(a[k]) for k in ("x", "dt", "z", "B", "C"))
    c0 = to_dev(synth.normal(SEED, "conv_state", (Bsz, Di, K), 0.5))
    s0 = to_dev(synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5))

    def scan(s_in, s_out):
        y = torch.empty((Bsz, T, Di), device="cuda")
        m.mamba_selective_scan_prefill(y, x, dt, Bm, Cm, p["A_log"], p["D"], p["dt_bias"], z, s_in, s_out,
                                       workspace=ws)
        return y

    def fused(c_in, c_out, s_in, s_out):
        y = torch.empty((Bsz, T, Di), device="cuda")
        m.mamba_mixer_prefill(y, x, dt, Bm, Cm, p["conv_w"], p["A_log"], p["conv_b"], p["D"], p["dt_bias"], z,
                              c_in, c_out, s_in, s_out, workspace=ws)
        return y

    s_ref = torch.empty_like(s0)
    y_ref = scan(s0, s_ref)
    s_off = _offset_like(torch.zeros_like(s0))
    y_off = scan(_offset_like(s0), s_off)
    s_inp = _offset_like(s0)
    y_inp = scan(s_inp, s_inp)
    c_ref, s_fref = torch.empty_like(c0), torch.empty_like(s0)
    yf_ref = fused(c0, c_ref, s0, s_fref)
    c_off, s_foff = _offset_like(torch.zeros_like(c0)), _offset_like(torch.zeros_like(s0))
    yf_off = fused(_offset_like(c0), c_off, _offset_like(s0), s_foff)
    torch.cuda.synchronize()
    assert s_off.data_ptr() % 16 == 4 and c_off.data_ptr() % 16 == 4
    assert torch.equal(y_ref, y_off) and torch.equal(s_ref, s_off)
    assert torch.equal(y_ref, y_inp) and torch.equal(s_ref, s_inp)
    assert torch.equal(yf_ref, yf_off) and torch.equal(c_ref, c_off) and torch.equal(s_fref, s_foff)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("route", ["auto", "sequential"])
def test_prefill_activations_one_element_off_alignment_match_aligned(cuda_lib, dtype, route):
    """Every activation (x / u, dt, z, B, C and y) one element past a 16-byte
    boundary takes the element-wise staging; the conv prefill, the scan and the
    fused prefill give the same bits as with aligned buffers."""
    m = cuda_lib
    Bsz, T, Di, N, K = 2, 900, 128, 16, 4
    assert m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N) > 0
    ws = None if route == "auto" else False
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    p = {k: to_dev(v) for k, v in _params(SEED + 6, Di, N, K).items()}
    a = synth.prefill_inputs(SEED + 6, Bsz, T, Di, N, dtype, names=("x", "dt", "z", "B", "C"))
    al = {k: to_dev(a[k], dtype) for k in ("x", "dt", "z", "B", "C")}
    off = {k: _offset_like(v) for k, v in al.items()}
    c0 = to_dev(synth.normal(SEED, "conv_state", (Bsz, Di, K), 0.5))
    s0 = to_dev(synth.normal(SEED, "ssm_state", (Bsz, Di, N), 0.5))

    def run(t, shift):
        mk = (lambda shape, dt_: _offset_like(torch.zeros(shape, device="cuda", dtype=dt_))) if shift else \
             (lambda shape, dt_: torch.zeros(shape, device="cuda", dtype=dt_))
        u, c1 = mk((Bsz, T, Di), td), torch.empty_like(c0)
        m.mamba_conv1d_silu_prefill(u, t["x"], p["conv_w"], p["conv_b"], c0, c1)
        y1, s1 = mk((Bsz, T, Di), torch.float32), torch.empty_like(s0)
        m.mamba_selective_scan_prefill(y1, u, t["dt"], t["B"], t["C"], p["A_log"], p["D"], p["dt_bias"], t["z"],
                                       s0, s1, workspace=ws)
        y2, c2, s2 = mk((Bsz, T, Di), torch.float32), torch.empty_like(c0), torch.empty_like(s0)
        m.mamba_mixer_prefill(y2, t["x"], t["dt"], t["B"], t["C"], p["conv_w"], p["A_log"], p["conv_b"], p["D"],
                              p["dt_bias"], t["z"], c0, c2, s0, s2, workspace=ws)
        return u, c1, y1, s1, y2, c2, s2

    ref = run(al, False)
    got = run(off, True)
    torch.cuda.synchronize()
    assert off["x"].data_ptr() % 16 != 0 and got[2].data_ptr() % 16 != 0
    for name, r, g in zip(("u", "conv state", "y", "ssm state", "fused y", "fused conv state", "fused ssm state"),
                          ref, got):
        assert torch.equal(r, g), name


def test_prefills_on_two_streams_with_the_cached_workspace_match_serial(cuda_lib):
    """T-split prefills enqueued on two streams at once, each with the
    binding's cached workspace, give the same bits as the same calls run one
    after the other: the cache keeps one workspace per stream."""
    m = cuda_lib
    Bsz, T, Di, N = 1, 2048, 256, 16
    assert m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N) > 0
    p = {k: to_dev(v) for k, v in _params(SEED + 7, Di, N, 4).items()}
    cases = []
    for i in range(2):
        a = synth.prefill_inputs(SEED + 70 + i, Bsz, T, Di, N, "f32", names=("x", "dt", "z", "B", "C"))
        cases.append({k: to_dev(a[k]) for k in ("x", "dt", "z", "B", "C")})

    def call(t, y, s_out, stream=None):
        m.mamba_mixer_prefill(y, t["x"], t["dt"], t["B"], t["C"], p["conv_w"], p["A_log"], p["conv_b"], p["D"],
                              p["dt_bias"], t["z"], None, None, None, s_out, stream=stream)

    ref = []
    for t in cases:
        y, so = torch.empty((Bsz, T, Di), device="cuda"), torch.empty((Bsz, Di, N), device="cuda")
        call(t, y, so)
        torch.cuda.synchronize()
        ref.append((y, so))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = [[(torch.empty((Bsz, T, Di), device="cuda"), torch.empty((Bsz, Di, N), device="cuda"))
             for _ in range(6)] for _ in range(2)]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for r in range(6):  # interleaved, so that the two streams' calls overlap on the GPU
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                call(cases[i], *outs[i][r])
    torch.cuda.synchronize()
    for i in range(2):
        for y, so in outs[i]:
            assert torch.equal(y, ref[i][0]) and torch.equal(so, ref[i][1])


# ------------------------------------------------------------ Mamba-3 step ----

@pytest.mark.parametrize("Bsz,H,P,N,dtype,y_dtype,with_D", [
    (3, 5, 64, 64, "f32", "f32", True), (2, 3, 32, 128, "bf16", "f32", True), (4, 2, 100, 16, "f32", "bf16", False),
    (1, 1, 256, 64, "f32", "f32", True), (2, 4, 48, 32, "bf16", "bf16", True),
])
def test_m3_step_matches_oracle(cuda_lib, Bsz, H, P, N, dtype, y_dtype, with_D):
    """Three Mamba-3 SISO steps on the middle layer of a 3-layer state: y and
    all three states against the oracle; the other layers untouched."""
    m = cuda_lib
    L, layer = 3, 1
    st_h, ks_h, vs_h = synth.m3_states(SEED, L, Bsz, H, P, N)
    st, ks, vs = to_dev(st_h), to_dev(ks_h), to_dev(vs_h)
    ref = [a.astype(np.float64).copy() for a in (st_h, ks_h, vs_h)]
    D_h = synth.normal(SEED, "m3_D", (H,), 1.0) if with_D else None
    D = to_dev(D_h) if with_D else None
    ytd = torch.bfloat16 if y_dtype == "bf16" else torch.float32
    for step in range(3):
        inp = synth.m3_step_inputs(SEED, layer, step, Bsz, H, P, N, dtype)
        x, k, q = (to_dev(inp[n], dtype) for n in ("x", "k", "q"))
        al, be, ga = (to_dev(inp[n]) for n in ("alpha", "beta", "gamma"))
        y = torch.empty((Bsz, H, P), device="cuda", dtype=ytd)
        m.mamba3_siso_step_batched(y, x, k, q, al, be, ga, st, ks, vs, layer, D)
        torch.cuda.synchronize()
        y_ref = oracle.m3_step(inp["x"], inp["k"], inp["q"], inp["alpha"], inp["beta"], inp["gamma"],
                               ref[0], ref[1], ref[2], layer, D_h)
        assert_within(to_host(y), y_ref, f"m3 y step {step}", bf16_out=y_dtype == "bf16")
        assert_within(to_host(st[layer]), ref[0][layer], f"m3 ssm state step {step}")
        assert np.array_equal(to_host(ks[layer]), ref[1][layer]) and np.array_equal(to_host(vs[layer]), ref[2][layer])
    for s_dev, s_h in ((st, st_h), (ks, ks_h), (vs, vs_h)):
        for l in (0, 2):
            assert np.array_equal(to_host(s_dev[l]), s_h[l])
    assert m.mamba_device_faults(clear=True) == 0


@pytest.mark.parametrize("P,N,dtype", [(64, 64, "f32"), (32, 128, "bf16"), (100, 16, "f32")])
def test_m3_ring_and_direct_paths_agree_bitwise(cuda_lib, P, N, dtype):
    """The copy-ring Mamba-3 kernel (aligned buffers) and the per-(batch, head)
    kernel (k_state 4 bytes off a 16-byte boundary) give identical results."""
    m = cuda_lib
    L, Bsz, H, layer = 2, 5, 3, 1
    st_h, ks_h, vs_h = synth.m3_states(SEED + 1, L, Bsz, H, P, N)
    sa, ka, va = to_dev(st_h), to_dev(ks_h), to_dev(vs_h)
    sb, kb, vb = to_dev(st_h), _offset_like(to_dev(ks_h)), to_dev(vs_h)
    D = to_dev(synth.normal(SEED, "m3_D", (H,), 1.0))
    for step in range(3):
        inp = synth.m3_step_inputs(SEED + 1, layer, step, Bsz, H, P, N, dtype)
        x, k, q = (to_dev(inp[n], dtype) for n in ("x", "k", "q"))
        al, be, ga = (to_dev(inp[n]) for n in ("alpha", "beta", "gamma"))
        ya = torch.empty((Bsz, H, P), device="cuda")
        yb = torch.empty((Bsz, H, P), device="cuda")
        m.mamba3_siso_step_batched(ya, x, k, q, al, be, ga, sa, ka, va, layer, D)
        m.mamba3_siso_step_batched(yb, x, k, q, al, be, ga, sb, kb, vb, layer, D)
        torch.cuda.synchronize()
        assert torch.equal(ya, yb), f"y differs at step {step}"
        assert torch.equal(sa, sb) and torch.equal(ka, kb) and torch.equal(va, vb)
    assert m.mamba_device_faults(clear=True) == 0


# ---------------------------------------------- Mamba-3 step preparation ----

def _m3p_call(m, inp, na, th, layer, kq_dtype=torch.float32, k=None):
    Bsz, H, N = inp["k_in"].shape
    d = {n: to_dev(v) for n, v in inp.items()}
    k = torch.empty((Bsz, H, N), device="cuda", dtype=kq_dtype) if k is None else k
    q = torch.empty((Bsz, H, N), device="cuda", dtype=kq_dtype)
    al, be, ga = (torch.empty((Bsz, H), device="cuda") for _ in range(3))
    m.mamba3_siso_step_prepare(k, q, al, be, ga, d["k_in"], d["q_in"], d["dt"], d["A"], d["lam"],
                               d["angles"] if na else None, th if na else None, layer)
    return k, q, al, be, ga


@pytest.mark.parametrize("Bsz,H,N,na,kq", [
    (3, 5, 64, 32, "f32"), (2, 3, 128, 16, "bf16"), (4, 2, 16, 0, "f32"), (1, 7, 32, 1, "f32"),
    (2, 4, 64, 32, "bf16"), (5, 3, 2, 1, "f32"),
])
def test_m3_prepare_matches_oracle(cuda_lib, Bsz, H, N, na, kq):
    """Three tokens of the step's preparation on the middle layer of a 3-layer
    angle state: k, q, alpha, beta, gamma and the angle state against the
    oracle; the other layers untouched, nothing written past k."""
    m = cuda_lib
    L, layer = 3, 1
    th_h = synth.m3_angle_state(SEED, L, Bsz, H, max(na, 1))
    th = to_dev(th_h)
    th_ref = th_h.astype(np.float64)
    kqd = torch.bfloat16 if kq == "bf16" else torch.float32
    for step in range(3):
        inp = synth.m3_prepare_inputs(SEED, layer, step, Bsz, H, N, na)
        kg = Guarded((Bsz, H, N), kq)
        k, q, al, be, ga = _m3p_call(m, inp, na, th, layer, kqd, kg.view)
        torch.cuda.synchronize()
        kg.check()
        rk, rq, ral, rbe, rga = oracle.m3_prepare(inp["k_in"], inp["q_in"], inp["dt"], inp["A"], inp["lam"],
                                                  inp["angles"] if na else None, th_ref if na else None, layer)
        assert_within(to_host(k), rk, f"m3 prepare k step {step}", bf16_out=kq == "bf16")
        assert_within(to_host(q), rq, f"m3 prepare q step {step}", bf16_out=kq == "bf16")
        for g, r, nm in ((al, ral, "alpha"), (be, rbe, "beta"), (ga, rga, "gamma")):
            assert_within(to_host(g), r, f"m3 prepare {nm} step {step}")
        if na:
            assert_within(to_host(th[layer]), th_ref[layer], f"m3 angle state step {step}")
    for l in (0, 2):
        assert np.array_equal(to_host(th[l]), th_h[l])
    if not na:
        assert np.array_equal(to_host(th), th_h)


def test_m3_prepare_rotates_by_the_stored_angle_at_any_size(cuda_lib):
    """Angles of order 1e4 (a long stream of tokens): the stored f32 angle is
    the oracle's sum rounded once, and k and q are turned by exactly that
    stored angle (the rotation reduces any argument accurately)."""
    m = cuda_lib
    Bsz, H, N, na = 4, 6, 64, 32
    th_h = synth.m3_angle_state(SEED + 3, 1, Bsz, H, na, span=2e4)
    th = to_dev(th_h)
    inp = synth.m3_prepare_inputs(SEED + 3, 0, 0, Bsz, H, N, na)
    k, q, *_ = _m3p_call(m, inp, na, th, 0)
    torch.cuda.synchronize()
    th_sum = th_h.astype(np.float64).copy()
    oracle.m3_prepare(inp["k_in"], inp["q_in"], inp["dt"], inp["A"], inp["lam"], inp["angles"], th_sum, 0)
    got = to_host(th)
    assert np.all(np.abs(got - th_sum) <= np.spacing(np.abs(th_sum).astype(np.float32)).astype(np.float64))
    # the rotation by the stored angle: the oracle from the stored state with no increment
    stored = got.copy()
    rk, rq, *_ = oracle.m3_prepare(inp["k_in"], inp["q_in"], np.zeros((Bsz, H)), inp["A"], inp["lam"],
                                   inp["angles"], stored, 0)
    assert_within(to_host(k), rk, "m3 prepare k at large angles")
    assert_within(to_host(q), rq, "m3 prepare q at large angles")


@pytest.mark.parametrize("P,N,na,dtype", [(64, 64, 32, "f32"), (32, 128, 8, "bf16"), (48, 16, 8, "f32")])
def test_m3_prepare_then_step_decodes_like_the_oracle(cuda_lib, P, N, na, dtype):
    """Six tokens of the Mamba-3 SISO decode on layer 1 of 2, each token the
    preparation (angle state, rotated k and q, alpha / beta / gamma) and then
    the step, against the same chain of oracle calls: y and all four states."""
    m = cuda_lib
    L, layer, Bsz, H = 2, 1, 3, 4
    st_h, ks_h, vs_h = synth.m3_states(SEED + 5, L, Bsz, H, P, N)
    th_h = synth.m3_angle_state(SEED + 5, L, Bsz, H, na)
    st, ks, vs, th = to_dev(st_h), to_dev(ks_h), to_dev(vs_h), to_dev(th_h)
    ref = [a.astype(np.float64).copy() for a in (st_h, ks_h, vs_h, th_h)]
    D_h = synth.normal(SEED + 5, "m3_D", (H,), 1.0)
    D = to_dev(D_h)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    for step in range(6):
        inp = synth.m3_prepare_inputs(SEED + 5, layer, step, Bsz, H, N, na)
        x_h = synth.normal(SEED + 5, "m3_x", (Bsz, H, P), 1.0, dtype, layer, step)
        k, q, al, be, ga = _m3p_call(m, inp, na, th, layer, tdt)
        y = torch.empty((Bsz, H, P), device="cuda")
        m.mamba3_siso_step_batched(y, to_dev(x_h, dtype), k, q, al, be, ga, st, ks, vs, layer, D)
        torch.cuda.synchronize()
        rk, rq, ral, rbe, rga = oracle.m3_prepare(inp["k_in"], inp["q_in"], inp["dt"], inp["A"], inp["lam"],
                                                  inp["angles"], ref[3], layer)
        if dtype == "bf16":  # the step reads k and q as stored; the oracle takes the same values
            rk, rq = to_host(k), to_host(q)
        y_ref = oracle.m3_step(x_h, rk, rq, ral, rbe, rga, ref[0], ref[1], ref[2], layer, D_h)
        assert_within(to_host(y), y_ref, f"m3 decode y token {step}")
        assert_within(to_host(st[layer]), ref[0][layer], f"m3 decode ssm state token {step}")
        assert_within(to_host(ks[layer]), ref[1][layer], f"m3 decode k state token {step}")
        assert_within(to_host(th[layer]), ref[3][layer], f"m3 decode angle state token {step}")
        assert np.array_equal(to_host(vs[layer]), ref[2][layer])
    for s_dev, s_h in ((st, st_h), (ks, ks_h), (vs, vs_h), (th, th_h)):
        assert np.array_equal(to_host(s_dev[0]), s_h[0])
    assert m.mamba_device_faults(clear=True) == 0


# ------------------------------------------ Mamba-3 token in one launch ----

@pytest.mark.parametrize("P,N,na,aligned,y_dtype", [
    (64, 64, 32, True, "f32"), (64, 64, 32, False, "f32"), (32, 128, 12, True, "bf16"), (48, 16, 3, True, "f32"),
    (100, 16, 8, False, "f32"), (64, 32, 0, True, "f32"),
])
def test_m3_fused_token_equals_prepare_then_step_bitwise(cuda_lib, P, N, na, aligned, y_dtype):
    """mamba3_siso_step_fused_batched equals mamba3_siso_step_prepare (f32 k,
    q) followed by mamba3_siso_step_batched, bit for bit, over four tokens: y
    and all four states.  Aligned buffers with n_angles a multiple of 4 take
    the fused copy ring; a k state 4 bytes off a 16-byte boundary, or an odd
    n_angles, the per-(batch, head) kernel."""
    m = cuda_lib
    L, layer, Bsz, H = 2, 1, 3, 5
    st_h, ks_h, vs_h = synth.m3_states(SEED + 7, L, Bsz, H, P, N)
    th_h = synth.m3_angle_state(SEED + 7, L, Bsz, H, max(na, 1))
    D = to_dev(synth.normal(SEED + 7, "m3_D", (H,), 1.0))
    two = [to_dev(a) for a in (st_h, ks_h, vs_h, th_h)]
    one = [to_dev(a) for a in (st_h, ks_h, vs_h, th_h)]
    if not aligned:
        one[1] = _offset_like(one[1])
    ytd = torch.bfloat16 if y_dtype == "bf16" else torch.float32
    for step in range(4):
        inp = synth.m3_prepare_inputs(SEED + 7, layer, step, Bsz, H, N, na)
        d = {n: to_dev(v) for n, v in inp.items()}
        x = to_dev(synth.normal(SEED + 7, "m3_x", (Bsz, H, P), 1.0, "f32", layer, step))
        ang = d["angles"] if na else None
        k, q, al, be, ga = _m3p_call(m, inp, na, two[3], layer)
        y2 = torch.empty((Bsz, H, P), device="cuda", dtype=ytd)
        m.mamba3_siso_step_batched(y2, x, k, q, al, be, ga, two[0], two[1], two[2], layer, D)
        y1 = torch.empty((Bsz, H, P), device="cuda", dtype=ytd)
        m.mamba3_siso_step_fused_batched(y1, x, d["k_in"], d["q_in"], d["dt"], d["A"], d["lam"], ang, one[0], one[1],
                                         one[2], one[3] if na else None, layer, D)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2), f"y differs at token {step}"
        for i, nm in enumerate(("ssm", "k", "v", "angle")):
            assert torch.equal(one[i], two[i]), f"{nm} state differs at token {step}"
    assert m.mamba_device_faults(clear=True) == 0


@pytest.mark.parametrize("P,N,na,x_dtype", [(64, 64, 32, "bf16"), (32, 16, 8, "f32"), (16, 128, 64, "bf16")])
def test_m3_fused_tokens_decode_like_the_oracle(cuda_lib, P, N, na, x_dtype):
    """Five Mamba-3 SISO tokens, each one fused launch, against the chain of
    oracle calls (the preparation, then the step): y and all four states."""
    m = cuda_lib
    L, layer, Bsz, H = 2, 0, 4, 3
    st_h, ks_h, vs_h = synth.m3_states(SEED + 9, L, Bsz, H, P, N)
    th_h = synth.m3_angle_state(SEED + 9, L, Bsz, H, na)
    st, ks, vs, th = to_dev(st_h), to_dev(ks_h), to_dev(vs_h), to_dev(th_h)
    ref = [a.astype(np.float64).copy() for a in (st_h, ks_h, vs_h, th_h)]
    D_h = synth.normal(SEED + 9, "m3_D", (H,), 1.0)
    for step in range(5):
        inp = synth.m3_prepare_inputs(SEED + 9, layer, step, Bsz, H, N, na)
        d = {n: to_dev(v) for n, v in inp.items()}
        x_h = synth.normal(SEED + 9, "m3_x", (Bsz, H, P), 1.0, x_dtype, layer, step)
        y = torch.empty((Bsz, H, P), device="cuda")
        m.mamba3_siso_step_fused_batched(y, to_dev(x_h, x_dtype), d["k_in"], d["q_in"], d["dt"], d["A"], d["lam"],
                                         d["angles"], st, ks, vs, th, layer, to_dev(D_h))
        torch.cuda.synchronize()
        rk, rq, ral, rbe, rga = oracle.m3_prepare(inp["k_in"], inp["q_in"], inp["dt"], inp["A"], inp["lam"],
                                                  inp["angles"], ref[3], layer)
        y_ref = oracle.m3_step(x_h, rk, rq, ral, rbe, rga, ref[0], ref[1], ref[2], layer, D_h)
        assert_within(to_host(y), y_ref, f"m3 fused y token {step}")
        assert_within(to_host(st[layer]), ref[0][layer], f"m3 fused ssm state token {step}")
        assert_within(to_host(ks[layer]), ref[1][layer], f"m3 fused k state token {step}")
        assert_within(to_host(th[layer]), ref[3][layer], f"m3 fused angle state token {step}")
        assert np.array_equal(to_host(vs[layer]), ref[2][layer])
    for s_dev, s_h in ((st, st_h), (ks, ks_h), (vs, vs_h), (th, th_h)):
        assert np.array_equal(to_host(s_dev[1]), s_h[1])
    assert m.mamba_device_faults(clear=True) == 0


@pytest.mark.parametrize("P,N,na,aligned", [(64, 64, 32, True), (48, 16, 3, True), (32, 32, 8, False)])
def test_m3_decode_graph_replays_the_direct_calls_bitwise(cuda_lib, P, N, na, aligned):
    """A recorded n_steps x n_layers Mamba-3 decode graph, launched twice, gives
    the same y and four states, bit for bit, as the same one-launch tokens
    called directly (both step kernels: a k state 4 bytes off a 16-byte
    boundary takes the per-(batch, head) one)."""
    m = cuda_lib
    L, S, Bsz, H = 3, 2, 4, 5
    st_h, ks_h, vs_h = synth.m3_states(SEED + 11, L, Bsz, H, P, N)
    th_h = synth.m3_angle_state(SEED + 11, L, Bsz, H, na)
    g_states = [to_dev(a) for a in (st_h, ks_h, vs_h, th_h)]
    d_states = [to_dev(a) for a in (st_h, ks_h, vs_h, th_h)]
    if not aligned:
        g_states[1], d_states[1] = _offset_like(g_states[1]), _offset_like(d_states[1])
    D = [to_dev(synth.normal(SEED + 11, "m3_D", (H,), 1.0, layer=l)) for l in range(L)]
    io = []
    for s in range(S):
        row = []
        for l in range(L):
            inp = {k: to_dev(v) for k, v in synth.m3_prepare_inputs(SEED + 11, l, s, Bsz, H, N, na).items()}
            inp["x"] = to_dev(synth.normal(SEED + 11, "m3_x", (Bsz, H, P), 1.0, "f32", l, s))
            inp["y"] = torch.empty((Bsz, H, P), device="cuda")
            row.append(inp)
        io.append(row)
    with m.Mamba3DecodeGraph(io, *g_states, D=D) as g:
        assert g.kernels == S * L
        for rep in range(2):
            g.launch()
            torch.cuda.synchronize()
            ys = {}
            for s in range(S):
                for l in range(L):
                    q = io[s][l]
                    ys[s, l] = torch.empty((Bsz, H, P), device="cuda")
                    m.mamba3_siso_step_fused_batched(ys[s, l], q["x"], q["k_in"], q["q_in"], q["dt"], q["A"],
                                                     q["lam"], q["angles"], *d_states, l, D[l])
            torch.cuda.synchronize()
            for (s, l), y in ys.items():
                assert torch.equal(y, io[s][l]["y"]), f"y differs (launch {rep}, token {s}, layer {l})"
            for i, nm in enumerate(("ssm", "k", "v", "angle")):
                assert torch.equal(g_states[i], d_states[i]), f"{nm} state differs after launch {rep}"
    assert m.mamba_device_faults(clear=True) == 0



def test_m3_fused_token_equals_prepare_then_step_at_the_decode_shape(cuda_lib):
    """At the bench's decode shape (batch 128 x 24 heads, headdim 64, d_state 64,
    32 rotated pairs) every copy-ring CTA walks several (batch, head) tiles and
    reuses its stages: the one-launch token still equals the preparation + step
    bit for bit over two tokens, and the other layer's slabs stay untouched."""
    m = cuda_lib
    L, layer, Bsz, H, P, N, na = 2, 1, 128, 24, 64, 64, 32
    st_h, ks_h, vs_h = synth.m3_states(SEED + 13, L, Bsz, H, P, N)
    th_h = synth.m3_angle_state(SEED + 13, L, Bsz, H, na)
    two = [to_dev(a) for a in (st_h, ks_h, vs_h, th_h)]
    one = [to_dev(a) for a in (st_h, ks_h, vs_h, th_h)]
    D = to_dev(synth.normal(SEED + 13, "m3_D", (H,), 1.0))
    for step in range(2):
        inp = synth.m3_prepare_inputs(SEED + 13, layer, step, Bsz, H, N, na)
        d = {n: to_dev(v) for n, v in inp.items()}
        x = to_dev(synth.normal(SEED + 13, "m3_x", (Bsz, H, P), 1.0, "f32", layer, step))
        k, q, al, be, ga = _m3p_call(m, inp, na, two[3], layer)
        y2 = torch.empty((Bsz, H, P), device="cuda")
        m.mamba3_siso_step_batched(y2, x, k, q, al, be, ga, two[0], two[1], two[2], layer, D)
        y1 = torch.empty((Bsz, H, P), device="cuda")
        m.mamba3_siso_step_fused_batched(y1, x, d["k_in"], d["q_in"], d["dt"], d["A"], d["lam"], d["angles"],
                                         *one, layer, D)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2), f"y differs at token {step}"
        for i, nm in enumerate(("ssm", "k", "v", "angle")):
            assert torch.equal(one[i], two[i]), f"{nm} state differs at token {step}"
    for i, a in enumerate((st_h, ks_h, vs_h, th_h)):
        assert np.array_equal(to_host(one[i][0]), a[0])
    assert m.mamba_device_faults(clear=True) == 0
