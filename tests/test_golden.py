"""Hand-derived worked examples (tests/golden/*.json) against the oracle (CPU)
and against the kernels (GPU).

The expected values are fixed by the mathematics of the definitions, derived by
hand in each file; neither the oracle nor the CUDA path produced them.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit

import oracle

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
LN2 = math.log(2.0)


def _load(name):
    with open(os.path.join(HERE, name)) as f:
        return json.load(f)


def _scan_case():
    g = _load("scan_worked_example.json")
    i, e = g["inputs"], g["expected"]
    T = len(i["u"])
    arr = lambda v: np.asarray(v, np.float64)
    inp = dict(u=arr(i["u"]).reshape(1, T, 1), dt=arr(i["dt"]).reshape(1, T, 1), Bm=arr(i["B"]).reshape(1, T, 2),
               Cm=arr(i["C"]).reshape(1, T, 2), A_log=arr(i["A_log"]), D=arr(i["D"]), dt_bias=arr(i["dt_bias"]),
               state_in=arr(i["state_in"]).reshape(1, 1, 2))
    y = (arr(e["y_ln2_coef"]) * LN2 + arr(e["y_const"])).reshape(1, T, 1)
    s = (arr(e["state_out_ln2_coef"]) * LN2).reshape(1, 1, 2)
    return inp, y, s


def _conv_case():
    g = _load("conv_worked_example.json")
    i, e = g["inputs"], g["expected"]
    T = len(i["x"])
    pre = np.asarray(e["pre"], np.float64)
    inp = dict(x=np.asarray(i["x"], np.float64).reshape(1, T, 1), w=np.asarray(i["w"], np.float64),
               bias=np.asarray(i["bias"], np.float64), state_in=np.asarray(i["state_in"], np.float64).reshape(1, 1, 3))
    u = (pre * expit(pre)).reshape(1, T, 1)  # SiLU from scipy, independent of both sides
    return inp, u, np.asarray(e["state_out"], np.float64).reshape(1, 1, 3)


def _m3_case(N=16):
    g = _load("m3_worked_example.json")
    i, e = g["inputs"], g["expected"]
    pad = lambda v: np.concatenate([np.asarray(v, np.float64), np.zeros(N - len(v))])
    inp = dict(h=pad(i["h"]).reshape(1, 1, 1, 1, N), k_prev=pad(i["k_prev"]).reshape(1, 1, 1, N),
               v_prev=np.asarray(i["v_prev"], np.float64).reshape(1, 1, 1, 1),
               x=np.asarray(i["x"], np.float64).reshape(1, 1, 1), k=pad(i["k"]).reshape(1, 1, N),
               q=pad(i["q"]).reshape(1, 1, N), alpha=np.full((1, 1), i["alpha"]), beta=np.full((1, 1), i["beta"]),
               gamma=np.full((1, 1), i["gamma"]), D=np.full(1, i["D"]))
    exp = dict(h=pad(e["h"]).reshape(1, 1, 1, 1, N), y=np.asarray(e["y"], np.float64).reshape(1, 1, 1),
               k_state=pad(e["k_state"]).reshape(1, 1, 1, N), v_state=np.asarray(e["v_state"]).reshape(1, 1, 1, 1))
    return inp, exp


# ------------------------------------------------------------------ oracle ----

def test_oracle_scan_worked_example():
    inp, y, s = _scan_case()
    yo, so = oracle.selective_scan_prefill(inp["u"], inp["dt"], inp["Bm"], inp["Cm"], inp["A_log"], inp["D"],
                                           inp["dt_bias"], None, inp["state_in"])
    np.testing.assert_allclose(yo, y, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(so, s, rtol=1e-14, atol=1e-15)


def test_oracle_conv_worked_example():
    inp, u, st = _conv_case()
    uo, so = oracle.conv1d_silu_prefill(inp["x"], inp["w"], inp["bias"], inp["state_in"])
    np.testing.assert_allclose(uo, u, rtol=1e-14, atol=1e-15)
    assert np.array_equal(so, st)


def test_oracle_m3_worked_example():
    inp, exp = _m3_case()
    h, ks, vs = inp["h"].copy(), inp["k_prev"].copy(), inp["v_prev"].copy()
    y = oracle.m3_step(inp["x"], inp["k"], inp["q"], inp["alpha"], inp["beta"], inp["gamma"], h, ks, vs, 0,
                       D=inp["D"])
    assert np.array_equal(y, exp["y"]) and np.array_equal(h, exp["h"])
    assert np.array_equal(ks, exp["k_state"]) and np.array_equal(vs, exp["v_state"])


# --------------------------------------------------------------------- GPU ----

def _within(got, ref):
    got = np.asarray(got, np.float64)
    assert np.all(np.abs(got - ref) <= 2e-4 * (1.0 + np.abs(ref))), (got, ref)


@pytest.mark.gpu
def test_kernels_scan_worked_example(cuda_lib):
    import torch

    m = cuda_lib
    inp, y_ref, s_ref = _scan_case()
    d = lambda a: torch.tensor(np.asarray(a, np.float32), device="cuda")
    y = torch.empty((1, 4, 1), device="cuda")
    s = torch.empty((1, 1, 2), device="cuda")
    m.mamba_selective_scan_prefill(y, d(inp["u"]), d(inp["dt"]), d(inp["Bm"]), d(inp["Cm"]), d(inp["A_log"]),
                                   d(inp["D"]), d(inp["dt_bias"]), None, d(inp["state_in"]), s)
    # the same tokens as four batched T=1 steps on a one-layer state
    st = d(inp["state_in"]).reshape(1, 1, 1, 2).contiguous()
    ys = []
    for t in range(4):
        yt = torch.empty((1, 1), device="cuda")
        m.mamba_ssm_step_batched(yt, d(inp["u"][:, t]), d(inp["dt"][:, t]), d(inp["Bm"][:, t]), d(inp["Cm"][:, t]),
                                 st, 0, d(inp["A_log"]), d(inp["D"]), d(inp["dt_bias"]), None)
        ys.append(yt)
    torch.cuda.synchronize()
    _within(y.cpu().numpy(), y_ref)
    _within(s.cpu().numpy(), s_ref)
    _within(torch.stack(ys, 1).cpu().numpy().reshape(1, 4, 1), y_ref)
    _within(st.cpu().numpy().reshape(1, 1, 2), s_ref)


@pytest.mark.gpu
def test_kernels_conv_worked_example(cuda_lib):
    import torch

    m = cuda_lib
    inp, u_ref, st_ref = _conv_case()
    d = lambda a: torch.tensor(np.asarray(a, np.float32), device="cuda")
    u = torch.empty((1, 2, 1), device="cuda")
    so = torch.empty((1, 1, 3), device="cuda")
    m.mamba_conv1d_silu_prefill(u, d(inp["x"]), d(inp["w"]), d(inp["bias"]), d(inp["state_in"]), so)
    cs = d(inp["state_in"]).reshape(1, 1, 1, 3).contiguous()
    us = []
    for t in range(2):
        ut = torch.empty((1, 1), device="cuda")
        m.mamba_conv1d_silu_step(ut, d(inp["x"][:, t]), cs, 0, d(inp["w"]), d(inp["bias"]))
        us.append(ut)
    torch.cuda.synchronize()
    _within(u.cpu().numpy(), u_ref)
    assert np.array_equal(so.cpu().numpy(), st_ref)
    _within(torch.stack(us, 1).cpu().numpy().reshape(1, 2, 1), u_ref)
    assert np.array_equal(cs.cpu().numpy().reshape(1, 1, 3), st_ref)


def _m3p_case():
    g = _load("m3_prepare_worked_example.json")
    i, e = g["inputs"], g["expected"]
    arr = lambda v, *shape: np.asarray(v, np.float64).reshape(*shape)
    inp = dict(k_in=arr(i["k_in"], 1, 1, 16), q_in=arr(i["q_in"], 1, 1, 16), dt=arr(i["dt"], 1, 1),
               A=arr(i["A"], 1, 1), lam=arr(i["lam"], 1, 1), angles=arr(i["angles"], 1, 2),
               angle_state=arr(i["angle_state"], 1, 1, 1, 2))
    exp = dict(angle_state=arr(e["angle_state"], 1, 1, 2), k=arr(e["k"], 1, 1, 16), q=arr(e["q"], 1, 1, 16),
               alpha=e["alpha_times_e"] / math.e, beta=e["beta_times_e"] / math.e, gamma=e["gamma"])
    return inp, exp


def test_oracle_m3_prepare_worked_example():
    inp, exp = _m3p_case()
    st = inp["angle_state"].copy()
    k, q, al, be, ga = oracle.m3_prepare(inp["k_in"], inp["q_in"], inp["dt"], inp["A"], inp["lam"], inp["angles"],
                                         st, 0)
    np.testing.assert_allclose(st[0], exp["angle_state"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(k, exp["k"], rtol=0, atol=1e-15)
    np.testing.assert_allclose(q, exp["q"], rtol=0, atol=1e-15)
    np.testing.assert_allclose([al[0, 0], be[0, 0], ga[0, 0]], [exp["alpha"], exp["beta"], exp["gamma"]],
                               rtol=1e-15, atol=0)


@pytest.mark.gpu
def test_kernels_m3_prepare_worked_example(cuda_lib):
    """The preparation kernel and the one-launch token (whose k state receives
    the turned k) against the hand-derived values."""
    import torch

    m = cuda_lib
    inp, exp = _m3p_case()
    d = lambda a: torch.tensor(np.asarray(a, np.float32), device="cuda").contiguous()
    st = d(inp["angle_state"])
    k, q = torch.empty((1, 1, 16), device="cuda"), torch.empty((1, 1, 16), device="cuda")
    al, be, ga = (torch.empty((1, 1), device="cuda") for _ in range(3))
    m.mamba3_siso_step_prepare(k, q, al, be, ga, d(inp["k_in"]), d(inp["q_in"]), d(inp["dt"]), d(inp["A"]),
                               d(inp["lam"]), d(inp["angles"]), st, 0)
    torch.cuda.synchronize()
    _within(st.cpu().numpy()[0], exp["angle_state"])
    _within(k.cpu().numpy(), exp["k"])
    _within(q.cpu().numpy(), exp["q"])
    _within(np.array([al.item(), be.item(), ga.item()]), np.array([exp["alpha"], exp["beta"], exp["gamma"]]))
    # the same token in one launch: the k state receives the turned k
    h, ks, vs = (torch.zeros(s, device="cuda") for s in ((1, 1, 1, 1, 16), (1, 1, 1, 16), (1, 1, 1, 1)))
    st2 = d(inp["angle_state"])
    y = torch.empty((1, 1, 1), device="cuda")
    m.mamba3_siso_step_fused_batched(y, torch.ones((1, 1, 1), device="cuda"), d(inp["k_in"]), d(inp["q_in"]),
                                     d(inp["dt"]), d(inp["A"]), d(inp["lam"]), d(inp["angles"]), h, ks, vs, st2, 0)
    torch.cuda.synchronize()
    _within(ks.cpu().numpy()[0], exp["k"])
    _within(st2.cpu().numpy()[0], exp["angle_state"])


@pytest.mark.gpu
def test_kernels_m3_worked_example(cuda_lib):
    import torch

    m = cuda_lib
    inp, exp = _m3_case()
    d = lambda a: torch.tensor(np.asarray(a, np.float32), device="cuda").contiguous()
    h, ks, vs = d(inp["h"]), d(inp["k_prev"]), d(inp["v_prev"])
    y = torch.empty((1, 1, 1), device="cuda")
    m.mamba3_siso_step_batched(y, d(inp["x"]), d(inp["k"]), d(inp["q"]), d(inp["alpha"]), d(inp["beta"]),
                               d(inp["gamma"]), h, ks, vs, 0, d(inp["D"]))
    torch.cuda.synchronize()
    _within(y.cpu().numpy(), exp["y"])
    _within(h.cpu().numpy(), exp["h"])
    assert np.array_equal(ks.cpu().numpy(), exp["k_state"]) and np.array_equal(vs.cpu().numpy(), exp["v_state"])
