"""Pins for the f64 CPU oracle, independent of the oracle's own code.

Each test checks the oracle against something the pages or the mathematics fix
(mamba-rs inference.rs / prefill.rs source views; the Mamba-1 recurrence):
library special functions, the unrolled closed form of the recurrence, the
geometric series for d_state = 1, continuation, T=1 prefill == step,
delta -> 0, A -> -inf, linearity in (u, h0), row independence, and the conv's
impulse response and shift-register state.  They are chosen so that a dropped
term, a wrong sign, an off-by-one index or a transposed operand in the oracle
fails at least one of them.
"""
import numpy as np
import pytest
from scipy.special import expit

import oracle
from selective_state_space_conv1d_gb300 import synth

RNG = np.random.default_rng(1234)


def _rand_scan_case(Bsz=2, T=24, Di=5, N=4, gate=True, state=True, seed=0):
    r = np.random.default_rng(seed)
    c = dict(
        u=r.standard_normal((Bsz, T, Di)),
        dt=0.3 * r.standard_normal((Bsz, T, Di)),
        Bm=r.standard_normal((Bsz, T, N)),
        Cm=r.standard_normal((Bsz, T, N)),
        A_log=r.uniform(-1.0, 1.5, (Di, N)),
        D=r.standard_normal(Di),
        dt_bias=r.uniform(-3.0, 0.5, Di),
        z=r.standard_normal((Bsz, T, Di)) if gate else None,
        state_in=r.standard_normal((Bsz, Di, N)) if state else None,
    )
    return c


def _unrolled(c):
    """Brute force: y_t = sum_{s<=t} C_t (prod_{r=s+1..t} exp(d_r A)) d_s B_s u_s
    + C_t (prod_{r<=t} exp(d_r A)) h0 + D u_t, gated; h_T likewise.  O(T^2 N)."""
    u, dt, Bm, Cm = c["u"], c["dt"], c["Bm"], c["Cm"]
    Bsz, T, Di = u.shape
    N = Bm.shape[2]
    A = -np.exp(c["A_log"])
    delta = np.logaddexp(0.0, dt + c["dt_bias"][None, None, :])  # library softplus
    h0 = c["state_in"] if c["state_in"] is not None else np.zeros((Bsz, Di, N))
    y = np.zeros((Bsz, T, Di))
    hT = np.zeros((Bsz, Di, N))
    for b in range(Bsz):
        for ch in range(Di):
            dA = np.exp(delta[b, :, ch][:, None] * A[ch][None, :])  # [T, N]
            for t in range(T + 1):
                # state after tokens 0..t-1 (t == T gives the final state)
                h = np.prod(dA[:t], axis=0) * h0[b, ch]
                for s in range(t):
                    h = h + np.prod(dA[s + 1:t], axis=0) * delta[b, s, ch] * Bm[b, s] * u[b, s, ch]
                if t < T:
                    # y_t uses the state after token t
                    ht = np.prod(dA[: t + 1], axis=0) * h0[b, ch]
                    for s in range(t + 1):
                        ht = ht + np.prod(dA[s + 1:t + 1], axis=0) * delta[b, s, ch] * Bm[b, s] * u[b, s, ch]
                    yt = Cm[b, t] @ ht + c["D"][ch] * u[b, t, ch]
                    if c["z"] is not None:
                        yt *= c["z"][b, t, ch] * expit(c["z"][b, t, ch])
                    y[b, t, ch] = yt
                else:
                    hT[b, ch] = h
    return y, hT


def _scan(c, **over):
    c = dict(c, **over)
    return oracle.selective_scan_prefill(
        c["u"], c["dt"], c["Bm"], c["Cm"], c["A_log"], D=c["D"], dt_bias=c["dt_bias"],
        z=c["z"], state_in=c["state_in"], nthreads=2)


# ---------------------------------------------------------------- functions --

def test_softplus_matches_library_and_identity():
    for v in [-750.0, -200.0, -40.0, -5.0, -1e-3, 0.0, 1e-8, 0.7, 5.0, 30.0, 700.0]:
        assert oracle.softplus(v) == pytest.approx(np.logaddexp(0.0, v), rel=1e-15, abs=1e-300)
        # softplus(v) - softplus(-v) = v
        assert oracle.softplus(v) - oracle.softplus(-v) == pytest.approx(v, rel=1e-14, abs=1e-14)
    assert oracle.softplus(0.0) == pytest.approx(np.log(2.0), rel=1e-16)


def test_silu_matches_library():
    for x in [-700.0, -30.0, -1.0, 0.0, 0.5, 3.0, 40.0]:
        assert oracle.silu(x) == pytest.approx(x * expit(x), rel=1e-15, abs=1e-300)
    assert oracle.silu(0.0) == 0.0


# --------------------------------------------------------------------- scan --

@pytest.mark.parametrize("gate,state", [(True, True), (False, False), (True, False)])
def test_scan_matches_unrolled_brute_force(gate, state):
    c = _rand_scan_case(Bsz=2, T=20, Di=3, N=4, gate=gate, state=state, seed=7)
    y, hT = _scan(c)
    y_ref, h_ref = _unrolled(c)
    np.testing.assert_allclose(y, y_ref, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(hT, h_ref, rtol=1e-11, atol=1e-12)


def test_scan_d_state_one_closed_form_geometric_series():
    # constant delta, B, u; N = 1:  h_t = a^t h0 + b (1 - a^t) / (1 - a)
    T, Di = 50, 3
    A_log = np.array([[0.0], [0.7], [-0.4]])
    dt_bias = np.array([0.2, -1.0, 0.0])
    dtv, uv, Bv, Cv, h0 = 0.05, 0.8, -1.3, 0.6, np.array([0.4, -2.0, 1.5])
    Dv = np.array([1.0, 0.5, -0.25])
    u = np.full((1, T, Di), uv)
    y, hT = oracle.selective_scan_prefill(
        u, np.full((1, T, Di), dtv), np.full((1, T, 1), Bv), np.full((1, T, 1), Cv), A_log,
        D=Dv, dt_bias=dt_bias, state_in=h0.reshape(1, Di, 1), nthreads=1)
    delta = np.log1p(np.exp(dtv + dt_bias))
    a = np.exp(-delta * np.exp(A_log[:, 0]))
    bb = delta * Bv * uv
    t = np.arange(1, T + 1)[:, None]
    h = a ** t * h0 + bb * (1 - a ** t) / (1 - a)
    np.testing.assert_allclose(y[0], Cv * h + Dv * uv, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(hT[0, :, 0], h[-1], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("T1", [1, 7, 16])
def test_scan_continuation_is_bitwise(T1):
    c = _rand_scan_case(Bsz=2, T=29, Di=4, N=8, seed=3)
    y, hT = _scan(c)
    sl = lambda a, s: None if a is None else a[:, s]
    c1 = {k: (sl(v, slice(0, T1)) if k in ("u", "dt", "Bm", "Cm", "z") else v) for k, v in c.items()}
    c2 = {k: (sl(v, slice(T1, None)) if k in ("u", "dt", "Bm", "Cm", "z") else v) for k, v in c.items()}
    y1, h1 = _scan(c1)
    c2["state_in"] = h1
    y2, h2 = _scan(c2)
    assert np.array_equal(np.concatenate([y1, y2], axis=1), y)
    assert np.array_equal(h2, hT)


@pytest.mark.parametrize("parts", [2, 3, 5])
def test_scan_split_along_T_and_folded_equals_the_whole_scan(parts):
    """The decomposition the T-split route rests on, in exact arithmetic: scan
    each part from a zero state, take each part's total decay exp(A * sum of
    its deltas), fold carry_{j+1} = decay_j * carry_j + end_j from carry_0 =
    h0, and rescan each part from its carry.  That reproduces the whole scan's
    y and final state (f64, to rounding)."""
    c = _rand_scan_case(Bsz=2, T=37, Di=3, N=5, seed=21)
    y_all, h_all = _scan(c)
    T = c["u"].shape[1]
    bounds = np.linspace(0, T, parts + 1).astype(int)
    A = -np.exp(c["A_log"])
    carry = c["state_in"].copy()
    ys = []
    for j in range(parts):
        sl = slice(bounds[j], bounds[j + 1])
        part = {k: (v[:, sl] if k in ("u", "dt", "Bm", "Cm", "z") else v) for k, v in c.items()}
        _, end = _scan(part, state_in=None)                       # this part from a zero state
        delta = np.logaddexp(0.0, part["dt"] + c["dt_bias"])      # [B, t, Di]
        decay = np.exp(A[None] * delta.sum(axis=1)[:, :, None])    # [B, Di, N]
        y_j, h_j = _scan(part, state_in=carry)                    # the rescan from the carry-in
        ys.append(y_j)
        np.testing.assert_allclose(h_j, decay * carry + end, rtol=1e-12, atol=1e-13)
        carry = decay * carry + end
    np.testing.assert_allclose(np.concatenate(ys, axis=1), y_all, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(carry, h_all, rtol=1e-12, atol=1e-13)


def test_scan_T1_prefill_equals_step_bitwise():
    c = _rand_scan_case(Bsz=3, T=1, Di=6, N=16, seed=11)
    y, hT = _scan(c)
    L = 3
    states = np.random.default_rng(5).standard_normal((L, 3, 6, 16))
    states[1] = c["state_in"]
    before = states.copy()
    ys = oracle.ssm_step(c["u"][:, 0], c["dt"][:, 0], c["Bm"][:, 0], c["Cm"][:, 0], states, 1,
                         c["A_log"], D=c["D"], dt_bias=c["dt_bias"], z=c["z"][:, 0])
    assert np.array_equal(ys, y[:, 0])
    assert np.array_equal(states[1], hT)
    assert np.array_equal(states[0], before[0]) and np.array_equal(states[2], before[2])


def test_scan_delta_to_zero_keeps_state():
    c = _rand_scan_case(Bsz=1, T=10, Di=4, N=4, gate=False, state=True, seed=2)
    c["dt"] = np.zeros_like(c["dt"])
    c["dt_bias"] = np.full(4, -800.0)  # softplus(-800) == 0 in f64
    y, hT = _scan(c)
    assert np.array_equal(hT, c["state_in"])
    expect = np.einsum("btn,bcn->btc", c["Cm"], c["state_in"]) + c["D"] * c["u"]
    np.testing.assert_allclose(y, expect, rtol=1e-14, atol=1e-14)
    # zero initial state: y = D * u exactly, state stays zero
    y0, h0 = _scan(c, state_in=None)
    assert np.array_equal(h0, np.zeros_like(h0))
    np.testing.assert_array_equal(y0, c["D"] * c["u"])


def test_scan_A_to_minus_infinity_is_memoryless():
    c = _rand_scan_case(Bsz=2, T=12, Di=3, N=4, gate=False, state=True, seed=4)
    c["A_log"] = np.full((3, 4), 80.0)  # A = -exp(80): exp(delta A) == 0
    y, hT = _scan(c)
    delta = np.logaddexp(0.0, c["dt"] + c["dt_bias"])
    h = delta[..., None] * c["Bm"][:, :, None, :] * c["u"][..., None]  # [B, T, Di, N]
    np.testing.assert_allclose(y, np.einsum("btn,btcn->btc", c["Cm"], h) + c["D"] * c["u"],
                               rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(hT, h[:, -1], rtol=1e-13, atol=1e-14)


def test_scan_is_linear_in_u_and_h0():
    c1 = _rand_scan_case(Bsz=1, T=15, Di=3, N=4, gate=False, state=True, seed=21)
    c2 = _rand_scan_case(Bsz=1, T=15, Di=3, N=4, gate=False, state=True, seed=22)
    c2.update({k: c1[k] for k in ("dt", "Bm", "Cm", "A_log", "D", "dt_bias")})
    al, be = 0.7, -1.9
    y1, h1 = _scan(c1)
    y2, h2 = _scan(c2)
    y3, h3 = _scan(c1, u=al * c1["u"] + be * c2["u"], state_in=al * c1["state_in"] + be * c2["state_in"])
    np.testing.assert_allclose(y3, al * y1 + be * y2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(h3, al * h1 + be * h2, rtol=1e-12, atol=1e-12)


def test_scan_rows_are_independent_and_permute():
    c = _rand_scan_case(Bsz=3, T=9, Di=6, N=4, seed=8)
    y, hT = _scan(c)
    perm = np.array([3, 0, 5, 1, 4, 2])
    cp = dict(c)
    for k in ("u", "dt", "z"):
        cp[k] = c[k][:, :, perm]
    for k in ("D", "dt_bias"):
        cp[k] = c[k][perm]
    cp["A_log"] = c["A_log"][perm]
    cp["state_in"] = c["state_in"][:, perm]
    yp, hp = _scan(cp)
    assert np.array_equal(yp, y[:, :, perm]) and np.array_equal(hp, hT[:, perm])
    # batch row 1 run alone
    c1 = {k: (v[1:2] if k in ("u", "dt", "z", "Bm", "Cm", "state_in") else v) for k, v in c.items()}
    y1, h1 = _scan(c1)
    assert np.array_equal(y1[0], y[1]) and np.array_equal(h1[0], hT[1])


def test_scan_gate_special_values():
    c = _rand_scan_case(Bsz=1, T=6, Di=2, N=4, gate=True, state=True, seed=9)
    y_nogate, _ = _scan(c, z=None)
    y_zero, _ = _scan(c, z=np.zeros_like(c["z"]))
    assert np.array_equal(y_zero, np.zeros_like(y_zero))
    y_big, _ = _scan(c, z=np.full_like(c["z"], 800.0))  # SiLU(800) == 800 exactly
    np.testing.assert_array_equal(y_big, y_nogate * 800.0)


# --------------------------------------------------------------------- conv --

def test_conv_impulse_response():
    K, Di, T, t0 = 4, 3, 12, 5
    w = RNG.uniform(-0.5, 0.5, (Di, K))
    bias = np.array([0.0, 0.3, -0.2])
    x = np.zeros((1, T, Di))
    x[0, t0] = 1.0
    u, st = oracle.conv1d_silu_prefill(x, w, bias, None, nthreads=1)
    pre = np.tile(bias, (T, 1))
    for j in range(K):
        pre[t0 + j] = w[:, K - 1 - j] + bias  # the newest tap w[:, K-1] meets x_t
    np.testing.assert_allclose(u[0], pre * expit(pre), rtol=1e-15, atol=1e-300)


def test_conv_constant_input_and_state_semantics():
    K, Di, T = 4, 2, 9
    w = RNG.uniform(-0.5, 0.5, (Di, K))
    bias = np.array([0.1, -0.4])
    x = np.full((1, T, Di), 0.75)
    u, st = oracle.conv1d_silu_prefill(x, w, bias, None, nthreads=1)
    pre = bias + 0.75 * w.sum(1)
    np.testing.assert_allclose(u[0, K - 1:], np.tile(pre * expit(pre), (T - K + 1, 1)), rtol=1e-15)
    assert np.array_equal(st[0], np.full((Di, K), 0.75))


@pytest.mark.parametrize("T", [1, 2, 3, 4, 7])
def test_conv_state_out_is_last_K_of_state_then_inputs(T):
    K, Di = 4, 3
    w = RNG.uniform(-0.5, 0.5, (Di, K))
    s0 = RNG.standard_normal((2, Di, K))
    x = RNG.standard_normal((2, T, Di))
    u, st = oracle.conv1d_silu_prefill(x, w, None, s0, nthreads=1)
    seq = np.concatenate([s0, np.transpose(x, (0, 2, 1))], axis=2)  # [B, Di, K+T]
    assert np.array_equal(st, seq[:, :, T:T + K])
    # every output uses slots 1..K-1 of the state then the inputs: pre_t = sum_k w_k seq[t+1+k]
    for t in range(T):
        pre = np.einsum("ck,bck->bc", w, seq[:, :, t + 1:t + 1 + K])
        np.testing.assert_allclose(u[:, t], pre * expit(pre), rtol=1e-14, atol=1e-15)


def test_conv_continuation_and_step_bitwise():
    K, Di, T = 4, 5, 13
    w = RNG.uniform(-0.5, 0.5, (Di, K))
    bias = RNG.standard_normal(Di)
    s0 = RNG.standard_normal((2, Di, K))
    x = RNG.standard_normal((2, T, Di))
    u, st = oracle.conv1d_silu_prefill(x, w, bias, s0)
    u1, st1 = oracle.conv1d_silu_prefill(x[:, :6], w, bias, s0)
    u2, st2 = oracle.conv1d_silu_prefill(x[:, 6:], w, bias, st1)
    assert np.array_equal(np.concatenate([u1, u2], 1), u) and np.array_equal(st2, st)
    # T token steps on layer 1 of a 2-layer state equal the prefill
    states = np.zeros((2, 2, Di, K))
    states[1] = s0
    for t in range(T):
        ut = oracle.conv1d_silu_step(x[:, t], states, 1, w, bias)
        assert np.array_equal(ut, u[:, t])
    assert np.array_equal(states[1], st) and np.array_equal(states[0], np.zeros((2, Di, K)))


# ---------------------------------------------------------------- workloads --

def test_tiny_workload_runs_and_is_finite():
    wl = synth.WORKLOADS[0]
    p = synth.mixer_params(wl.seed, wl.d_inner, wl.d_state, wl.d_conv)
    a = synth.prefill_inputs(wl.seed, wl.batch, wl.seqlen, wl.d_inner, wl.d_state)
    u, cst = oracle.conv1d_silu_prefill(a["x"], p["conv_w"], p["conv_b"], None)
    y, sst = oracle.selective_scan_prefill(u, a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                           p["dt_bias"], a["z"], None)
    assert np.isfinite(y).all() and np.isfinite(sst).all() and np.isfinite(cst).all()
    # delta lies in the log-uniform range widened by dt ~ N(0, 0.1^2)
    delta = np.logaddexp(0.0, a["dt"].astype(np.float64) + p["dt_bias"])
    assert 1e-4 < delta.min() and delta.max() < 0.3


# ---------------------------------------------------------------- Mamba-3 step ----
# Pins of oracle.m3_step (Mamba-3 SISO trapezoidal step, mamba-rs 0.2.1
# mamba3_siso/gpu/inference.rs: state buffers and the F6 m3_step_fwd launch).

def _m3_case(rng, B=2, H=3, P=4, N=5, L=2):
    st = np.ascontiguousarray(rng.normal(size=(L, B, H, P, N)))
    ks = np.ascontiguousarray(rng.normal(size=(L, B, H, N)))
    vs = np.ascontiguousarray(rng.normal(size=(L, B, H, P)))
    return st, ks, vs


def test_m3_constant_inputs_follow_the_geometric_series():
    """Constant k, x (and the states' previous k, v equal to them): after T steps
    h_T = a^T h0 + (b + g) k x (1 - a^T) / (1 - a), y_T = q . h_T + D x."""
    rng = np.random.default_rng(31)
    B, H, P, N, T = 2, 3, 4, 5, 37
    k, q, x = rng.normal(size=(B, H, N)), rng.normal(size=(B, H, N)), rng.normal(size=(B, H, P))
    a = rng.uniform(0.5, 0.99, size=(B, H))
    be, g = rng.uniform(0.0, 0.3, size=(B, H)), rng.uniform(0.0, 0.3, size=(B, H))
    D = rng.normal(size=H)
    h0 = rng.normal(size=(1, B, H, P, N))
    st = h0.copy()
    ks, vs = k[None].copy(), x[None].copy()
    for _ in range(T):
        y = oracle.m3_step(x, k, q, a, be, g, st, ks, vs, 0, D)
    aT = a[..., None, None] ** T
    outer = k[:, :, None, :] * x[:, :, :, None]
    h_ref = aT * h0[0] + (be + g)[..., None, None] * outer * (1 - aT) / (1 - a)[..., None, None]
    np.testing.assert_allclose(st[0], h_ref, rtol=1e-12, atol=1e-12)
    y_ref = np.einsum("bhn,bhpn->bhp", q, h_ref) + D[None, :, None] * x
    np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12)


def test_m3_hands_the_current_k_and_x_to_the_next_step_and_keeps_other_layers():
    rng = np.random.default_rng(32)
    st, ks, vs = _m3_case(rng)
    st0, ks0, vs0 = st.copy(), ks.copy(), vs.copy()
    B, H, P, N = 2, 3, 4, 5
    x, k, q = rng.normal(size=(B, H, P)), rng.normal(size=(B, H, N)), rng.normal(size=(B, H, N))
    ones = np.ones((B, H))
    oracle.m3_step(x, k, q, ones, ones, ones, st, ks, vs, 1)
    assert np.array_equal(ks[1], k) and np.array_equal(vs[1], x)
    assert np.array_equal(st[0], st0[0]) and np.array_equal(ks[0], ks0[0]) and np.array_equal(vs[0], vs0[0])
    # the previous (k, v) enter with weight beta, the current (k, x) with gamma
    zero = np.zeros((B, H))
    st2, ks2, vs2 = st0.copy(), ks0.copy(), vs0.copy()
    oracle.m3_step(x, k, q, zero, ones, zero, st2, ks2, vs2, 1)
    np.testing.assert_allclose(st2[1], ks0[1][:, :, None, :] * vs0[1][:, :, :, None], rtol=1e-15)
    st3, ks3, vs3 = st0.copy(), ks0.copy(), vs0.copy()
    y3 = oracle.m3_step(x, k, q, zero, zero, ones, st3, ks3, vs3, 1)
    np.testing.assert_allclose(st3[1], k[:, :, None, :] * x[:, :, :, None], rtol=1e-15)
    np.testing.assert_allclose(y3, np.einsum("bhn,bhn,bhp->bhp", q, k, x), rtol=1e-12)


def test_m3_pure_decay_and_skip():
    rng = np.random.default_rng(33)
    st, ks, vs = _m3_case(rng)
    B, H, P, N = 2, 3, 4, 5
    x, k, q = rng.normal(size=(B, H, P)), rng.normal(size=(B, H, N)), rng.normal(size=(B, H, N))
    a = rng.uniform(0.1, 1.0, size=(B, H))
    zero = np.zeros((B, H))
    D = rng.normal(size=H)
    h0 = st[0].copy()
    y = oracle.m3_step(x, k, q, a, zero, zero, st, ks, vs, 0, D)
    np.testing.assert_allclose(st[0], a[..., None, None] * h0, rtol=1e-15)
    np.testing.assert_allclose(y, np.einsum("bhn,bhpn->bhp", q, st[0]) + D[None, :, None] * x, rtol=1e-12)


def test_m3_is_jointly_linear_in_state_previous_v_and_x():
    rng = np.random.default_rng(34)
    B, H, P, N = 2, 3, 4, 5
    k, q = rng.normal(size=(B, H, N)), rng.normal(size=(B, H, N))
    kprev = rng.normal(size=(1, B, H, N))
    a, be, g = (rng.uniform(0.2, 0.9, size=(B, H)) for _ in range(3))
    D = rng.normal(size=H)

    def run(h0, v0, x):
        st, ks, vs = h0[None].copy(), kprev.copy(), v0[None].copy()
        y = oracle.m3_step(x, k, q, a, be, g, st, ks, vs, 0, D)
        return st[0], y

    s1 = (rng.normal(size=(B, H, P, N)), rng.normal(size=(B, H, P)), rng.normal(size=(B, H, P)))
    s2 = (rng.normal(size=(B, H, P, N)), rng.normal(size=(B, H, P)), rng.normal(size=(B, H, P)))
    c1, c2 = 0.7, -1.3
    h1, y1 = run(*s1)
    h2, y2 = run(*s2)
    h12, y12 = run(*(c1 * u + c2 * v for u, v in zip(s1, s2)))
    np.testing.assert_allclose(h12, c1 * h1 + c2 * h2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(y12, c1 * y1 + c2 * y2, rtol=1e-12, atol=1e-12)


def test_m3_batch_and_head_independence():
    rng = np.random.default_rng(35)
    B, H, P, N = 3, 4, 2, 3
    st, ks, vs = _m3_case(rng, B, H, P, N, L=1)
    x, k, q = rng.normal(size=(B, H, P)), rng.normal(size=(B, H, N)), rng.normal(size=(B, H, N))
    a, be, g = (rng.uniform(0.2, 0.9, size=(B, H)) for _ in range(3))
    D = rng.normal(size=H)
    pb, ph = np.array([2, 0, 1]), np.array([3, 1, 0, 2])
    sA, kA, vA = st.copy(), ks.copy(), vs.copy()
    y = oracle.m3_step(x, k, q, a, be, g, sA, kA, vA, 0, D)
    perm = lambda t: np.ascontiguousarray(t[pb][:, ph])
    sB, kB, vB = (np.ascontiguousarray(s_[:, pb][:, :, ph]) for s_ in (st, ks, vs))
    yB = oracle.m3_step(perm(x), perm(k), perm(q), perm(a), perm(be), perm(g), sB, kB, vB, 0, D[ph])
    np.testing.assert_array_equal(yB, perm(y))
    np.testing.assert_array_equal(sB[0], perm(sA[0]))


# ------------------------------------------------------- Mamba-3 step inputs ----
# Pins of oracle.m3_prepare (mamba-rs 0.2.1 mamba3_siso/gpu/inference.rs: step
# F4c, the angle accumulation into the layer's angle state and the rotation of
# B and C in pairs, and step F5, alpha / beta / gamma of the
# exponential-trapezoidal rule).

def _m3p_inputs(rng, B=2, H=3, N=8):
    k_in, q_in = rng.normal(size=(B, H, N)), rng.normal(size=(B, H, N))
    dt = rng.uniform(0.01, 0.2, size=(B, H))
    A = -rng.uniform(0.2, 3.0, size=(B, H))
    lam = rng.uniform(0.0, 1.0, size=(B, H))
    return k_in, q_in, dt, A, lam


def test_m3_prepare_quarter_and_half_turns_move_each_pair_and_copy_the_rest():
    """From a zero angle state, dt * angle = pi/2 turns each pair (x, y) into
    (-y, x) and pi turns it into (-x, -y); the components past the rotated
    pairs are copied.  Batch row 0 takes the quarter turn, row 1 the half."""
    rng = np.random.default_rng(41)
    B, H, N, na = 2, 3, 8, 3
    k_in, q_in, _, A, lam = _m3p_inputs(rng, B, H, N)
    dt = np.full((B, H), 0.5)
    angles = np.empty((B, na))
    angles[0], angles[1] = np.pi, 2 * np.pi
    st = np.zeros((1, B, H, na))
    k, q, *_ = oracle.m3_prepare(k_in, q_in, dt, A, lam, angles, st, 0)
    for src, out in ((k_in, k), (q_in, q)):
        exp_ = src.copy()
        e, o = src[..., 0:2 * na:2], src[..., 1:2 * na:2]
        exp_[0, :, 0:2 * na:2], exp_[0, :, 1:2 * na:2] = -o[0], e[0]
        exp_[1, :, 0:2 * na:2], exp_[1, :, 1:2 * na:2] = -e[1], -o[1]
        np.testing.assert_allclose(out, exp_, rtol=0, atol=1e-14)
        assert np.array_equal(out[..., 2 * na:], src[..., 2 * na:])
    np.testing.assert_allclose(st[0, 0], np.pi / 2, rtol=1e-15)
    np.testing.assert_allclose(st[0, 1], np.pi, rtol=1e-15)


def test_m3_prepare_angle_state_continues_over_tokens():
    """Two tokens' increments add up in the angle state, and the rotation is a
    function of the accumulated angle: the second token's k equals k_in turned
    once by the total, from a zero state."""
    rng = np.random.default_rng(42)
    B, H, N, na = 2, 3, 8, 4
    k_in, q_in, dt1, A, lam = _m3p_inputs(rng, B, H, N)
    dt2 = rng.uniform(0.01, 0.2, size=(B, H))
    a1, a2 = rng.normal(size=(B, na)), rng.normal(size=(B, na))
    th0 = rng.normal(size=(1, B, H, na))
    st = th0.copy()
    oracle.m3_prepare(k_in, q_in, dt1, A, lam, a1, st, 0)
    k2, q2, *_ = oracle.m3_prepare(k_in, q_in, dt2, A, lam, a2, st, 0)
    # one token carrying both increments (the state is per (b, h), the angles per b)
    total = th0[0] + dt1[..., None] * a1[:, None, :] + dt2[..., None] * a2[:, None, :]
    np.testing.assert_allclose(st[0], total, rtol=1e-14, atol=1e-14)
    for b in range(B):
        for h in range(H):
            z = np.zeros((1, 1, 1, na))
            kk, qq, *_ = oracle.m3_prepare(k_in[b:b + 1, h:h + 1], q_in[b:b + 1, h:h + 1], np.ones((1, 1)),
                                           A[b:b + 1, h:h + 1], lam[b:b + 1, h:h + 1], total[b:b + 1, h], z, 0)
            np.testing.assert_allclose(k2[b, h], kk[0, 0], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(q2[b, h], qq[0, 0], rtol=1e-12, atol=1e-12)


def test_m3_prepare_rotation_keeps_pair_norms_and_the_q_k_product():
    """A rotation keeps each pair's length, and turning k and q by the same
    angles keeps q . k (only relative angles reach the read-out)."""
    rng = np.random.default_rng(43)
    B, H, N, na = 3, 2, 16, 8
    k_in, q_in, dt, A, lam = _m3p_inputs(rng, B, H, N)
    st = rng.normal(scale=50.0, size=(2, B, H, na))
    k, q, *_ = oracle.m3_prepare(k_in, q_in, dt, A, lam, rng.normal(size=(B, na)), st, 1)
    pn = lambda v: np.hypot(v[..., 0::2], v[..., 1::2])
    np.testing.assert_allclose(pn(k), pn(k_in), rtol=1e-13)
    np.testing.assert_allclose(pn(q), pn(q_in), rtol=1e-13)
    np.testing.assert_allclose(np.einsum("bhn,bhn->bh", q, k), np.einsum("bhn,bhn->bh", q_in, k_in),
                               rtol=1e-12, atol=1e-12)
    assert not np.allclose(k, k_in)


def test_m3_prepare_weights_are_the_trapezoid_rule_of_the_decay():
    """Over one step the input weight is the integral of exp(A s) for s in
    [0, dt], (exp(A dt) - 1) / A.  lam = 1/2 takes the trapezoid rule: beta +
    gamma is within its error bound dt^3 A^2 / 12.  lam = 1 is the right
    end-point rule (only the current input, undecayed: beta = 0, gamma = dt),
    lam = 0 the left one (only the previous input, decayed over the step:
    gamma = 0, beta = dt alpha).  alpha is the decay exp(A dt): a semigroup in
    dt (alpha(d1) alpha(d2) = alpha(d1 + d2)) with alpha(0) = 1 and slope A at 0."""
    rng = np.random.default_rng(44)
    B, H, N = 2, 5, 4
    k_in, q_in, dt, A, _ = _m3p_inputs(rng, B, H, N)
    prep = lambda d, l: oracle.m3_prepare(k_in, q_in, d, A, np.full((B, H), l), None, None, 0)[2:]
    al, be, ga = prep(dt, 0.5)
    integral = np.expm1(A * dt) / A
    assert np.all(np.abs(be + ga - integral) <= dt ** 3 * A ** 2 / 12 * (1 + 1e-9))
    assert np.all(np.abs(be + ga - integral) > 0)
    al1, be1, ga1 = prep(dt, 1.0)
    assert np.array_equal(be1, np.zeros((B, H))) and np.array_equal(ga1, dt)
    al0, be0, ga0 = prep(dt, 0.0)
    assert np.array_equal(ga0, np.zeros((B, H)))
    np.testing.assert_allclose(be0, dt * al0, rtol=1e-15)
    # alpha: the decay semigroup with generator A
    d2 = rng.uniform(0.01, 0.2, size=(B, H))
    np.testing.assert_allclose(prep(dt, 0.5)[0] * prep(d2, 0.5)[0], prep(dt + d2, 0.5)[0], rtol=1e-14)
    assert np.array_equal(prep(np.zeros((B, H)), 0.5)[0], np.ones((B, H)))
    eps = 1e-7
    np.testing.assert_allclose((prep(np.full((B, H), eps), 0.5)[0] - 1) / eps, A, rtol=1e-6)


def test_m3_prepare_without_angles_copies_and_keeps_other_slabs():
    """n_angles = 0 leaves k and q as they come; with angles, only the named
    layer's slab of the angle state moves, and each (b, h) only sees its own
    dt, its batch row's angles and its own slot."""
    rng = np.random.default_rng(45)
    B, H, N, na = 3, 4, 8, 2
    k_in, q_in, dt, A, lam = _m3p_inputs(rng, B, H, N)
    k, q, *_ = oracle.m3_prepare(k_in, q_in, dt, A, lam, None, None, 0)
    assert np.array_equal(k, k_in) and np.array_equal(q, q_in)
    st = rng.normal(size=(3, B, H, na))
    st0 = st.copy()
    angles = rng.normal(size=(B, na))
    k, q, al, be, ga = oracle.m3_prepare(k_in, q_in, dt, A, lam, angles, st, 1)
    assert np.array_equal(st[0], st0[0]) and np.array_equal(st[2], st0[2])
    assert not np.allclose(st[1], st0[1])
    pb, ph = np.array([2, 0, 1]), np.array([3, 1, 0, 2])
    perm = lambda t: np.ascontiguousarray(t[pb][:, ph])
    stP = np.ascontiguousarray(st0[:, pb][:, :, ph])
    kP, qP, alP, beP, gaP = oracle.m3_prepare(perm(k_in), perm(q_in), perm(dt), perm(A), perm(lam),
                                              np.ascontiguousarray(angles[pb]), stP, 1)
    for u, v in ((kP, k), (qP, q), (alP, al), (beP, be), (gaP, ga), (stP[1], st[1])):
        np.testing.assert_array_equal(u, perm(v))


def test_m3_prepare_and_step_discretise_the_ode_to_the_rule_s_order():
    """The preparation's weights and the step together integrate
    dh/dt = A h + k x(t).  For x(t) = sin(w t), h(0) = 0 the exact state is
    k (w e^{At} - A sin wt - w cos wt) / (A^2 + w^2).  The trapezoid weights
    (lam = 1/2) are second order: halving dt quarters the error at t = 1; the
    end-point rule (lam = 1) is first order: halving dt halves it."""
    A, w = -2.0, 3.0
    exact = (w * np.exp(A) - A * np.sin(w) - w * np.cos(w)) / (A * A + w * w)

    def run(n, lam):
        d = 1.0 / n
        st = np.zeros((1, 1, 1, 1, 2))
        ks = np.array([1.0, 0.0]).reshape(1, 1, 1, 2)   # the previous token's k (constant)
        vs = np.zeros((1, 1, 1, 1))                      # the previous token's x: x(0) = 0
        k_in = np.array([1.0, 0.0]).reshape(1, 1, 2)
        for i in range(1, n + 1):
            k, q, al, be, ga = oracle.m3_prepare(k_in, k_in, np.full((1, 1), d), np.full((1, 1), A),
                                                 np.full((1, 1), lam), None, None, 0)
            x = np.full((1, 1, 1), np.sin(w * i * d))
            oracle.m3_step(x, k, q, al, be, ga, st, ks, vs, 0)
        return abs(st[0, 0, 0, 0, 0] - exact)

    e1, e2, e3 = (run(n, 0.5) for n in (50, 100, 200))
    assert 3.6 < e1 / e2 < 4.4 and 3.6 < e2 / e3 < 4.4, (e1, e2, e3)
    f1, f2 = run(100, 1.0), run(200, 1.0)
    assert 1.8 < f1 / f2 < 2.2, (f1, f2)
    assert e2 < f1 / 10
