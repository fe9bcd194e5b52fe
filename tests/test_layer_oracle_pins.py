"""Pins for the f64 layer oracle (RMSNorm, the projections, one Mamba-1 block),
independent of the oracle's own code.

What the mathematics fixes: brute-force sums on tiny inputs (math.fsum, no
numpy matmul), the RMSNorm of a constant row and its scale invariance, the
closed form of one token from given states (one step of the recurrence,
h = exp(delta A) h0 + delta B u, so the whole block is a few explicit sums;
from zero state h = delta B u), prefill == T steps,
prefill continuation through the states, and the residual identity when
out_proj is zero.  The closed form is written in plain Python loops over the
pages' step order (mamba-rs inference.rs step chain F1-F12); a plausible
mistake -- x and the gate swapped, B and C swapped, dt_rank columns taken from
the wrong end, the conv taps reversed, a dropped D term, bias, norm weight
or residual -- fails it, which the
mutant cases below check by planting each mistake in the inputs the oracle
sees.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import layer as L

SEED = 0x1A7E4


def _params(seed, dm=6, Di=8, N=3, R=2, K=4, scale=0.5):
    r = np.random.default_rng(seed)
    return dict(
        norm_w=r.uniform(0.5, 1.5, dm),
        in_proj_w=scale * r.standard_normal((2 * Di, dm)),
        conv_w=scale * r.standard_normal((Di, K)),
        conv_b=0.2 * r.standard_normal(Di),
        x_proj_w=scale * r.standard_normal((R + 2 * N, Di)),
        dt_proj_w=scale * r.standard_normal((Di, R)),
        dt_bias=r.uniform(-2.0, 0.5, Di),
        A_log=np.log(r.uniform(0.5, 4.0, (Di, N))),
        D=1.0 + 0.5 * r.standard_normal(Di),
        out_proj_w=scale * r.standard_normal((dm, Di)),
    )


def _silu(v):
    return v / (1.0 + math.exp(-v))


def _softplus(v):
    return math.log1p(math.exp(v)) if v < 30 else v


# ---------------------------------------------------------------- RMSNorm ----

def test_rmsnorm_matches_brute_force_sums():
    r = np.random.default_rng(SEED)
    x = r.standard_normal((5, 7))
    w = r.uniform(0.5, 2.0, 7)
    got = L.rmsnorm(x, w, eps=1e-5)
    for i in range(5):
        ms = math.fsum(v * v for v in x[i]) / 7
        for j in range(7):
            assert got[i, j] == pytest.approx(x[i, j] / math.sqrt(ms + 1e-5) * w[j], rel=1e-14)


def test_rmsnorm_constant_row_closed_form():
    # a row of c's has mean square c^2: h = c / sqrt(c^2 + eps) * w
    for c in (3.0, -0.25, 1e-3):
        x = np.full((1, 16), c)
        w = np.linspace(0.5, 2.0, 16)
        np.testing.assert_allclose(L.rmsnorm(x, w)[0], c / math.sqrt(c * c + 1e-5) * w, rtol=1e-15)


def test_rmsnorm_worked_example():
    # x = (3, 4): mean square 12.5, eps 0 -> (3, 4) / sqrt(12.5)
    got = L.rmsnorm(np.array([[3.0, 4.0]]), np.ones(2), eps=0.0)
    np.testing.assert_allclose(got[0], [0.848528137423857, 1.131370849898476], rtol=1e-15)


def test_rmsnorm_scale_invariance_and_eps_placement():
    r = np.random.default_rng(SEED + 1)
    x = r.standard_normal((3, 32)) * 10
    w = r.uniform(0.5, 2.0, 32)
    np.testing.assert_allclose(L.rmsnorm(7.5 * x, w, eps=0.0), L.rmsnorm(x, w, eps=0.0), rtol=1e-14)
    # eps sits inside the square root: a zero row stays zero, a tiny row is
    # damped by sqrt(eps) rather than blown up
    assert np.all(L.rmsnorm(np.zeros((1, 8)), np.ones(8)) == 0.0)
    tiny = np.full((1, 8), 1e-6)
    np.testing.assert_allclose(L.rmsnorm(tiny, np.ones(8)), 1e-6 / math.sqrt(1e-12 + 1e-5), rtol=1e-14)


# ----------------------------------------------------------------- linear ----

def test_linear_matches_brute_force_sums_nonsquare():
    r = np.random.default_rng(SEED + 2)
    a = r.standard_normal((3, 5))
    w = r.standard_normal((4, 5))  # [out, in]: the product is a w^T, shape [3, 4]
    res = r.standard_normal((3, 4))
    got = L.linear(a, w, res)
    assert got.shape == (3, 4)
    for i in range(3):
        for j in range(4):
            assert got[i, j] == pytest.approx(math.fsum(a[i, k] * w[j, k] for k in range(5)) + res[i, j], rel=1e-13)
    np.testing.assert_array_equal(L.linear(a, np.eye(5)), a)


# ------------------------------------------------------------------ block ----

def _closed_form_one_token(x, p, conv_s=None, h0=None):
    """One token from given states, in explicit sums.  The conv window is the
    state shifted left by one with x appended (slot K-1 newest, weight
    w[:, K-1] on x); the state is h = exp(delta A) h0 + delta B u with
    A = -exp(A_log); y = (C . h + D u) SiLU(z) and x' = x + W_out y.  From a
    zero state the conv sees only its newest tap and h = delta B u."""
    dm = x.shape[0]
    Di, K = p["conv_w"].shape
    N = p["A_log"].shape[1]
    R = p["dt_proj_w"].shape[1]
    conv_s = np.zeros((Di, K)) if conv_s is None else conv_s
    h0 = np.zeros((Di, N)) if h0 is None else h0
    ms = math.fsum(v * v for v in x) / dm
    h = [x[j] / math.sqrt(ms + 1e-5) * p["norm_w"][j] for j in range(dm)]
    xz = [math.fsum(p["in_proj_w"][o, j] * h[j] for j in range(dm)) for o in range(2 * Di)]
    xb, z = xz[:Di], xz[Di:]
    u = []
    for c in range(Di):
        taps = [p["conv_w"][c, k] * conv_s[c, k + 1] for k in range(K - 1)] + [p["conv_w"][c, K - 1] * xb[c]]
        u.append(_silu(math.fsum(taps) + p["conv_b"][c]))
    xd = [math.fsum(p["x_proj_w"][o, c] * u[c] for c in range(Di)) for o in range(R + 2 * N)]
    dt_low, Bv, Cv = xd[:R], xd[R:R + N], xd[R + N:]
    y = []
    for c in range(Di):
        delta = _softplus(math.fsum(p["dt_proj_w"][c, q] * dt_low[q] for q in range(R)) + p["dt_bias"][c])
        hs = [math.exp(-delta * math.exp(p["A_log"][c, n])) * h0[c, n] + delta * Bv[n] * u[c] for n in range(N)]
        core = math.fsum(Cv[n] * hs[n] for n in range(N)) + p["D"][c] * u[c]
        y.append(core * _silu(z[c]))
    return [x[j] + math.fsum(p["out_proj_w"][j, c] * y[c] for c in range(Di)) for j in range(dm)]


def test_block_one_token_from_zero_state_closed_form():
    p = _params(SEED + 3)
    r = np.random.default_rng(SEED + 4)
    x = r.standard_normal((3, 6))
    got, _, _, _ = L.layer_prefill(x, p, 3, 1)
    for b in range(3):
        np.testing.assert_allclose(got[b], _closed_form_one_token(x[b], p), rtol=1e-12, atol=1e-13)


def test_block_one_token_from_given_states_closed_form():
    p = _params(SEED + 17)
    r = np.random.default_rng(SEED + 18)
    x = r.standard_normal((2, 6))
    c0 = r.standard_normal((2, 8, 4))
    s0 = r.standard_normal((2, 8, 3))
    got, _, _, _ = L.layer_prefill(x, p, 2, 1, c0, s0)
    for b in range(2):
        np.testing.assert_allclose(got[b], _closed_form_one_token(x[b], p, c0[b], s0[b]), rtol=1e-12, atol=1e-13)


def _swap_rows(w, a, b, n):
    w = w.copy()
    w[[*range(a, a + n), *range(b, b + n)]] = w[[*range(b, b + n), *range(a, a + n)]]
    return w


@pytest.mark.parametrize("mistake", ["x_z_swapped", "B_C_swapped", "dt_cols_from_end", "no_D", "no_dt_bias",
                                     "no_norm_w", "conv_taps_reversed"])
def test_closed_form_catches_planted_mistakes(mistake):
    """Each mistake is planted in what the oracle is given (equivalent to the
    same index or term mistake in its code): the closed form must notice."""
    p = _params(SEED + 5)
    Di, N, R = 8, 3, 2
    r = np.random.default_rng(SEED + 6)
    x = r.standard_normal((2, 6))
    q = dict(p)
    if mistake == "x_z_swapped":
        q["in_proj_w"] = _swap_rows(p["in_proj_w"], 0, Di, Di)
    elif mistake == "B_C_swapped":
        q["x_proj_w"] = _swap_rows(p["x_proj_w"], R, R + N, N)
    elif mistake == "dt_cols_from_end":
        q["x_proj_w"] = np.concatenate([p["x_proj_w"][2 * N:], p["x_proj_w"][:2 * N]])
    elif mistake == "no_D":
        q["D"] = np.zeros(Di)
    elif mistake == "no_dt_bias":
        q["dt_bias"] = np.zeros(Di)
    elif mistake == "no_norm_w":
        q["norm_w"] = np.ones(6)
    elif mistake == "conv_taps_reversed":
        q["conv_w"] = p["conv_w"][:, ::-1].copy()
    c0 = r.standard_normal((2, Di, 4))
    s0 = r.standard_normal((2, Di, N))
    got, _, _, _ = L.layer_prefill(x, q, 2, 1, c0, s0)
    want = np.array([_closed_form_one_token(x[b], p, c0[b], s0[b]) for b in range(2)])
    assert np.max(np.abs(got - want)) > 1e-6, mistake


def test_block_zero_out_proj_is_the_residual_identity():
    p = _params(SEED + 7)
    p["out_proj_w"] = np.zeros_like(p["out_proj_w"])
    x = np.random.default_rng(SEED + 8).standard_normal((2 * 5, 6))
    got, _, _, _ = L.layer_prefill(x, p, 2, 5)
    np.testing.assert_array_equal(got, x)


def test_block_residual_scales_with_out_proj():
    # x' - x is linear in W_out: a dropped or doubled residual breaks this
    p = _params(SEED + 9)
    x = np.random.default_rng(SEED + 10).standard_normal((4, 6))
    d1 = L.layer_prefill(x, p, 1, 4)[0] - x
    p2 = dict(p, out_proj_w=2.5 * p["out_proj_w"])
    d2 = L.layer_prefill(x, p2, 1, 4)[0] - x
    np.testing.assert_allclose(d2, 2.5 * d1, rtol=1e-12, atol=1e-14)


def test_block_prefill_equals_t_steps():
    """The prefill (C prefill kernels, whole-sequence projections) and T calls
    of the step (C step kernels, per-token projections) agree."""
    Bsz, T, dm, Di, N, R, K = 2, 9, 6, 8, 3, 2, 4
    p = _params(SEED + 11, dm, Di, N, R, K)
    r = np.random.default_rng(SEED + 12)
    x = r.standard_normal((Bsz, T, dm))
    c0 = r.standard_normal((Bsz, Di, K))
    s0 = r.standard_normal((Bsz, Di, N))
    xp, cp, sp, _ = L.layer_prefill(x.reshape(Bsz * T, dm), p, Bsz, T, c0, s0)
    cs = np.ascontiguousarray(c0[None])
    ss = np.ascontiguousarray(s0[None])
    for t in range(T):
        xt, _ = L.layer_step(x[:, t], p, cs, ss, 0)
        np.testing.assert_allclose(xt, xp.reshape(Bsz, T, dm)[:, t], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(cs[0], cp, rtol=0, atol=0)
    np.testing.assert_allclose(ss[0], sp, rtol=1e-11, atol=1e-12)


def test_block_prefill_continuation():
    Bsz, T1, T2, dm = 2, 7, 5, 6
    p = _params(SEED + 13)
    x = np.random.default_rng(SEED + 14).standard_normal((Bsz, T1 + T2, dm))
    whole, cw, sw, _ = L.layer_prefill(x.reshape(-1, dm), p, Bsz, T1 + T2)
    a, ca, sa, _ = L.layer_prefill(x[:, :T1].reshape(-1, dm), p, Bsz, T1)
    b, cb, sb, _ = L.layer_prefill(x[:, T1:].reshape(-1, dm), p, Bsz, T2, ca, sa)
    whole = whole.reshape(Bsz, T1 + T2, dm)
    np.testing.assert_allclose(a.reshape(Bsz, T1, dm), whole[:, :T1], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(b.reshape(Bsz, T2, dm), whole[:, T1:], rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(cb, cw)
    np.testing.assert_allclose(sb, sw, rtol=1e-11, atol=1e-12)


def test_block_stages_are_the_step_outputs():
    # the stages returned are the values each step produced: spot-check two
    p = _params(SEED + 15)
    x = np.random.default_rng(SEED + 16).standard_normal((3, 6))
    _, _, _, st = L.layer_prefill(x, p, 1, 3)
    np.testing.assert_allclose(st["h"], L.rmsnorm(x, p["norm_w"]), rtol=0, atol=0)
    u_ref, _ = oracle.conv1d_silu_prefill(st["xz"][:, :8].reshape(1, 3, 8), p["conv_w"], p["conv_b"])
    np.testing.assert_array_equal(st["u"], u_ref.reshape(3, 8))
