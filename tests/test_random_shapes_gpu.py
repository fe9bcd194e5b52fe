"""A seeded sweep of random shapes and layouts (GPU).

Each case draws batch, T, d_inner, d_state, d_conv, the storage dtype, the gate,
the initial states and a row stride for the activations, then checks:
  - the conv prefill against the oracle (u within the bound, the new conv state
    exactly);
  - the scan prefill, on the conv's own stored u, against the oracle (y and the
    final state within the bound);
  - for d_conv 4, the fused prefill against the two calls, bit for bit;
  - for T = 1, one fused decode step against the T=1 prefill, bit for bit.
The shapes cover ragged channel tails, both prefill routes and every d_state.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_conv1d_gb300 import synth
from _helpers import assert_within, strided_copy, to_dev, to_host

pytestmark = pytest.mark.gpu

N_CASES = 24


def _draw(i):
    r = np.random.default_rng(0x5EED_2000 + i)
    case = dict(
        Bsz=int(r.integers(1, 5)),
        T=int(r.choice([1, 2, 3, int(r.integers(4, 200)), int(r.integers(200, 1400))])),
        Di=int(r.integers(1, 300)),
        N=int(r.choice([1, 2, 4, 8, 16, 32, 64])),
        K=int(r.choice([2, 3, 4, 4])),
        dtype=str(r.choice(["f32", "bf16"])),
        gate=bool(r.integers(0, 2)),
        states=bool(r.integers(0, 2)),
        pad=int(r.choice([0, 0, 1, 8])),  # extra row stride, in elements
    )
    return case


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_shape_matches_oracle(cuda_lib, i):
    m = cuda_lib
    c = _draw(i)
    Bsz, T, Di, N, K, dtype = c["Bsz"], c["T"], c["Di"], c["N"], c["K"], c["dtype"]
    seed = 0x5EED_2100 + i
    p = synth.parity_params(seed, Di, N, K)
    pd = {k: to_dev(v) for k, v in p.items()}
    a = synth.prefill_inputs(seed, Bsz, T, Di, N, dtype, names=("x", "dt", "z", "B", "C"))
    ld = Di + c["pad"]
    x = strided_copy(a["x"], dtype, ld)
    dt = strided_copy(a["dt"], dtype, ld)
    z = strided_copy(a["z"], dtype, ld) if c["gate"] else None
    Bm, Cm = to_dev(a["B"], dtype), to_dev(a["C"], dtype)
    c0 = synth.normal(seed, "conv_state", (Bsz, Di, K), 0.5) if c["states"] else None
    s0 = synth.normal(seed, "ssm_state", (Bsz, Di, N), 0.5) if c["states"] else None
    c0d = to_dev(c0) if c0 is not None else None
    s0d = to_dev(s0) if s0 is not None else None

    u = torch.empty((Bsz, T, Di), device="cuda", dtype=x.dtype)
    c1 = torch.empty((Bsz, Di, K), device="cuda")
    m.mamba_conv1d_silu_prefill(u, x, pd["conv_w"], pd["conv_b"], c0d, c1)
    y1 = torch.empty((Bsz, T, Di), device="cuda")
    s1 = torch.empty((Bsz, Di, N), device="cuda")
    m.mamba_selective_scan_prefill(y1, u, dt, Bm, Cm, pd["A_log"], pd["D"], pd["dt_bias"], z, s0d, s1)
    torch.cuda.synchronize()

    u_ref, c_ref = oracle.conv1d_silu_prefill(a["x"], p["conv_w"], p["conv_b"], c0)
    assert_within(to_host(u), u_ref, f"case {i} {c}: u", bf16_out=dtype == "bf16")
    assert np.array_equal(to_host(c1), c_ref), f"case {i} {c}: conv state"
    u_stored = to_host(u)  # the scan's input as stored (bf16 values are exact in f64)
    y_ref, s_ref = oracle.selective_scan_prefill(u_stored, a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                 p["dt_bias"], a["z"] if c["gate"] else None, s0)
    assert_within(to_host(y1), y_ref, f"case {i} {c}: y")
    assert_within(to_host(s1), s_ref, f"case {i} {c}: ssm state")

    if K <= m.MAMBA_MAX_FUSED_D_CONV:
        y2 = torch.empty_like(y1)
        c2, s2 = torch.empty_like(c1), torch.empty_like(s1)
        m.mamba_mixer_prefill(y2, x, dt, Bm, Cm, pd["conv_w"], pd["A_log"], pd["conv_b"], pd["D"], pd["dt_bias"],
                              z, c0d, c2, s0d, s2)
        torch.cuda.synchronize()
        assert torch.equal(y2, y1) and torch.equal(c2, c1) and torch.equal(s2, s1), f"case {i} {c}: fused"

    if T == 1:
        # one layer of a [1][B][Di][K|N] state, continuing from the same states
        conv = (c0d.clone() if c0d is not None else torch.zeros((Bsz, Di, K), device="cuda")).unsqueeze(0)
        ssm = (s0d.clone() if s0d is not None else torch.zeros((Bsz, Di, N), device="cuda")).unsqueeze(0)
        ys = torch.empty((Bsz, Di), device="cuda")
        m.mamba_mixer_step_batched(ys, x[:, 0].contiguous(), dt[:, 0].contiguous(), Bm[:, 0].contiguous(),
                                   Cm[:, 0].contiguous(), conv, ssm, 0, pd["conv_w"], pd["A_log"], pd["conv_b"],
                                   pd["D"], pd["dt_bias"], z[:, 0].contiguous() if z is not None else None)
        torch.cuda.synchronize()
        assert torch.equal(ys, y1[:, 0]), f"case {i} {c}: step y"
        assert torch.equal(conv[0], c1) and torch.equal(ssm[0], s1), f"case {i} {c}: step states"


def _draw_m3(i):
    r = np.random.default_rng(0x5EED_3000 + i)
    N = int(r.choice([16, 32, 64, 128]))
    P = int(r.choice([1, 3, 8, 17, 32, 64, 100, 2048 * 8 // N]))  # up to the P*N/8 <= 2048 limit
    return dict(Bsz=int(r.integers(1, 4)), H=int(r.integers(1, 6)), P=P, N=N, L=int(r.integers(1, 4)),
                dtype=str(r.choice(["f32", "bf16"])), y_dtype=str(r.choice(["f32", "bf16"])),
                with_D=bool(r.integers(0, 2)))


@pytest.mark.parametrize("i", range(12))
def test_random_m3_shape_matches_oracle(cuda_lib, i):
    """Random Mamba-3 SISO shapes (both kernels: headdim * 4 % 16 picks the
    copy ring or the any-alignment one): two steps on the last layer against
    the oracle, the other layers untouched."""
    m = cuda_lib
    c = _draw_m3(i)
    Bsz, H, P, N, L, dtype, y_dtype = c["Bsz"], c["H"], c["P"], c["N"], c["L"], c["dtype"], c["y_dtype"]
    seed, layer = 0x5EED_3100 + i, c["L"] - 1
    st_h, ks_h, vs_h = synth.m3_states(seed, L, Bsz, H, P, N)
    st, ks, vs = to_dev(st_h), to_dev(ks_h), to_dev(vs_h)
    ref = [a.astype(np.float64).copy() for a in (st_h, ks_h, vs_h)]
    D_h = synth.normal(seed, "m3_D", (H,), 1.0) if c["with_D"] else None
    D = to_dev(D_h) if D_h is not None else None
    ytd = torch.bfloat16 if y_dtype == "bf16" else torch.float32
    for step in range(2):
        inp = synth.m3_step_inputs(seed, layer, step, Bsz, H, P, N, dtype)
        x, k, q = (to_dev(inp[n], dtype) for n in ("x", "k", "q"))
        al, be, ga = (to_dev(inp[n]) for n in ("alpha", "beta", "gamma"))
        y = torch.empty((Bsz, H, P), device="cuda", dtype=ytd)
        m.mamba3_siso_step_batched(y, x, k, q, al, be, ga, st, ks, vs, layer, D)
        torch.cuda.synchronize()
        y_ref = oracle.m3_step(inp["x"], inp["k"], inp["q"], inp["alpha"], inp["beta"], inp["gamma"],
                               ref[0], ref[1], ref[2], layer, D_h)
        assert_within(to_host(y), y_ref, f"case {i} {c}: y step {step}", bf16_out=y_dtype == "bf16")
        assert_within(to_host(st[layer]), ref[0][layer], f"case {i} {c}: ssm state step {step}")
        assert np.array_equal(to_host(ks[layer]), ref[1][layer]) and np.array_equal(to_host(vs[layer]), ref[2][layer])
    for s_dev, s_h in ((st, st_h), (ks, ks_h), (vs, vs_h)):
        for l in range(L - 1):
            assert np.array_equal(to_host(s_dev[l]), s_h[l])
    assert m.mamba_device_faults(clear=True) == 0


@pytest.mark.parametrize("i", range(10))
def test_random_m3_prepare_shape_matches_oracle(cuda_lib, i):
    """Random shapes of the Mamba-3 step's preparation (any even d_state, any
    number of rotated pairs up to all of them, f32 or bf16 k and q): two tokens
    on the last layer against the oracle, the other layers' angle state
    untouched."""
    m = cuda_lib
    r = np.random.default_rng(0x5EED_3200 + i)
    N = 2 * int(r.integers(1, 65))
    na = int(r.integers(0, N // 2 + 1))
    Bsz, H, L = int(r.integers(1, 9)), int(r.integers(1, 33)), int(r.integers(1, 4))
    kq = str(r.choice(["f32", "bf16"]))
    seed, layer = 0x5EED_3300 + i, L - 1
    th_h = synth.m3_angle_state(seed, L, Bsz, H, max(na, 1))
    th = to_dev(th_h)
    th_ref = th_h.astype(np.float64)
    kqd = torch.bfloat16 if kq == "bf16" else torch.float32
    what = f"case {i} (B={Bsz} H={H} N={N} n_angles={na} {kq})"
    for step in range(2):
        inp = synth.m3_prepare_inputs(seed, layer, step, Bsz, H, N, na)
        d = {n: to_dev(v) for n, v in inp.items()}
        k = torch.empty((Bsz, H, N), device="cuda", dtype=kqd)
        q = torch.empty_like(k)
        al, be, ga = (torch.empty((Bsz, H), device="cuda") for _ in range(3))
        m.mamba3_siso_step_prepare(k, q, al, be, ga, d["k_in"], d["q_in"], d["dt"], d["A"], d["lam"],
                                   d["angles"] if na else None, th if na else None, layer)
        torch.cuda.synchronize()
        rk, rq, ral, rbe, rga = oracle.m3_prepare(inp["k_in"], inp["q_in"], inp["dt"], inp["A"], inp["lam"],
                                                  inp["angles"] if na else None, th_ref if na else None, layer)
        assert_within(to_host(k), rk, f"{what}: k step {step}", bf16_out=kq == "bf16")
        assert_within(to_host(q), rq, f"{what}: q step {step}", bf16_out=kq == "bf16")
        for g, rr, nm in ((al, ral, "alpha"), (be, rbe, "beta"), (ga, rga, "gamma")):
            assert_within(to_host(g), rr, f"{what}: {nm} step {step}")
        if na:
            assert_within(to_host(th[layer]), th_ref[layer], f"{what}: angle state step {step}")
    for l in range(L - 1):
        assert np.array_equal(to_host(th[l]), th_h[l])
