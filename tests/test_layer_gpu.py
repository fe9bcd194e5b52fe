"""GPU parity of the rest of the Mamba-1 block: the tcgen05 projection GEMM,
the RMSNorm, and the whole block (prefill and T=1 step) through the C ABI.

Each stage is checked element by element against the f64 oracle on the
stage's own GPU inputs (a bf16 activation is rounded once by the GPU; the
oracle then consumes the GPU's rounded values, so a rounding decision on one
side never cascades into the next stage): |gpu - ref| <= 2e-4 (1 + |ref|),
plus one bf16 unit in the last place for a bf16 output.  The block call is
checked to be exactly the documented sequence of ABI calls (bit for bit), and
end to end against the oracle that mirrors the GPU's bf16 storage.
"""
import numpy as np
import pytest
import torch

from oracle import layer as OL
from selective_state_space_conv1d_gb300 import synth
from _helpers import assert_within, to_dev, to_host

pytestmark = pytest.mark.gpu

SEED = 0x5EED4000


def _bf16_dev(a):
    return to_dev(a, "bf16")


# ----------------------------------------------------------------- linear ----

@pytest.mark.parametrize("M,N,K", [
    (128, 128, 64),        # one tile
    (333, 96, 200),        # ragged M, N and K
    (2048, 3072, 768),     # 130m in_proj
    (2048, 80, 1536),      # 130m x_proj (narrow N)
    (2048, 1536, 48),      # 130m dt_proj (K below one 64-wide stage)
    (2048, 768, 1536),     # 130m out_proj
    (1, 3072, 768),        # one row (a T=1 step at batch 1)
    (130, 200, 1000),
    (128, 768, 1536),      # decode out_proj: few tiles, K split over a cluster of 8
    (128, 80, 1536),       # decode x_proj
    (300, 380, 256),       # 192-wide tiles, ragged second column block
    (2048, 4096, 256),     # 128 x 256 tiles, more tiles than SMs: both accumulators in turn
    (640, 2560, 2560),     # 2.8b out_proj-shaped K and N
])
@pytest.mark.parametrize("out", ["f32", "bf16", "f32+residual"])
def test_linear_matches_oracle(cuda_lib, M, N, K, out):
    m = cuda_lib
    r = np.random.default_rng(SEED + M + N + K)
    a = synth.store(r.standard_normal((M, K)).astype(np.float32), "bf16")
    w = synth.store((r.standard_normal((N, K)) * K ** -0.5).astype(np.float32), "bf16")
    res = r.standard_normal((M, N)).astype(np.float32) if out == "f32+residual" else None
    c = torch.full((M, N), float("nan"), device="cuda", dtype=torch.bfloat16 if out == "bf16" else torch.float32)
    if res is not None:
        c.copy_(to_dev(res))
    m.mamba_linear_bf16(c, _bf16_dev(a), _bf16_dev(w), c if res is not None else None)
    torch.cuda.synchronize()
    assert m.mamba_device_faults(clear=True) == 0
    assert_within(to_host(c), OL.linear(a, w, res), f"linear {M}x{N}x{K} {out}", bf16_out=out == "bf16")


def test_linear_strided_operands_and_output(cuda_lib):
    """A column slice of a wider buffer as A (the dt_proj reading the first
    dt_rank columns of the x_proj output) and as C; the columns around the
    output slice stay untouched."""
    m = cuda_lib
    M, N, K, ld_a, ld_c = 300, 160, 48, 88, 200
    r = np.random.default_rng(SEED + 7)
    abuf = _bf16_dev(synth.store(r.standard_normal((M, ld_a)).astype(np.float32), "bf16"))
    a = abuf[:, :K]
    w = _bf16_dev(synth.store((r.standard_normal((N, K)) * 0.2).astype(np.float32), "bf16"))
    cbuf = torch.full((M, ld_c), 5.5, device="cuda", dtype=torch.bfloat16)
    c = cbuf[:, 16:16 + N]
    m.mamba_linear_bf16(c, a, w)
    torch.cuda.synchronize()
    assert_within(to_host(c), OL.linear(to_host(a), to_host(w)), "strided linear", bf16_out=True)
    assert bool((cbuf[:, :16] == 5.5).all()) and bool((cbuf[:, 16 + N:] == 5.5).all())


@pytest.mark.parametrize("out", ["bf16", "f32+residual"])
def test_linear_misaligned_output_takes_the_element_path(cuda_lib, out):
    """An output at an odd element offset with an odd row stride (no 16-byte
    rows: neither tensor stores nor vector stores apply) gives the same values."""
    m = cuda_lib
    M, N, K, ld_c, off = 260, 136, 192, 151, 3
    r = np.random.default_rng(SEED + 9)
    a = synth.store(r.standard_normal((M, K)).astype(np.float32), "bf16")
    w = synth.store((r.standard_normal((N, K)) * K ** -0.5).astype(np.float32), "bf16")
    dt = torch.bfloat16 if out == "bf16" else torch.float32
    cbuf = torch.full((M, ld_c), 9.0, device="cuda", dtype=dt)
    c = cbuf[:, off:off + N]
    res = None
    if out != "bf16":
        res = r.standard_normal((M, N)).astype(np.float32)
        c.copy_(to_dev(res))
    m.mamba_linear_bf16(c, _bf16_dev(a), _bf16_dev(w), c if res is not None else None)
    torch.cuda.synchronize()
    assert_within(to_host(c), OL.linear(a, w, res), f"misaligned {out}", bf16_out=out == "bf16")
    assert bool((cbuf[:, :off] == 9.0).all()) and bool((cbuf[:, off + N:] == 9.0).all())


def test_linear_is_row_independent_bitwise(cuda_lib):
    """A row's result does not depend on M or on the row's place in its tile:
    the K order of every output element is fixed."""
    m = cuda_lib
    M, N, K = 500, 256, 640
    r = np.random.default_rng(SEED + 8)
    a = _bf16_dev(synth.store(r.standard_normal((M, K)).astype(np.float32), "bf16"))
    w = _bf16_dev(synth.store((r.standard_normal((N, K)) * 0.05).astype(np.float32), "bf16"))
    c = torch.empty(M, N, device="cuda")
    m.mamba_linear_bf16(c, a, w)
    c2 = torch.empty(7, N, device="cuda")
    m.mamba_linear_bf16(c2, a[301:308].contiguous(), w)
    torch.cuda.synchronize()
    assert torch.equal(c[301:308], c2)


# ---------------------------------------------------------------- RMSNorm ----

@pytest.mark.parametrize("M,D,out,ld_x", [
    (2048, 768, "bf16", 768), (100, 2560, "bf16", 2560), (37, 768, "f32", 800),
    (64, 100, "f32", 100),    # D not a multiple of 4: element path
    (5, 7, "bf16", 9),
])
def test_rmsnorm_matches_oracle(cuda_lib, M, D, out, ld_x):
    m = cuda_lib
    r = np.random.default_rng(SEED + M + D)
    xb = (r.standard_normal((M, ld_x)) * r.uniform(0.1, 10.0, (M, 1))).astype(np.float32)
    w = r.uniform(0.5, 1.5, D).astype(np.float32)
    x = to_dev(xb)[:, :D]
    o = torch.empty(M, D, device="cuda", dtype=torch.bfloat16 if out == "bf16" else torch.float32)
    m.mamba_rmsnorm(o, x, to_dev(w), 1e-5)
    torch.cuda.synchronize()
    assert_within(to_host(o), OL.rmsnorm(xb[:, :D], w), f"rmsnorm {M}x{D}", bf16_out=out == "bf16")


# ------------------------------------------------------------------ block ----

SHAPES = {
    # name: (d_model, d_inner, d_state, d_conv, dt_rank)
    "small": (64, 128, 16, 4, 8),
    "130m": (768, 1536, 16, 4, 48),
    "n8_k3": (128, 256, 8, 3, 16),
}


def _block(name, seed, Bsz, T, state=True):
    dm, Di, N, K, R = SHAPES[name]
    p = synth.layer_params(seed, dm, Di, N, K, R, parity=True)
    x = synth.normal(seed, "hidden", (Bsz * T, dm), 1.0)
    c0 = synth.normal(seed, "conv_state", (Bsz, Di, K), 1.0) if state else None
    s0 = synth.normal(seed, "ssm_state", (Bsz, Di, N), 0.5) if state else None
    return p, x, c0, s0


def _dev_weights(p):
    return {k: (_bf16_dev(v) if k.endswith("proj_w") else to_dev(v)) for k, v in p.items()}


def _staged(m, wd, hidden, Bsz, T, c_in, c_out, s_in, s_out):
    """The block as its documented sequence of ABI calls, every stage kept."""
    dm = hidden.shape[-1]
    Di, K = wd["conv_w"].shape
    N = wd["A_log"].shape[1]
    R = wd["dt_proj_w"].shape[1]
    rows = Bsz * T
    bf = dict(device="cuda", dtype=torch.bfloat16)
    ldx = (R + 2 * N + 7) // 8 * 8
    h = torch.empty(rows, dm, **bf)
    xz = torch.empty(rows, 2 * Di, **bf)
    u = torch.empty(Bsz, T, Di, **bf)
    xdb = torch.empty(rows, ldx, **bf)
    xd = xdb[:, :R + 2 * N]
    dt = torch.empty(rows, Di, **bf)
    y = torch.empty(Bsz, T, Di, **bf)
    hid = hidden.reshape(rows, dm)
    m.mamba_rmsnorm(h, hid, wd["norm_w"], 1e-5)
    m.mamba_linear_bf16(xz, h, wd["in_proj_w"])
    xz3 = xz.view(Bsz, T, 2 * Di)
    m.mamba_conv1d_silu_prefill(u, xz3[:, :, :Di], wd["conv_w"], wd["conv_b"], c_in, c_out)
    m.mamba_linear_bf16(xd, u.view(rows, Di), wd["x_proj_w"])
    m.mamba_linear_bf16(dt, xdb[:, :R], wd["dt_proj_w"])
    xd3 = xdb.view(Bsz, T, ldx)
    m.mamba_selective_scan_prefill(y, u, dt.view(Bsz, T, Di), xd3[:, :, R:R + N], xd3[:, :, R + N:R + 2 * N],
                                   wd["A_log"], wd["D"], wd["dt_bias"], xz3[:, :, Di:], s_in, s_out)
    m.mamba_linear_bf16(hid, y.view(rows, Di), wd["out_proj_w"], hid)
    return dict(h=h, xz=xz, u=u.view(rows, Di), x_dbl=xd, dt=dt, y=y.view(rows, Di))


def _check_block(m, p, x, c0, s0, Bsz, T, end_to_end=True):
    """Every stage against the oracle on its own GPU inputs; the block call
    equal to its call sequence bit for bit; optionally end to end against the
    storage-mirroring oracle."""
    import oracle

    Di, K = p["conv_w"].shape
    N = p["A_log"].shape[1]
    R = p["dt_proj_w"].shape[1]
    dm = p["norm_w"].shape[0]
    wd = _dev_weights(p)
    hidden = to_dev(x).view(Bsz, T, dm)
    cs, ss = to_dev(c0), to_dev(s0)
    c_out, s_out = torch.empty_like(cs), torch.empty_like(ss)
    st = _staged(m, wd, hidden, Bsz, T, cs, c_out, ss, s_out)
    torch.cuda.synchronize()
    assert m.mamba_device_faults(clear=True) == 0
    g = {k: to_host(v) for k, v in st.items()}
    # every stage against the oracle on the GPU's own (rounded) inputs
    assert_within(g["h"], OL.rmsnorm(x, p["norm_w"]), "h = RMSNorm(x)", bf16_out=True)
    assert_within(g["xz"], OL.linear(g["h"], p["in_proj_w"]), "xz = in_proj(h)", bf16_out=True)
    u_ref, c_ref = oracle.conv1d_silu_prefill(g["xz"][:, :Di].reshape(Bsz, T, Di), p["conv_w"], p["conv_b"], c0)
    assert_within(g["u"], u_ref.reshape(-1, Di), "u = SiLU(conv(x))", bf16_out=True)
    assert np.array_equal(to_host(c_out), c_ref)
    assert_within(g["x_dbl"], OL.linear(g["u"], p["x_proj_w"]), "x_dbl = x_proj(u)", bf16_out=True)
    assert_within(g["dt"], OL.linear(g["x_dbl"][:, :R], p["dt_proj_w"]), "dt = dt_proj(x_dbl)", bf16_out=True)
    y_ref, s_ref = oracle.selective_scan_prefill(
        g["u"].reshape(Bsz, T, Di), g["dt"].reshape(Bsz, T, Di), g["x_dbl"][:, R:R + N].reshape(Bsz, T, N),
        g["x_dbl"][:, R + N:].reshape(Bsz, T, N), p["A_log"], p["D"], p["dt_bias"],
        g["xz"][:, Di:].reshape(Bsz, T, Di), s0)
    assert_within(g["y"], y_ref.reshape(-1, Di), "y = scan(...) * SiLU(z)", bf16_out=True)
    assert_within(to_host(s_out), s_ref, "ssm state")
    assert_within(to_host(hidden).reshape(-1, dm), OL.linear(g["y"], p["out_proj_w"], x), "x + out_proj(y)")

    # the block call is exactly that sequence, bit for bit
    hidden2 = to_dev(x).view(Bsz, T, dm)
    c2, s2 = torch.empty_like(cs), torch.empty_like(ss)
    m.mamba_layer_prefill(hidden2, wd, cs, c2, ss, s2)
    torch.cuda.synchronize()
    assert torch.equal(hidden2, hidden)
    assert torch.equal(c2, c_out) and torch.equal(s2, s_out)
    assert m.mamba_device_faults(clear=True) == 0
    if not end_to_end:
        return
    # end to end against the oracle that stores every activation in bf16 as
    # the GPU does: only rounding decisions taken on f32 vs f64 values differ,
    # each by one bf16 unit, so the block output stays within the bound of the
    # out_proj term's scale
    store = lambda v: synth.round_to_bf16(np.asarray(v, np.float32)).astype(np.float64)
    x_ref, c_e, s_e, _ = OL.layer_prefill(x, p, Bsz, T, c0, s0, store=store)
    scale = np.sqrt(np.mean((x_ref - x) ** 2))
    err = np.max(np.abs(to_host(hidden2).reshape(-1, dm) - x_ref))
    assert err <= 0.05 * scale + 2e-4, (err, scale)
    # the conv state holds bf16 x values: the two sides may round one of them
    # to neighbouring bf16 values (one unit apart, at most 2^-7 |ref|)
    c_err = np.abs(to_host(c2) - c_e)
    assert np.all(c_err <= 2.0 ** -7 * np.abs(c_e) + 1e-30), np.max(c_err)
    assert np.mean(c_err > 0) < 1e-2


@pytest.mark.parametrize("name,Bsz,T", [("small", 2, 300), ("130m", 1, 256), ("n8_k3", 3, 70), ("small", 1, 1)])
def test_block_prefill_stages_match_oracle(cuda_lib, name, Bsz, T):
    p, x, c0, s0 = _block(name, SEED + T, Bsz, T)
    _check_block(cuda_lib, p, x, c0, s0, Bsz, T)


@pytest.mark.parametrize("case", range(10))
def test_block_random_shapes(cuda_lib, case):
    """Seeded random block shapes: d_model, d_inner and dt_rank any multiples of
    8, every supported d_state, d_conv 1..8, batch 1..4, T 1..400 (ragged GEMM
    tiles and scan tiles, element and vector paths); stages against the
    oracle, the block call against its call sequence, and the T = 1 block step
    against the T = 1 block prefill, bit for bit."""
    m = cuda_lib
    r = np.random.default_rng(SEED + 900 + case)
    dm = 8 * int(r.integers(1, 41))
    Di = 8 * int(r.integers(1, 65))
    N = int(r.choice([1, 2, 4, 8, 16, 32, 64]))
    K = int(r.integers(1, 9))
    R = 8 * int(r.integers(1, 7))
    Bsz = int(r.integers(1, 5))
    T = int(r.integers(1, 401))
    seed = SEED + 1000 + case
    p = synth.layer_params(seed, dm, Di, N, K, R, parity=True)
    x = synth.normal(seed, "hidden", (Bsz * T, dm), 1.0)
    c0 = synth.normal(seed, "conv_state", (Bsz, Di, K), 1.0)
    s0 = synth.normal(seed, "ssm_state", (Bsz, Di, N), 0.5)
    _check_block(m, p, x, c0, s0, Bsz, T, end_to_end=False)
    # the step on slab 1 of 2 layers equals the T = 1 prefill
    wd = _dev_weights(p)
    x1 = to_dev(x[:Bsz])
    cst = torch.stack([to_dev(c0), to_dev(c0) + 1.0]).contiguous()
    sst = torch.stack([to_dev(s0), to_dev(s0) - 1.0]).contiguous()
    h_step = x1.clone()
    c_before = cst[0].clone()
    s_before = sst[0].clone()
    m.mamba_layer_step(h_step, wd, cst, sst, 1)
    h_pre = x1.clone().view(Bsz, 1, dm)
    c1, s1 = (to_dev(c0) + 1.0), (to_dev(s0) - 1.0)
    m.mamba_layer_prefill(h_pre, wd, c1, c1, s1, s1)
    torch.cuda.synchronize()
    assert torch.equal(h_step, h_pre.view(Bsz, dm))
    assert torch.equal(cst[1], c1) and torch.equal(sst[1], s1)
    assert torch.equal(cst[0], c_before) and torch.equal(sst[0], s_before)
    assert m.mamba_device_faults(clear=True) == 0


def test_block_prefill_zero_state_defaults_and_in_place_states(cuda_lib):
    """NULL states mean zeros; in-place states equal separate in/out buffers."""
    m = cuda_lib
    Bsz, T = 2, 150
    p, x, _, _ = _block("small", SEED + 11, Bsz, T, state=False)
    dm, Di, N, K, R = SHAPES["small"]
    wd = _dev_weights(p)
    h1 = to_dev(x).view(Bsz, T, dm)
    c1, s1 = torch.empty(Bsz, Di, K, device="cuda"), torch.empty(Bsz, Di, N, device="cuda")
    m.mamba_layer_prefill(h1, wd, None, c1, None, s1)
    h2 = to_dev(x).view(Bsz, T, dm)
    c2, s2 = torch.zeros(Bsz, Di, K, device="cuda"), torch.zeros(Bsz, Di, N, device="cuda")
    m.mamba_layer_prefill(h2, wd, c2, c2, s2, s2)
    torch.cuda.synchronize()
    assert torch.equal(h1, h2) and torch.equal(c1, c2) and torch.equal(s1, s2)


def test_block_prefill_continuation(cuda_lib):
    """prefill(T1) then prefill(T2) from the returned states equals prefill(T1 + T2)."""
    m = cuda_lib
    Bsz, T1, T2 = 2, 130, 77
    p, x, c0, s0 = _block("small", SEED + 12, Bsz, T1 + T2)
    dm, Di, N, K, R = SHAPES["small"]
    wd = _dev_weights(p)
    x3 = to_dev(x).view(Bsz, T1 + T2, dm)
    whole = x3.clone()
    cw, sw = to_dev(c0), to_dev(s0)
    m.mamba_layer_prefill(whole, wd, cw, cw, sw, sw)
    a, b = x3[:, :T1].contiguous(), x3[:, T1:].contiguous()
    cs, ss = to_dev(c0), to_dev(s0)
    m.mamba_layer_prefill(a, wd, cs, cs, ss, ss)
    m.mamba_layer_prefill(b, wd, cs, cs, ss, ss)
    torch.cuda.synchronize()
    assert torch.equal(cs, cw)
    assert_within(to_host(ss), to_host(sw), "ssm state")
    assert_within(to_host(torch.cat([a, b], 1)), to_host(whole), "hidden")


def test_block_step_equals_t1_prefill_on_its_slab(cuda_lib):
    """A T=1 block step on slab l of layer-major states is the T=1 prefill
    (bit for bit), and leaves every other slab untouched."""
    m = cuda_lib
    L, l, Bsz = 3, 1, 5
    p, _, _, _ = _block("130m", SEED + 13, Bsz, 1)
    dm, Di, N, K, R = SHAPES["130m"]
    wd = _dev_weights(p)
    x = to_dev(synth.normal(SEED + 13, "hidden", (Bsz, dm), 1.0))
    cst = to_dev(synth.normal(SEED + 13, "conv_state", (L, Bsz, Di, K), 1.0))
    sst = to_dev(synth.normal(SEED + 13, "ssm_state", (L, Bsz, Di, N), 0.5))
    c_ref, s_ref = cst.clone(), sst.clone()
    h_step = x.clone()
    m.mamba_layer_step(h_step, wd, cst, sst, l)
    h_pre = x.clone().view(Bsz, 1, dm)
    c1, s1 = c_ref[l].clone(), s_ref[l].clone()
    m.mamba_layer_prefill(h_pre, wd, c1, c1, s1, s1)
    torch.cuda.synchronize()
    assert m.mamba_device_faults(clear=True) == 0
    assert torch.equal(h_step, h_pre.view(Bsz, dm))
    assert torch.equal(cst[l], c1) and torch.equal(sst[l], s1)
    for o in range(L):
        if o != l:
            assert torch.equal(cst[o], c_ref[o]) and torch.equal(sst[o], s_ref[o])


def test_block_steps_continue_a_prefill(cuda_lib):
    """prefill(T) then 3 block steps == prefill(T + 3) on the last 3 tokens."""
    m = cuda_lib
    Bsz, T, S = 2, 60, 3
    p, x, c0, s0 = _block("small", SEED + 14, Bsz, T + S)
    dm, Di, N, K, R = SHAPES["small"]
    wd = _dev_weights(p)
    x3 = to_dev(x).view(Bsz, T + S, dm)
    whole = x3.clone()
    cw, sw = to_dev(c0), to_dev(s0)
    m.mamba_layer_prefill(whole, wd, cw, cw, sw, sw)
    head = x3[:, :T].contiguous()
    cs, ss = to_dev(c0)[None].contiguous(), to_dev(s0)[None].contiguous()
    m.mamba_layer_prefill(head, wd, cs[0], cs[0], ss[0], ss[0])
    outs = []
    for t in range(S):
        h = x3[:, T + t].contiguous()
        m.mamba_layer_step(h, wd, cs, ss, 0)
        outs.append(h)
    torch.cuda.synchronize()
    assert_within(to_host(torch.stack(outs, 1)), to_host(whole[:, T:]), "hidden after the steps")
    assert torch.equal(cs[0], cw)
    assert_within(to_host(ss[0]), to_host(sw), "ssm state")


def test_block_workspace_smaller_scan_share_same_result(cuda_lib):
    """A workspace with only the activations' bytes runs the scan's one-pass
    route instead of the chained one (wide enough a shape for it): the same
    numbers, since the two routes scan every row once in the same order."""
    m = cuda_lib
    Bsz, T = 26, 160
    dm, Di, N, K, R = SHAPES["130m"]
    p, x, c0, s0 = _block("130m", SEED + 15, Bsz, T)
    wd = _dev_weights(p)
    full = m.mamba_layer_workspace_bytes(wd, Bsz, T)
    rows = Bsz * T
    r256 = lambda b: (b + 255) // 256 * 256
    act = (r256(rows * dm * 2) + r256(rows * 2 * Di * 2) + 3 * r256(rows * Di * 2)
           + r256(rows * ((R + 2 * N + 7) // 8 * 8) * 2))
    assert full >= act
    outs = []
    for nbytes in (full, act):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        h = to_dev(x).view(Bsz, T, dm)
        c, s = to_dev(c0), to_dev(s0)
        m.mamba_layer_prefill(h, wd, c, c, s, s, workspace=ws)
        outs.append((h, c, s))
    torch.cuda.synchronize()
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    with pytest.raises(m.MambaError):
        ws = torch.empty(act - 256, dtype=torch.uint8, device="cuda")
        m.mamba_layer_prefill(to_dev(x).view(Bsz, T, dm), wd, workspace=ws)


def test_block_prefill_2p8b_full_size_sampled(cuda_lib):
    """The mamba-2.8b-shaped block over batch 8 x T 4096 (the launch shapes the
    benchmark times): the block call equals its call sequence bit for bit, and
    each stage matches the oracle on sampled rows (the norm and the
    projections are row-independent) and on sampled channels of one batch row
    (the conv and the scan are channel-independent)."""
    m = cuda_lib
    dm, Di, N, K, R = 2560, 5120, 16, 4, 160
    Bsz, T = 8, 4096
    rows = Bsz * T
    seed = SEED + 2800
    p = synth.layer_params(seed, dm, Di, N, K, R, parity=True)
    wd = _dev_weights(p)
    x = synth.torch_normal((Bsz, T, dm), 1.0, seed + 1, "cuda")
    c0 = synth.torch_normal((Bsz, Di, K), 1.0, seed + 2, "cuda")
    s0 = synth.torch_normal((Bsz, Di, N), 0.5, seed + 3, "cuda")
    hidden = x.clone()
    c_out, s_out = torch.empty_like(c0), torch.empty_like(s0)
    st = _staged(m, wd, hidden, Bsz, T, c0, c_out, s0, s_out)
    hidden2 = x.clone()
    c2, s2 = torch.empty_like(c0), torch.empty_like(s0)
    m.mamba_layer_prefill(hidden2, wd, c0, c2, s0, s2)
    torch.cuda.synchronize()
    assert m.mamba_device_faults(clear=True) == 0
    assert torch.equal(hidden2, hidden) and torch.equal(c2, c_out) and torch.equal(s2, s_out)

    r = np.random.default_rng(seed)
    sel = np.unique(np.concatenate([r.choice(rows, 96, replace=False), [0, 127, 128, rows - 1]]))
    idx = torch.as_tensor(sel, device="cuda")
    pick = lambda t: to_host(t.reshape(rows, -1).index_select(0, idx))
    xh = pick(x)
    g = {k: pick(v) for k, v in st.items()}
    assert_within(g["h"], OL.rmsnorm(xh, p["norm_w"]), "h (sampled rows)", bf16_out=True)
    assert_within(g["xz"], OL.linear(g["h"], p["in_proj_w"]), "xz (sampled rows)", bf16_out=True)
    assert_within(g["x_dbl"], OL.linear(g["u"], p["x_proj_w"]), "x_dbl (sampled rows)", bf16_out=True)
    assert_within(g["dt"], OL.linear(g["x_dbl"][:, :R], p["dt_proj_w"]), "dt (sampled rows)", bf16_out=True)
    assert_within(pick(hidden), OL.linear(g["y"], p["out_proj_w"], xh), "x + out_proj(y) (sampled rows)")

    # one batch row, sampled channels, through the conv and the scan
    import oracle

    b = 5
    ch = np.unique(np.concatenate([r.choice(Di, 40, replace=False), [0, 31, 32, Di - 1]]))
    cidx = torch.as_tensor(ch, device="cuda")
    col = lambda t, off=0: to_host(t.view(Bsz, T, -1)[b:b + 1].index_select(2, cidx + off))
    ps = {k: np.ascontiguousarray(v[ch]) for k, v in p.items() if k in ("conv_w", "conv_b", "A_log", "D", "dt_bias")}
    u_ref, c_ref = oracle.conv1d_silu_prefill(col(st["xz"]), ps["conv_w"], ps["conv_b"], to_host(c0[b:b + 1, ch]))
    assert_within(col(st["u"]), u_ref, "u (one row, sampled channels)", bf16_out=True)
    assert np.array_equal(to_host(c_out[b:b + 1, ch]), c_ref)
    xdb = to_host(st["x_dbl"].view(Bsz, T, -1)[b:b + 1])
    y_ref, s_ref = oracle.selective_scan_prefill(col(st["u"]), col(st["dt"]), xdb[:, :, R:R + N],
                                                 xdb[:, :, R + N:R + 2 * N], ps["A_log"], ps["D"], ps["dt_bias"],
                                                 col(st["xz"], Di), to_host(s0[b:b + 1, ch]))
    assert_within(col(st["y"]), y_ref, "y (one row, sampled channels)", bf16_out=True)
    assert_within(to_host(s_out[b:b + 1, ch]), s_ref, "ssm state (one row, sampled channels)")


def test_layer_decode_graph_replays_the_block_steps_bitwise(cuda_lib):
    """The whole-block decode graph (n_layers block steps recorded once) gives
    the direct calls' bits, launch after launch, and records 7 kernels per layer."""
    m = cuda_lib
    L, Bsz, S = 3, 5, 3
    dm, Di, N, K, R = SHAPES["130m"]
    wds = [_dev_weights(synth.layer_params(SEED + 70 + l, dm, Di, N, K, R, parity=True)) for l in range(L)]
    xs = [to_dev(synth.normal(SEED + 80 + s_, "hidden", (Bsz, dm), 1.0)) for s_ in range(S)]
    c0 = to_dev(synth.normal(SEED + 90, "conv_state", (L, Bsz, Di, K), 1.0))
    s0 = to_dev(synth.normal(SEED + 90, "ssm_state", (L, Bsz, Di, N), 0.5))
    hg, cg, sg = torch.empty(Bsz, dm, device="cuda"), c0.clone(), s0.clone()
    hd, cd, sd = torch.empty(Bsz, dm, device="cuda"), c0.clone(), s0.clone()
    with m.LayerDecodeGraph(wds, hg, cg, sg) as g:
        assert g.kernels == 7 * L
        for s_ in range(S):
            hg.copy_(xs[s_])
            g.launch()
            hd.copy_(xs[s_])
            for l in range(L):
                m.mamba_layer_step(hd, wds[l], cd, sd, l)
            torch.cuda.synchronize()
            assert torch.equal(hg, hd), f"step {s_}"
            assert torch.equal(cg, cd) and torch.equal(sg, sd)
    assert m.mamba_device_faults(clear=True) == 0
