"""Parity on the five synthetic workloads at full size, in the launch
configuration bench.py times (default workspace, so narrow prefills take the
T-split route; decode as a CUDA graph).  Where the oracle cannot run the whole
workload in seconds it checks sampled channels / rows, which are independent
recurrences, so a sample is a full-fidelity check of those rows.
"""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_conv1d_gb300 import synth
from _helpers import assert_within, to_dev, to_host

pytestmark = pytest.mark.gpu


def _conv_scan_gpu(m, a, p, dtype, conv_state=None, ssm_state=None):
    x = to_dev(a["x"], dtype)
    u = torch.empty_like(x)
    cst = torch.empty((x.shape[0], x.shape[2], p["conv_w"].shape[1]), device="cuda")
    m.mamba_conv1d_silu_prefill(u, x, to_dev(p["conv_w"]), to_dev(p["conv_b"]),
                                to_dev(conv_state) if conv_state is not None else None, cst)
    y = torch.empty(x.shape, device="cuda")
    sst = torch.empty((x.shape[0], x.shape[2], a["B"].shape[2]), device="cuda")
    m.mamba_selective_scan_prefill(y, u, to_dev(a["dt"], dtype), to_dev(a["B"], dtype), to_dev(a["C"], dtype),
                                   to_dev(p["A_log"]), to_dev(p["D"]), to_dev(p["dt_bias"]),
                                   to_dev(a["z"], dtype), to_dev(ssm_state) if ssm_state is not None else None,
                                   sst)
    torch.cuda.synchronize()
    return u, y, cst, sst


@pytest.mark.parametrize("wl_index", [0, 1])
def test_f32_prefill_workloads_full(cuda_lib, wl_index):
    """Tiny mixer and the mamba-130m layer: conv then scan, every element."""
    m = cuda_lib
    wl = synth.WORKLOADS[wl_index]
    Bsz, T, Di, N, K = wl.batch, wl.seqlen, wl.d_inner, wl.d_state, wl.d_conv
    p = synth.mixer_params(wl.seed, Di, N, K)
    a = synth.prefill_inputs(wl.seed, Bsz, T, Di, N, "f32", names=("x", "dt", "z", "B", "C"))
    u, y, cst, sst = _conv_scan_gpu(m, a, p, "f32")
    u_ref, c_ref = oracle.conv1d_silu_prefill(a["x"], p["conv_w"], p["conv_b"], None)
    y_ref, s_ref = oracle.selective_scan_prefill(u_ref, a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                                 p["dt_bias"], a["z"], None)
    assert_within(to_host(u), u_ref, "u")
    assert_within(to_host(y), y_ref, "y")
    assert np.array_equal(to_host(cst), c_ref)
    assert_within(to_host(sst), s_ref, "ssm state")
    # the fused prefill, as the benchmark's step runs it (default workspace)
    y2 = torch.empty_like(y)
    c2, s2 = torch.empty_like(cst), torch.empty_like(sst)
    m.mamba_mixer_prefill(y2, to_dev(a["x"]), to_dev(a["dt"]), to_dev(a["B"]), to_dev(a["C"]), to_dev(p["conv_w"]),
                          to_dev(p["A_log"]), to_dev(p["conv_b"]), to_dev(p["D"]), to_dev(p["dt_bias"]),
                          to_dev(a["z"]), None, c2, None, s2)
    torch.cuda.synchronize()
    assert_within(to_host(y2), y_ref, "fused y")
    assert np.array_equal(to_host(c2), c_ref)
    assert_within(to_host(s2), s_ref, "fused ssm state")
    assert torch.equal(y2, y) and torch.equal(s2, sst), "fused prefill != conv + scan"


def test_2p8b_bf16_fused_prefill_equals_the_two_calls(cuda_lib):
    """mamba-2.8b layer at full size, as the benchmark's step runs it: the
    fused prefill equals the conv prefill followed by the scan on its bf16 u,
    bit for bit; and the fused call's own y and states match the oracle on 64
    channels spread over d_inner, run from the same x.  u is stored in bf16
    between the conv and the scan, and where that rounding falls on a tie
    boundary an f32 and an f64 conv may round to neighbouring bf16 values; so
    the oracle's scan takes the kernel's rounded u (the rounding decision made
    in the kernel's precision), and the conv's u itself is held to the oracle
    within one bf16 unit."""
    m = cuda_lib
    wl = synth.WORKLOADS[3]
    Bsz, T, Di, N, K = wl.batch, wl.seqlen, wl.d_inner, wl.d_state, wl.d_conv
    ph = synth.mixer_params(wl.seed, Di, N, K)
    p = {k: to_dev(v) for k, v in ph.items()}
    a = synth.prefill_inputs(wl.seed, Bsz, T, Di, N, "bf16", names=("x", "dt", "z", "B", "C"))
    x, dt, z, Bm, Cm = (to_dev(a[k], "bf16") for k in ("x", "dt", "z", "B", "C"))
    u = torch.empty_like(x)
    c1 = torch.empty((Bsz, Di, K), device="cuda")
    m.mamba_conv1d_silu_prefill(u, x, p["conv_w"], p["conv_b"], None, c1)
    y1 = torch.empty((Bsz, T, Di), device="cuda")
    s1 = torch.empty((Bsz, Di, N), device="cuda")
    m.mamba_selective_scan_prefill(y1, u, dt, Bm, Cm, p["A_log"], p["D"], p["dt_bias"], z, None, s1)
    y2 = torch.empty_like(y1)
    c2, s2 = torch.empty_like(c1), torch.empty_like(s1)
    m.mamba_mixer_prefill(y2, x, dt, Bm, Cm, p["conv_w"], p["A_log"], p["conv_b"], p["D"], p["dt_bias"], z,
                          None, c2, None, s2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(c1, c2) and torch.equal(s1, s2)

    sel = np.arange(11, Di, Di // 64)[:64]
    col = lambda t: np.ascontiguousarray(t[:, :, sel])
    ps = {k: np.ascontiguousarray(v[sel]) for k, v in ph.items()}
    u_ref, c_ref = oracle.conv1d_silu_prefill(col(a["x"]), ps["conv_w"], ps["conv_b"], None)
    u_gpu = to_host(u[:, :, sel])
    assert_within(u_gpu, u_ref, "u (bf16)", bf16_out=True)
    y_ref, s_ref = oracle.selective_scan_prefill(u_gpu, col(a["dt"]), a["B"], a["C"], ps["A_log"], ps["D"],
                                                 ps["dt_bias"], col(a["z"]), None)
    assert_within(to_host(y2[:, :, sel]), y_ref, "fused y (64 sampled channels, every token)")
    assert_within(to_host(s2[:, sel]), s_ref, "fused ssm state")
    assert np.array_equal(to_host(c2[:, sel]), c_ref)


def test_2p8b_bf16_prefill_sampled(cuda_lib):
    """mamba-2.8b layer (8 x 4096 x 5120, bf16 storage): conv and scan on the
    GPU at full size; the oracle checks 64 channels spread over d_inner."""
    m = cuda_lib
    wl = synth.WORKLOADS[3]
    Bsz, T, Di, N, K = wl.batch, wl.seqlen, wl.d_inner, wl.d_state, wl.d_conv
    p = synth.mixer_params(wl.seed, Di, N, K)
    a = synth.prefill_inputs(wl.seed, Bsz, T, Di, N, "bf16", names=("x", "u", "dt", "z", "B", "C"))
    x = to_dev(a["x"], "bf16")
    u = torch.empty_like(x)
    cst = torch.empty((Bsz, Di, K), device="cuda")
    m.mamba_conv1d_silu_prefill(u, x, to_dev(p["conv_w"]), to_dev(p["conv_b"]), None, cst)
    y = torch.empty((Bsz, T, Di), device="cuda")
    sst = torch.empty((Bsz, Di, N), device="cuda")
    # the scan is checked on its own seeded bf16 input u (not the conv's output)
    m.mamba_selective_scan_prefill(y, to_dev(a["u"], "bf16"), to_dev(a["dt"], "bf16"), to_dev(a["B"], "bf16"),
                                   to_dev(a["C"], "bf16"), to_dev(p["A_log"]), to_dev(p["D"]),
                                   to_dev(p["dt_bias"]), to_dev(a["z"], "bf16"), None, sst)
    torch.cuda.synchronize()
    sel = np.arange(7, Di, Di // 64)[:64]
    col = lambda t: np.ascontiguousarray(t[:, :, sel])
    ps = {k: np.ascontiguousarray(v[sel]) for k, v in p.items()}
    u_ref, c_ref = oracle.conv1d_silu_prefill(col(a["x"]), ps["conv_w"], ps["conv_b"], None)
    y_ref, s_ref = oracle.selective_scan_prefill(col(a["u"]), col(a["dt"]), a["B"], a["C"], ps["A_log"],
                                                 ps["D"], ps["dt_bias"], col(a["z"]), None)
    assert_within(to_host(u[:, :, sel]), u_ref, "u (bf16)", bf16_out=True)
    assert np.array_equal(to_host(cst[:, sel]), c_ref)
    assert_within(to_host(y[:, :, sel]), y_ref, "y")
    assert_within(to_host(sst[:, sel]), s_ref, "ssm state")


def _decode_layer_params(wl):
    return [synth.mixer_params(wl.seed, wl.d_inner, wl.d_state, wl.d_conv, layer=l) for l in range(wl.n_layers)]


def test_decode_24_layers_first_steps_full(cuda_lib):
    """24-layer batch-128 decode from the seeded state: 4 steps, every output
    of every layer and the whole state checked (conv step then SSM step)."""
    m = cuda_lib
    wl = synth.WORKLOADS[2]
    L, Bsz, Di, N, K = wl.n_layers, wl.batch, wl.d_inner, wl.d_state, wl.d_conv
    conv_h, ssm_h = synth.seeded_states(wl.seed, L, Bsz, Di, N, K)
    conv, ssm = to_dev(conv_h), to_dev(ssm_h)
    conv_ref, ssm_ref = conv_h.astype(np.float64), ssm_h.astype(np.float64)
    params = _decode_layer_params(wl)
    pd = [{k: to_dev(v) for k, v in p.items()} for p in params]
    for step in range(4):
        for l in range(L):
            inp = synth.decode_step_inputs(wl.seed, l, step, Bsz, Di, N)
            u = torch.empty((Bsz, Di), device="cuda")
            y = torch.empty((Bsz, Di), device="cuda")
            m.mamba_conv1d_silu_step(u, to_dev(inp["x"]), conv, l, pd[l]["conv_w"], pd[l]["conv_b"])
            m.mamba_ssm_step_batched(y, u, to_dev(inp["dt"]), to_dev(inp["B"]), to_dev(inp["C"]), ssm, l,
                                     pd[l]["A_log"], pd[l]["D"], pd[l]["dt_bias"], to_dev(inp["z"]))
            u_ref = oracle.conv1d_silu_step(inp["x"], conv_ref, l, params[l]["conv_w"], params[l]["conv_b"])
            y_ref = oracle.ssm_step(u_ref, inp["dt"], inp["B"], inp["C"], ssm_ref, l, params[l]["A_log"],
                                    params[l]["D"], params[l]["dt_bias"], inp["z"])
            torch.cuda.synchronize()
            assert_within(to_host(u), u_ref, f"u step {step} layer {l}")
            assert_within(to_host(y), y_ref, f"y step {step} layer {l}")
    assert np.array_equal(to_host(conv), conv_ref)
    assert_within(to_host(ssm), ssm_ref, "ssm state after 4 steps")


def test_decode_256_steps_as_captured_graph_sampled_rows(cuda_lib):
    """The bench's configuration: 256 steps x 24 layers in one CUDA graph with
    fresh inputs per (layer, step) drawn on the device; the oracle replays 24
    sampled (batch, channel) rows through all 256 steps and 24 layers."""
    m = cuda_lib
    wl = synth.WORKLOADS[2]
    L, Bsz, Di, N, K, S = wl.n_layers, wl.batch, wl.d_inner, wl.d_state, wl.d_conv, 256
    conv_h, ssm_h = synth.seeded_states(wl.seed, L, Bsz, Di, N, K)
    conv, ssm = to_dev(conv_h), to_dev(ssm_h)
    params = _decode_layer_params(wl)
    pd = [{k: to_dev(v) for k, v in p.items()} for p in params]
    x = synth.torch_normal((S, L, Bsz, Di), 1.0, wl.seed + 11, "cuda")
    z = synth.torch_normal((S, L, Bsz, Di), 1.0, wl.seed + 12, "cuda")
    dt = synth.torch_normal((S, L, Bsz, Di), 0.1, wl.seed + 13, "cuda")
    Bm = synth.torch_normal((S, L, Bsz, N), 1.0, wl.seed + 14, "cuda")
    Cm = synth.torch_normal((S, L, Bsz, N), 1.0, wl.seed + 15, "cuda")
    u = torch.empty((L, Bsz, Di), device="cuda")
    y = torch.empty((S, L, Bsz, Di), device="cuda")

    def body():
        for s in range(S):
            for l in range(L):
                m.mamba_conv1d_silu_step(u[l], x[s, l], conv, l, pd[l]["conv_w"], pd[l]["conv_b"])
                m.mamba_ssm_step_batched(y[s, l], u[l], dt[s, l], Bm[s, l], Cm[s, l], ssm, l, pd[l]["A_log"],
                                         pd[l]["D"], pd[l]["dt_bias"], z[s, l])

    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        with torch.cuda.graph(g, stream=st, capture_error_mode="relaxed"):
            body()
    torch.cuda.current_stream().wait_stream(st)
    g.replay()
    torch.cuda.synchronize()

    # oracle: the cross product of 24 sampled batch rows x 24 sampled channels
    # (576 independent rows) replayed through all steps and layers
    rng = np.random.default_rng(7)
    bs = np.sort(rng.choice(Bsz, 24, replace=False))
    cs = np.sort(rng.choice(Di, 24, replace=False))
    pick = lambda t: to_host(t[:, :, bs][:, :, :, cs])               # [S, L, 24, 24]
    xs, zs, dts = pick(x), pick(z), pick(dt)
    Bs, Cs = to_host(Bm[:, :, bs]), to_host(Cm[:, :, bs])            # [S, L, 24, N]
    conv_r = np.ascontiguousarray(conv_h[:, bs][:, :, cs].astype(np.float64))   # [L, 24, 24, K]
    ssm_r = np.ascontiguousarray(ssm_h[:, bs][:, :, cs].astype(np.float64))     # [L, 24, 24, N]
    ps = [{k: np.ascontiguousarray(v[cs]) for k, v in p.items()} for p in params]
    y_ref = np.empty((S, L, 24, 24))
    for s in range(S):
        for l in range(L):
            ur = oracle.conv1d_silu_step(xs[s, l], conv_r, l, ps[l]["conv_w"], ps[l]["conv_b"], nthreads=4)
            y_ref[s, l] = oracle.ssm_step(ur, dts[s, l], Bs[s, l], Cs[s, l], ssm_r, l, ps[l]["A_log"], ps[l]["D"],
                                          ps[l]["dt_bias"], zs[s, l], nthreads=4)
    assert_within(pick(y), y_ref, "y (24 x 24 sampled rows, 256 steps x 24 layers)")
    assert_within(to_host(ssm[:, bs][:, :, cs]), ssm_r, "ssm state (sampled rows)")
    assert np.array_equal(to_host(conv[:, bs][:, :, cs]), conv_r)


def test_long_context_continuation(cuda_lib):
    """Batch 4, d_inner 2048: prefill 16384 tokens from a seeded state, then 64
    T=1 decode steps, must match one 16448-token prefill (GPU vs GPU, every
    element) and the oracle on 32 sampled channels (every token)."""
    m = cuda_lib
    wl = synth.WORKLOADS[4]
    Bsz, T, Di, N, K, S = wl.batch, wl.seqlen, wl.d_inner, wl.d_state, wl.d_conv, wl.steps
    TT = T + S
    p = synth.mixer_params(wl.seed, Di, N, K)
    a = synth.prefill_inputs(wl.seed, Bsz, TT, Di, N, "f32", names=("x", "dt", "z", "B", "C"))
    conv0, ssm0 = synth.seeded_states(wl.seed, 1, Bsz, Di, N, K, ssm_std=0.5, conv_std=1.0)
    conv0, ssm0 = conv0[0], ssm0[0]
    pd = {k: to_dev(v) for k, v in p.items()}
    dev = {k: to_dev(v) for k, v in a.items()}

    # one prefill of all 16448 tokens
    u1 = torch.empty_like(dev["x"])
    c1 = torch.empty((Bsz, Di, K), device="cuda")
    m.mamba_conv1d_silu_prefill(u1, dev["x"], pd["conv_w"], pd["conv_b"], to_dev(conv0), c1)
    y1 = torch.empty_like(dev["x"])
    s1 = torch.empty((Bsz, Di, N), device="cuda")
    m.mamba_selective_scan_prefill(y1, u1, dev["dt"], dev["B"], dev["C"], pd["A_log"], pd["D"], pd["dt_bias"],
                                   dev["z"], to_dev(ssm0), s1)

    # prefill 16384, then 64 steps on a 1-layer persistent state (the ABI takes
    # a batch stride of T rows, so the first-T slices are copied out)
    head = lambda k: dev[k][:, :T].contiguous()
    x2 = head("x")
    u2 = torch.empty_like(x2)
    conv = torch.empty((1, Bsz, Di, K), device="cuda")
    ssm = torch.empty((1, Bsz, Di, N), device="cuda")
    m.mamba_conv1d_silu_prefill(u2, x2, pd["conv_w"], pd["conv_b"], to_dev(conv0), conv[0])
    y2 = torch.empty_like(dev["x"])
    y2h = torch.empty_like(x2)
    m.mamba_selective_scan_prefill(y2h, u2, head("dt"), head("B"), head("C"), pd["A_log"],
                                   pd["D"], pd["dt_bias"], head("z"), to_dev(ssm0), ssm[0])
    y2[:, :T].copy_(y2h)
    for s in range(S):
        t = T + s
        us = torch.empty((Bsz, Di), device="cuda")
        ys = torch.empty((Bsz, Di), device="cuda")
        m.mamba_conv1d_silu_step(us, dev["x"][:, t].contiguous(), conv, 0, pd["conv_w"], pd["conv_b"])
        m.mamba_ssm_step_batched(ys, us, dev["dt"][:, t].contiguous(), dev["B"][:, t].contiguous(),
                                 dev["C"][:, t].contiguous(), ssm, 0, pd["A_log"], pd["D"], pd["dt_bias"],
                                 dev["z"][:, t].contiguous())
        y2[:, t].copy_(ys)
    torch.cuda.synchronize()

    # the same continuation through the fused calls: mamba_mixer_prefill over
    # the first 16384 tokens, then 64 mamba_mixer_step_batched steps
    conv_f = torch.empty((1, Bsz, Di, K), device="cuda")
    ssm_f = torch.empty((1, Bsz, Di, N), device="cuda")
    y3 = torch.empty_like(dev["x"])
    y3h = torch.empty_like(x2)
    m.mamba_mixer_prefill(y3h, x2, head("dt"), head("B"), head("C"), pd["conv_w"], pd["A_log"], pd["conv_b"],
                          pd["D"], pd["dt_bias"], head("z"), to_dev(conv0), conv_f[0], to_dev(ssm0), ssm_f[0])
    y3[:, :T].copy_(y3h)
    for s in range(S):
        t = T + s
        ys = torch.empty((Bsz, Di), device="cuda")
        m.mamba_mixer_step_batched(ys, dev["x"][:, t].contiguous(), dev["dt"][:, t].contiguous(),
                                   dev["B"][:, t].contiguous(), dev["C"][:, t].contiguous(), conv_f, ssm_f, 0,
                                   pd["conv_w"], pd["A_log"], pd["conv_b"], pd["D"], pd["dt_bias"],
                                   dev["z"][:, t].contiguous())
        y3[:, t].copy_(ys)
    torch.cuda.synchronize()
    # the fused forms equal the separate calls bit for bit (u is f32 here)
    assert torch.equal(y3, y2), "fused prefill + fused steps != conv/scan prefill + conv/ssm steps"
    assert torch.equal(ssm_f, ssm) and torch.equal(conv_f, conv)

    Y1, Y2 = to_host(y1), to_host(y2)
    assert_within(Y2, Y1, "y: prefill+steps vs one prefill")
    assert_within(to_host(ssm[0]), to_host(s1), "ssm state: prefill+steps vs one prefill")
    assert np.array_equal(to_host(conv[0]), to_host(c1))

    sel = np.arange(3, Di, Di // 32)[:32]
    col = lambda t: np.ascontiguousarray(t[:, :, sel])
    ps = {k: np.ascontiguousarray(v[sel]) for k, v in p.items()}
    u_ref, c_ref = oracle.conv1d_silu_prefill(col(a["x"]), ps["conv_w"], ps["conv_b"],
                                              np.ascontiguousarray(conv0[:, sel]))
    y_ref, s_ref = oracle.selective_scan_prefill(u_ref, col(a["dt"]), a["B"], a["C"], ps["A_log"], ps["D"],
                                                 ps["dt_bias"], col(a["z"]), np.ascontiguousarray(ssm0[:, sel]))
    assert_within(Y2[:, :, sel], y_ref, "y vs oracle (sampled channels, 16448 tokens)")
    assert_within(to_host(ssm[0][:, sel]), s_ref, "ssm state vs oracle")
    assert np.array_equal(to_host(conv[0][:, sel]), c_ref)


def test_prefill_beyond_2pow31_activation_elements(cuda_lib):
    """B*T*Di = 2.2e9 > 2^31 activation elements (every index 64-bit): the fused
    prefill equals conv prefill + scan prefill bit for bit at full size, and
    both match the oracle on 4 channels (first, last, two in between) over all
    2.1M tokens, with the final states."""
    m = cuda_lib
    Bsz, T, Di, N, K = 1, (1 << 21) + 17, 1056, 16, 4
    assert Bsz * T * Di > 2 ** 31
    SEED = 0x5EED0B16
    p = synth.mixer_params(SEED, Di, N, K)
    pd = {k: to_dev(v) for k, v in p.items()}
    x = synth.torch_normal((Bsz, T, Di), 1.0, SEED + 901, "cuda")
    dt = synth.torch_normal((Bsz, T, Di), 0.1, SEED + 902, "cuda")
    z = synth.torch_normal((Bsz, T, Di), 1.0, SEED + 903, "cuda")
    Bm = synth.torch_normal((Bsz, T, N), 1.0, SEED + 904, "cuda")
    Cm = synth.torch_normal((Bsz, T, N), 1.0, SEED + 905, "cuda")
    y = torch.empty((Bsz, T, Di), device="cuda")
    c1, s1 = torch.empty((Bsz, Di, K), device="cuda"), torch.empty((Bsz, Di, N), device="cuda")
    m.mamba_mixer_prefill(y, x, dt, Bm, Cm, pd["conv_w"], pd["A_log"], pd["conv_b"], pd["D"], pd["dt_bias"], z,
                          None, c1, None, s1)
    u = torch.empty_like(x)
    c2, s2 = torch.empty_like(c1), torch.empty_like(s1)
    m.mamba_conv1d_silu_prefill(u, x, pd["conv_w"], pd["conv_b"], None, c2)
    y2 = torch.empty_like(y)
    m.mamba_selective_scan_prefill(y2, u, dt, Bm, Cm, pd["A_log"], pd["D"], pd["dt_bias"], z, None, s2)
    torch.cuda.synchronize()
    assert torch.equal(y, y2), "fused prefill != conv prefill + scan prefill at > 2^31 elements"
    assert torch.equal(c1, c2) and torch.equal(s1, s2)
    del u, y2
    sel = np.array([0, 517, 1030, Di - 1])
    idx = torch.as_tensor(sel, device="cuda")
    col = lambda t: np.ascontiguousarray(t.index_select(2, idx).cpu().numpy().astype(np.float64))
    ps = {k: np.ascontiguousarray(v[sel]) for k, v in p.items()}
    u_ref, c_ref = oracle.conv1d_silu_prefill(col(x), ps["conv_w"], ps["conv_b"], None)
    y_ref, s_ref = oracle.selective_scan_prefill(u_ref, col(dt), to_host(Bm).astype(np.float64),
                                                 to_host(Cm).astype(np.float64), ps["A_log"], ps["D"],
                                                 ps["dt_bias"], col(z), None)
    assert_within(col(y), y_ref, "y (4 channels, all tokens)")
    assert_within(to_host(s1[:, sel]), s_ref, "ssm state")
    assert np.array_equal(to_host(c1[:, sel]), c_ref)
