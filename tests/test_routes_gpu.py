"""GPU parity of the chained route: a wide prefill (at least as many
32-channel tiles as the GPU holds warps) is laid out as one run of tile-rows
and cut into equal roles, one per warp; a tile cut between two roles is handed
from one to the next through the workspace.  Every row is scanned once, in the
same order and with the same arithmetic as the one-pass route (no workspace),
so the two agree bit for bit; sampled channels are also checked against the
oracle (channels are independent recurrences, so a sample is a full-fidelity
check of those channels)."""
import numpy as np
import pytest
import torch

import oracle
from selective_state_space_conv1d_gb300 import synth
from _helpers import assert_within, to_dev, to_host

pytestmark = pytest.mark.gpu

SEED = 0x5EED3000


def _sample(Di):
    return np.unique(np.concatenate([np.arange(5, Di, Di // 12)[:12], [0, 31, 32, Di - 1]]))


@pytest.mark.parametrize("dtype,fused,gate,inplace,Di,T,K", [
    ("f32", False, True, False, 8184, 1300, 4),   # ragged last tile
    ("bf16", False, True, True, 8192, 1100, 4),
    ("f32", True, True, True, 8184, 1300, 4),
    ("bf16", True, False, False, 8192, 1537, 4),
    ("f32", True, True, False, 8184, 333, 3),      # roles span several whole tiles
    ("bf16", True, True, False, 8192, 1030, 2),
])
def test_chained_route_equals_one_pass_and_matches_oracle(cuda_lib, dtype, fused, gate, inplace, Di, T, K):
    m = cuda_lib
    Bsz, N = 6, 16
    need = m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
    assert need > 0, "expected the chained route for this wide shape"
    p = synth.parity_params(SEED + K, Di, N, K)
    pd = {k: to_dev(v) for k, v in p.items()}
    x = synth.torch_normal((Bsz, T, Di), 1.0, SEED + 1, "cuda", torch.bfloat16 if dtype == "bf16" else None)
    dt = synth.torch_normal((Bsz, T, Di), 0.1, SEED + 2, "cuda", x.dtype)
    z = synth.torch_normal((Bsz, T, Di), 1.0, SEED + 3, "cuda", x.dtype) if gate else None
    Bm = synth.torch_normal((Bsz, T, N), 1.0, SEED + 4, "cuda", x.dtype)
    Cm = synth.torch_normal((Bsz, T, N), 1.0, SEED + 5, "cuda", x.dtype)
    s0 = synth.torch_normal((Bsz, Di, N), 0.5, SEED + 6, "cuda")
    c0 = synth.torch_normal((Bsz, Di, K), 1.0, SEED + 7, "cuda")

    def run(workspace):
        y = torch.empty((Bsz, T, Di), device="cuda")
        s_in = s0.clone()
        s_out = s_in if inplace else torch.empty_like(s0)
        c_in = c0.clone()
        c_out = c_in if inplace else torch.empty_like(c0)
        if fused:
            m.mamba_mixer_prefill(y, x, dt, Bm, Cm, pd["conv_w"], pd["A_log"], pd["conv_b"], pd["D"], pd["dt_bias"],
                                  z, c_in, c_out, s_in, s_out, workspace=workspace)
        else:
            m.mamba_selective_scan_prefill(y, x, dt, Bm, Cm, pd["A_log"], pd["D"], pd["dt_bias"], z, s_in, s_out,
                                           workspace=workspace)
        torch.cuda.synchronize()
        return y, s_out, c_out

    y1, s1, c1 = run(None)    # chained (the default workspace)
    y2, s2, c2 = run(False)   # one pass per tile
    assert torch.equal(y1, y2), "chained route != one-pass route"
    assert torch.equal(s1, s2)
    if fused:
        assert torch.equal(c1, c2)
    assert m.mamba_device_faults(clear=True) == 0

    sel = _sample(Di)
    idx = torch.as_tensor(sel, device="cuda")
    col = lambda t: np.ascontiguousarray(t.index_select(2, idx).float().cpu().numpy().astype(np.float64))
    ps = {k: np.ascontiguousarray(v[sel]) for k, v in p.items()}
    s0h = np.ascontiguousarray(s0.cpu().numpy()[:, sel])
    if fused:
        u = torch.empty_like(x)
        m.mamba_conv1d_silu_prefill(u, x, pd["conv_w"], pd["conv_b"], c0, None)
        torch.cuda.synchronize()
        u_ref, c_ref = oracle.conv1d_silu_prefill(col(x), ps["conv_w"], ps["conv_b"],
                                                  np.ascontiguousarray(c0.cpu().numpy()[:, sel]))
        # a bf16 u is rounded once between the conv and the scan: the oracle's scan
        # takes the kernel's rounding (checked against the oracle's u here)
        assert_within(col(u), u_ref, "u", bf16_out=dtype == "bf16")
        u_in = col(u)
        assert np.array_equal(to_host(c1[:, sel]), c_ref)
    else:
        u_in = col(x)
    y_ref, s_ref = oracle.selective_scan_prefill(u_in, col(dt), to_host(Bm), to_host(Cm), ps["A_log"], ps["D"],
                                                 ps["dt_bias"], col(z) if gate else None, s0h)
    assert_within(col(y1), y_ref, "y (sampled channels)")
    assert_within(to_host(s1[:, sel]), s_ref, "ssm state (sampled channels)")


def test_chained_route_two_calls_in_a_row_reuse_the_workspace(cuda_lib):
    """The workspace header is cleared by every call: a second call with the
    same workspace and other inputs gives the one-pass result again."""
    m = cuda_lib
    Bsz, T, Di, N = 6, 1200, 8192, 16
    need = m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
    assert need > 0, "expected the chained route for this wide shape"
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ws.fill_(0xAB)  # contents on entry are ignored
    p = {k: to_dev(v) for k, v in synth.parity_params(SEED, Di, N, 4).items()}
    for call in range(2):
        u, dt, z = (synth.torch_normal((Bsz, T, Di), s, SEED + 10 * call + i, "cuda")
                    for i, s in ((1, 1.0), (2, 0.1), (3, 1.0)))
        Bm, Cm = (synth.torch_normal((Bsz, T, N), 1.0, SEED + 10 * call + i, "cuda") for i in (4, 5))
        out = []
        for w in (ws, False):
            y = torch.empty_like(u)
            s = torch.empty((Bsz, Di, N), device="cuda")
            m.mamba_selective_scan_prefill(y, u, dt, Bm, Cm, p["A_log"], p["D"], p["dt_bias"], z, None, s,
                                           workspace=w)
            out.append((y, s))
        torch.cuda.synchronize()
        assert torch.equal(out[0][0], out[1][0]) and torch.equal(out[0][1], out[1][1]), f"call {call}"
    assert m.mamba_device_faults(clear=True) == 0
