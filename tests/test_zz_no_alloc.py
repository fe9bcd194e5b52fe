"""mamba_selective_scan_prefill_noalloc against mamba_selective_scan_prefill.

The no-allocation variant serves callers that cannot allocate device memory:
its T-split scratch is a static array inside the library instead of a caller
workspace.  On a narrow shape that the planner splits along T it must give the
same y and final state as the regular entry point (same kernels, same plan),
on two calls in a row with different inputs, so the shared scratch is reused.
This file is named to run last: it must pass both alone and after the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

from selective_state_space_conv1d_gb300 import synth
from _helpers import assert_within, to_dev, to_host

pytestmark = pytest.mark.gpu


def _inputs(seed, Bsz, T, Di, N):
    a = synth.prefill_inputs(seed, Bsz, T, Di, N, "f32", names=("u", "dt", "z", "B", "C"))
    p = synth.mixer_params(seed, Di, N, 4)
    s0 = synth.normal(seed, "ssm_state", (Bsz, Di, N), 0.5)
    return {k: to_dev(v) for k, v in a.items()}, {k: to_dev(v) for k, v in p.items()}, to_dev(s0)


def _call_regular(m, a, p, s0, ws):
    y = torch.empty_like(a["u"])
    s = torch.empty_like(s0)
    m.mamba_selective_scan_prefill(y, a["u"], a["dt"], a["B"], a["C"], p["A_log"], p["D"], p["dt_bias"],
                                   a["z"], s0, s, workspace=ws)
    return y, s


def _call_noalloc_through_c_abi(m, a, p, s0):
    """Direct C-ABI call: plain pointers and sizes, no workspace argument."""
    lib = m.load()
    y = torch.empty_like(a["u"])
    s = torch.empty_like(s0)
    Bsz, T, Di = a["u"].shape
    N = p["A_log"].shape[1]
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lib.mamba_selective_scan_prefill_noalloc(
        y.data_ptr(), Di, 0, a["u"].data_ptr(), Di, a["dt"].data_ptr(), Di, a["z"].data_ptr(), Di,
        a["B"].data_ptr(), N, a["C"].data_ptr(), N, 0, p["A_log"].data_ptr(), p["D"].data_ptr(),
        p["dt_bias"].data_ptr(), s0.data_ptr(), s.data_ptr(), Bsz, T, Di, N, stream)
    assert rc == 0, m.mamba_last_error()
    return y, s


def test_noalloc_matches_regular_entry_point_on_two_calls(cuda_lib):
    m = cuda_lib
    Bsz, T, Di, N = 1, 2048, 1536, 16  # one 130m layer at batch 1: split along T
    need = m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
    assert 0 < need <= m.MAMBA_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((0x5EED2000, 0x5EED2001)):
        a, p, s0 = _inputs(seed, Bsz, T, Di, N)
        y_ref, s_ref = _call_regular(m, a, p, s0, ws)
        y, s = _call_noalloc_through_c_abi(m, a, p, s0)
        torch.cuda.synchronize()
        assert_within(to_host(y), to_host(y_ref), f"y, call {call}")
        assert_within(to_host(s), to_host(s_ref), f"state, call {call}")


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_lib):
    m = cuda_lib
    # a long batch-1 prefill with d_state 64 splits along T and needs more
    # scratch than the static array holds (nothing is allocated or launched)
    Bsz, T, Di, N = 1, 1 << 20, 2048, 64
    need = m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
    if need <= m.MAMBA_NOALLOC_SCRATCH_BYTES:
        pytest.skip("planner does not split this shape on this device")
    lib = m.load()
    fake = ctypes.c_void_p(0x100000)  # rejected before any pointer is used
    rc = lib.mamba_selective_scan_prefill_noalloc(
        fake, Di, 0, fake, Di, fake, Di, None, 0, fake, N, fake, N, 0, fake, None, None, None, None,
        Bsz, T, Di, N, None)
    assert rc == m.MAMBA_ERR_UNSUPPORTED
    assert "scratch" in m.mamba_last_error()
