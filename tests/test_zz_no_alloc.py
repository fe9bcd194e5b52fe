"""mamba_selective_scan_prefill_noalloc against mamba_selective_scan_prefill.

The no-allocation variant serves callers that cannot allocate device memory
when they run the prefill (an engine whose device memory is fixed at start-up,
a plugin inside a framework that owns the allocator): its T-split scratch is a
static array inside the library instead of a caller workspace.  It runs the
same plan and the same kernels as the regular entry point given a workspace of
min(required size, the array), so the two must agree bit for bit, on two calls
in a row with different inputs (the shared scratch is reused).
This file is named to run last: it must pass both alone and after the rest.
"""
import ctypes

import numpy as np
import pytest
import torch

from selective_state_space_conv1d_gb300 import synth
from _helpers import to_dev

pytestmark = pytest.mark.gpu


def _inputs(seed, Bsz, T, Di, N):
    a = synth.prefill_inputs(seed, Bsz, T, Di, N, "f32", names=("u", "dt", "z", "B", "C"))
    p = synth.parity_params(seed, Di, N, 4)
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
        assert torch.equal(y, y_ref), f"y differs from the regular entry point, call {call}"
        assert torch.equal(s, s_ref), f"state differs from the regular entry point, call {call}"


def test_noalloc_splits_a_long_context_shape_within_its_scratch(cuda_lib):
    """Batch 4 x T 16384 x d_inner 2048: the planned split needs more than the
    array; the variant splits into as many parts as fit, exactly as the regular
    entry point does when given a workspace the size of the array."""
    m = cuda_lib
    Bsz, T, Di, N = 4, 16384, 2048, 16
    need = m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
    if need <= m.MAMBA_NOALLOC_SCRATCH_BYTES:
        pytest.skip("the plan for this shape fits the array on this device")
    ws = torch.empty(m.MAMBA_NOALLOC_SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
    for call, seed in enumerate((0x5EED2010, 0x5EED2011)):
        a, p, s0 = _inputs(seed, Bsz, T, Di, N)
        y_ref, s_ref = _call_regular(m, a, p, s0, ws)
        y, s = _call_noalloc_through_c_abi(m, a, p, s0)
        torch.cuda.synchronize()
        assert torch.equal(y, y_ref), f"y differs from the regular entry point, call {call}"
        assert torch.equal(s, s_ref), f"state differs from the regular entry point, call {call}"


def test_noalloc_python_wrapper_matches_the_c_abi_call(cuda_lib):
    m = cuda_lib
    a, p, s0 = _inputs(0x5EED2020, 1, 1500, 512, 16)
    y1, s1 = _call_noalloc_through_c_abi(m, a, p, s0)
    y2, s2 = torch.empty_like(y1), torch.empty_like(s1)
    m.mamba_selective_scan_prefill_noalloc(y2, a["u"], a["dt"], a["B"], a["C"], p["A_log"], p["D"],
                                           p["dt_bias"], a["z"], s0, s2)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2) and torch.equal(s1, s2)


def test_noalloc_rejects_shapes_beyond_its_scratch(cuda_lib):
    """A shape split along T (fewer 32-channel tiles than half the warps the GPU
    holds, eight per SM) whose two parts need three state slots of more than a
    third of the array is refused before anything is allocated or launched."""
    m = cuda_lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    tiles = (8 * sms + 1) // 2 - 1  # the widest shape the planner still splits
    Bsz, T, Di, N = 1, 1 << 20, tiles * 32, 64
    if 3 * Bsz * Di * N * 4 <= m.MAMBA_NOALLOC_SCRATCH_BYTES:
        pytest.skip(f"with {sms} SMs every shape split along T fits two parts in the static array")
    lib = m.load()
    fake = ctypes.c_void_p(0x100000)  # rejected before any pointer is used
    rc = lib.mamba_selective_scan_prefill_noalloc(
        fake, Di, 0, fake, Di, fake, Di, None, 0, fake, N, fake, N, 0, fake, None, None, None, None,
        Bsz, T, Di, N, None)
    assert rc == m.MAMBA_ERR_UNSUPPORTED
    assert "scratch" in m.mamba_last_error()
