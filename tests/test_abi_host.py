"""Host-side checks of the C ABI (no GPU needed).

The library must build for sm_103a, load, export every symbol include/*.h
declares, and reject bad arguments on the host before touching a device.
"""
import ctypes
import glob
import os
import re
import subprocess

import pytest

import selective_state_space_conv1d_gb300 as m
from selective_state_space_conv1d_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = ctypes.c_void_p(0x100000)  # never dereferenced: the calls below fail before any device work


@pytest.fixture(scope="module")
def lib():
    B.build()
    return m.load()


def header_symbols():
    syms = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        txt = open(h).read()
        syms |= set(re.findall(r"MAMBA_API\s+[\w\s\*]+?\b(mamba\w+)\s*\(", txt))
    return syms


def test_header_declares_the_four_entry_points():
    syms = header_symbols()
    for s in ("mamba_conv1d_silu_prefill", "mamba_conv1d_silu_step",
              "mamba_selective_scan_prefill", "mamba_ssm_step_batched", "mamba_last_error"):
        assert s in syms
    assert syms == set(m.ABI_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(mamba\w+)", out))
    assert header_symbols() <= exported
    for s in header_symbols():
        assert hasattr(lib, s)
    # nothing but the ABI leaks out of the library
    assert exported == header_symbols()


def test_library_is_built_for_sm_103a_only(lib):
    out = subprocess.run(["cuobjdump", "--list-elf", B.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("cuobjdump unavailable")
    arches = set(re.findall(r"sm_(\d+a?)", out.stdout))
    assert arches == {"103a"}, arches


def test_version_and_error_string(lib):
    assert m.mamba_version() == "0.1.0"
    assert isinstance(m.mamba_last_error(), str)


def _scan(lib, **kw):
    a = dict(y=FAKE, ld_y=8, y_dtype=0, u=FAKE, ld_u=8, dt=FAKE, ld_dt=8, z=None, ld_z=0,
             Bm=FAKE, ld_B=16, Cm=FAKE, ld_C=16, in_dtype=0, A_log=FAKE, D=None, dt_bias=None,
             s_in=None, s_out=None, B=1, T=4, Di=8, N=16, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return lib.mamba_selective_scan_prefill(
        a["y"], a["ld_y"], a["y_dtype"], a["u"], a["ld_u"], a["dt"], a["ld_dt"], a["z"], a["ld_z"],
        a["Bm"], a["ld_B"], a["Cm"], a["ld_C"], a["in_dtype"], a["A_log"], a["D"], a["dt_bias"],
        a["s_in"], a["s_out"], a["B"], a["T"], a["Di"], a["N"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(y_dtype=7), m.MAMBA_ERR_INVALID_ARG),
    (dict(in_dtype=-1), m.MAMBA_ERR_INVALID_ARG),
    (dict(B=-1), m.MAMBA_ERR_INVALID_ARG),
    (dict(T=-5), m.MAMBA_ERR_INVALID_ARG),
    (dict(N=3), m.MAMBA_ERR_UNSUPPORTED),
    (dict(N=65), m.MAMBA_ERR_UNSUPPORTED),
    (dict(N=128), m.MAMBA_ERR_UNSUPPORTED),
    (dict(u=None), m.MAMBA_ERR_INVALID_ARG),
    (dict(y=None), m.MAMBA_ERR_INVALID_ARG),
    (dict(A_log=None), m.MAMBA_ERR_INVALID_ARG),
    (dict(ld_u=7), m.MAMBA_ERR_INVALID_ARG),
    (dict(ld_z=4, z=FAKE), m.MAMBA_ERR_INVALID_ARG),
    (dict(ld_B=15), m.MAMBA_ERR_INVALID_ARG),
    (dict(B=1 << 40, T=1 << 40), m.MAMBA_ERR_INVALID_ARG),
    (dict(ws=FAKE, ws_bytes=-1), m.MAMBA_ERR_INVALID_ARG),
])
def test_scan_rejects_bad_arguments_on_host(lib, kw, code):
    assert _scan(lib, **kw) == code
    assert m.mamba_last_error() != ""


def test_zero_sized_calls_are_noops(lib):
    assert _scan(lib, B=0) == m.MAMBA_OK
    assert _scan(lib, Di=0) == m.MAMBA_OK
    assert m.mamba_last_error() == ""
    assert lib.mamba_conv1d_silu_prefill(None, 0, None, 0, 0, None, None, FAKE, None, 0, 5, 8, 4, None) == 0


def test_workspace_query_rejects_bad_sizes(lib):
    assert lib.mamba_selective_scan_workspace_bytes(1, 10, 8, 3) == m.MAMBA_ERR_UNSUPPORTED
    assert lib.mamba_selective_scan_workspace_bytes(-1, 10, 8, 16) == m.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_selective_scan_workspace_bytes(0, 10, 8, 16) == 0
    assert lib.mamba_selective_scan_workspace_bytes(2, 0, 8, 16) == 0


@pytest.mark.parametrize("K,code", [(0, m.MAMBA_ERR_UNSUPPORTED), (9, m.MAMBA_ERR_UNSUPPORTED)])
def test_conv_rejects_unsupported_d_conv(lib, K, code):
    assert lib.mamba_conv1d_silu_prefill(FAKE, 8, FAKE, 8, 0, None, None, FAKE, None, 1, 4, 8, K, None) == code
    assert lib.mamba_conv1d_silu_step(FAKE, FAKE, 0, FAKE, 0, 1, FAKE, None, 1, 8, K, None) == code


def test_conv_rejects_bad_arguments(lib):
    E = m.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_conv1d_silu_prefill(FAKE, 4, FAKE, 8, 0, None, None, FAKE, None, 1, 4, 8, 4, None) == E
    assert lib.mamba_conv1d_silu_prefill(None, 8, FAKE, 8, 0, None, None, FAKE, None, 1, 4, 8, 4, None) == E
    assert lib.mamba_conv1d_silu_prefill(FAKE, 8, FAKE, 8, 0, None, None, None, None, 1, 4, 8, 4, None) == E
    assert lib.mamba_conv1d_silu_prefill(FAKE, 8, FAKE, 8, 2, None, None, FAKE, None, 1, 4, 8, 4, None) == E
    # layer outside [0, n_layers)
    assert lib.mamba_conv1d_silu_step(FAKE, FAKE, 0, FAKE, 3, 3, FAKE, None, 1, 8, 4, None) == E
    assert lib.mamba_conv1d_silu_step(FAKE, FAKE, 0, FAKE, -1, 3, FAKE, None, 1, 8, 4, None) == E


def test_step_rejects_bad_arguments(lib):
    E, U = m.MAMBA_ERR_INVALID_ARG, m.MAMBA_ERR_UNSUPPORTED
    f = lib.mamba_ssm_step_batched
    assert f(FAKE, 0, FAKE, FAKE, None, FAKE, FAKE, 0, FAKE, None, None, FAKE, 0, 1, 2, 8, 65, None) == U
    assert f(FAKE, 0, FAKE, FAKE, None, FAKE, FAKE, 0, FAKE, None, None, FAKE, 1, 1, 2, 8, 16, None) == E
    assert f(FAKE, 0, None, FAKE, None, FAKE, FAKE, 0, FAKE, None, None, FAKE, 0, 1, 2, 8, 16, None) == E
    assert f(FAKE, 0, FAKE, FAKE, None, FAKE, FAKE, 0, FAKE, None, None, None, 0, 1, 2, 8, 16, None) == E


def test_valid_call_without_a_gpu_fails_cleanly(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    rc = _scan(lib)
    assert rc in (m.MAMBA_ERR_CUDA, m.MAMBA_ERR_UNSUPPORTED)
    assert m.mamba_last_error()


def test_python_binding_raises_when_library_missing(tmp_path):
    from selective_state_space_conv1d_gb300 import _binding

    saved = _binding._lib
    _binding._lib = None
    try:
        with pytest.raises(RuntimeError, match="missing"):
            _binding.load(str(tmp_path / "nope.so"))
    finally:
        _binding._lib = saved


def test_decode_graph_rejects_bad_arguments_on_host(lib):
    h = ctypes.c_void_p()
    # out NULL, params / io NULL, no steps or layers: refused before any device call
    assert lib.mamba_decode_graph_create(None, FAKE, FAKE, 1, 1, 0, 0, FAKE, FAKE, 1, 8, 4, 16) == m.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_decode_graph_create(ctypes.byref(h), None, FAKE, 1, 1, 0, 0, FAKE, FAKE, 1, 8, 4, 16) \
        == m.MAMBA_ERR_INVALID_ARG
    assert h.value is None
    for n_steps, n_layers in ((0, 1), (1, 0), (-1, 4), (1 << 21, 1)):
        assert lib.mamba_decode_graph_create(ctypes.byref(h), FAKE, FAKE, n_steps, n_layers, 0, 0, FAKE, FAKE,
                                             1, 8, 4, 16) == m.MAMBA_ERR_INVALID_ARG
        assert "n_steps" in m.mamba_last_error()
    assert lib.mamba_decode_graph_launch(None, None) == m.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_decode_graph_kernels(None) == m.MAMBA_ERR_INVALID_ARG
    assert lib.mamba_decode_graph_destroy(None) == m.MAMBA_OK


def test_m3_decode_graph_rejects_bad_arguments_on_host(lib):
    h = ctypes.c_void_p()
    # out NULL, io NULL, no tokens or layers: refused before any device call
    args = lambda n_steps=1, n_layers=1: (FAKE, None, n_steps, n_layers, 0, 0, FAKE, FAKE, FAKE, FAKE, 2, 3, 64, 64, 32)
    assert lib.mamba3_decode_graph_create(None, *args()) == m.MAMBA_ERR_INVALID_ARG
    assert lib.mamba3_decode_graph_create(ctypes.byref(h), None, *args()[1:]) == m.MAMBA_ERR_INVALID_ARG
    assert h.value is None
    for n_steps, n_layers in ((0, 1), (1, 0), (-1, 4), (1 << 21, 1)):
        assert lib.mamba3_decode_graph_create(ctypes.byref(h), *args(n_steps, n_layers)) == m.MAMBA_ERR_INVALID_ARG
        assert "n_steps" in m.mamba_last_error()


def test_mixer_prefill_refuses_other_d_conv_on_host(lib):
    for K, code in ((0, m.MAMBA_ERR_UNSUPPORTED), (5, m.MAMBA_ERR_UNSUPPORTED), (8, m.MAMBA_ERR_UNSUPPORTED)):
        rc = lib.mamba_mixer_prefill(FAKE, 64, 0, FAKE, 64, FAKE, 64, None, 0, FAKE, 16, FAKE, 16, 0,
                                     FAKE, None, None, None, FAKE, None, None, None, None,
                                     1, 8, 64, K, 16, None, 0, None)
        assert rc == code and "d_conv 1..4" in m.mamba_last_error()
    rc = lib.mamba_mixer_prefill(FAKE, 64, 0, FAKE, 64, FAKE, 64, None, 0, FAKE, 16, FAKE, 16, 7,
                                 FAKE, None, None, None, FAKE, None, None, None, None, 1, 8, 64, 4, 16, None, 0, None)
    assert rc == m.MAMBA_ERR_INVALID_ARG


def test_m3_step_rejects_bad_arguments_on_host(lib):
    args = lambda P=64, N=64, layer=0, L=1: (FAKE, 0, FAKE, FAKE, FAKE, 0, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE,
                                            layer, L, 2, 3, P, N, None)
    assert lib.mamba3_siso_step_batched(*args(N=8)) == m.MAMBA_ERR_UNSUPPORTED
    assert lib.mamba3_siso_step_batched(*args(P=1024, N=128)) == m.MAMBA_ERR_UNSUPPORTED
    assert lib.mamba3_siso_step_batched(*args(layer=1, L=1)) == m.MAMBA_ERR_INVALID_ARG
    assert lib.mamba3_siso_step_batched(*args(P=-1)) == m.MAMBA_ERR_INVALID_ARG


def test_m3_prepare_rejects_bad_arguments_on_host(lib):
    def call(N=64, na=32, layer=0, L=1, dtype=0, angles=FAKE, state=FAKE, k_in=FAKE, B=2):
        return lib.mamba3_siso_step_prepare(FAKE, FAKE, dtype, FAKE, FAKE, FAKE, k_in, FAKE, FAKE, FAKE, FAKE,
                                            angles, state, layer, L, B, 3, N, na, None)
    assert call(N=15, na=4) == m.MAMBA_ERR_UNSUPPORTED          # odd d_state
    assert call(N=16, na=9) == m.MAMBA_ERR_INVALID_ARG          # more angles than pairs
    assert call(na=-1) == m.MAMBA_ERR_INVALID_ARG
    assert call(layer=1, L=1) == m.MAMBA_ERR_INVALID_ARG
    assert call(layer=1, L=1, na=0, angles=None, state=None, B=0) == m.MAMBA_OK  # no angle state: layer unused
    assert call(dtype=7) == m.MAMBA_ERR_INVALID_ARG
    assert call(angles=None) == m.MAMBA_ERR_INVALID_ARG         # angles needed when n_angles > 0
    assert "angles" in m.mamba_last_error()
    assert call(state=None) == m.MAMBA_ERR_INVALID_ARG
    assert call(k_in=None) == m.MAMBA_ERR_INVALID_ARG
    assert call(B=0, k_in=None) == m.MAMBA_OK                   # empty batch: nothing to do


def test_m3_fused_rejects_bad_arguments_on_host(lib):
    def call(N=64, na=32, layer=0, L=1, P=64, angles=FAKE, state=FAKE, k_in=FAKE, B=2):
        return lib.mamba3_siso_step_fused_batched(FAKE, 0, FAKE, 0, k_in, FAKE, FAKE, FAKE, FAKE, angles, None, FAKE,
                                                  FAKE, FAKE, state, layer, L, B, 3, P, N, na, None)
    assert call(N=8, na=4) == m.MAMBA_ERR_UNSUPPORTED           # d_state outside {16, 32, 64, 128}
    assert call(N=16, na=9) == m.MAMBA_ERR_INVALID_ARG          # more angles than pairs
    assert call(P=1024, N=128) == m.MAMBA_ERR_UNSUPPORTED       # headdim * d_state / 8 too large
    assert call(layer=1, L=1) == m.MAMBA_ERR_INVALID_ARG
    assert call(angles=None) == m.MAMBA_ERR_INVALID_ARG
    assert call(state=None) == m.MAMBA_ERR_INVALID_ARG
    assert call(k_in=None) == m.MAMBA_ERR_INVALID_ARG
    assert call(B=0, k_in=None) == m.MAMBA_OK


def test_m3_fused_and_graph_wrappers_refuse_mismatched_tensors_before_any_call():
    import torch
    B, H, P, N, na, L = 2, 3, 8, 16, 4, 2
    f = lambda *s: torch.zeros(*s)
    tok = dict(y=f(B, H, P), x=f(B, H, P), k_in=f(B, H, N), q_in=f(B, H, N), dt=f(B, H), A=f(B, H), lam=f(B, H),
               angles=f(B, na))
    states = dict(ssm_state=f(L, B, H, P, N), k_state=f(L, B, H, N), v_state=f(L, B, H, P), angle_state=f(L, B, H, na))
    bad = [dict(k_in=f(B, H, N + 2)), dict(dt=f(B, H + 1)), dict(angles=None), dict(x=f(B, H, P + 1)),
           dict(lam=f(B, H).double()), dict(angle_state=f(L, B, H, na + 1)), dict(ssm_state=f(L, B, H, P, N)[:, :, :, :, ::2])]
    for b in bad:
        kw = {**tok, **states, **b}
        with pytest.raises(ValueError):
            m.mamba3_siso_step_fused_batched(kw["y"], kw["x"], kw["k_in"], kw["q_in"], kw["dt"], kw["A"], kw["lam"],
                                             kw["angles"], kw["ssm_state"], kw["k_state"], kw["v_state"],
                                             kw["angle_state"], 0)
    for b in bad:
        kw = {**tok, **states, **b}
        io = [[{k: kw[k] for k in tok}] * L]
        with pytest.raises(ValueError):
            m.Mamba3DecodeGraph(io, kw["ssm_state"], kw["k_state"], kw["v_state"], kw["angle_state"])
    with pytest.raises(ValueError):  # D needs one entry per layer
        m.Mamba3DecodeGraph([[dict(tok)] * L], *states.values(), D=[f(H)])


def test_m3_prepare_wrapper_refuses_mismatched_tensors_before_any_call():
    import torch
    B, H, N, na = 2, 3, 8, 2
    f = lambda *s: torch.zeros(*s)
    good = dict(k=f(B, H, N), q=f(B, H, N), alpha=f(B, H), beta=f(B, H), gamma=f(B, H), k_in=f(B, H, N),
                q_in=f(B, H, N), dt=f(B, H), A=f(B, H), lam=f(B, H), angles=f(B, na), angle_state=f(1, B, H, na),
                layer=0)
    bad = [dict(q=f(B, H, N).to(torch.bfloat16)), dict(k_in=f(B, H, N + 2)), dict(dt=f(B, H + 1)),
           dict(angles=None), dict(angle_state=f(1, B, H, na + 1)), dict(k=f(B, H, N // 2)),
           dict(lam=f(B, H).double())]
    for b in bad:
        with pytest.raises(ValueError):
            m.mamba3_siso_step_prepare(**{**good, **b})


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "mamba_ssm.h"

int main(void) {
    int fails = 0;
    if (strlen(mamba_version()) == 0) { puts("empty version"); ++fails; }
    /* refused on the host, before any device work */
    if (mamba_selective_scan_prefill(NULL, 0, MAMBA_F32, NULL, 0, NULL, 0, NULL, 0, NULL, 0, NULL, 0, MAMBA_F32,
                                     NULL, NULL, NULL, NULL, NULL, 1, 8, 32, 3, NULL, 0, NULL) != MAMBA_ERR_UNSUPPORTED)
        { puts("d_state 3 accepted"); ++fails; }
    if (strstr(mamba_last_error(), "d_state") == NULL) { puts("no message"); ++fails; }
    if (mamba_conv1d_silu_step(NULL, NULL, 7, NULL, 0, 1, NULL, NULL, 1, 8, 4, NULL) != MAMBA_ERR_INVALID_ARG)
        { puts("bad dtype accepted"); ++fails; }
    if (mamba_decode_graph_destroy(NULL) != MAMBA_OK) { puts("destroy(NULL)"); ++fails; }
    if (mamba_selftest_bounded_wait(0, 0, NULL) != MAMBA_ERR_INVALID_ARG) { puts("limit 0 accepted"); ++fails; }
    if (mamba_selective_scan_prefill(NULL, 0, MAMBA_F32, NULL, 0, NULL, 0, NULL, 0, NULL, 0, NULL, 0, MAMBA_F32,
                                     NULL, NULL, NULL, NULL, NULL, 0, 8, 32, 16, NULL, 0, NULL) != MAMBA_OK)
        { puts("empty batch not a no-op"); ++fails; }
    printf("%s\n", fails ? "FAIL" : "OK");
    return fails;
}
"""


def test_header_compiles_as_c99_and_library_links(lib, tmp_path):
    """The ABI is plain C: a C99 program built with gcc against include/ and
    linked to the library runs the host-side paths."""
    src = tmp_path / "abi_check.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi_check"
    pkg = os.path.dirname(B.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-o", str(exe), "-L", pkg, "-lmamba_ssm", f"-Wl,-rpath,{pkg}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip().endswith("OK"), run.stdout + run.stderr


def test_noalloc_scratch_size_matches_the_header():
    """The binding's copy of MAMBA_NOALLOC_SCRATCH_BYTES is the header's value."""
    txt = open(os.path.join(ROOT, "include", "mamba_ssm.h")).read()
    mm = re.search(r"#define\s+MAMBA_NOALLOC_SCRATCH_BYTES\s+\(([0-9L\s\*]+)\)", txt)
    assert mm, "MAMBA_NOALLOC_SCRATCH_BYTES not found in the header"
    value = 1
    for factor in mm.group(1).split("*"):
        value *= int(factor.strip().rstrip("L"))
    assert value == m.MAMBA_NOALLOC_SCRATCH_BYTES


@pytest.mark.parametrize("fn", ["mamba_selective_scan_prefill", "mamba_selective_scan_prefill_noalloc"])
@pytest.mark.parametrize("bad", ["dt_dtype", "B_dtype", "short_B", "short_C", "short_z", "short_y", "short_dt",
                                 "state_shape"])
def test_scan_wrappers_refuse_mismatched_tensors_before_any_call(fn, bad):
    """The C ABI cannot see allocation sizes, so both scan wrappers refuse a
    tensor of another dtype or of fewer rows than the sizes say (host tensors:
    nothing is loaded or launched)."""
    import torch

    Bsz, T, Di, N = 2, 8, 32, 16
    f = lambda *s, dtype=torch.float32: torch.zeros(*s, dtype=dtype)
    args = dict(y=f(Bsz, T, Di), u=f(Bsz, T, Di), dt=f(Bsz, T, Di), Bm=f(Bsz, T, N), Cm=f(Bsz, T, N),
                A_log=f(Di, N), z=f(Bsz, T, Di), ssm_state_out=f(Bsz, Di, N))
    if bad == "dt_dtype":
        args["dt"] = f(Bsz, T, Di, dtype=torch.bfloat16)
    elif bad == "B_dtype":
        args["Bm"] = f(Bsz, T, N, dtype=torch.bfloat16)
    elif bad == "short_B":
        args["Bm"] = f(Bsz, T - 1, N)
    elif bad == "short_C":
        args["Cm"] = f(Bsz, T, N - 1)
    elif bad == "short_z":
        args["z"] = f(Bsz, T - 1, Di)
    elif bad == "short_y":
        args["y"] = f(Bsz, T - 1, Di)
    elif bad == "short_dt":
        args["dt"] = f(Bsz, T, Di - 1)
    elif bad == "state_shape":
        args["ssm_state_out"] = f(Bsz, Di, N - 1)
    with pytest.raises(ValueError):
        getattr(m, fn)(**args)


def _layer(dm=64, Di=128, N=16, K=4, R=8, eps=1e-5, null=()):
    S = m._binding._MambaLayer(dm, Di, N, K, R, eps, *([FAKE.value] * 10))
    for f in null:
        setattr(S, f, None)
    return S


@pytest.mark.parametrize("kw,code", [
    (dict(dm=60), m.MAMBA_ERR_UNSUPPORTED),     # d_model not a multiple of 8
    (dict(Di=100), m.MAMBA_ERR_UNSUPPORTED),    # d_inner not a multiple of 8
    (dict(R=6), m.MAMBA_ERR_UNSUPPORTED),       # dt_rank not a multiple of 8
    (dict(N=3), m.MAMBA_ERR_UNSUPPORTED),
    (dict(K=9), m.MAMBA_ERR_UNSUPPORTED),
    (dict(dm=0), m.MAMBA_ERR_INVALID_ARG),
    (dict(eps=-1.0), m.MAMBA_ERR_INVALID_ARG),
    (dict(eps=float("nan")), m.MAMBA_ERR_INVALID_ARG),
])
def test_layer_rejects_bad_dims_on_host(lib, kw, code):
    S = _layer(**kw)
    assert lib.mamba_layer_workspace_bytes(ctypes.byref(S), 2, 16) == code
    assert lib.mamba_layer_prefill(FAKE, ctypes.byref(S), None, None, None, None, 2, 16, FAKE, 1 << 30, None) == code
    assert lib.mamba_layer_step(FAKE, ctypes.byref(S), FAKE, FAKE, 0, 1, 2, FAKE, 1 << 30, None) == code
    assert m.mamba_last_error()


def test_layer_rejects_bad_arguments_on_host(lib):
    E = m.MAMBA_ERR_INVALID_ARG
    S = _layer()
    assert lib.mamba_layer_workspace_bytes(None, 2, 16) == E
    assert lib.mamba_layer_workspace_bytes(ctypes.byref(S), -1, 16) == E
    assert lib.mamba_layer_prefill(FAKE, None, None, None, None, None, 2, 16, FAKE, 1 << 30, None) == E
    assert lib.mamba_layer_prefill(FAKE, ctypes.byref(S), None, None, None, None, 2, 16, FAKE, -1, None) == E
    # the block over B x T rows needs at least its activations' bytes
    assert lib.mamba_layer_prefill(FAKE, ctypes.byref(S), None, None, None, None, 2, 16, FAKE, 1024, None) == E
    # a misaligned workspace or bf16 weight, a missing weight
    assert lib.mamba_layer_prefill(FAKE, ctypes.byref(S), None, None, None, None, 2, 16,
                                   ctypes.c_void_p(FAKE.value + 8), 1 << 30, None) == E
    S2 = _layer()
    S2.in_proj_w = FAKE.value + 2
    assert lib.mamba_layer_prefill(FAKE, ctypes.byref(S2), None, None, None, None, 2, 16, FAKE, 1 << 30, None) == E
    for f in ("norm_w", "in_proj_w", "conv_w", "x_proj_w", "dt_proj_w", "A_log", "out_proj_w"):
        assert lib.mamba_layer_prefill(FAKE, ctypes.byref(_layer(null=(f,))), None, None, None, None, 2, 16, FAKE,
                                       1 << 30, None) == E, f
    # step: layer index outside [0, n_layers), missing states
    assert lib.mamba_layer_step(FAKE, ctypes.byref(S), FAKE, FAKE, 2, 2, 2, FAKE, 1 << 30, None) == E
    assert lib.mamba_layer_step(FAKE, ctypes.byref(S), None, FAKE, 0, 2, 2, FAKE, 1 << 30, None) == E
    # B == 0 is a no-op
    assert lib.mamba_layer_prefill(None, ctypes.byref(S), None, None, None, None, 0, 16, None, 0, None) == 0


def test_rmsnorm_and_linear_reject_bad_arguments_on_host(lib):
    E = m.MAMBA_ERR_INVALID_ARG
    f = lib.mamba_rmsnorm
    assert f(FAKE, 32, 1, FAKE, 64, FAKE, 1e-5, 4, 64, None) == E         # ld_out < D
    assert f(None, 64, 1, FAKE, 64, FAKE, 1e-5, 4, 64, None) == E
    assert f(FAKE, 64, 1, FAKE, 64, None, 1e-5, 4, 64, None) == E
    assert f(FAKE, 64, 7, FAKE, 64, FAKE, 1e-5, 4, 64, None) == E          # unknown dtype
    assert f(FAKE, 64, 1, FAKE, 64, FAKE, -1.0, 4, 64, None) == E
    assert f(None, 0, 1, None, 0, None, 1e-5, 0, 64, None) == 0           # M == 0
    g = lib.mamba_linear_bf16
    assert g(FAKE, 64, 0, ctypes.c_void_p(FAKE.value + 2), 64, FAKE, 64, None, 0, 8, 64, 64, None) == E
    assert g(FAKE, 64, 0, FAKE, 60, FAKE, 64, None, 0, 8, 64, 60, None) == E   # ld_a not a multiple of 8
    assert g(FAKE, 32, 0, FAKE, 64, FAKE, 64, None, 0, 8, 64, 64, None) == E   # ld_c < N
    assert g(FAKE, 64, 0, FAKE, 64, FAKE, 64, None, 0, 8, 64, 0, None) == E    # K == 0


def test_layer_wrappers_refuse_mismatched_tensors_before_any_call():
    import torch

    dm, Di, N, K, R = 64, 128, 16, 4, 8
    bf = lambda *s: torch.zeros(*s, dtype=torch.bfloat16)
    f = lambda *s: torch.zeros(*s)
    w = dict(norm_w=f(dm), in_proj_w=bf(2 * Di, dm), conv_w=f(Di, K), x_proj_w=bf(R + 2 * N, Di),
             dt_proj_w=bf(Di, R), A_log=f(Di, N), out_proj_w=bf(dm, Di))
    m.layer_struct(w)  # consistent shapes pass
    for k, bad in (("in_proj_w", f(2 * Di, dm)), ("x_proj_w", bf(R + 2 * N + 1, Di)), ("out_proj_w", bf(Di, dm)),
                   ("norm_w", f(dm + 1)), ("D", f(Di - 1))):
        with pytest.raises(ValueError):
            m.layer_struct(dict(w, **{k: bad}))
    with pytest.raises(ValueError):
        m.mamba_layer_prefill(torch.zeros(2, 4, dm, dtype=torch.bfloat16), w)
    with pytest.raises(ValueError):
        m.mamba_layer_prefill(torch.zeros(2, 4, dm + 8), w)
    with pytest.raises(ValueError):
        m.mamba_layer_prefill(torch.zeros(2, 4, dm), w, conv_state_in=f(2, Di, K + 1))
    with pytest.raises(ValueError):
        m.mamba_layer_step(torch.zeros(2, dm), w, f(3, 2, Di, K), f(2, 2, Di, N), 0)


def test_layer_decode_graph_rejects_bad_arguments_on_host(lib):
    E = m.MAMBA_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    two = (m._binding._MambaLayer * 2)(_layer(), _layer(dm=72))
    assert lib.mamba_layer_decode_graph_create(ctypes.byref(h), two, 2, FAKE, FAKE, FAKE, 4, FAKE, 1 << 30) == E
    assert "dims of layer 0" in m.mamba_last_error()
    assert lib.mamba_layer_decode_graph_create(None, two, 2, FAKE, FAKE, FAKE, 4, FAKE, 1 << 30) == E
    assert lib.mamba_layer_decode_graph_create(ctypes.byref(h), None, 2, FAKE, FAKE, FAKE, 4, FAKE, 1 << 30) == E
    assert lib.mamba_layer_decode_graph_create(ctypes.byref(h), two, 0, FAKE, FAKE, FAKE, 4, FAKE, 1 << 30) == E
    assert h.value is None
