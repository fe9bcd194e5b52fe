"""Run one kernel of the mixer core on one synthetic shape, a few times.

A small, self-contained target for a profiler (for example
`ncu -k regex:scan_kernel -s 1 -c 1 python -m selective_state_space_conv1d_gb300.profile_case --what scan ...`):
it builds its inputs on the device with torch's RNG, calls the C ABI `--reps`
times, then times one more call with CUDA events and prints it.

  --what scan      selective-scan prefill  [B, T, Di] inputs, d_state N
  --what conv      conv1d + SiLU prefill    [B, T, Di], d_conv 4
  --what step      T=1 SSM step on layer 1 of an [L][B][Di][N] state
  --what mixer     fused conv step + SSM step on layer 1
  --what convstep  T=1 conv step on layer 1 of an [L][B][Di][4] state
  --what fused     fused conv1d + SiLU and selective-scan prefill  [B, T, Di]
  --what m3        Mamba-3 SISO step on layer 1: --B batch, --H heads, --P headdim, --N d_state
  --what m3prep    one Mamba-3 SISO token on layer 1: the step's inputs prepared (N/2 rotated pairs), then the step
  --what m3fused   the same token in one launch (the preparation inside the step)
  --what linear    projection GEMM: --M rows, --Nout outputs, --K inputs (--out f32|bf16, --residual)
  --what rmsnorm   RMSNorm of --M rows of --dm (f32 in, bf16 out)
  --what block     whole Mamba-1 block prefill: --B, --T, --dm, --Di, --N, --R (dt_rank), d_conv 4
  --what blockstep whole-block T=1 step on layer 1 of --L layers: --B, --dm, --Di, --N, --R
  --route plain    prefills without a workspace (one warp per 32-channel tile)
  --flush          write a 256 MB buffer before every call, so each call starts with a cold L2
                   (for counters taken with ncu --cache-control none: the launches inside one call
                   then see the cache state they see in a real run)
"""
import argparse
import math

import torch

from . import _binding as m


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--what", default="scan", choices=("scan", "conv", "step", "mixer", "convstep", "fused", "m3", "m3prep", "m3fused", "linear",
                                                           "rmsnorm", "block", "blockstep"))
    ap.add_argument("--M", type=int, default=2048)
    ap.add_argument("--Nout", type=int, default=3072)
    ap.add_argument("--K", type=int, default=768)
    ap.add_argument("--out", default="bf16", choices=("f32", "bf16"))
    ap.add_argument("--residual", action="store_true")
    ap.add_argument("--dm", type=int, default=768)
    ap.add_argument("--R", type=int, default=48)
    ap.add_argument("--H", type=int, default=24)
    ap.add_argument("--P", type=int, default=64)
    ap.add_argument("--B", type=int, default=1)
    ap.add_argument("--T", type=int, default=2048)
    ap.add_argument("--Di", type=int, default=1536)
    ap.add_argument("--N", type=int, default=16)
    ap.add_argument("--L", type=int, default=24)
    ap.add_argument("--dtype", default="f32", choices=("f32", "bf16"))
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--flush", action="store_true", help="cold L2 before every call")
    ap.add_argument("--route", default="auto", choices=("auto", "plain"),
                    help="prefills: the planned route, or one warp per tile with no workspace")
    a = ap.parse_args(argv)
    td = torch.float32 if a.dtype == "f32" else torch.bfloat16
    g = torch.Generator(device="cuda")
    g.manual_seed(1)
    r = lambda s, std=1.0: (torch.randn(s, generator=g, device="cuda") * std).to(td)
    A = torch.log(torch.arange(1, a.N + 1, device="cuda", dtype=torch.float32)).repeat(a.Di, 1).contiguous()
    D = torch.ones(a.Di, device="cuda")
    dtb = torch.full((a.Di,), -4.0, device="cuda")
    w = torch.rand((a.Di, 4), generator=g, device="cuda") - 0.5
    m.load()
    bf = torch.bfloat16
    if a.what in ("block", "blockstep"):
        wts = {"norm_w": torch.ones(a.dm, device="cuda"),
               "in_proj_w": (torch.randn((2 * a.Di, a.dm), generator=g, device="cuda") * a.dm ** -0.5).to(bf),
               "conv_w": w, "conv_b": torch.zeros(a.Di, device="cuda"),
               "x_proj_w": (torch.randn((a.R + 2 * a.N, a.Di), generator=g, device="cuda") * a.Di ** -0.5).to(bf),
               "dt_proj_w": (torch.randn((a.Di, a.R), generator=g, device="cuda") * a.R ** -0.5).to(bf),
               "dt_bias": dtb, "A_log": A, "D": D,
               "out_proj_w": (torch.randn((a.dm, a.Di), generator=g, device="cuda") * a.Di ** -0.5).to(bf)}
    if a.what == "linear":
        A_ = torch.randn((a.M, a.K), generator=g, device="cuda").to(bf)
        W_ = (torch.randn((a.Nout, a.K), generator=g, device="cuda") * a.K ** -0.5).to(bf)
        C_ = torch.zeros((a.M, a.Nout), device="cuda", dtype=bf if a.out == "bf16" else torch.float32)
        f = lambda: m.mamba_linear_bf16(C_, A_, W_, C_ if a.residual else None)
    elif a.what == "rmsnorm":
        X_ = torch.randn((a.M, a.dm), generator=g, device="cuda")
        O_ = torch.empty((a.M, a.dm), device="cuda", dtype=bf)
        nw = torch.ones(a.dm, device="cuda")
        f = lambda: m.mamba_rmsnorm(O_, X_, nw)
    elif a.what == "block":
        hid = torch.randn((a.B, a.T, a.dm), generator=g, device="cuda")
        cs = torch.zeros((a.B, a.Di, 4), device="cuda")
        ss = torch.zeros((a.B, a.Di, a.N), device="cuda")
        f = lambda: m.mamba_layer_prefill(hid, wts, cs, cs, ss, ss)
    elif a.what == "blockstep":
        hid = torch.randn((a.B, a.dm), generator=g, device="cuda")
        cs = torch.zeros((a.L, a.B, a.Di, 4), device="cuda")
        ss = torch.zeros((a.L, a.B, a.Di, a.N), device="cuda")
        f = lambda: m.mamba_layer_step(hid, wts, cs, ss, 1)
    elif a.what in ("m3", "m3prep", "m3fused"):
        BH = (a.B, a.H)
        st = torch.randn((a.L, a.B, a.H, a.P, a.N), generator=g, device="cuda")
        ks = torch.randn((a.L, a.B, a.H, a.N), generator=g, device="cuda")
        vs = torch.randn((a.L, a.B, a.H, a.P), generator=g, device="cuda")
        x, k, q = r((a.B, a.H, a.P)), r((a.B, a.H, a.N)), r((a.B, a.H, a.N))
        al = torch.exp(-torch.rand(BH, generator=g, device="cuda") * 0.2)
        be = torch.rand(BH, generator=g, device="cuda") * 0.1
        ga = torch.rand(BH, generator=g, device="cuda") * 0.1
        Dh = torch.ones(a.H, device="cuda")
        y = torch.empty((a.B, a.H, a.P), device="cuda")
        f = lambda: m.mamba3_siso_step_batched(y, x, k, q, al, be, ga, st, ks, vs, 1, Dh)
        if a.what in ("m3prep", "m3fused"):
            na = a.N // 2
            u01 = lambda s_: torch.rand(s_, generator=g, device="cuda")
            th = (u01((a.L, a.B, a.H, na)) - 0.5) * 100.0
            kin = torch.randn((a.B, a.H, a.N), generator=g, device="cuda")
            qin = torch.randn((a.B, a.H, a.N), generator=g, device="cuda")
            dt = torch.exp(math.log(1e-3) + u01(BH) * math.log(100.0))
            Ad, lam = -(0.05 + 3.95 * u01(BH)), u01(BH)
            ang = (u01((a.B, na)) * 2.0 - 1.0) * math.pi

            def f():
                m.mamba3_siso_step_prepare(k, q, al, be, ga, kin, qin, dt, Ad, lam, ang, th, 1)
                m.mamba3_siso_step_batched(y, x, k, q, al, be, ga, st, ks, vs, 1, Dh)

            if a.what == "m3fused":
                def f():
                    m.mamba3_siso_step_fused_batched(y, x, kin, qin, dt, Ad, lam, ang, st, ks, vs, th, 1, Dh)
    elif a.what in ("scan", "conv", "fused"):
        sh = (a.B, a.T, a.Di)
        x, u, dt, z = r(sh), r(sh), r(sh, 0.1), r(sh)
        Bm, Cm = r((a.B, a.T, a.N)), r((a.B, a.T, a.N))
        y = torch.empty(sh, device="cuda")
        uo = torch.empty_like(x)
        so = torch.empty((a.B, a.Di, a.N), device="cuda")
        co = torch.empty((a.B, a.Di, 4), device="cuda")
        ws = False if a.route == "plain" else None
        if a.what == "conv":
            f = lambda: m.mamba_conv1d_silu_prefill(uo, x, w, None, None, co)
        elif a.what == "fused":
            f = lambda: m.mamba_mixer_prefill(y, x, dt, Bm, Cm, w, A, None, D, dtb, z, None, co, None, so,
                                              workspace=ws)
        else:
            f = lambda: m.mamba_selective_scan_prefill(y, u, dt, Bm, Cm, A, D, dtb, z, None, so, workspace=ws)
    else:
        st = torch.randn((a.L, a.B, a.Di, a.N if a.what in ("step", "mixer") else 4), generator=g, device="cuda")
        x, u, dt, z = r((a.B, a.Di)), r((a.B, a.Di)), r((a.B, a.Di), 0.1), r((a.B, a.Di))
        Bm, Cm = r((a.B, a.N)), r((a.B, a.N))
        y = torch.empty((a.B, a.Di), device="cuda", dtype=td)
        if a.what == "step":
            f = lambda: m.mamba_ssm_step_batched(y, u, dt, Bm, Cm, st, 1, A, D, dtb, z)
        elif a.what == "mixer":
            cs = torch.randn((a.L, a.B, a.Di, 4), generator=g, device="cuda")
            f = lambda: m.mamba_mixer_step_batched(y, x, dt, Bm, Cm, cs, st, 1, w, A, None, D, dtb, z)
        else:
            f = lambda: m.mamba_conv1d_silu_step(y, x, st, 1, w, None)
    if a.flush:
        scratch = torch.empty(64 * 1024 * 1024, device="cuda")  # 256 MB, twice the L2
        call = f
        f = lambda: (scratch.zero_(), call())
    for _ in range(a.reps):
        f()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    f()
    e1.record()
    torch.cuda.synchronize()
    print(f"{a.what} B={a.B} T={a.T} Di={a.Di} N={a.N} {a.dtype}: {e0.elapsed_time(e1) * 1e3:.1f} us", flush=True)


if __name__ == "__main__":
    main()
