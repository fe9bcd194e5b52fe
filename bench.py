#!/usr/bin/env python3
"""Benchmark of the GB300 Mamba-1 mixer core.

Headline (one JSON line on rank 0): prefill tokens/s of one mamba-2.8b-shaped
layer (batch 8, T 4096, d_inner 5120, d_state 16, d_conv 4; x/dt/z/B/C stored
in bf16, f32 arithmetic, f32 y) -- one step is the whole mixer-core prefill
(conv1d+SiLU and the selective scan with its gate, fused or as two calls,
whichever is faster: the two give the same bits), through the C ABI, on seeded
synthetic inputs already resident in HBM.  The same line carries the roofline
of the dominant call, the end-to-end figure (host buffers, copies inside the
timed region), the f64 CPU oracle timed on the host cores for every workload,
the SM clocks seen, and under "extra" the other workloads: the mamba-130m
layer prefill (f32), the long-context continuation, the 24-layer batch-128
decode, the Mamba-3 SISO decode, the prefill-versus-steps comparison, and the
whole Mamba-1 block (RMSNorm, projections on the tensor cores, mixer,
residual): the mamba-2.8b block prefill and the 24-layer block decode.

Launch: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
N > 1 runs under torch.distributed.run: every rank runs an independent replica
on its own GPU (the mixer shards over batch and channels with no exchange).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s and decode steps/s (batch×layers) at 1 GB300; HBM GB/s % of peak"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = {
    "scan": ["selective_state_space_conv1d_gb300/csrc/scan_prefill.cu",
             "selective_state_space_conv1d_gb300/csrc/scan_kernel.cuh",
             "selective_state_space_conv1d_gb300/csrc/scan_inst.cu",
             "selective_state_space_conv1d_gb300/csrc/device_math.cuh"],
    "conv": ["selective_state_space_conv1d_gb300/csrc/conv1d.cu",
             "selective_state_space_conv1d_gb300/csrc/device_math.cuh"],
    "step": ["selective_state_space_conv1d_gb300/csrc/ssm_step.cu",
             "selective_state_space_conv1d_gb300/csrc/async_copy.cuh",
             "selective_state_space_conv1d_gb300/csrc/device_math.cuh"],
}
KERNEL_SOURCES["mixer_step"] = KERNEL_SOURCES["step"]
KERNEL_SOURCES["fused"] = KERNEL_SOURCES["scan"]
KERNEL_SOURCES["gemm"] = ["selective_state_space_conv1d_gb300/csrc/gemm.cu",
                          "selective_state_space_conv1d_gb300/csrc/async_copy.cuh"]
KERNEL_SOURCES["rmsnorm"] = ["selective_state_space_conv1d_gb300/csrc/rmsnorm.cu"]
# the whole block step: every kernel it launches
KERNEL_SOURCES["block"] = ["selective_state_space_conv1d_gb300/csrc/api.cu",
                           "selective_state_space_conv1d_gb300/csrc/gemm.cu",
                           "selective_state_space_conv1d_gb300/csrc/rmsnorm.cu",
                           "selective_state_space_conv1d_gb300/csrc/conv1d.cu",
                           "selective_state_space_conv1d_gb300/csrc/ssm_step.cu",
                           "selective_state_space_conv1d_gb300/csrc/async_copy.cuh",
                           "selective_state_space_conv1d_gb300/csrc/device_math.cuh"]
KERNEL_SOURCES["m3_step"] = ["selective_state_space_conv1d_gb300/csrc/m3_step.cu",
                             "selective_state_space_conv1d_gb300/csrc/m3_math.cuh",
                             "selective_state_space_conv1d_gb300/csrc/device_math.cuh"]


# ---------------------------------------------------------------- utilities --

def source_hash(kind: str) -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def bf16_peak():
    """Dense bf16 tensor peak of the GB300s: (burst, sustained, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 1900.0, 1700.0, "fallback"


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def ncu_traffic(kind: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it is for this source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)[f"{kind}:{workload}"]
    except Exception:
        return None
    if rec.get("source_hash") != source_hash(kind):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="mamba_clocks_", suffix=".csv")
            self.fh = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    return g


# ------------------------------------------------------------- workloads ----

class PrefillSet:
    """Device buffers of one prefill step (conv then scan), all resident in HBM."""

    def __init__(self, torch, host, params, dtype, device):
        td = torch.float32 if dtype == "f32" else torch.bfloat16
        dev = lambda a, d=td: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device).to(d)
        self.x, self.dt, self.z = dev(host["x"]), dev(host["dt"]), dev(host["z"])
        self.B, self.C = dev(host["B"]), dev(host["C"])
        self.u = torch.empty_like(self.x)
        self.y = torch.empty(self.x.shape, device=device, dtype=torch.float32)
        Bsz, T, Di = self.x.shape
        N = self.B.shape[2]
        K = params["conv_w"].shape[1]
        self.conv_out = torch.empty((Bsz, Di, K), device=device)
        self.ssm_out = torch.empty((Bsz, Di, N), device=device)
        self.p = {k: dev(v, torch.float32) for k, v in params.items()}

    @classmethod
    def from_device(cls, torch, shape, N, params, dtype, device, seed):
        """Large workloads: same distributions drawn with torch's device RNG."""
        from selective_state_space_conv1d_gb300 import synth

        self = cls.__new__(cls)
        td = torch.float32 if dtype == "f32" else torch.bfloat16
        Bsz, T, Di = shape
        self.x = synth.torch_normal(shape, 1.0, seed + 1, device, td)
        self.dt = synth.torch_normal(shape, 0.1, seed + 2, device, td)
        self.z = synth.torch_normal(shape, 1.0, seed + 3, device, td)
        self.B = synth.torch_normal((Bsz, T, N), 1.0, seed + 4, device, td)
        self.C = synth.torch_normal((Bsz, T, N), 1.0, seed + 5, device, td)
        self.u = torch.empty_like(self.x)
        self.y = torch.empty(shape, device=device, dtype=torch.float32)
        K = params["conv_w"].shape[1]
        self.conv_out = torch.empty((Bsz, Di, K), device=device)
        self.ssm_out = torch.empty((Bsz, Di, N), device=device)
        self.p = {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(device)
                  for k, v in params.items()}
        return self

    def conv(self, m):
        m.mamba_conv1d_silu_prefill(self.u, self.x, self.p["conv_w"], self.p["conv_b"], None,
                                    self.conv_out)

    def scan(self, m):
        m.mamba_selective_scan_prefill(self.y, self.u, self.dt, self.B, self.C, self.p["A_log"],
                                       self.p["D"], self.p["dt_bias"], self.z, None, self.ssm_out)

    def fused(self, m):
        m.mamba_mixer_prefill(self.y, self.x, self.dt, self.B, self.C, self.p["conv_w"], self.p["A_log"],
                              self.p["conv_b"], self.p["D"], self.p["dt_bias"], self.z, None, self.conv_out,
                              None, self.ssm_out)

    def bytes_per_step(self):
        """Algorithmic HBM bytes of (conv, scan): every input read once, every output written once."""
        es = self.x.element_size()
        Bsz, T, Di = self.x.shape
        N = self.B.shape[2]
        K = self.conv_out.shape[2]
        conv = Bsz * T * Di * 2 * es + Bsz * Di * K * 4 + Di * (K + 1) * 4
        scan = (Bsz * T * Di * (3 * es + self.y.element_size()) + Bsz * T * N * 2 * es
                + Bsz * Di * N * 4 + Di * (N + 2) * 4)
        return conv, scan


def timed_graph_run(torch, m, sets, n_steps, per_graph, clocks=None, dist=None, fused=False):
    """Time n_steps prefill steps (conv then scan, or the fused call) as replays
    of captured graphs."""
    per_graph = max(1, min(per_graph, n_steps))

    def build(nsteps):
        def body():
            for i in range(nsteps):
                s = sets[i % len(sets)]
                if fused:
                    s.fused(m)
                else:
                    s.conv(m)
                    s.scan(m)
        return capture(torch, body)

    g_main = build(per_graph)
    reps, tail = divmod(n_steps, per_graph)
    g_tail = build(tail) if tail else None
    g_main.replay()
    if g_tail:
        g_tail.replay()
    torch.cuda.synchronize()

    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    start.record()
    for _ in range(reps):
        g_main.replay()
    if g_tail:
        g_tail.replay()
    end.record()
    torch.cuda.synchronize()
    ck = clocks.stop() if clocks else None
    if dist is not None:
        dist.barrier()
    return start.elapsed_time(end), ck


def kernel_time(torch, calls, n, reps=3):
    """Average duration of one call: a captured graph of n back-to-back calls
    (calls[i % len]) replayed `reps` times between CUDA events on its stream."""
    def body():
        for i in range(n):
            calls[i % len(calls)]()
    g = capture(torch, body)
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / (n * reps)


def roofline(bytes_per_launch, ms, peak, peak_src, traffic):
    gbs = bytes_per_launch / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
            "frac": round(gbs / peak, 4), "traffic": traffic, "peak_source": peak_src,
            "algorithmic_bytes_per_launch": int(bytes_per_launch), "avg_launch_ms": round(ms, 6)}


GB300_SMS = 152
GB300_MAX_SM_MHZ = 2070.0
# FP32 pipe of GB300: 128 lanes/clk/SM (an FMA counts as one operation)
FP32_LANES_PER_CLK_SM = 128

# MUFU throughput probe: every thread runs 8 independent chains of
# ex2.approx.ftz.f32 (or fma.rn.f32), and each CTA times itself with clock64;
# lanes per clock per SM = operations / (cycles of the slowest CTA on an SM).
_PROBE_SRC = r"""
#include <cuda_runtime.h>
template <int OP>
__global__ void probe(float* out, long long* cyc, int iters) {
  float v[8];
  for (int j = 0; j < 8; ++j) v[j] = -1e-3f * (threadIdx.x + j);
  const long long t0 = clock64();
  for (int i = 0; i < iters; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (OP == 0) asm volatile("ex2.approx.ftz.f32 %0, %0;" : "+f"(v[j]));
      else asm volatile("fma.rn.f32 %0, %0, 0f3F7FFFF0, 0f3A83126F;" : "+f"(v[j]));
    }
  }
  const long long t1 = clock64();
  float s = 0.f;
  for (int j = 0; j < 8; ++j) s += v[j];
  out[blockIdx.x * blockDim.x + threadIdx.x] = s;
  if (threadIdx.x == 0) cyc[blockIdx.x] = t1 - t0;
}
extern "C" int run_probe(int op, int blocks, int threads, int iters, double* lanes_per_clk_sm) {
  float* out; long long* cyc;
  if (cudaMalloc(&out, sizeof(float) * blocks * threads) != cudaSuccess) return 1;
  if (cudaMalloc(&cyc, sizeof(long long) * blocks) != cudaSuccess) return 1;
  for (int rep = 0; rep < 2; ++rep) {
    if (op == 0) probe<0><<<blocks, threads>>>(out, cyc, iters);
    else probe<1><<<blocks, threads>>>(out, cyc, iters);
  }
  if (cudaDeviceSynchronize() != cudaSuccess) return 2;
  long long* h = new long long[blocks];
  cudaMemcpy(h, cyc, sizeof(long long) * blocks, cudaMemcpyDeviceToHost);
  long long mx = 0;
  for (int i = 0; i < blocks; ++i) mx = h[i] > mx ? h[i] : mx;
  delete[] h;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const double ops_per_sm = (double)blocks / sms * threads * iters * 8.0;
  *lanes_per_clk_sm = ops_per_sm / (double)mx;
  cudaFree(out); cudaFree(cyc);
  return 0;
}
"""


def alu_probe():
    """ex2 and FP32-FMA lanes per SM clock, measured on this GPU (None if nvcc
    or the run fails).  Eight CTAs of 256 threads per SM, chains long enough to
    run for milliseconds."""
    import ctypes

    try:
        d = tempfile.mkdtemp(prefix="mamba_probe_")
        src, lib = os.path.join(d, "probe.cu"), os.path.join(d, "probe.so")
        with open(src, "w") as f:
            f.write(_PROBE_SRC)
        nvcc = "nvcc" if subprocess.run(["which", "nvcc"], capture_output=True).returncode == 0 \
            else "/usr/local/cuda/bin/nvcc"
        r = subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared", "-Xcompiler",
                            "-fPIC", "-o", lib, src], capture_output=True, text=True)
        if r.returncode != 0:
            return None
        so = ctypes.CDLL(lib)
        so.run_probe.argtypes = (ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                 ctypes.POINTER(ctypes.c_double))
        import torch

        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
        res = {}
        for name, op, iters in (("ex2", 0, 20000), ("ffma", 1, 40000)):
            v = ctypes.c_double(0.0)
            if so.run_probe(op, 8 * sms, 256, iters, ctypes.byref(v)) != 0:
                return None
            res[name] = round(v.value, 2)
        return res
    except Exception:
        return None


_ALU = {"probe": None}


def mufu_lanes_per_clk():
    """Measured ex2 lanes per clock per SM (the probe), else the unit count 32."""
    p = _ALU["probe"]
    if p and p.get("ex2"):
        return p["ex2"], "measured: ex2.approx.ftz.f32 throughput probe (8 independent chains per thread)"
    return 32.0, "derived: 32 ex2 lanes/clk/SM (unit count; the probe did not run)"


def mufu_peak_tops(sm_count=GB300_SMS):
    lanes, _ = mufu_lanes_per_clk()
    return lanes * sm_count * GB300_MAX_SM_MHZ * 1e6 / 1e12


def fp32_peak_tops(sm_count=GB300_SMS):
    return FP32_LANES_PER_CLK_SM * sm_count * GB300_MAX_SM_MHZ * 1e6 / 1e12


def scan_roofline(tc, N, gate, bytes_per_launch, ms, hbm_peak_gbs, peak_src, traffic, sm_count, conv=False):
    """The scan is bound by MUFU (and FMA) throughput, not HBM: per (token,
    channel) it needs N ex2 for the states, ex2 + lg2 for softplus and, with a
    gate, ex2 + rcp for SiLU (lg2/rcp at half rate count twice): N + 3 (+ 3)
    ex2-equivalent MUFU slots; the fused prefill adds the conv's SiLU (+ 3).
    Reported against the MUFU peak, with the HBM and FP32-pipe views alongside."""
    slots = tc * (N + 3 + (3 if gate else 0) + (3 if conv else 0))
    tops = slots / (ms * 1e-3) / 1e12
    peak = mufu_peak_tops(sm_count)
    gbs = bytes_per_launch / (ms * 1e-3) / 1e9
    # FP32 operations per (token, channel): 4 per state (delta*A, delta*u*B, the
    # h update and the C.h term), 8 scalars (softplus 5, delta*u, the D term,
    # the gate product), the gate's SiLU 3, the conv's taps and SiLU 7
    ops = tc * (4 * N + 8 + (3 if gate else 0) + (7 if conv else 0))
    fops = ops / (ms * 1e-3) / 1e12
    fpeak = fp32_peak_tops(sm_count)
    return {"bound": "alu", "achieved": round(tops, 3), "peak": round(peak, 3),
            "unit": "T MUFU-slot/s", "frac": round(tops / peak, 4), "traffic": traffic,
            "peak_source": f"{mufu_lanes_per_clk()[1]}: {mufu_lanes_per_clk()[0]} ex2 lanes/clk/SM x "
                           f"{sm_count} SMs x {GB300_MAX_SM_MHZ:.0f} MHz",
            "algorithmic_mufu_slots_per_launch": int(slots),
            "algorithmic_bytes_per_launch": int(bytes_per_launch), "avg_launch_ms": round(ms, 6),
            "hbm": {"achieved": round(gbs, 1), "peak": hbm_peak_gbs, "unit": "GB/s",
                    "frac": round(gbs / hbm_peak_gbs, 4), "peak_source": peak_src},
            "fp32": {"achieved": round(fops, 3), "peak": round(fpeak, 3), "unit": "T FP32-op/s",
                     "frac": round(fops / fpeak, 4), "algorithmic_fp32_ops_per_launch": int(ops),
                     "peak_source": f"derived: {FP32_LANES_PER_CLK_SM} lanes/clk/SM x {sm_count} SMs x "
                                    f"{GB300_MAX_SM_MHZ:.0f} MHz"}}


def run_prefill(torch, m, synth, wl_index, steps, warmup, device, dist, clocks, host_inputs=True):
    wl = synth.WORKLOADS[wl_index]
    Bsz, T, Di, N, K = wl.batch, wl.seqlen, wl.d_inner, wl.d_state, wl.d_conv
    params = synth.mixer_params(wl.seed, Di, N, K)
    props = torch.cuda.get_device_properties(device)
    if host_inputs:
        host = synth.prefill_inputs(wl.seed, Bsz, T, Di, N, wl.dtype, names=("x", "dt", "z", "B", "C"))
        first = PrefillSet(torch, host, params, wl.dtype, device)
    else:
        host = None
        first = PrefillSet.from_device(torch, (Bsz, T, Di), N, params, wl.dtype, device, wl.seed)
    conv_b, scan_b = first.bytes_per_step()
    set_bytes = conv_b + scan_b
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    n_sets = 1 if set_bytes > 3 * l2 else int(math.ceil(3 * l2 / set_bytes)) + 1
    sets = [first]
    for _ in range(n_sets - 1):
        s = PrefillSet.__new__(PrefillSet)
        s.__dict__.update({k: (v.clone() if hasattr(v, "clone") else v) for k, v in first.__dict__.items()})
        s.p = first.p
        sets.append(s)
    # the clock record spans the warm-up, the per-kernel timings and the timed
    # steps, so that it holds samples even when the timed steps last milliseconds
    if clocks:
        clocks.start()
    # warm-up steps (eager), then graphs
    for i in range(max(warmup, 3)):
        sets[i % n_sets].conv(m)
        sets[i % n_sets].scan(m)
    torch.cuda.synchronize()
    n_k = 40 if set_bytes < 1e9 else 10
    conv_ms = kernel_time(torch, [lambda s=s: s.conv(m) for s in sets], n_k)
    scan_ms = kernel_time(torch, [lambda s=s: s.scan(m) for s in sets], n_k)
    fused_ms = kernel_time(torch, [lambda s=s: s.fused(m) for s in sets], n_k)
    # both forms compute the same result bit for bit: the step is the faster one
    use_fused = fused_ms < conv_ms + scan_ms
    total_ms, _ = timed_graph_run(torch, m, sets, steps, 100, None, dist, fused=use_fused)
    ck = clocks.stop() if clocks else None
    if ck is not None:
        ck["window"] = "this workload's warm-up, per-kernel timing graphs and timed steps"
    u_bytes = 2 * first.u.numel() * first.u.element_size()  # the u write + read the fusion drops
    route = scan_route(m, Bsz, T, Di, N, props.multi_processor_count)
    l2_note = (f"inputs > 3x L2 ({set_bytes / 1e6:.0f} MB per step)" if n_sets == 1 else
               f"rotating {n_sets} resident buffer sets ({n_sets * set_bytes / 1e6:.0f} MB > 3x the "
               f"{l2 / 1e6:.0f} MB L2)")
    return {
        "wl": wl, "sets": sets, "host": host, "params": params, "total_ms": total_ms,
        "ms_per_step": total_ms / steps, "conv_ms": conv_ms, "scan_ms": scan_ms, "fused_ms": fused_ms,
        "use_fused": use_fused,
        "fused_bytes": conv_b + scan_b - u_bytes,
        "route": route, "conv_bytes": conv_b, "scan_bytes": scan_b,
        "tokens_per_step": Bsz * T, "clocks": ck, "l2_note": l2_note,
    }


def scan_route(m, Bsz, T, Di, N, sms):
    """The route the library plans for a prefill with its default workspace:
    chained (one launch of persistent CTAs) for at least eight 32-channel tiles
    per SM, the T split (state-only pass, fold, full pass: three launches) for
    narrower shapes that get a workspace, else one warp per tile (one launch)."""
    ws = m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N)
    tiles = Bsz * ((Di + 31) // 32)
    if ws > 0:
        return "chained" if tiles >= 8 * sms else "split"
    return "plain"


ROUTE_DESC = {
    "chained": "one launch: persistent CTAs, rows cut into equal roles, tiles handed between roles",
    "split": "T-split: state-only pass, fold, full pass: 3 launches",
    "plain": "one launch: one warp per 32-channel tile",
}


def step_desc(res, fused):
    r = ROUTE_DESC[res["route"]]
    if fused:
        return "mamba_mixer_prefill: conv1d+SiLU fused into the selective scan (" + r + ")"
    return "mamba_conv1d_silu_prefill (1 launch) then mamba_selective_scan_prefill (" + r + ")"


def launches_per_step(res, fused):
    return (0 if fused else 1) + (3 if res["route"] == "split" else 1)


def other_form_line(res):
    """The step in the form the line's value did not use (same result, bit for bit)."""
    fused = not res["use_fused"]
    ms = res["fused_ms"] if fused else res["conv_ms"] + res["scan_ms"]
    b = res["fused_bytes"] if fused else res["conv_bytes"] + res["scan_bytes"]
    return {"step": step_desc(res, fused), "value": round(res["tokens_per_step"] / (ms * 1e-3), 1),
            "unit": "tokens/s", "ms_per_step": round(ms, 5), "algorithmic_bytes_per_step": int(b),
            "hbm_gbs": round(b / (ms * 1e-3) / 1e9, 1), "launches_per_step": launches_per_step(res, fused),
            "timing": "graphs of back-to-back calls per kernel kind, rotating buffer sets"}


def prefill_roofline(res, peak, peak_src, sms):
    """Roofline of the dominant call of the step the line times: the fused
    prefill call, or the selective-scan call of the two-call form."""
    wl = res["wl"]
    tc = wl.batch * wl.seqlen * wl.d_inner
    if res["use_fused"]:
        return scan_roofline(tc, wl.d_state, True, res["fused_bytes"], res["fused_ms"], peak, peak_src,
                             ncu_traffic("fused", wl.name), sms, conv=True)
    return scan_roofline(tc, wl.d_state, True, res["scan_bytes"], res["scan_ms"], peak, peak_src,
                         ncu_traffic("scan", wl.name), sms)


def run_e2e(torch, m, res, steps, device):
    """Same metric through the public API with pinned host buffers: every step
    copies its inputs host->device and reads y and both final states back."""
    wl, host = res["wl"], res["host"]
    s = res["sets"][0]
    if host is not None:
        pin = lambda a, like: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(like.dtype).pin_memory()
        hin = {k: pin(host[k], getattr(s, k)) for k in ("x", "dt", "z", "B", "C")}
    else:  # inputs drawn on the device: their pinned host copies are the step's inputs
        hin = {k: getattr(s, k).cpu().pin_memory() for k in ("x", "dt", "z", "B", "C")}
    hy = torch.empty(s.y.shape, dtype=s.y.dtype).pin_memory()
    hc = torch.empty(s.conv_out.shape).pin_memory()
    hs = torch.empty(s.ssm_out.shape).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in hin.values())
    d2h = hy.numel() * hy.element_size() + hc.numel() * 4 + hs.numel() * 4

    def step():
        for k, t in hin.items():
            getattr(s, k).copy_(t, non_blocking=True)
        if res["use_fused"]:
            s.fused(m)
        else:
            s.conv(m)
            s.scan(m)
        hy.copy_(s.y, non_blocking=True)
        hc.copy_(s.conv_out, non_blocking=True)
        hs.copy_(s.ssm_out, non_blocking=True)

    per = 20

    def time_graph(body):
        g = capture(torch, body)
        g.replay()
        torch.cuda.synchronize()
        reps = max(1, steps // per)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        del g
        return a.elapsed_time(b) / (reps * per)

    ms_serial = time_graph(lambda: [step() for _ in range(per)])

    # pipelined: two device buffer sets; step i's inputs go up on one copy
    # stream and step i's outputs come down on another, so the copies of
    # neighbouring steps overlap step i's kernels (every step still moves
    # all of its bytes inside the timed region)
    if len(res["sets"]) >= 2:
        sets2 = res["sets"][:2]
    else:  # a second buffer set, so that neighbouring steps never share buffers
        s2 = PrefillSet.__new__(PrefillSet)
        s2.__dict__.update({k: (v.clone() if hasattr(v, "clone") else v) for k, v in s.__dict__.items()})
        s2.p = s.p
        sets2 = [s, s2]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def pipelined():
        main = torch.cuda.current_stream()
        ev_comp, ev_d2h = [], []
        s_in.wait_stream(main)
        s_out.wait_stream(main)
        for i in range(per):
            st = sets2[i % 2]
            if i >= 2:
                s_in.wait_event(ev_comp[i - 2])  # this set's inputs are free again
            with torch.cuda.stream(s_in):
                for k, t in hin.items():
                    getattr(st, k).copy_(t, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            main.wait_event(ev_in)
            if i >= 2:
                main.wait_event(ev_d2h[i - 2])  # this set's outputs have been read
            if res["use_fused"]:
                st.fused(m)
            else:
                st.conv(m)
                st.scan(m)
            ev = torch.cuda.Event()
            ev.record(main)
            ev_comp.append(ev)
            s_out.wait_event(ev)
            with torch.cuda.stream(s_out):
                hy.copy_(st.y, non_blocking=True)
                hc.copy_(st.conv_out, non_blocking=True)
                hs.copy_(st.ssm_out, non_blocking=True)
                ev2 = torch.cuda.Event()
                ev2.record(s_out)
            ev_d2h.append(ev2)
        main.wait_stream(s_in)
        main.wait_stream(s_out)

    ms = time_graph(pipelined)
    return {"value": round(res["tokens_per_step"] / (ms * 1e-3), 1), "unit": "tokens/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms, 5), "api": "C ABI via the Python binding, pinned host buffers",
            "schedule": "pipelined over two buffer sets: H2D / kernels / D2H of neighbouring steps overlap",
            "serial": {"value": round(res["tokens_per_step"] / (ms_serial * 1e-3), 1),
                       "ms_per_step": round(ms_serial, 5), "schedule": "H2D, kernels, D2H one after another"}}


def run_decode(torch, m, synth, device, peak, peak_src, n_steps=256):
    """24-layer T=1 decode at batch 128 over a persistent state, graph-replayed."""
    wl = synth.WORKLOADS[2]
    L, Bsz, Di, N, K = wl.n_layers, wl.batch, wl.d_inner, wl.d_state, wl.d_conv
    conv_h, ssm_h = synth.seeded_states(wl.seed, L, Bsz, Di, N, K)
    conv = torch.from_numpy(conv_h).to(device)
    ssm = torch.from_numpy(ssm_h).to(device)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)
    params = [{k: dev(v) for k, v in synth.mixer_params(wl.seed, Di, N, K, layer=l).items()}
              for l in range(L)]
    shape = (n_steps, L, Bsz, Di)
    x = synth.torch_normal(shape, 1.0, wl.seed + 11, device)
    z = synth.torch_normal(shape, 1.0, wl.seed + 12, device)
    dt = synth.torch_normal(shape, 0.1, wl.seed + 13, device)
    Bm = synth.torch_normal((n_steps, L, Bsz, N), 1.0, wl.seed + 14, device)
    Cm = synth.torch_normal((n_steps, L, Bsz, N), 1.0, wl.seed + 15, device)
    u = torch.empty((L, Bsz, Di), device=device)
    y = torch.empty((L, Bsz, Di), device=device)

    def layer_step(s, l):
        p = params[l]
        m.mamba_conv1d_silu_step(u[l], x[s, l], conv, l, p["conv_w"], p["conv_b"])
        m.mamba_ssm_step_batched(y[l], u[l], dt[s, l], Bm[s, l], Cm[s, l], ssm, l, p["A_log"],
                                 p["D"], p["dt_bias"], z[s, l])

    def layer_step_fused(s, l):
        p = params[l]
        m.mamba_mixer_step_batched(y[l], x[s, l], dt[s, l], Bm[s, l], Cm[s, l], conv, ssm, l, p["conv_w"],
                                   p["A_log"], p["conv_b"], p["D"], p["dt_bias"], z[s, l])

    def time_decode(fn):
        for s in range(3):  # warm-up steps
            for l in range(L):
                fn(s, l)
        torch.cuda.synchronize()
        g = capture(torch, lambda: [fn(s, l) for s in range(n_steps) for l in range(L)])
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 4
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        del g
        return a.elapsed_time(b) / (reps * n_steps)

    def time_decode_driver():
        # the library's graph-captured decode driver: 256 steps x 24 layers of
        # fused mixer steps recorded once, replayed with one call
        io = [[{"y": y[l], "x": x[s, l], "dt": dt[s, l], "z": z[s, l], "Bm": Bm[s, l], "Cm": Cm[s, l]}
               for l in range(L)] for s in range(n_steps)]
        for s in range(3):  # warm-up steps
            for l in range(L):
                layer_step_fused(s, l)
        torch.cuda.synchronize()
        with m.DecodeGraph(params, io, conv, ssm) as g:
            g.launch()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            reps = 4
            a.record()
            for _ in range(reps):
                g.launch()
            b.record()
            torch.cuda.synchronize()
            kernels = g.kernels
        return a.elapsed_time(b) / (reps * n_steps), kernels

    ms_sep = time_decode(layer_step)
    ms_fused, driver_kernels = time_decode_driver()
    # per-kernel durations: graphs of one kernel kind over 4 steps x 24 layers
    conv_calls = [lambda s=s, l=l: m.mamba_conv1d_silu_step(u[l], x[s, l], conv, l, params[l]["conv_w"],
                                                             params[l]["conv_b"])
                  for s in range(4) for l in range(L)]
    step_calls = [lambda s=s, l=l: m.mamba_ssm_step_batched(y[l], u[l], dt[s, l], Bm[s, l], Cm[s, l], ssm, l,
                                                             params[l]["A_log"], params[l]["D"],
                                                             params[l]["dt_bias"], z[s, l])
                  for s in range(4) for l in range(L)]
    fused_calls = [lambda s=s, l=l: layer_step_fused(s, l) for s in range(4) for l in range(L)]
    conv_ms = kernel_time(torch, conv_calls, len(conv_calls))
    step_ms = kernel_time(torch, step_calls, len(step_calls))
    fused_ms = kernel_time(torch, fused_calls, len(fused_calls))
    rows = Bsz * Di
    step_bytes = rows * (2 * 4 * N + 5 * 4) + Bsz * N * 2 * 4 + Di * (N + 2) * 4
    conv_bytes = rows * (2 * 4 * K + 2 * 4) + Di * (K + 1) * 4
    fused_bytes = rows * (2 * 4 * N + 2 * 4 * K + 4 * 4) + Bsz * N * 2 * 4 + Di * (N + K + 3) * 4
    out = {
        "workload": wl.name, "value": round(1e3 / ms_fused, 2), "unit": "steps/s",
        "ms_per_step": round(ms_fused, 5),
        "layer_token_updates_per_s": round(1e3 / ms_fused * L * Bsz, 1),
        "algorithmic_bytes_per_step": int(L * fused_bytes),
        "hbm_gbs_per_step": round(L * fused_bytes / (ms_fused * 1e-3) / 1e9, 1),
        "step": "fused mixer step (conv1d+SiLU step then SSM step, 1 launch per layer)",
        "driver": f"mamba_decode_graph: {n_steps} steps x {L} layers recorded once ({driver_kernels} kernels), "
                  "replayed per call",
        "separate_calls": {"value": round(1e3 / ms_sep, 2), "unit": "steps/s", "ms_per_step": round(ms_sep, 5),
                           "hbm_gbs_per_step": round(L * (step_bytes + conv_bytes) / (ms_sep * 1e-3) / 1e9, 1),
                           "step": "conv1d step + SSM step, 2 launches per layer"},
        "config": {"n_layers": L, "batch": Bsz, "d_inner": Di, "d_state": N, "d_conv": K,
                   "steps_per_replay": n_steps,
                   "launch": "library decode graph (fused); CUDA graph of 256 steps x 24 layers (separate calls)",
                   "l2": f"state {L * rows * (N + K) * 4 / 1e6:.0f} MB > L2"},
        "gpu_launches_per_step": L, "separate_calls_launches_per_step": 2 * L,
    }
    out["roofline"] = roofline(fused_bytes, fused_ms, peak, peak_src, ncu_traffic("mixer_step", wl.name))
    out["ssm_step_roofline"] = roofline(step_bytes, step_ms, peak, peak_src, ncu_traffic("step", wl.name))
    out["conv_step_roofline"] = roofline(conv_bytes, conv_ms, peak, peak_src,
                                         ncu_traffic("conv", wl.name + "-step"))
    out["frac_of_hbm_peak"] = round(out["hbm_gbs_per_step"] / peak, 4)
    return out


def run_long_context(torch, m, synth, device, peak, peak_src, sms):
    """Long-context continuation (batch 4, d_inner 2048, d_state 16, d_conv 4,
    f32): one mamba_mixer_prefill of 16384 tokens from a seeded state, then 64
    fused T=1 steps replayed by the library's decode graph.  tokens/s counts
    all 4 x 16448 tokens over the time of both."""
    wl = synth.WORKLOADS[4]
    Bsz, T, Di, N, K, S = wl.batch, wl.seqlen, wl.d_inner, wl.d_state, wl.d_conv, wl.steps
    params = synth.mixer_params(wl.seed, Di, N, K)
    pre = PrefillSet.from_device(torch, (Bsz, T, Di), N, params, "f32", device, wl.seed)
    c0 = synth.torch_normal((Bsz, Di, K), 1.0, wl.seed + 41, device)
    s0 = synth.torch_normal((Bsz, Di, N), 0.5, wl.seed + 42, device)
    conv = torch.empty((1, Bsz, Di, K), device=device)
    ssm = torch.empty((1, Bsz, Di, N), device=device)
    xs = synth.torch_normal((S, Bsz, Di), 1.0, wl.seed + 43, device)
    zs = synth.torch_normal((S, Bsz, Di), 1.0, wl.seed + 44, device)
    dts = synth.torch_normal((S, Bsz, Di), 0.1, wl.seed + 45, device)
    Bs = synth.torch_normal((S, Bsz, N), 1.0, wl.seed + 46, device)
    Cs = synth.torch_normal((S, Bsz, N), 1.0, wl.seed + 47, device)
    ys = torch.empty((S, Bsz, Di), device=device)
    p = pre.p

    def prefill():
        m.mamba_mixer_prefill(pre.y, pre.x, pre.dt, pre.B, pre.C, p["conv_w"], p["A_log"], p["conv_b"], p["D"],
                              p["dt_bias"], pre.z, c0, conv[0], s0, ssm[0])

    io = [[{"y": ys[t], "x": xs[t], "dt": dts[t], "z": zs[t], "Bm": Bs[t], "Cm": Cs[t]}] for t in range(S)]
    prefill()
    torch.cuda.synchronize()
    with m.DecodeGraph([p], io, conv, ssm) as g:
        def step():
            prefill()
            g.launch()
        step()
        torch.cuda.synchronize()
        pre_g = capture(torch, prefill)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        a.record()
        for _ in range(reps):
            pre_g.replay()
            g.launch()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / reps
        pre_ms = kernel_time(torch, [prefill], 5)
        decode_kernels = g.kernels
        del pre_g
    route = scan_route(m, Bsz, T, Di, N, sms)
    _, scan_b = pre.bytes_per_step()
    conv_b, _ = pre.bytes_per_step()
    fused_bytes = conv_b + scan_b - 2 * pre.x.numel() * pre.x.element_size()
    tokens = Bsz * (T + S)
    out = {
        "workload": wl.name, "value": round(tokens / (ms * 1e-3), 1), "unit": "tokens/s", "ms_per_step": round(ms, 5),
        "step": f"mamba_mixer_prefill over {T} tokens ({ROUTE_DESC[route]}) then {S} fused T=1 steps "
                f"(mamba_decode_graph, {decode_kernels} kernels)",
        "prefill_ms": round(pre_ms, 5), "decode_ms": round(ms - pre_ms, 5),
        "config": {"batch": Bsz, "seq_len": T, "decode_steps": S, "d_inner": Di, "d_state": N, "d_conv": K,
                   "state": "seeded (ssm N(0, 0.5^2), conv N(0, 1))",
                   "inputs": "torch device RNG, the tiny-mixer distributions",
                   "l2": f"{fused_bytes / 1e9:.2f} GB per prefill > L2"},
        "gpu_launches_per_step": (3 if route == "split" else 1) + decode_kernels,
    }
    tc = Bsz * T * Di
    out["roofline"] = scan_roofline(tc, N, True, fused_bytes, pre_ms, peak, peak_src,
                                    ncu_traffic("fused", wl.name), sms, conv=True)
    return out


def run_prefill_vs_steps(torch, m, synth, device, lengths=(128, 512, 2048), prompt=5, n_layers=24):
    """Parallel prefill against step-by-step prefill on the 130m layer shape
    (batch 1, d_inner 1536, d_state 16, d_conv 4, f32): one mamba_mixer_prefill
    call over T tokens against T fused T=1 steps replayed by the library's
    decode graph; and a `prompt`-token prompt through `n_layers` layers both
    ways.  Both paths start from the same seeded state; their final states and
    y agree within 2e-4 (1 + |ref|), checked here before timing."""
    wl = synth.WORKLOADS[1]
    Di, N, K = wl.d_inner, wl.d_state, wl.d_conv
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(device)

    def time_fn(fn, reps=5):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def setup(T, L):
        params = [{k: dev(v) for k, v in synth.mixer_params(wl.seed, Di, N, K, layer=l).items()} for l in range(L)]
        x = synth.torch_normal((L, T, 1, Di), 1.0, wl.seed + 31, device)
        z = synth.torch_normal((L, T, 1, Di), 1.0, wl.seed + 32, device)
        dt = synth.torch_normal((L, T, 1, Di), 0.1, wl.seed + 33, device)
        Bm = synth.torch_normal((L, T, 1, N), 1.0, wl.seed + 34, device)
        Cm = synth.torch_normal((L, T, 1, N), 1.0, wl.seed + 35, device)
        c0 = synth.torch_normal((L, 1, Di, K), 0.5, wl.seed + 36, device)
        s0 = synth.torch_normal((L, 1, Di, N), 0.5, wl.seed + 37, device)
        return params, x, z, dt, Bm, Cm, c0, s0

    def both(T, L):
        params, x, z, dt, Bm, Cm, c0, s0 = setup(T, L)
        yp = torch.empty((L, T, 1, Di), device=device)
        cp, sp = torch.empty_like(c0), torch.empty_like(s0)

        def prefill():
            for l in range(L):
                p = params[l]
                m.mamba_mixer_prefill(yp[l].view(1, T, Di), x[l].view(1, T, Di), dt[l].view(1, T, Di),
                                      Bm[l].view(1, T, N), Cm[l].view(1, T, N), p["conv_w"], p["A_log"],
                                      p["conv_b"], p["D"], p["dt_bias"], z[l].view(1, T, Di), c0[l], cp[l],
                                      s0[l], sp[l])
        ys = torch.empty_like(yp)
        cs, ss = c0.clone(), s0.clone()
        io = [[{"y": ys[l, t], "x": x[l, t], "dt": dt[l, t], "z": z[l, t], "Bm": Bm[l, t], "Cm": Cm[l, t]}
               for l in range(L)] for t in range(T)]
        with m.DecodeGraph(params, io, cs, ss) as g:
            g.launch()
            torch.cuda.synchronize()
            prefill()
            torch.cuda.synchronize()
            for got, ref, nm in ((ys, yp, "y"), (cs, cp, "conv state"), (ss, sp, "ssm state")):
                err = ((got - ref).abs() / (1.0 + ref.abs())).max().item()
                if not err <= 2e-4:
                    raise RuntimeError(f"step-by-step and parallel prefill disagree on {nm}: {err:.3g}")

            def steps():
                cs.copy_(c0)
                ss.copy_(s0)
                g.launch()
            reset_ms = time_fn(lambda: (cs.copy_(c0), ss.copy_(s0)))
            step_ms = time_fn(steps) - reset_ms
        pre_g = capture(torch, prefill)  # both paths replay graphs: no host launch cost in either
        pre_ms = time_fn(pre_g.replay)
        del pre_g
        return pre_ms, step_ms

    out = {"workload": "mamba130m-layer, batch 1", "unit": "ms",
           "method": "parallel: mamba_mixer_prefill per layer; step-by-step: T x layers fused T=1 steps replayed "
                     "by mamba_decode_graph (state reset excluded); both as CUDA graphs, L2-resident inputs",
           "single_layer": {}}
    for T in lengths:
        pre_ms, step_ms = both(T, 1)
        out["single_layer"][f"T{T}"] = {"prefill_ms": round(pre_ms, 5), "steps_ms": round(step_ms, 5),
                                        "speedup": round(step_ms / pre_ms, 1)}
    pre_ms, step_ms = both(prompt, n_layers)
    out[f"prompt{prompt}_layers{n_layers}"] = {"prefill_ms": round(pre_ms, 5), "steps_ms": round(step_ms, 5),
                                               "extra_ms_step_path": round(step_ms - pre_ms, 5)}
    return out


# ------------------------------------------------------------ the whole block ----

BLOCK_SHAPES = {  # name: (d_model, d_inner, d_state, d_conv, dt_rank)
    "mamba2.8b": (2560, 5120, 16, 4, 160),
    "mamba130m": (768, 1536, 16, 4, 48),
}


def block_weights(torch, synth, seed, shape, device, layer=0):
    dm, Di, N, K, R = shape
    p = synth.layer_params(seed, dm, Di, N, K, R, layer=layer)
    return {k: torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(device).to(
        torch.bfloat16 if k.endswith("proj_w") else torch.float32) for k, v in p.items()}


def block_stage_calls(torch, m, wd, hidden, Bsz, T, conv_state, ssm_state):
    """The block's seven calls on buffers of their own (the sequence the block
    call makes), for per-stage timing: [(name, call, flops or None)]."""
    dm = hidden.shape[-1]
    Di, K = wd["conv_w"].shape
    N = wd["A_log"].shape[1]
    R = wd["dt_proj_w"].shape[1]
    rows = Bsz * T
    dev = hidden.device
    bf = dict(device=dev, dtype=torch.bfloat16)
    ldx = (R + 2 * N + 7) // 8 * 8
    h = torch.empty(rows, dm, **bf)
    xz = torch.empty(Bsz, T, 2 * Di, **bf)
    u = torch.empty(Bsz, T, Di, **bf)
    xd = torch.empty(Bsz, T, ldx, **bf)
    dt = torch.empty(Bsz, T, Di, **bf)
    y = torch.empty(Bsz, T, Di, **bf)
    hid = hidden.view(rows, dm)
    ws = torch.empty(max(m.mamba_selective_scan_workspace_bytes(Bsz, T, Di, N), 16), dtype=torch.uint8, device=dev)
    return [
        ("rmsnorm", lambda: m.mamba_rmsnorm(h, hid, wd["norm_w"]), None),
        ("in_proj", lambda: m.mamba_linear_bf16(xz.view(rows, 2 * Di), h, wd["in_proj_w"]), 2 * rows * 2 * Di * dm),
        ("conv", lambda: m.mamba_conv1d_silu_prefill(u, xz[:, :, :Di], wd["conv_w"], wd["conv_b"], conv_state,
                                                     conv_state), None),
        ("x_proj", lambda: m.mamba_linear_bf16(xd.view(rows, ldx)[:, :R + 2 * N], u.view(rows, Di), wd["x_proj_w"]),
         2 * rows * (R + 2 * N) * Di),
        ("dt_proj", lambda: m.mamba_linear_bf16(dt.view(rows, Di), xd.view(rows, ldx)[:, :R], wd["dt_proj_w"]),
         2 * rows * Di * R),
        ("scan", lambda: m.mamba_selective_scan_prefill(y, u, dt, xd[:, :, R:R + N], xd[:, :, R + N:R + 2 * N],
                                                        wd["A_log"], wd["D"], wd["dt_bias"], xz[:, :, Di:],
                                                        ssm_state, ssm_state, workspace=ws), None),
        ("out_proj", lambda: m.mamba_linear_bf16(hid, y.view(rows, Di), wd["out_proj_w"], hid), 2 * rows * dm * Di),
    ]


def run_block_prefill_small(torch, m, synth, device, steps=50, warmup=3):
    """One mamba-130m-shaped block prefill (batch 1 x T 2048, d_model 768): the
    narrow shape, where the scan takes its T split and the x_proj its K split;
    tokens/s = 2048 / time per block."""
    shape = BLOCK_SHAPES["mamba130m"]
    dm, Di, N, K, R = shape
    Bsz, T = 1, 2048
    seed = synth.SEED_BASE + 1
    wd = block_weights(torch, synth, seed, shape, device)
    hidden = synth.torch_normal((Bsz, T, dm), 1.0, seed + 31, device)
    conv = torch.zeros((Bsz, Di, K), device=device)
    ssm = torch.zeros((Bsz, Di, N), device=device)
    ws = torch.empty(m.mamba_layer_workspace_bytes(wd, Bsz, T), dtype=torch.uint8, device=device)

    def block():
        m.mamba_layer_prefill(hidden, wd, conv, conv, ssm, ssm, workspace=ws)

    for _ in range(warmup):
        block()
    torch.cuda.synchronize()
    ms = kernel_time(torch, [block], steps, reps=2)
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    route = scan_route(m, Bsz, T, Di, N, sms)
    return {"workload": "mamba130m-block-prefill", "value": round(Bsz * T / (ms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_block": round(ms, 5),
            "config": {"batch": Bsz, "seq_len": T, "d_model": dm, "d_inner": Di, "d_state": N, "d_conv": K,
                       "dt_rank": R, "launch": f"CUDA graph of {steps} blocks", "weights": "random init",
                       "l2": "the block's working set (~40 MB) fits the L2: an upper bound for a cold layer"},
            "scan_route": ROUTE_DESC[route], "gpu_launches_per_block": 6 + (3 if route == "split" else 1)}


def run_block_prefill(torch, m, synth, device, steps=100, warmup=3):
    """One whole mamba-2.8b-shaped Mamba-1 block (RMSNorm, in_proj, conv,
    x_proj, dt_proj, scan, out_proj + residual) over batch 8 x T 4096 through
    mamba_layer_prefill, graph-replayed; tokens/s = 32768 / time per block.
    The roofline is the tensor one of the dominant kernel, the in_proj GEMM."""
    shape = BLOCK_SHAPES["mamba2.8b"]
    dm, Di, N, K, R = shape
    Bsz, T = 8, 4096
    seed = synth.SEED_BASE + 3
    wd = block_weights(torch, synth, seed, shape, device)
    hidden = synth.torch_normal((Bsz, T, dm), 1.0, seed + 31, device)
    conv = synth.torch_normal((Bsz, Di, K), 1.0, seed + 32, device)
    ssm = synth.torch_normal((Bsz, Di, N), 0.5, seed + 33, device)
    ws = torch.empty(m.mamba_layer_workspace_bytes(wd, Bsz, T), dtype=torch.uint8, device=device)

    def block():
        m.mamba_layer_prefill(hidden, wd, conv, conv, ssm, ssm, workspace=ws)

    # the block's GEMMs run the GPU at its power cap: the clocks seen while the
    # block and while its stages are timed go into the line
    ck = ClockSampler(device.index if device.index is not None else 0)
    ck.start()
    for _ in range(warmup):
        block()
    torch.cuda.synchronize()
    ms = kernel_time(torch, [block], steps, reps=1)
    block_clocks = ck.stop()
    stages = block_stage_calls(torch, m, wd, hidden, Bsz, T, conv, ssm)
    stage_ms = {}
    tflops = {}
    ck = ClockSampler(device.index if device.index is not None else 0)
    ck.start()
    for name, fn, flops in stages:
        fn()
        torch.cuda.synchronize()
        stage_ms[name] = kernel_time(torch, [fn], 10 if flops else 5, reps=2)
        if flops:
            tflops[name] = round(flops / (stage_ms[name] * 1e-3) / 1e12, 1)
    stage_clocks = ck.stop()
    burst, sustained, src = bf16_peak()
    in_flops = 2 * Bsz * T * 2 * Di * dm
    ach = in_flops / (stage_ms["in_proj"] * 1e-3) / 1e12
    gemm_flops = sum(f for _, _, f in stages if f)
    gemm_ms = sum(stage_ms[n] for n, _, f in stages if f)
    rows = Bsz * T
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    route = scan_route(m, Bsz, T, Di, N, sms)
    del stages
    return {
        "workload": "mamba2.8b-block-prefill", "value": round(rows / (ms * 1e-3), 1), "unit": "tokens/s",
        "ms_per_block": round(ms, 4),
        "config": {"batch": Bsz, "seq_len": T, "d_model": dm, "d_inner": Di, "d_state": N, "d_conv": K,
                   "dt_rank": R, "storage": "bf16 weights and activations, f32 residual stream/params/states; "
                                            "f32 accumulation", "launch": f"CUDA graph of {steps} blocks",
                   "weights": "random init (no trained weights)"},
        "stage_ms": {k: round(v, 4) for k, v in stage_ms.items()},
        "gemm_tflops": tflops,
        "gemm_share": round(gemm_ms / sum(stage_ms.values()), 3),
        "gemm_tflops_all": round(gemm_flops / (gemm_ms * 1e-3) / 1e12, 1),
        "roofline": {"bound": "tensor", "achieved": round(ach, 1), "peak": burst, "unit": "TFLOP/s",
                     "frac": round(ach / burst, 4), "traffic": ncu_traffic("gemm", "mamba2.8b-in_proj"),
                     "peak_source": f"{src} cuBLAS bf16 burst (sustained {sustained})",
                     "algorithmic_flops_per_launch": int(in_flops), "avg_launch_ms": round(stage_ms["in_proj"], 6)},
        "roofline_kernel": "in_proj GEMM (tcgen05, 128 x 256 tiles)",
        "scan_route": ROUTE_DESC[route],
        "gpu_launches_per_block": 6 + (3 if route == "split" else 1),
        "clocks": block_clocks, "stage_clocks": stage_clocks,
    }


def run_block_decode(torch, m, synth, device, n_steps=32, L=24, Bsz=128):
    """Whole-block T=1 decode on mamba-130m shapes: 24 layers x batch 128, each
    layer the block step (RMSNorm, projections, conv and scan on the layer's
    state slab, out_proj + residual), graph-replayed; steps/s."""
    shape = BLOCK_SHAPES["mamba130m"]
    dm, Di, N, K, R = shape
    seed = synth.SEED_BASE + 2
    wds = [block_weights(torch, synth, seed, shape, device, layer=l) for l in range(L)]
    conv = synth.torch_normal((L, Bsz, Di, K), 0.5, seed + 41, device)
    ssm = synth.torch_normal((L, Bsz, Di, N), 0.5, seed + 42, device)
    emb = synth.torch_normal((n_steps, Bsz, dm), 1.0, seed + 43, device)
    hidden = torch.empty(Bsz, dm, device=device)
    ws = torch.empty(m.mamba_layer_workspace_bytes(wds[0], Bsz, 1), dtype=torch.uint8, device=device)

    def step(s):
        hidden.copy_(emb[s])
        for l in range(L):
            m.mamba_layer_step(hidden, wds[l], conv, ssm, l, workspace=ws)

    for s in range(3):
        step(s)
    torch.cuda.synchronize()
    g = capture(torch, lambda: [step(s) for s in range(n_steps)])
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 4
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (reps * n_steps)
    del g
    # the library's own graph of one token through the 24 blocks, launched
    # per token after the token's hidden state is copied in
    with m.LayerDecodeGraph(wds, hidden, conv, ssm, workspace=ws) as lg:
        kernels = lg.kernels
        for s_ in range(3):
            hidden.copy_(emb[s_])
            lg.launch()
        torch.cuda.synchronize()
        a.record()
        for s_ in range(n_steps):
            hidden.copy_(emb[s_])
            lg.launch()
        b.record()
        torch.cuda.synchronize()
        ms_driver = a.elapsed_time(b) / n_steps
    w_bytes = 2 * (2 * Di * dm + (R + 2 * N) * Di + Di * R + dm * Di)
    state_bytes = Bsz * Di * (N + K) * 4 * 2
    out = {
        "workload": "mamba130m-block-decode-b128-l24", "value": round(1e3 / ms, 2), "unit": "steps/s",
        "ms_per_step": round(ms, 5), "layer_token_updates_per_s": round(1e3 / ms * L * Bsz, 1),
        "config": {"n_layers": L, "batch": Bsz, "d_model": dm, "d_inner": Di, "d_state": N, "d_conv": K,
                   "dt_rank": R, "launch": f"CUDA graph of {n_steps} steps x {L} layers",
                   "weights": "random init, distinct per layer"},
        "bytes_per_step_weights_and_state": int(L * (w_bytes + state_bytes)),
        "hbm_gbs_weights_and_state": round(L * (w_bytes + state_bytes) / (ms * 1e-3) / 1e9, 1),
        "gpu_launches_per_step": L * 7,
        "driver": {"value": round(1e3 / ms_driver, 2), "unit": "steps/s", "ms_per_step": round(ms_driver, 5),
                   "how": f"mamba_layer_decode_graph: one token through {L} blocks recorded once ({kernels} "
                          "kernels), launched per token after a copy of the token's hidden state"},
    }
    peak, peak_src = hbm_peak()
    out["roofline"] = roofline(L * (w_bytes + state_bytes), ms, peak, peak_src, ncu_traffic("block", out["workload"]))
    out["roofline_kernel"] = ("whole 24-layer step (7 kernels per layer; each is latency-bound: the bytes are "
                              "the layers' weights and the state read and written once)")
    return out



def run_m3_decode(torch, m, device, peak, peak_src, n_steps=16, L=24, Bsz=128, H=24, P=64, N=64):
    """Mamba-3 SISO T=1 decode: L layers x batch B, H heads of headdim P and
    d_state N (a synthetic shape: the pages give none), graph-replayed."""
    g = torch.Generator(device=device)
    g.manual_seed(0x5EED0005)
    rn = lambda *shape: torch.randn(shape, generator=g, device=device)
    st = rn(L, Bsz, H, P, N) * 0.5
    ks, vs = rn(L, Bsz, H, N), rn(L, Bsz, H, P)
    x, k, q = rn(n_steps, L, Bsz, H, P), rn(n_steps, L, Bsz, H, N), rn(n_steps, L, Bsz, H, N)
    al = torch.exp(-torch.rand((n_steps, L, Bsz, H), generator=g, device=device) * 0.2)
    be = torch.rand((n_steps, L, Bsz, H), generator=g, device=device) * 0.1
    ga = torch.rand((n_steps, L, Bsz, H), generator=g, device=device) * 0.1
    D = rn(L, H)
    y = torch.empty((L, Bsz, H, P), device=device)

    def step(s_, l):
        m.mamba3_siso_step_batched(y[l], x[s_, l], k[s_, l], q[s_, l], al[s_, l], be[s_, l], ga[s_, l], st, ks, vs,
                                   l, D[l])

    for s_ in range(3):
        for l in range(L):
            step(s_, l)
    torch.cuda.synchronize()
    gr = capture(torch, lambda: [step(s_, l) for s_ in range(n_steps) for l in range(L)])
    gr.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 4
    a.record()
    for _ in range(reps):
        gr.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (reps * n_steps)
    del gr
    kms = kernel_time(torch, [lambda s_=s_, l=l: step(s_, l) for s_ in range(4) for l in range(L)], 4 * L)
    BH = Bsz * H
    per_launch = BH * P * N * 8 + BH * P * 16 + BH * N * 16 + BH * 12 + H * 4
    out = {
        "workload": f"mamba3-siso-decode-b{Bsz}-l{L}-h{H}-p{P}-n{N}", "value": round(1e3 / ms, 2),
        "unit": "steps/s", "ms_per_step": round(ms, 5),
        "config": {"n_layers": L, "batch": Bsz, "nheads": H, "headdim": P, "d_state": N,
                   "shape": "synthetic (the pages give no Mamba-3 shapes)",
                   "launch": f"CUDA graph of {n_steps} steps x {L} layers",
                   "l2": f"state {L * BH * P * N * 4 / 1e9:.2f} GB > L2"},
        "gpu_launches_per_step": L,
    }
    out["roofline"] = roofline(per_launch, kms, peak, peak_src, ncu_traffic("m3_step", out["workload"]))
    del x, k, q, al, be, ga

    # The same decode with each token's step inputs prepared on the GPU first
    # (the fourth state, the angles, advanced by dt * angles; B and C rotated in
    # pairs into k and q; alpha / beta / gamma): two launches per layer.
    na = N // 2
    th = (torch.rand((L, Bsz, H, na), generator=g, device=device) - 0.5) * 100.0
    k_in, q_in = rn(n_steps, L, Bsz, H, N), rn(n_steps, L, Bsz, H, N)
    x = rn(n_steps, L, Bsz, H, P)
    u01 = lambda *shape: torch.rand(shape, generator=g, device=device)
    dt = torch.exp(math.log(1e-3) + u01(n_steps, L, Bsz, H) * math.log(100.0))
    A = -(0.05 + 3.95 * u01(n_steps, L, Bsz, H))
    lam = u01(n_steps, L, Bsz, H)
    ang = (u01(n_steps, L, Bsz, na) * 2.0 - 1.0) * math.pi
    kc, qc = torch.empty((L, Bsz, H, N), device=device), torch.empty((L, Bsz, H, N), device=device)
    alc, bec, gac = (torch.empty((L, Bsz, H), device=device) for _ in range(3))

    def prep(s_, l):
        m.mamba3_siso_step_prepare(kc[l], qc[l], alc[l], bec[l], gac[l], k_in[s_, l], q_in[s_, l], dt[s_, l],
                                   A[s_, l], lam[s_, l], ang[s_, l], th, l)

    def prep_step(s_, l):
        prep(s_, l)
        m.mamba3_siso_step_batched(y[l], x[s_, l], kc[l], qc[l], alc[l], bec[l], gac[l], st, ks, vs, l, D[l])

    for s_ in range(3):
        for l in range(L):
            prep_step(s_, l)
    torch.cuda.synchronize()
    gr = capture(torch, lambda: [prep_step(s_, l) for s_ in range(n_steps) for l in range(L)])
    gr.replay()
    torch.cuda.synchronize()
    a.record()
    for _ in range(reps):
        gr.replay()
    b.record()
    torch.cuda.synchronize()
    ms2 = a.elapsed_time(b) / (reps * n_steps)
    del gr
    pms = kernel_time(torch, [lambda s_=s_, l=l: prep(s_, l) for s_ in range(4) for l in range(L)], 4 * L)

    # the same tokens with the preparation inside the step (one launch per layer)
    def fused(s_, l):
        m.mamba3_siso_step_fused_batched(y[l], x[s_, l], k_in[s_, l], q_in[s_, l], dt[s_, l], A[s_, l], lam[s_, l],
                                         ang[s_, l], st, ks, vs, th, l, D[l])

    for s_ in range(3):
        for l in range(L):
            fused(s_, l)
    torch.cuda.synchronize()
    # replayed through the library's Mamba-3 decode graph (mamba3_decode_graph_create)
    io = [[{"y": y[l], "x": x[s_, l], "k_in": k_in[s_, l], "q_in": q_in[s_, l], "dt": dt[s_, l], "A": A[s_, l],
            "lam": lam[s_, l], "angles": ang[s_, l]} for l in range(L)] for s_ in range(n_steps)]
    with m.Mamba3DecodeGraph(io, st, ks, vs, th, D=[D[l] for l in range(L)]) as gr:
        n_graph_kernels = gr.kernels
        gr.launch()
        torch.cuda.synchronize()
        a.record()
        for _ in range(reps):
            gr.launch()
        b.record()
        torch.cuda.synchronize()
    ms3 = a.elapsed_time(b) / (reps * n_steps)
    fms = kernel_time(torch, [lambda s_=s_, l=l: fused(s_, l) for s_ in range(4) for l in range(L)], 4 * L)
    # k_in, q_in replace k, q and dt, A, lam replace alpha, beta, gamma (same bytes); plus the angles
    fused_bytes = per_launch + BH * na * 8 + Bsz * na * 4
    out["fused"] = {
        "value": round(1e3 / ms3, 2), "unit": "steps/s", "ms_per_step": round(ms3, 5), "n_angles": na,
        "gpu_launches_per_step": n_graph_kernels // n_steps,
        "note": "each layer: mamba3_siso_step_fused_batched (the preparation inside the step); the library's Mamba-3 "
                "decode graph of {} tokens x {} layers".format(n_steps, L),
        "roofline": roofline(fused_bytes, fms, peak, peak_src, ncu_traffic("m3_step", out["workload"] + "-fused")),
    }
    out["with_prepare"] = {
        "value": round(1e3 / ms2, 2), "unit": "steps/s", "ms_per_step": round(ms2, 5),
        "n_angles": na, "gpu_launches_per_step": 2 * L,
        "prepare_us_per_launch": round(pms * 1e3, 3),
        "prepare_bytes_per_launch": int(BH * N * 4 * 4 + BH * na * 8 + BH * 6 * 4 + Bsz * na * 4),
        "note": "each layer: mamba3_siso_step_prepare (angle state, rotated k and q, alpha/beta/gamma) then "
                "mamba3_siso_step_batched",
    }
    return out


# ----------------------------------------------------------- CPU oracle arm --

def oracle_prefill_sample(synth, wl_index, n_channels, nthreads, stride=1):
    """Run the f64 oracle (conv then scan, from the workload's initial state) on
    n_channels channels of the workload (every `stride`-th); returns (seconds,
    tokens-equivalent processed = B*T*n_channels/Di).  Channels are independent
    recurrences, so a sample is a full-fidelity run of those channels."""
    import oracle

    wl = synth.WORKLOADS[wl_index]
    Bsz, T, Di, N, K = wl.batch, wl.seqlen, wl.d_inner, wl.d_state, wl.d_conv
    sel = np.arange(0, Di, stride)[:n_channels]
    g = np.random.default_rng(wl.seed)
    # the sample's inputs, drawn from the workload's distributions (only the
    # sampled channels: drawing a whole 2.8b layer on the host takes longer than
    # the oracle's sample)
    x = g.standard_normal((Bsz, T, len(sel)))
    dt = 0.1 * g.standard_normal((Bsz, T, len(sel)))
    z = g.standard_normal((Bsz, T, len(sel)))
    if wl.dtype == "bf16":
        x, dt, z = (synth.round_to_bf16(v.astype(np.float32)).astype(np.float64) for v in (x, dt, z))
    Bm = g.standard_normal((Bsz, T, N))
    Cm = g.standard_normal((Bsz, T, N))
    params = synth.mixer_params(wl.seed, Di, N, K)
    p = {k: np.ascontiguousarray(v[sel], np.float64) for k, v in params.items()}
    s0 = 0.5 * g.standard_normal((Bsz, len(sel), N)) if wl.state == "seeded" else None
    c0 = g.standard_normal((Bsz, len(sel), K)) if wl.state == "seeded" else None
    t0 = time.perf_counter()
    u, _ = oracle.conv1d_silu_prefill(x, p["conv_w"], p["conv_b"], c0, nthreads=nthreads)
    oracle.selective_scan_prefill(u, dt, Bm, Cm, p["A_log"], p["D"], p["dt_bias"], z, s0, nthreads=nthreads)
    dtm = time.perf_counter() - t0
    return dtm, Bsz * T * len(sel) / Di


def oracle_decode_sample(synth, n_rows, n_layers, n_steps, nthreads):
    """The oracle's fused T=1 step (conv step then SSM step) over n_rows batch
    rows x channels of the 24-layer decode state, n_steps steps of n_layers
    layers; returns (seconds, full 24-layer batch-128 steps equivalent)."""
    import oracle

    wl = synth.WORKLOADS[2]
    L, Bsz, Di, N, K = wl.n_layers, wl.batch, wl.d_inner, wl.d_state, wl.d_conv
    g = np.random.default_rng(wl.seed)
    ch = max(1, n_rows // Bsz)
    conv = 0.5 * g.standard_normal((n_layers, Bsz, ch, K))
    ssm = 0.5 * g.standard_normal((n_layers, Bsz, ch, N))
    params = [synth.mixer_params(wl.seed, Di, N, K, layer=l) for l in range(n_layers)]
    ps = [{k: np.ascontiguousarray(v[:ch], np.float64) for k, v in pl.items()} for pl in params]
    inp = [[(g.standard_normal((Bsz, ch)), 0.1 * g.standard_normal((Bsz, ch)), g.standard_normal((Bsz, ch)),
             g.standard_normal((Bsz, N)), g.standard_normal((Bsz, N))) for _ in range(n_layers)]
           for _ in range(n_steps)]
    t0 = time.perf_counter()
    for s_ in range(n_steps):
        for l in range(n_layers):
            x, dt, z, Bm, Cm = inp[s_][l]
            u = oracle.conv1d_silu_step(x, conv, l, ps[l]["conv_w"], ps[l]["conv_b"], nthreads=nthreads)
            oracle.ssm_step(u, dt, Bm, Cm, ssm, l, ps[l]["A_log"], ps[l]["D"], ps[l]["dt_bias"], z,
                            nthreads=nthreads)
    dtm = time.perf_counter() - t0
    full = n_steps * (n_layers / L) * (Bsz * ch) / (Bsz * Di)
    return dtm, full


def oracle_block_samples(synth, nthreads):
    """The f64 block oracle (oracle/layer.py: numpy matmuls, the C conv and
    scan) on bounded samples of the two block workloads: the mamba-2.8b block
    over 256 tokens of one sequence (every token costs the same, so tokens/s
    carries over to batch 8 x 4096), and one whole-block decode step (24
    layers, batch 128) on mamba-130m shapes."""
    from oracle import layer as OL

    out = {}
    dm, Di, N, K, R = BLOCK_SHAPES["mamba2.8b"]
    seed = synth.SEED_BASE + 3
    p = {k: np.asarray(v, np.float64) for k, v in synth.layer_params(seed, dm, Di, N, K, R).items()}
    x = synth.normal(seed, "hidden", (1024, dm), 1.0).astype(np.float64)
    t0 = time.perf_counter()
    OL.layer_prefill(x, p, 1, 1024)
    sec = time.perf_counter() - t0
    out["mamba2.8b-block-prefill"] = {
        "value": round(1024 / sec, 1), "unit": "tokens/s", "cores": nthreads,
        "sample": f"one sequence of 1024 tokens through the f64 block oracle, {sec:.2f} s; per-token work is the "
                  f"workload's (batch 8 x 4096)"}
    dm, Di, N, K, R = BLOCK_SHAPES["mamba130m"]
    seed = synth.SEED_BASE + 2
    L, Bsz = 24, 128
    ps = [{k: np.asarray(v, np.float64) for k, v in synth.layer_params(seed, dm, Di, N, K, R, layer=l).items()}
          for l in range(L)]
    conv = np.ascontiguousarray(0.5 * np.random.default_rng(seed).standard_normal((L, Bsz, Di, K)))
    ssm = np.ascontiguousarray(0.5 * np.random.default_rng(seed + 1).standard_normal((L, Bsz, Di, N)))
    h = synth.normal(seed, "hidden", (Bsz, dm), 1.0).astype(np.float64)
    t0 = time.perf_counter()
    for l in range(L):
        h, _ = OL.layer_step(h, ps[l], conv, ssm, l)
    sec = time.perf_counter() - t0
    out["mamba130m-block-decode-b128-l24"] = {
        "value": round(1.0 / sec, 3), "unit": "steps/s", "cores": nthreads,
        "sample": f"one whole-block decode step (24 layers, batch 128) through the f64 block oracle, {sec:.2f} s"}
    return out


def cpu_baseline(synth, headline_wl=3):
    """The f64 oracle as it stands, on all host cores, per workload: bounded
    samples of independent channels (or rows), each about 2-10 s, with the
    throughput scaled to the whole workload; plus one thread on the headline
    workload."""
    import oracle

    nthreads = oracle.default_threads()
    per = {}

    def timed(fn, budget):
        tot_s, tot_u, reps = 0.0, 0.0, 0
        while tot_s < budget:
            s_, u_ = fn()
            tot_s += s_
            tot_u += u_
            reps += 1
        return tot_s, tot_u, reps

    for wl_index, n_ch, budget in ((1, 1536, 6.0), (3, 256, 6.0), (4, 128, 4.0)):
        wl = synth.WORKLOADS[wl_index]
        stride = max(1, wl.d_inner // n_ch)
        sec, tok, reps = timed(lambda: oracle_prefill_sample(synth, wl_index, n_ch, nthreads, stride), budget)
        per[wl.name] = {"value": round(tok / sec, 1), "unit": "tokens/s", "cores": nthreads,
                        "sample": f"{reps} x {n_ch} of {wl.d_inner} channels (every {stride}-th), all "
                                  f"{wl.batch} x {wl.seqlen} tokens, f64 conv+scan; {sec:.1f} s of wall time; "
                                  f"tokens/s scaled by d_inner / channels"}
    sec, steps, reps = timed(lambda: oracle_decode_sample(synth, 128 * 16, 24, 2, nthreads), 4.0)
    per[synth.WORKLOADS[2].name] = {
        "value": round(steps / sec, 3), "unit": "steps/s", "cores": nthreads,
        "sample": f"{reps} x 2 steps x 24 layers on batch 128 x 16 of 1536 channels, f64 conv step + SSM step; "
                  f"{sec:.1f} s; steps/s scaled to all 1536 channels"}
    per.update(oracle_block_samples(synth, nthreads))
    wl = synth.WORKLOADS[headline_wl]
    s1, t1, _ = timed(lambda: oracle_prefill_sample(synth, headline_wl, 16, 1, wl.d_inner // 16), 1.5)
    head = per[wl.name]
    return {"value": head["value"], "unit": "tokens/s", "cores": nthreads, "kind": "oracle",
            "sample": head["sample"],
            "single_core": {"value": round(t1 / s1, 1), "unit": "tokens/s",
                            "sample": f"16 channels of the same workload on 1 thread, {s1:.2f} s"},
            "per_workload": per}


def replica_throughput(torch, local_ms, tokens_per_step, steps, world, dist=None, device=None):
    """Whole-job throughput of `world` independent replicas: every rank ran
    `steps` steps of `tokens_per_step` tokens in local_ms; the job took the
    slowest rank's time.  Returns (max_ms, tokens/s over all ranks)."""
    total_ms = local_ms
    if dist is not None:
        t = torch.tensor([float(local_ms)], device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    return total_ms, world * tokens_per_step * steps / (total_ms * 1e-3)


def run_reference(args, rank, world):
    """The oracle as the reference arm: the f64 CPU oracle on this host's cores,
    on the headline workload (the mamba-2.8b layer prefill), each step a
    bounded sample of its channels."""
    from selective_state_space_conv1d_gb300 import synth
    import oracle

    if rank != 0:
        return
    nthreads = oracle.default_threads()
    wl = synth.WORKLOADS[HEADLINE_WL]
    n_steps = args.steps + args.warmup
    # size the per-step sample so the whole run stays within --ref-budget seconds
    one_s, _ = oracle_prefill_sample(synth, HEADLINE_WL, 8, nthreads, wl.d_inner // 8)
    per_ch = one_s / 8
    n_ch = int(max(1, min(wl.d_inner, (args.ref_budget / max(n_steps, 1)) / max(per_ch, 1e-9))))
    stride = max(1, wl.d_inner // n_ch)
    for _ in range(args.warmup):
        oracle_prefill_sample(synth, HEADLINE_WL, n_ch, nthreads, stride)
    tot_s, tot_tok = 0.0, 0.0
    for _ in range(args.steps):
        s_, tok = oracle_prefill_sample(synth, HEADLINE_WL, n_ch, nthreads, stride)
        tot_s += s_
        tot_tok += tok
    value = tot_tok / tot_s
    sample = (f"{n_ch} of {wl.d_inner} channels (every {stride}-th) of the 2.8b-layer prefill per step "
              f"({wl.batch}x{wl.seqlen}, d_state 16, bf16-rounded inputs), f64 conv+scan; tokens/s scaled by "
              f"d_inner / channels")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_s / max(args.steps, 1), 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "batch": wl.batch, "seq_len": wl.seqlen,
                   "d_inner": wl.d_inner, "d_state": wl.d_state, "d_conv": wl.d_conv},
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": nthreads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- main --

HEADLINE_WL = 3  # the mamba-2.8b layer prefill: the largest single-GPU prefill workload


def prefill_line(res, peak, peak_src, sms):
    """One prefill workload as an extra line: value, dominant call's roofline, the other form."""
    wl = res["wl"]
    return {
        "workload": wl.name, "value": round(res["tokens_per_step"] / (res["ms_per_step"] * 1e-3), 1),
        "unit": "tokens/s", "ms_per_step": round(res["ms_per_step"], 5),
        "hbm_gbs_per_step": round((res["fused_bytes"] if res["use_fused"] else res["conv_bytes"] + res["scan_bytes"])
                                  / (res["ms_per_step"] * 1e-3) / 1e9, 1),
        "step": step_desc(res, res["use_fused"]),
        "gpu_launches_per_step": launches_per_step(res, res["use_fused"]),
        "roofline": prefill_roofline(res, peak, peak_src, sms),
        "conv_roofline": roofline(res["conv_bytes"], res["conv_ms"], peak, peak_src, ncu_traffic("conv", wl.name)),
        "other_form": other_form_line(res),
        "config": {"batch": wl.batch, "seq_len": wl.seqlen, "d_inner": wl.d_inner, "d_state": wl.d_state,
                   "d_conv": wl.d_conv, "storage": wl.dtype + " activations, f32 y/params/state",
                   "l2": res["l2_note"]},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-extra", action="store_true", help="headline workload only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="--impl reference: seconds of oracle work for the whole run")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch

    import selective_state_space_conv1d_gb300 as m
    from selective_state_space_conv1d_gb300 import synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as td

        td.init_process_group("nccl", device_id=device)
        dist = td
    m.load()
    _ALU["probe"] = alu_probe()
    peak, peak_src = hbm_peak()
    clocks = ClockSampler(local_rank)
    sms = torch.cuda.get_device_properties(device).multi_processor_count

    # headline: the mamba-2.8b layer prefill (inputs drawn on the device: too
    # large to draw on the host quickly; > 3x L2, so every step reads HBM)
    res = run_prefill(torch, m, synth, HEADLINE_WL, args.steps, args.warmup, device, dist, clocks,
                      host_inputs=False)
    total_ms, value = replica_throughput(torch, res["total_ms"], res["tokens_per_step"], args.steps, world, dist,
                                         device)
    ms_step = total_ms / args.steps
    head_roof = prefill_roofline(res, peak, peak_src, sms)
    conv_roof = roofline(res["conv_bytes"], res["conv_ms"], peak, peak_src, ncu_traffic("conv", res["wl"].name))
    step_bytes = res["fused_bytes"] if res["use_fused"] else res["conv_bytes"] + res["scan_bytes"]
    step_gbs = step_bytes / (ms_step * 1e-3) / 1e9

    extra = {}
    if not args.no_extra:
        r1 = run_prefill(torch, m, synth, 1, 2000, 3, device, None, None)
        extra["prefill_130m_f32"] = prefill_line(r1, peak, peak_src, sms)
        extra["prefill_130m_f32"]["e2e"] = run_e2e(torch, m, r1, 400, device)
        del r1
        torch.cuda.empty_cache()
        extra["long_context_b4_t16384"] = run_long_context(torch, m, synth, device, peak, peak_src, sms)
        torch.cuda.empty_cache()
        extra["decode_130m_b128_l24"] = run_decode(torch, m, synth, device, peak, peak_src)
        extra["decode_mamba3_siso"] = run_m3_decode(torch, m, device, peak, peak_src)
        extra["prefill_vs_steps"] = run_prefill_vs_steps(torch, m, synth, device)
        torch.cuda.empty_cache()
        extra["block_prefill_2p8b"] = run_block_prefill(torch, m, synth, device)
        torch.cuda.empty_cache()
        extra["block_decode_130m_b128_l24"] = run_block_decode(torch, m, synth, device)
        extra["block_prefill_130m"] = run_block_prefill_small(torch, m, synth, device)

    e2e = run_e2e(torch, m, res, min(args.steps, 100), device)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(synth, HEADLINE_WL)

    if cpu is not None:
        for key, name in (("block_prefill_2p8b", "mamba2.8b-block-prefill"),
                          ("block_decode_130m_b128_l24", "mamba130m-block-decode-b128-l24")):
            if key in extra and name in cpu["per_workload"]:
                extra[key]["cpu_baseline"] = dict(cpu["per_workload"][name], kind="oracle")

    if rank == 0:
        wl = res["wl"]
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 6),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded, the tiny-mixer distributions; inputs drawn on the device)",
            "config": {"workload": wl.name, "batch": wl.batch, "seq_len": wl.seqlen,
                       "d_inner": wl.d_inner, "d_state": wl.d_state, "d_conv": wl.d_conv,
                       "storage": "bf16 x/dt/z/B/C, f32 y/params/state; arithmetic f32",
                       "step": step_desc(res, res["use_fused"]),
                       "parallelism": f"replicas x{world}", "l2": res["l2_note"],
                       "launch": "CUDA graph replays of up to 100 steps"},
            "hbm_gbs_per_step": round(step_gbs, 1),
            "roofline": head_roof,
            "roofline_kernel": ("fused conv+scan prefill call" if res["use_fused"] else "selective-scan prefill call")
                               + f" ({ROUTE_DESC[res['route']]})",
            "conv_roofline": conv_roof,
            "other_form": other_form_line(res),
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches_per_step(res, res["use_fused"]) * args.steps,
            "clocks": res["clocks"],
            "alu_probe": _ALU["probe"],
            "extra": extra,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
