"""Build libmamba_ssm.so (the C-ABI library) in-tree with nvcc for sm_103a.

The translation units compile in parallel; the result lands next to this file
so the Python binding (and any C caller) loads it from the package directory.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libmamba_ssm.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)

SOURCES = ["api.cu", "conv1d.cu", "scan_prefill.cu", "ssm_step.cu", "noalloc.cu", "decode_graph.cu", "m3_step.cu",
           "m3_prepare.cu", "selftest.cu", "gemm.cu", "rmsnorm.cu"]
# scan_inst.cu is compiled once per (storage dtype, d_state): small parallel units
SCAN_INST = [(bf16, n) for n in (1, 2, 4, 8, 16, 32, 64) for bf16 in (0, 1)]
HEADERS = [os.path.join(CSRC, h) for h in ("async_copy.cuh", "device_math.cuh", "launch.h", "m3_math.cuh", "scan_kernel.cuh")] + [
    os.path.join(INCLUDE, "mamba_ssm.h")
]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr", "-I", INCLUDE,
]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmamba_ssm.so")
    return cand


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = ([os.path.join(CSRC, s) for s in SOURCES + ["scan_inst.cu"]] + HEADERS
            + [os.path.abspath(__file__)])
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile (if stale) and return the path of libmamba_ssm.so."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(job) -> str:
        src, obj_name, defines = job
        obj = os.path.join(BUILD_DIR, obj_name)
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, *defines, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} {defines}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        return obj

    jobs = [(f"scan_inst.cu", f"scan_{'bf16' if b else 'f32'}_{n}.o", [f"-DSCAN_BF16={b}", f"-DSCAN_N={n}"])
            for b, n in SCAN_INST]
    jobs.sort(key=lambda j: -int(j[2][1].split("=")[1]))  # largest d_state first
    jobs += [(src, os.path.splitext(src)[0] + ".o", []) for src in SOURCES]
    workers = max(1, min(len(jobs), os.cpu_count() or 4))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(compile_one, jobs))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
