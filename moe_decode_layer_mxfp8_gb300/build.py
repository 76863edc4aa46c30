"""Builds libmono_layer.so (the layer's C ABI and sm_103a kernels) in-tree.

Each .cu file compiles to an object in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo``; the objects link into a
shared library with the CUDA runtime linked statically.  Run ``python -m
moe_decode_layer_mxfp8_gb300.build`` or call ``build()``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmono_layer.so")
SOURCES = ["k_gemm.cu", "k_expert_tc.cu", "k_dense_tc.cu", "k_norm.cu", "k_attn.cu", "k_route.cu", "mono_layer.cu",
           "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the layer")


def _flags(verbose_ptxas: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "mono_layer.h"))
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True) -> str:
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    jobs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(OUT_DIR, s.replace(".cu", ".o"))
        if force or verbose_ptxas or _stale(obj, src):
            jobs.append((src, obj))

    def run(job):
        src, obj = job
        cmd = [nvcc] + _flags(verbose_ptxas) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r

    with cf.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        for src, r in ex.map(run, jobs):
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
            if verbose_ptxas or (not quiet and r.stderr.strip()):
                sys.stderr.write(r.stderr)
    objs = [os.path.join(OUT_DIR, s.replace(".cu", ".o")) for s in SOURCES]
    if jobs or not os.path.exists(LIB):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-lcuda"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            # libcuda.so may be absent on a machine without a driver; the library only needs
            # the runtime (driver entry points are fetched at run time)
            cmd = cmd[:-1]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("link failed:\n" + r.stderr)
        os.replace(tmp, LIB)
    return LIB


PROBE_LIB = os.path.join(HERE, "libmono_probe.so")


def build_probe(force: bool = False) -> str:
    """The schedule probe (csrc/probe_schedule.cu), its own small library."""
    src = os.path.join(CSRC, "probe_schedule.cu")
    if force or not os.path.exists(PROBE_LIB) or os.path.getmtime(src) > os.path.getmtime(PROBE_LIB):
        tmp = PROBE_LIB + f".tmp{os.getpid()}"
        cmd = [_nvcc()] + ARCH + ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                                  "-cudart", "static", src, "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on probe_schedule.cu:\n" + r.stderr)
        os.replace(tmp, PROBE_LIB)
    return PROBE_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, quiet=False))
