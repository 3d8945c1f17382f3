"""Build the CUDA library libnanoflow.so in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel and linked into
``nano_intra_device_gb300/_build/libnanoflow.so``.  The CUDA runtime is linked
statically and the driver is reached through the runtime's entry-point query,
so the library loads on a machine without a GPU driver (its calls then fail
cleanly).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libnanoflow.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "gemm_tc.cu", "gemm_wrows.cu", "attn_mma.cu", "attn_prefill.cu", "meta.cu", "moe.cu", "rmsnorm.cu", "runtime.cu",
           "profile.cu", "search.cpp", "noalloc.cu", "selftest.cu"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O3",
                   "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
                   "-I", CSRC] + list(extra)


def _stale(obj, src):
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    deps.append(os.path.join(ROOT, "include", "nanoflow.h"))
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    objs, jobs = [], []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(OUT_DIR, s.rsplit(".", 1)[0] + ".o")
        objs.append(obj)
        if force or _stale(obj, src):
            extra = ["-Xptxas", "-v"] if ptxas_info and s.endswith(".cu") else []
            jobs.append([cc] + _flags(extra) + ["-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        for out in ex.map(run, jobs):
            if verbose and out.strip():
                print(out, file=sys.stderr)
    if jobs or not os.path.exists(LIB):
        tmp = LIB + ".tmp"
        run([cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv, ptxas_info="--ptxas" in sys.argv))
