"""Build libfa.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each translation unit compiles in its own nvcc process (in parallel), then one
link step produces ``io_aware_exact_14_gb300/libfa.so``.  The CUDA runtime is
linked statically, so loading the library needs no libcudart on the path and
works on a machine without a GPU (only the calls need a device).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libfa.so")

SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_fwd_q4.cu", "fa_fwd_d256.cu", "fa_bwd.cu", "fa_bwd_d256.cu", "fa_fp8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfa.so")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "fa.h")]
    return [f for f in files if os.path.isfile(f)]


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in _deps() + [src, __file__])


def build(verbose: bool = False, force: bool = False, ptxas_info: bool = False) -> str:
    """Compile (as needed) and link libfa.so; returns its path."""
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    jobs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        if force or _stale(obj, path):
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c", path, "-o", obj]
            if ptxas_info:
                cmd += ["-Xptxas", "-v"]
            jobs.append((src, cmd))

    def run(job):
        src, cmd = job
        p = subprocess.run(cmd, capture_output=True, text=True)
        return src, cmd, p

    if jobs:
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for src, cmd, p in ex.map(run, jobs):
                if verbose or ptxas_info or p.returncode != 0:
                    sys.stderr.write(f"[build] {' '.join(cmd)}\n{p.stdout}{p.stderr}")
                if p.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {src}")
    objs = [os.path.join(BUILD_DIR, s.replace(".cu", ".o")) for s in SOURCES]
    if jobs or not os.path.exists(LIB_PATH) or any(os.path.getmtime(o) > os.path.getmtime(LIB_PATH) for o in objs):
        tmp = LIB_PATH + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or p.returncode != 0:
            sys.stderr.write(f"[build] {' '.join(cmd)}\n{p.stdout}{p.stderr}")
        if p.returncode != 0:
            raise RuntimeError("link of libfa.so failed")
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, force="-f" in sys.argv, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)
