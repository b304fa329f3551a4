"""Builds the C-ABI library libseqsum.so from csrc/ with nvcc, for sm_103a.

Every device translation unit is compiled with --fmad=false (no contraction
anywhere on the device path), and the result is a plain shared library that
Python loads with ctypes; no PyTorch extension machinery is involved.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libseqsum.so")
# self-checking variant (-DSEQSUM_CHECKS): bounds checks on every computed index
CHECK_BUILD = os.path.join(BUILD, "check")
CHECK_LIB = os.path.join(CHECK_BUILD, "libseqsum.so")
SOURCES = ["seqsum_kernel.cu", "seqsum_api.cu", "seqsum_static.cu"]
HEADERS = ["binade_math.cuh", "seqsum_internal.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "--fmad=false", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fno-fast-math", "-Xcompiler", "-ffp-contract=off",
                     "--expt-relaxed-constexpr"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libseqsum")
    return exe


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


# profiling variant (-DSEQSUM_PROFILE): a timeline of two streaming CTAs and the walk's phases in the diagnostic words
PROFILE_BUILD = os.path.join(BUILD, "profile")
PROFILE_LIB = os.path.join(PROFILE_BUILD, "libseqsum.so")


def build(force: bool = False, extra_flags=(), verbose: bool = False, checks: bool = False,
          profile: bool = False) -> str:
    bdir, lib = (CHECK_BUILD, CHECK_LIB) if checks else ((PROFILE_BUILD, PROFILE_LIB) if profile else (BUILD, LIB))
    if checks:
        extra_flags = tuple(extra_flags) + ("-DSEQSUM_CHECKS",)
    if profile:
        extra_flags = tuple(extra_flags) + ("-DSEQSUM_PROFILE",)
    os.makedirs(bdir, exist_ok=True)
    inc = os.path.join(os.path.dirname(HERE), "include")
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(inc, "seqsum.h"), __file__]
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-I", inc, "-c", s, "-o", o + ".tmp"]
            jobs.append((cmd, o))

    def run(job):
        cmd, o = job
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        os.replace(o + ".tmp", o)
        return r.stderr

    with ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(force="--force" in sys.argv or bool(extra), extra_flags=extra, verbose=v or bool(extra),
                checks="--checks" in sys.argv))
