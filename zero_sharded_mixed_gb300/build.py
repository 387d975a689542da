"""Build libzero_gb300.so in-tree: nvcc for sm_103a only, no cmake.

    python -m zero_sharded_mixed_gb300.build [--verbose] [--force]

Each translation unit is compiled in parallel into ``_build/`` and linked into
``zero_sharded_mixed_gb300/libzero_gb300.so`` (the CUDA runtime is linked
statically, so the library needs only the driver at run time).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "zero_gb300")
LIB = os.path.join(PKG, "libzero_gb300.so")

CUDA_SOURCES = ["zero_runtime.cu", "zero_rs_adamw.cu", "zero_accumulate.cu", "zero_gather.cu",
                "zero_norm.cu", "zero_quant.cu", "zero_rs_adamw_tma.cu", "zero_qgrad.cu",
                "zero_schedule.cu", "zero_cast.cu"]
HOST_SOURCES = ["zero_host.cpp", "zero_ckpt.cpp"]
HEADERS = ["zero_common.cuh", "zero_update.cuh", "zero_quant.cuh", "zero_tma.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Host code: no FMA contraction either (the bias corrections are formed on the host).
HOST_FLAGS = ["-O2", "-fPIC", "-ffp-contract=off", "-std=c++17"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzero_gb300.so")


def _nvcc_flags(verbose: bool, defines=()) -> list[str]:
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-I", INCLUDE, "-I", CSRC,
             "-Xcompiler", ",".join(HOST_FLAGS)]
    if verbose:
        flags += ["-Xptxas", "-v"]
    flags += [f"-D{d}" for d in defines]
    return flags


def _stale(out: str, deps: list[str]) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, defines=(), out: str = LIB) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "zero_gb300.h")]
    jobs = []
    objs = []
    tag = "" if not defines else "_" + "_".join(d.replace("=", "") for d in defines)
    for src in CUDA_SOURCES + HOST_SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + tag + ".o")
        objs.append(obj)
        if force or _stale(obj, [path, *headers, __file__]):
            if src.endswith(".cu"):
                cmd = [nvcc(), *_nvcc_flags(verbose, defines), "-c", path, "-o", obj]
            else:
                cmd = ["g++", *HOST_FLAGS, "-I", INCLUDE, "-c", path, "-o", obj]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with cf.ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose and (r.stdout or r.stderr):
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("compile failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if force or jobs or _stale(out, objs):
        tmp = out + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        os.replace(tmp, out)
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose))


if __name__ == "__main__":
    main()
