"""Builds the package's CUDA libraries in-tree with nvcc, for sm_103a only.

    python -m engram_hashed_gram_gb300.build [--force] [--ptxas-info]

produces ``engram_hashed_gram_gb300/libengram.so`` (the layer's C ABI,
include/engram.h) and ``engram_hashed_gram_gb300/libengram_synth.so`` (the
device twin of the seeded table generator, include/engram_synth.h).
Translation units compile in parallel; a library is rebuilt only when one of
its sources or headers is newer than it.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                     "-I", INCLUDE]

LIBS = {
    "libengram.so": ["gather.cu", "gemm.cu", "gate.cu", "engram_api.cu", "noalloc.cu", "hash.cu"],
    "libengram_synth.so": ["synth.cu"],
}
HEADERS = [os.path.join(CSRC, h) for h in ("common.cuh", "internal.cuh")] + \
          [os.path.join(INCLUDE, h) for h in ("engram.h", "engram_synth.h")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the Engram CUDA libraries cannot be built")


def lib_path(name: str) -> str:
    return os.path.join(HERE, name)


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd: list[str]) -> None:
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        print(r.stderr.strip())


def build(force: bool = False, ptxas_info: bool = False, verbose: bool = False) -> dict[str, str]:
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    for lib, srcs in LIBS.items():
        for s in srcs:
            src = os.path.join(CSRC, s)
            obj = os.path.join(BUILD, s.replace(".cu", ".o"))
            if force or ptxas_info or _stale(obj, [src] + HEADERS):
                jobs.append([exe, *NVCC_FLAGS, *extra, "-c", src, "-o", obj])
    if jobs:
        with ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
            list(ex.map(_run, jobs))
    out = {}
    for lib, srcs in LIBS.items():
        objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in srcs]
        target = lib_path(lib)
        if force or _stale(target, objs):
            _run([exe, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", target, *objs])
            if verbose:
                print("built", target)
        out[lib] = target
    return out


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true")
    args = ap.parse_args()
    for k, v in build(force=args.force, ptxas_info=args.ptxas_info, verbose=True).items():
        print(k, "->", v)


if __name__ == "__main__":
    main()
