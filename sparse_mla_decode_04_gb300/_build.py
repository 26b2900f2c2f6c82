"""Builds libsmla.so in-tree with nvcc for sm_103a.

The translation units (kernels + host C ABI) are compiled in parallel and
linked against the static CUDA runtime.  Host code is compiled with
-ffp-contract=off so that the planner's floating-point cost model evaluates
identically on x86-64 and aarch64.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
BUILD = PKG / "_build"
LIB_DIR = PKG / "lib"
LIB_NAME = "libsmla.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

SOURCES = ["smla_decode.cu", "smla_host.cpp", "smla_static_scratch.cu", "smla_cache_write.cu", "smla_topk.cu"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsmla.so")
    return cand


def lib_path() -> Path:
    return LIB_DIR / LIB_NAME


def _stale(target: Path, deps) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(Path(d).stat().st_mtime > t for d in deps)


def build(verbose: bool = False, force: bool = False) -> Path:
    """Compile (if out of date) and return the path of libsmla.so."""
    nvcc = nvcc_path()
    BUILD.mkdir(exist_ok=True)
    LIB_DIR.mkdir(exist_ok=True)
    headers = list(CSRC.glob("*.h")) + list(CSRC.glob("*.cuh")) + list(INCLUDE.glob("*.h"))
    common = [nvcc, *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-ffp-contract=off",
              f"-I{INCLUDE}", f"-I{CSRC}"]
    objs, jobs = [], []
    for src in SOURCES:
        s = CSRC / src
        o = BUILD / (s.stem + ".o")
        objs.append(o)
        if force or _stale(o, [s, *headers]):
            jobs.append(common + ["-c", str(s), "-o", str(o)])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            print(" ".join(cmd))
            print(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed ({r.returncode}) for {cmd[-3]}")

    if jobs:
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            list(ex.map(run, jobs))
    lib = lib_path()
    if force or jobs or _stale(lib, objs):
        tmp = lib.with_suffix(".so.tmp")
        run([nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
