"""Build libmagicpig.so in-tree with nvcc for sm_103a (one translation unit per .cu, in parallel).

    python -m lsh_sampled_sparse_gb300.build [--force] [--verbose] [--checks]

--checks builds libmagicpig_checks.so instead: the same sources with -DMP_CHECKS=1, whose kernels
check the indices of their global accesses and raise MP_ERR_BOUNDS instead of making an
out-of-range one (the binding loads it when MAGICPIG_CHECKS=1 is set).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(ROOT, "_build", "obj")
LIB = os.path.join(PKG, "libmagicpig.so")
OBJDIR_CHECKS = os.path.join(ROOT, "_build", "obj_checks")
LIB_CHECKS = os.path.join(PKG, "libmagicpig_checks.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libmagicpig")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hdrs + sources() + [os.path.abspath(__file__)]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _run(cmd: list[str], verbose: bool) -> None:
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)


def build(force: bool = False, verbose: bool = False, checks: bool = False) -> str:
    """Compile every .cu under csrc/ and link libmagicpig.so (libmagicpig_checks.so with
    checks=True) next to this file; returns its path."""
    lib, objdir = (LIB_CHECKS, OBJDIR_CHECKS) if checks else (LIB, OBJDIR)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (["-DMP_CHECKS=1"] if checks else [])
    objs = []
    cmds = []
    for src in sources():
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmds.append([cc] + flags + ["-c", src, "-o", obj])
    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, len(cmds))) as ex:
        for f in [ex.submit(_run, c, verbose) for c in cmds]:
            f.result()
    tmp = lib + ".tmp"
    _run([cc] + ARCH + ["-shared", "-o", tmp] + objs, verbose)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
                checks="--checks" in sys.argv))
