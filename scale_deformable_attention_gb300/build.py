"""Build the sm_103a CUDA library ``libmsda.so`` in-tree.

    python -m scale_deformable_attention_gb300.build [--force] [--verbose]

Each translation unit under ``csrc/`` is compiled in parallel with nvcc for
``sm_103a`` only, then linked into a shared library against the shared CUDA
runtime (so it shares one runtime instance with PyTorch in a process).
"""
from __future__ import annotations

import argparse
import fcntl
import glob
import hashlib
import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmsda.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library needs the CUDA 13 toolkit to build")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h")) + [
        os.path.abspath(__file__)]


STAMP = LIB + ".stamp"


def _stamp() -> str:
    """Digest of every source the library is built from, of the build flags and
    of the machine it is built on: a library built elsewhere, or from other
    sources, is rebuilt whatever its file times say."""
    h = hashlib.sha256()
    for p in sorted(_deps()):
        with open(p, "rb") as f:
            h.update(os.path.relpath(p, ROOT).encode() + b"\0" + f.read())
    h.update(" ".join(ARCH).encode() + platform.machine().encode())
    return h.hexdigest()


def stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(STAMP):
        return True
    with open(STAMP) as f:
        return f.read().strip() != _stamp()


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    # one builder at a time (parallel test workers may all find the library stale)
    with open(os.path.join(BUILD, ".lock"), "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        if not force and not stale():
            return LIB
        return _build_locked(verbose, ptxas_info)


def _build_locked(verbose: bool, ptxas_info: bool) -> str:
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
                     "--expt-relaxed-constexpr"]
    if ptxas_info:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [cc] + common + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr[-6000:]}")
        return obj, r.stderr

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_info:
        for obj, err in results:
            sys.stderr.write(err)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    with open(STAMP + ".tmp", "w") as f:
        f.write(_stamp())
    os.replace(STAMP + ".tmp", STAMP)
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers / spills / shared memory per kernel")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose, ptxas_info=args.ptxas_info))


if __name__ == "__main__":
    main()
