"""Builds the CUDA library ``libattn_sm103.so`` in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library (CUDA runtime linked statically; the driver's tensor-map
encoder is looked up at run time, so the library loads on machines without a
GPU driver).  Rebuilds only when a source or header is newer than the library.

``build(debug=True)`` makes the checking build ``libattn_sm103_debug.so``
(compiled with -DATTN_DEBUG): the same entry points, with device-side bounds
checks before every tensor-map copy and global store that record
ATTN_ERR_DEVICE_BOUNDS and skip the access instead of faulting.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libattn_sm103.so")
LIB_DEBUG = os.path.join(HERE, "libattn_sm103_debug.so")
SOURCES = ["api.cu", "meta.cu", "fwd.cu", "bwd.cu", "bwd_bf16.cu", "bwd_f16.cu", "dkdv128.cu",
           "dq128.cu", "fwd2t.cu", "fwd_fp8.cu"]
HEADERS = ["attn_internal.cuh", "chunk_mask.h", "sm103_ptx.cuh", "bwd_passes.cuh", "debug_checks.h",
           os.path.join("..", "..", "include", "attn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def _stale(lib=LIB):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    build_dir = os.path.join(BUILD, "debug") if debug else BUILD
    os.makedirs(build_dir, exist_ok=True)
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                    "-I" + os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if debug:
        flags.append("-DATTN_DEBUG")
    procs = []
    objs = []
    for s in SOURCES:
        o = os.path.join(build_dir, s.replace(".cu", ".o"))
        objs.append(o)
        cmd = [nvcc()] + flags + ["-c", os.path.join(CSRC, s), "-o", o]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((s, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"), file=sys.stderr)
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))
