"""Build liblora.so in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel to an object file
under _build/, then linked into lora_serving_device_gb300/liblora.so.  The
CUDA runtime is linked statically; the driver is reached through the
runtime's entry-point query, so nothing else needs to be on the link line.

With debug=True the same sources are built with -DLORA_DEBUG into
_build_debug/ and liblora_debug.so: indices handed from one kernel to
another are checked on the device, and one outside its buffer sets
LORA_DEVERR_BOUNDS instead of being used.

    python -m lora_serving_device_gb300.build [--force] [--verbose] [--debug]
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "liblora.so")
BUILD_DEBUG = os.path.join(ROOT, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "liblora_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "-I", INCLUDE, "-I", CSRC]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    for c in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          debug: bool = False) -> str:
    """Compile (if stale) and return the path of liblora.so (liblora_debug.so
    with debug=True)."""
    nvcc = nvcc_path()
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = CFLAGS + (["-DLORA_DEBUG"] if debug else [])
    os.makedirs(build_dir, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    procs = []
    objs = []
    for src in srcs:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs):
            cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
            if ptxas_verbose:
                cmd[1:1] = ["-Xptxas", "-v"]
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_verbose or p.returncode):
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(f) for f in failed))
    if force or procs or _stale(lib, objs):
        tmp = lib + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
                ptxas_verbose="--ptxas" in sys.argv, debug="--debug" in sys.argv))
