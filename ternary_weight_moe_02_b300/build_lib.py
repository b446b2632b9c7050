"""Build libmaple.so in-tree: every csrc/*.cu compiled for sm_103a with nvcc.

Usage: python -m ternary_weight_moe_02_b300.build_lib [--force] [--verbose]
Object files go to _build/ at the repository root; the shared library is written next
to this file so that the binding loads it from the package directory.
"""
from __future__ import annotations

import glob
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libmaple.so")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                 "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]
LDFLAGS = ARCH + ["-shared", "-cudart", "static", "-Xlinker", "--exclude-libs=ALL",
                  "-Xlinker", "-Bsymbolic"]


def _deps_hash(src: str, extra_flags) -> str:
    h = hashlib.sha256()
    h.update(" ".join(CFLAGS + list(extra_flags)).encode())
    for f in sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                    [os.path.join(INCLUDE, "maple.h"), src]):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    objs, changed = [], force or not os.path.exists(LIB)
    for src in sorted(glob.glob(os.path.join(CSRC, "*.cu"))):
        name = os.path.splitext(os.path.basename(src))[0]
        obj = os.path.join(BUILD, f"{name}.{_deps_hash(src, extra_flags)}.o")
        if force or not os.path.exists(obj):
            cmd = [NVCC] + CFLAGS + list(extra_flags) + (["-Xptxas", "-v"] if verbose else []) + \
                  ["-c", src, "-o", obj + ".tmp"]
            if verbose:
                print(" ".join(cmd), flush=True)
            subprocess.check_call(cmd)
            os.replace(obj + ".tmp", obj)
            changed = True
        objs.append(obj)
    # the objects a library was linked from: a source switched back to an earlier
    # version finds its (older) object cached, which a time comparison would miss
    manifest = LIB + ".objs"
    linked = ""
    if os.path.exists(manifest) and os.path.exists(LIB):
        with open(manifest) as fh:
            linked = fh.read()
    names = "\n".join(os.path.basename(o) for o in objs)
    if changed or linked != names:
        tmp = LIB + f".tmp{os.getpid()}"
        subprocess.check_call([NVCC] + LDFLAGS + objs + ["-o", tmp])
        os.replace(tmp, LIB)
        with open(manifest, "w") as fh:
            fh.write(names)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
