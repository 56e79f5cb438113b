"""Build libfattn.so in-tree (tiled_online_softmax_fwd_gb300/_build/) with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
into one shared library with the CUDA runtime linked statically and only the
C-ABI symbols exported.

    python -m tiled_online_softmax_fwd_gb300.build [--verbose] [--force]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libfattn.so")

SOURCES = ["fattn_api.cu", "fattn_fwd_sm103.cu", "fattn_bwd_sm103.cu", "fattn_fwd_simt.cu",
           "fattn_rowops.cu"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
EXPORTS = "{ global: attn_fwd*; attn_bwd*; fattn_*; local: *; };\n"


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found (CUDA 13 toolkit required)")
    return path


def _inputs_newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(INCLUDE, "fattn.h")]


def _compile(src: str, verbose: bool, force: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    deps = [os.path.join(CSRC, src)] + _headers()
    if not force and not _inputs_newer(obj, deps):
        return obj
    cmd = [nvcc(), *GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj + ".tmp"]
    if verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, res.stdout, res.stderr))
    if verbose and (res.stdout or res.stderr):
        sys.stderr.write(res.stdout + res.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile and link libfattn.so; returns its path.  Rebuilds only what changed."""
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, force), SOURCES))
    if force or _inputs_newer(LIB, objs):
        vmap = os.path.join(BUILD, "exports.map")
        with open(vmap, "w") as f:
            f.write(EXPORTS)
        cmd = [nvcc(), *GENCODE, "-shared", "-cudart", "static", "-o", LIB + ".tmp", *objs,
               "-Xlinker", "--version-script=" + vmap]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n%s%s" % (res.stdout, res.stderr))
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true", help="print ptxas register/smem usage")
    ap.add_argument("--force", action="store_true")
    a = ap.parse_args()
    print(build(verbose=a.verbose, force=a.force))
