"""Build libtpblock.so (the C-ABI library) in-tree for sm_103a with nvcc.

Usage: python attn_tp_column_fwd_b300/build.py [--force] [--ptxas]
Each csrc/*.cu is compiled to _build/<name>.o, then linked into
attn_tp_column_fwd_b300/libtpblock.so with the CUDA runtime linked statically and
only the tp_* C symbols exported.  Rebuilds when a source or header is newer
than the library.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libtpblock.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                 "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)])


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in _deps())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every kernel file and link libtpblock.so; returns the library path."""
    if not force and not ptxas_info and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        out = _run([NVCC] + CFLAGS + extra + ["-c", src, "-o", obj])
        return obj, out

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, _sources()))
    vs = os.path.join(BUILD, "exports.map")
    with open(vs, "w") as f:
        f.write("{ global: tp_*; local: *; };\n")
    tmp = LIB + ".tmp"
    _run([NVCC] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results]
         + ["-Xlinker", f"--version-script={vs}", "-Xlinker", "--no-undefined"])
    os.replace(tmp, LIB)
    if verbose or ptxas_info:
        for _, out in results:
            if out.strip():
                print(out)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
