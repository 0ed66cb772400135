"""Build libtwell.so (the C-ABI library) in-tree for sm_103a with nvcc.

Every translation unit under ``csrc/`` is compiled in parallel and linked
into ``activation_sparse_gated_gate_gb300/libtwell.so``; the same sources
compiled with -DTWELL_BOUNDS_CHECK give ``libtwell_bounds.so``, the
bounds-checking build (every data-dependent gather and scatter index range
checked, TWELL_FLAG_BOUNDS instead of an out-of-range access), which the
tests load to run the parity cases under those checks.  Run as
``python -m activation_sparse_gated_gate_gb300.build`` or call ``build()``.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtwell.so")
BOUNDS_OUT_DIR = os.path.join(HERE, "_build_bounds")
BOUNDS_LIB = os.path.join(HERE, "libtwell_bounds.so")
VARIANTS = {"normal": (OUT_DIR, LIB, []),
            "bounds": (BOUNDS_OUT_DIR, BOUNDS_LIB, ["-DTWELL_BOUNDS_CHECK"])}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I" + os.path.join(os.path.dirname(HERE), "include")]


def _nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _compile(src, extra, out_dir=OUT_DIR):
    obj = os.path.join(out_dir, os.path.basename(src).replace(".cu", ".o"))
    cmd = [_nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, extra=(), variants=("normal", "bounds")) -> str:
    """Compile csrc/*.cu for each variant (all objects in one parallel pool)
    and link its library; returns the normal library's path."""
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = list(extra) + (["-Xptxas", "-v"] if verbose else [])
    jobs = []
    for v in variants:
        out_dir, _, defs = VARIANTS[v]
        os.makedirs(out_dir, exist_ok=True)
        jobs += [(v, src, extra + defs, out_dir) for src in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(16, len(jobs))) as ex:
        results = list(ex.map(lambda j: (j[0],) + _compile(j[1], j[2], j[3]), jobs))
    if verbose:
        for _, _, log in results:
            sys.stderr.write(log)
    for v in variants:
        lib_path = VARIANTS[v][1]
        objs = [o for vv, o, _ in results if vv == v]
        tmp = lib_path + ".tmp"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
