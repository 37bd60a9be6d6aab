"""Build the library in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` is compiled to an object, in parallel, twice: once as is
(``libringattn.so``, the product) and once with ``-DRA_CHECKS=1``
(``libringattn_checked.so``, the bounds-checked build the tests also run; see
``csrc/checks.cuh``).  Each set is linked with the CUDA runtime linked
statically, so the libraries need only the driver at run time.  Usage:

    python -m ring_attention_fwd_gb300.build [--verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "libringattn.so")
OUT_CHECKED = os.path.join(PKG, "libringattn_checked.so")
BUILD_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          "--expt-relaxed-constexpr"]
VARIANTS = {"release": (OUT, []), "checked": (OUT_CHECKED, ["-DRA_CHECKS=1"])}


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libringattn.so")
    return exe


def _compile(job) -> str:
    src, variant, verbose = job
    odir = os.path.join(BUILD_DIR, variant)
    obj = os.path.join(odir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *CFLAGS, *VARIANTS[variant][1], "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src} ({variant}):\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(f"[{variant}] " + r.stdout + r.stderr)
    return obj


def _link(objs, out: str) -> None:
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)


def build(verbose: bool = False, variants=("release", "checked")) -> str:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    jobs = [(s, v, verbose) for v in variants for s in srcs]
    for v in variants:
        os.makedirs(os.path.join(BUILD_DIR, v), exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(16, len(jobs), (os.cpu_count() or 8))) as ex:
        objs = list(ex.map(_compile, jobs))
    for v in variants:
        _link([o for o, j in zip(objs, jobs) if j[1] == v], VARIANTS[v][0])
    return OUT


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv))
