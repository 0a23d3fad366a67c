"""In-tree build of libmxg.so for sm_103a (nvcc only, no cmake).

Each ``csrc/*.cu`` compiles to ``_build/<name>.o`` in parallel; the objects link into
``mxfp8_mlp_gqa_gb300/libmxg.so``. A rebuild happens only when a source or header is
newer than its output. Usage: ``python -m mxfp8_mlp_gqa_gb300.build [--force] [--timeline]``.

``--timeline`` builds a separate, instrumented copy (``libmxg_tl.so`` from ``_build_tl/``,
compiled with ``-DMXG_TIMELINE``) whose decode-step kernels record per-warp device timestamps;
``mxfp8_mlp_gqa_gb300.timeline`` reads them. The production library never contains that code.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmxg.so")
BUILD_TL = os.path.join(PKG, "_build_tl")
LIB_TL = os.path.join(PKG, "libmxg_tl.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
    "-I" + INCLUDE, "-I" + CSRC,
]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required to build libmxg")
    return p


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _newer(srcs, out) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


def _compile(src: str, extra, bdir: str = BUILD) -> str:
    obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
    if _newer([src] + _headers(), obj):
        cmd = [nvcc()] + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False, extra=(), timeline: bool = False) -> str:
    bdir, out = (BUILD_TL, LIB_TL) if timeline else (BUILD, LIB)
    extra = list(extra) + (["-DMXG_TIMELINE"] if timeline else [])
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    if force:
        for o in glob.glob(os.path.join(bdir, "*.o")):
            os.remove(o)
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, bdir), srcs))
    if force or _newer(objs, out):
        tmp = out + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, out)
    if verbose:
        print(out)
    return out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, timeline="--timeline" in sys.argv)
