"""Builds libfo.so in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in its own nvcc process (in parallel), then
linked into one shared library.  The CUDA runtime is linked statically; driver
entry points are resolved at run time, so the library loads on hosts without
a GPU driver (symbols can be inspected there; compute needs a GB300).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfo.so")
SOURCES = ["fo_api.cu", "fo_gemm.cu", "fo_gemm2.cu", "fo_attn.cu", "fo_elem.cu", "fo_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, verbose: bool, build_dir: str = BUILD, extra=()) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose:
        sys.stderr.write(res.stderr)
    return obj


def build(verbose: bool = False, debug_bounds: bool = False, out: str = LIB) -> str:
    """Builds the library into `out` (default: the package's libfo.so, which the binding
    loads).  debug_bounds: the kernels check their tile coordinates, operand maps and
    flag indices and record FO_ERR_INTERNAL instead of making an out-of-range access."""
    build_dir = BUILD + ("_debug" if debug_bounds else "")
    extra = ("-DFO_DEBUG_BOUNDS",) if debug_bounds else ()
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, build_dir, extra), SOURCES))
    tmp = out + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
