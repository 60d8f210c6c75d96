"""Build libsanta.so in-tree: every csrc/*.cu compiled for sm_103a in parallel, then linked.

    python -m sampled_sparse_decode_gb300.build [--force]
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsanta.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-Xptxas", "-v",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsanta.so")


def _inputs():
    return (sorted(glob.glob(os.path.join(CSRC, "*.cu"))),
            sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                   glob.glob(os.path.join(INCLUDE, "*.h"))))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    srcs, hdrs = _inputs()
    return any(os.path.getmtime(f) > t for f in srcs + hdrs + [os.path.abspath(__file__)])


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libsanta.so if any source is newer than it; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    srcs, _ = _inputs()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + ".o")
        r = subprocess.run([cc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr[-6000:]}")
        return obj, r.stderr

    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(compile_one, srcs))
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as log:
        for (obj, err) in results:
            log.write(f"== {os.path.basename(obj)}\n{err}\n")
    if verbose:
        print(open(os.path.join(BUILD_DIR, "ptxas.log")).read())
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp,
                        *[o for o, _ in results]], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of libsanta.so failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
