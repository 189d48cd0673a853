"""Build of the in-tree shared library ``libk2t.so`` (sm_103a, CUDA 13).

Every translation unit compiles in parallel with nvcc (one -gencode, no
cmake), then nvcc links them into one shared object next to this file.
The library links the CUDA runtime dynamically so it shares the runtime
(and the primary context) of the PyTorch process that loads it.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libk2t.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-O3", "-I" + os.path.join(ROOT, "include")]
SOURCES = ["k2t_host.cpp", "k2t_device.cu", "k2t_sr_plus_times.cu", "k2t_sr_boolean.cu", "k2t_sr_min_plus.cu",
           "k2t_static.cu", "k2t_probe.cu", "k2t_product.cu"]
HEADERS = ["k2t_internal.h", "k2t_kernels.cuh", os.path.join("..", "..", "include", "k2t.h")]


def _newest_input() -> float:
    paths = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [__file__]
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, extra) -> str:
    obj = os.path.join(BUILD, src + ".o")
    cmd = [NVCC] + COMMON + ARCH + list(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd = [NVCC, "-x", "c++"] + COMMON + ["-Xcompiler", "-pthread", "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("compile failed: %s\n%s\n%s" % (" ".join(cmd), r.stdout, r.stderr))
    return obj


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile libk2t.so if any source is newer than it; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [NVCC, "-shared"] + ARCH + ["-cudart", "shared", "-o", tmp] + objs + \
        ["-Xlinker", "-rpath,/usr/local/cuda/lib64", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed: %s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    if verbose:
        print("built", LIB, file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
