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
CHECKED_LIB = os.path.join(HERE, "libk2t_checked.so")   # same ABI, kernels with bounds tests (K2T_CHECKED)
PROBE_LIB = os.path.join(HERE, "libk2t_probe.so")   # benchmark instrumentation, not the product ABI
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# hidden visibility: only the K2T_API calls of include/k2t.h are exported
COMMON = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-O3,-fvisibility=hidden",
          "-I" + os.path.join(ROOT, "include")]
SOURCES = ["k2t_host.cpp", "k2t_device.cu", "k2t_sr_plus_times.cu", "k2t_sr_boolean.cu", "k2t_sr_min_plus.cu",
           "k2t_static.cu", "k2t_product.cu"]
PROBE_SOURCES = [os.path.join("probe", "k2t_probe.cu")]
HEADERS = ["k2t_internal.h", "k2t_kernels.cuh", os.path.join("..", "..", "include", "k2t.h")]


def _newest_input(sources) -> float:
    paths = [os.path.join(CSRC, s) for s in list(sources) + HEADERS] + [__file__]
    return max(os.path.getmtime(p) for p in paths)


def _compile(src: str, extra, tag: str) -> str:
    obj = os.path.join(BUILD, tag, src.replace(os.sep, "_") + ".o")
    cmd = [NVCC] + COMMON + ARCH + list(extra) + ["-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd = [NVCC, "-x", "c++"] + COMMON + list(extra) + ["-Xcompiler", "-pthread", "-c", os.path.join(CSRC, src),
                                                           "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("compile failed: %s\n%s\n%s" % (" ".join(cmd), r.stdout, r.stderr))
    return obj


def _link(objs, out: str) -> None:
    tmp = out + ".tmp%d" % os.getpid()
    cmd = [NVCC, "-shared"] + ARCH + ["-cudart", "shared", "-o", tmp] + objs + \
        ["-Xlinker", "-rpath,/usr/local/cuda/lib64", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed: %s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, out)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile the product library libk2t.so, its bounds-checked twin
    libk2t_checked.so (-DK2T_CHECKED: the same ABI, kernels that test their
    indexes and report a failure in the device status word) and the
    benchmark's probe library libk2t_probe.so where a source is newer than
    the library (all translation units in parallel); return the product
    library's path."""
    targets = [(LIB, SOURCES, list(extra), "lib"), (CHECKED_LIB, SOURCES, list(extra) + ["-DK2T_CHECKED"], "checked"),
               (PROBE_LIB, PROBE_SOURCES, [], "probe")]
    todo = [t for t in targets
            if force or not os.path.exists(t[0]) or os.path.getmtime(t[0]) < _newest_input(t[1])]
    if not todo:
        return LIB
    jobs = []
    for out, srcs, flags, tag in todo:
        os.makedirs(os.path.join(BUILD, tag), exist_ok=True)
        jobs += [(src, flags, tag) for src in srcs]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(*j), jobs))
    k = 0
    for out, srcs, flags, tag in todo:
        _link(objs[k:k + len(srcs)], out)
        k += len(srcs)
        if verbose:
            print("built", out, file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
