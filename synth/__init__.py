"""Seeded synthetic inputs for k^2-tree SpMV: graphs (COO) and dense vectors.

This package is the only code that both the library's tests/benchmark and
the CPU oracle consume.  It contains no part of the product's arithmetic.
Graph generators are native (``synth.cpp``, counter-based randomness, the
same output for any thread count); dense vectors come from numpy's PCG64.

The five workloads stand in for the datasets of "A GPU Engine for Sparse
Matrix-Vector Products on k^2-Tree-Compressed Graphs" (Wikidata relations,
the Software Heritage subgraph and the LAW web and social graphs of its
Table 2), which are not available here; each keeps the shape, degree
distribution and vector distribution its description states.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.cpp")
_LIB = os.path.join(_HERE, "libk2t_synth.so")
_lib = None


def build() -> str:
    if (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["g++", "-O3", "-std=c++17", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.synth_edges_size.argtypes = [P]
        lib.synth_edges_size.restype = ctypes.c_uint64
        lib.synth_edges_copy.argtypes = [P, P, P]
        lib.synth_edges_free.argtypes = [P]
        lib.synth_rmat.argtypes = [ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                   ctypes.c_uint64, ctypes.c_uint64, ctypes.c_int]
        lib.synth_rmat.restype = P
        lib.synth_weblike.argtypes = [ctypes.c_uint64, ctypes.c_double, ctypes.c_double,
                                      ctypes.c_int64, ctypes.c_uint64]
        lib.synth_weblike.restype = P
        lib.synth_permute_bfs.argtypes = [ctypes.c_uint64, P, P, ctypes.c_uint64, ctypes.c_uint64]
        _lib = lib
    return _lib


def _take(h):
    lib = _load()
    if not h:
        raise ValueError("generator rejected its arguments")
    try:
        n = int(lib.synth_edges_size(h))
        rows = np.empty(n, dtype=np.uint32)
        cols = np.empty(n, dtype=np.uint32)
        if n:
            lib.synth_edges_copy(h, rows.ctypes.data, cols.ctypes.data)
        return rows, cols
    finally:
        lib.synth_edges_free(h)


def rmat(scale: int, a: float, b: float, c: float, target: int, seed: int,
         symmetric: bool = False):
    """R-MAT edges: distinct, no self-loops, sorted by (row, col)."""
    return _take(_load().synth_rmat(scale, a, b, c, target, seed, int(symmetric)))


def weblike(n: int, lam: float = 14.0, local_frac: float = 0.8, window: int = 256, seed: int = 2):
    """Poisson(lam) out-degrees; targets near the source w.p. local_frac."""
    return _take(_load().synth_weblike(n, lam, local_frac, window, seed))


def permute_bfs(n: int, rows: np.ndarray, cols: np.ndarray, seed: int):
    """Random relabelling followed by BFS order (in place)."""
    assert rows.dtype == np.uint32 and cols.dtype == np.uint32
    _load().synth_permute_bfs(n, rows.ctypes.data, cols.ctypes.data, rows.size, seed)
    return rows, cols


def uniform(n: int, nnz: int, seed: int):
    """nnz distinct (row, col) pairs, uniform over n x n without replacement."""
    rng = np.random.default_rng(seed)
    idx = rng.choice(n * n, size=nnz, replace=False)
    return (idx // n).astype(np.uint32), (idx % n).astype(np.uint32), rng


# --- workloads -------------------------------------------------------------
PLUS_TIMES, BOOLEAN, TROPICAL = 0, 1, 2


@dataclass
class Workload:
    name: str
    rows: np.ndarray
    cols: np.ndarray
    n_rows: int
    n_cols: int
    semiring: int
    B: int
    w: float
    n_k4: int = 0                 # leading k = 4 levels
    cache_last_internal: bool = False
    xs: dict = field(default_factory=dict)   # direction -> input vector(s)
    extra: dict = field(default_factory=dict)

    @property
    def nnz(self) -> int:
        return int(self.rows.size)


def _fp32_uniform(rng, shape, lo, hi):
    return rng.uniform(lo, hi, size=shape).astype(np.float32)


def uniform_c1(seed: int = 0) -> Workload:
    """Tiny uniform matrix: n = 1024, 8192 distinct cells, x ~ U(-1, 1), B = 1."""
    n = 1024
    r, c, rng = uniform(n, 8192, seed)
    x_right = _fp32_uniform(rng, (n, 1), -1.0, 1.0)
    x_left = _fp32_uniform(rng, (n, 1), -1.0, 1.0)
    return Workload("uniform-n1024-m8192", r, c, n, n, PLUS_TIMES, 1, 1.0,
                    xs={0: x_right, 1: x_left})


def uniform_large(log_n: int = 20, edges_per_vertex: int = 16, seed: int = 5) -> Workload:
    """Uniform random matrix of the R-MAT workload's size (no hub rows): a
    control for contention effects.  Drawn as R-MAT with equal quadrants."""
    n = 1 << log_n
    r, c = rmat(log_n, 0.25, 0.25, 0.25, edges_per_vertex * n, seed)
    rng = np.random.default_rng(seed)
    xs = {d: rng.uniform(0.0, 1.0, size=(n, 1)).astype(np.float32) for d in (0, 1)}
    return Workload("uniform%d-m%d" % (log_n, edges_per_vertex * n), r, c, n, n, PLUS_TIMES, 1, 1.0, xs=xs)


def rmat_c2(scale: int = 20, edges_per_vertex: int = 16, seed: int = 1) -> Workload:
    """Power-law R-MAT (.57,.19,.19,.05), 16 edges per vertex, x ~ U(0,1)/sum."""
    n = 1 << scale
    r, c = rmat(scale, 0.57, 0.19, 0.19, edges_per_vertex * n, seed)
    rng = np.random.default_rng(seed)
    xs = {}
    for d in (0, 1):
        x = rng.uniform(0.0, 1.0, size=(n, 1))
        xs[d] = (x / x.sum()).astype(np.float32)
    return Workload("rmat%d-pagerank" % scale, r, c, n, n, PLUS_TIMES, 1, 1.0, xs=xs)


def weblike_c3(log_n: int = 22, B: int = 32, seed: int = 2, n_k4: int = 2) -> Workload:
    """Web-like locality graph; 32 bit-packed Boolean frontiers with 1% set."""
    n = 1 << log_n
    r, c = weblike(n, 14.0, 0.8, 256, seed)
    rng = np.random.default_rng(seed)
    k = int(round(0.01 * n))
    xs = {}
    for d in (0, 1):
        words = np.zeros(n, dtype=np.uint32)
        for b in range(B):
            idx = rng.choice(n, size=k, replace=False)
            words[idx] |= np.uint32(1 << b)
        xs[d] = words
    return Workload("weblike%d-bool-B%d" % (log_n, B), r, c, n, n, BOOLEAN, B, 1.0,
                    n_k4=n_k4, xs=xs)


def social_c4(scale: int = 24, edges_per_vertex: int = 16, B: int = 8, seed: int = 3,
              w: float = 0.0) -> Workload:
    """Symmetric R-MAT (.45,.15,.15,.25); tropical; x ~ U(0,100), 90% +inf."""
    n = 1 << scale
    r, c = rmat(scale, 0.45, 0.15, 0.15, edges_per_vertex * n, seed, symmetric=True)
    rng = np.random.default_rng(seed)
    xs = {}
    for d in (0, 1):
        x = _fp32_uniform(rng, (n, B), 0.0, 100.0)
        inf_mask = rng.random(size=(n, B)) < 0.9
        x[inf_mask] = np.inf
        xs[d] = x
    return Workload("social-rmat%d-tropical-B%d" % (scale, B), r, c, n, n, TROPICAL, B, w, xs=xs)


def large_c5(scale: int = 27, edges: int = 1_200_000_000, B: int = 1, seed: int = 4) -> Workload:
    """R-MAT (.57,.19,.19,.05), ids permuted then BFS-ordered; cached last level.
    x ~ U(0,1) fp32; the square matrix uses one x for both directions."""
    n = 1 << scale
    r, c = rmat(scale, 0.57, 0.19, 0.19, edges, seed)
    permute_bfs(n, r, c, seed)
    rng = np.random.default_rng(seed)
    x = rng.random(size=(n, B), dtype=np.float32)
    return Workload("rmat%d-bfs-%dM" % (scale, edges // 1_000_000), r, c, n, n, PLUS_TIMES, B, 1.0,
                    cache_last_internal=True, xs={0: x, 1: x})


def clustered(scale: int = 22, block: int = 16, per_row: int = 8, seed: int = 6):
    """A clustered graph: every row i draws per_row distinct columns inside its
    own block-aligned window [i - i % block, i - i % block + block), so the
    matrix is block diagonal with blocks per_row/block full.  Dense leaves
    (several non-zeros per 2x2 or 4x4 block), as on locality-ordered crawls.
    x ~ U(0,1) fp32, plus-times, right and left, B = 1."""
    n = 1 << scale
    rng = np.random.default_rng(seed)
    rows = np.repeat(np.arange(n, dtype=np.uint32), per_row)
    offs = np.argsort(rng.random((n, block)), axis=1)[:, :per_row].astype(np.uint32).reshape(-1)
    cols = (rows - rows % block) + offs
    x = rng.random(size=(n, 1), dtype=np.float32)
    return Workload("clustered%d-b%d-d%d" % (scale, block, per_row), rows, cols, n, n, PLUS_TIMES, 1, 1.0,
                    cache_last_internal=True, xs={0: x, 1: x})


def random_small(seed: int, n_rows: int, n_cols: int, density: float):
    """Small random Boolean matrix (with repeated coordinates) for exhaustive checks."""
    rng = np.random.default_rng(seed)
    m = int(density * n_rows * n_cols) + 1
    rows = rng.integers(0, n_rows, size=m, dtype=np.uint32)
    cols = rng.integers(0, n_cols, size=m, dtype=np.uint32)
    return rows, cols, rng
