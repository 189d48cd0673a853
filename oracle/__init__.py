"""CPU oracle for k^2-tree semiring SpMV -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library under test never imports
it and shares no code with it; the only module both sides use is the seeded
input generator package ``synth``.

Two independent layers, both written from "A GPU Engine for Sparse
Matrix-Vector Products on k^2-Tree-Compressed Graphs" (Tosoni & Mencagli):

* ``spmv_edges`` -- the definition of section 2.2, y_i = (+)_{j: A_ij=1} w (x) x_j,
  evaluated straight from the (deduplicated) edge list with numpy.  This is
  the pages' "CPU CSR oracle" of section 5.9, here as a COO scatter.
* ``OracleTree`` / ``OracleTree.spmv`` -- the tree of section 2.1 built by
  recursive subdivision, and the product computed by a recursive top-down
  descent in which every step down is a rank query (section 2.1), in plain C
  (``k2t_oracle.c``).

Semirings follow Table 1: 0 plus-times (fp64 accumulation here), 1 Boolean
(bit-packed: one uint32 word per vertex, up to 32 vectors), 2 tropical
(fp32 w + x, min in the IEEE total order with -0 < +0, empty min = +inf).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k2t_oracle.c")
_LIB = os.path.join(_HERE, "libk2t_oracle.so")

PLUS_TIMES, BOOLEAN, TROPICAL = 0, 1, 2
RIGHT, LEFT = 0, 1
_MAX_LEVELS = 64


def build() -> str:
    """Compile the C oracle with gcc (no vector contraction: -ffp-contract=off)."""
    if (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
                               "-ffp-contract=off", "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


class _Tree(ctypes.Structure):
    _fields_ = [("levels", ctypes.c_int32), ("n_k4", ctypes.c_int32),
                ("dim_bits", ctypes.c_int32), ("leaf_k4", ctypes.c_int32),
                ("nodes", ctypes.c_uint64 * _MAX_LEVELS),
                ("start", ctypes.c_uint64 * (_MAX_LEVELS + 1)),
                ("t_bits", ctypes.c_uint64), ("nwords", ctypes.c_uint64),
                ("bits", ctypes.c_void_p), ("cum", ctypes.c_void_p)]


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        lib.orc_build.argtypes = [P, P, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64,
                                  ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(_Tree)]
        lib.orc_build.restype = ctypes.c_int
        lib.orc_free.argtypes = [ctypes.POINTER(_Tree)]
        lib.orc_rank1.argtypes = [ctypes.POINTER(_Tree), ctypes.c_uint64]
        lib.orc_rank1.restype = ctypes.c_uint64
        lib.orc_child_pos.argtypes = [ctypes.POINTER(_Tree), ctypes.c_int, ctypes.c_uint64]
        lib.orc_child_pos.restype = ctypes.c_uint64
        lib.orc_spmv.argtypes = [ctypes.POINTER(_Tree), ctypes.c_uint64, ctypes.c_uint64,
                                 ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_uint32,
                                 P, P, P]
        lib.orc_spmv.restype = ctypes.c_uint64
        lib.orc_spmv_bands.argtypes = [ctypes.POINTER(_Tree), ctypes.c_uint64, ctypes.c_uint64,
                                       ctypes.c_int32, ctypes.c_int32, ctypes.c_float, ctypes.c_uint32,
                                       P, P, P, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
        lib.orc_spmv_bands.restype = ctypes.c_uint64
        lib.orc_decode.argtypes = [ctypes.POINTER(_Tree), P, P, ctypes.c_uint64]
        lib.orc_decode.restype = ctypes.c_uint64
        lib.orc_copy_bits.argtypes = [ctypes.POINTER(_Tree), P]
        lib.orc_rows_product.argtypes = [P, P, ctypes.c_uint64, ctypes.c_int32, ctypes.c_int32,
                                         ctypes.c_float, ctypes.c_uint32, P, P, ctypes.c_uint64,
                                         P, P]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data) if a.size else ctypes.c_void_p(0)


def _batch_shape(semiring: int, n: int, B: int):
    return (n,) if semiring == BOOLEAN else (n, B)


@dataclass
class OracleResult:
    y: np.ndarray            # float64 (plus-times), uint32 words (Boolean), float32 (tropical)
    scale: np.ndarray | None  # plus-times: sum_j |w * x_j| per output entry
    cells: int


class OracleTree:
    """k^2-tree of section 2.1 built by recursive subdivision (test oracle).
    n_k4: leading levels with k = 4; leaf_k = 4: 4x4 leaf bitmaps (section 5.6)."""

    def __init__(self, rows, cols, n_rows: int, n_cols: int, n_k4: int = 0, leaf_k: int = 2):
        lib = _load()
        if leaf_k not in (2, 4):
            raise ValueError("leaf_k must be 2 or 4")
        self.rows = np.ascontiguousarray(rows, dtype=np.uint32)
        self.cols = np.ascontiguousarray(cols, dtype=np.uint32)
        self.n_rows, self.n_cols = int(n_rows), int(n_cols)
        self._t = _Tree()
        rc = lib.orc_build(_ptr(self.rows), _ptr(self.cols), self.rows.size,
                           self.n_rows, self.n_cols, int(n_k4), int(leaf_k == 4), ctypes.byref(self._t))
        if rc != 0:
            raise ValueError("oracle build failed (%d)" % rc)

    def __del__(self):
        try:
            _load().orc_free(ctypes.byref(self._t))
        except Exception:
            pass

    # --- shape ---------------------------------------------------------
    @property
    def levels(self) -> int:
        return self._t.levels

    @property
    def n_k4(self) -> int:
        return self._t.n_k4

    @property
    def leaf_k(self) -> int:
        return 4 if self._t.leaf_k4 else 2

    @property
    def dim_bits(self) -> int:
        return self._t.dim_bits

    def level_nodes(self):
        return [int(self._t.nodes[d]) for d in range(self.levels)]

    def level_start(self):
        return [int(self._t.start[d]) for d in range(self.levels + 1)]

    @property
    def t_bits(self) -> int:
        return int(self._t.t_bits)

    def bits(self) -> np.ndarray:
        """The bitstring T followed by L as a uint8 array of 0/1, one per position."""
        w = np.zeros(int(self._t.nwords), dtype=np.uint64)
        _load().orc_copy_bits(ctypes.byref(self._t), _ptr(w))
        total = int(self._t.start[self.levels])
        b = np.unpackbits(w.view(np.uint8), bitorder="little")
        return b[:total].copy()

    def bitstring(self, level: int) -> str:
        s = self.level_start()
        b = self.bits()[s[level]:s[level + 1]]
        return "".join("1" if v else "0" for v in b)

    def rank1(self, p: int) -> int:
        return int(_load().orc_rank1(ctypes.byref(self._t), p))

    def child_pos(self, level: int, p: int) -> int:
        return int(_load().orc_child_pos(ctypes.byref(self._t), level, p))

    def decode(self):
        lib = _load()
        n = lib.orc_decode(ctypes.byref(self._t), None, None, 0)
        r = np.zeros(n, dtype=np.uint32)
        c = np.zeros(n, dtype=np.uint32)
        lib.orc_decode(ctypes.byref(self._t), _ptr(r), _ptr(c), n)
        return r, c

    # --- product -------------------------------------------------------
    def spmv(self, direction: int, semiring: int, x: np.ndarray, B: int = 1,
             w: float | None = None, threads: int = 1, band_level: int = -1) -> OracleResult:
        """Product by recursive rank-based descent (see module docstring).
        threads != 1: the descent shared among threads by row bands (right)
        or column bands (left) of the level-band_level subtrees (-1: picked
        from the thread count; threads 0: one per core); the result is the
        same, and ``threads_used`` records how many ran."""
        if w is None:
            w = 1.0
        n_in = self.n_cols if direction == RIGHT else self.n_rows
        n_out = self.n_rows if direction == RIGHT else self.n_cols
        if semiring == BOOLEAN:
            x = np.ascontiguousarray(x, dtype=np.uint32).reshape(n_in)
            y = np.zeros(n_out, dtype=np.uint32)
            scale = None
        elif semiring == PLUS_TIMES:
            x = np.ascontiguousarray(x, dtype=np.float32).reshape(n_in, B)
            y = np.zeros((n_out, B), dtype=np.float64)
            scale = np.zeros((n_out, B), dtype=np.float64)
        else:
            x = np.ascontiguousarray(x, dtype=np.float32).reshape(n_in, B)
            y = np.zeros((n_out, B), dtype=np.float32)
            scale = None
        sc = _ptr(scale) if scale is not None else None
        if threads == 1:
            cells = _load().orc_spmv(ctypes.byref(self._t), self.n_rows, self.n_cols, direction,
                                     semiring, ctypes.c_float(w), B, _ptr(x), _ptr(y), sc)
            self.threads_used = 1
        else:
            used = ctypes.c_int32(0)
            cells = _load().orc_spmv_bands(ctypes.byref(self._t), self.n_rows, self.n_cols, direction,
                                           semiring, ctypes.c_float(w), B, _ptr(x), _ptr(y), sc,
                                           int(band_level), int(threads), ctypes.byref(used))
            if cells == (1 << 64) - 1:
                raise MemoryError("oracle band descent ran out of memory")
            self.threads_used = int(used.value)
        return OracleResult(y, scale, int(cells))


# --- definition from the edge list (numpy) ------------------------------
def dedup_edges(rows, cols):
    """Distinct (row, col) pairs of a COO list, sorted by (row, col)."""
    r = np.asarray(rows, dtype=np.uint64)
    c = np.asarray(cols, dtype=np.uint64)
    key = np.unique((r << np.uint64(32)) | c)
    return (key >> np.uint64(32)).astype(np.uint32), (key & np.uint64(0xffffffff)).astype(np.uint32)


def _total_order_key(v: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    k = np.where(u & np.uint32(0x80000000), u ^ np.uint32(0x7fffffff), u)
    return k.astype(np.uint32).view(np.int32)


def spmv_edges(rows, cols, n_rows: int, n_cols: int, direction: int, semiring: int,
               x: np.ndarray, B: int = 1, w: float | None = None) -> OracleResult:
    """y = (+)_{edges} w (x) x by the definition (section 2.2), from the edge list."""
    if w is None:
        w = 1.0
    r, c = dedup_edges(rows, cols)
    src = c if direction == RIGHT else r
    dst = r if direction == RIGHT else c
    n_in = n_cols if direction == RIGHT else n_rows
    n_out = n_rows if direction == RIGHT else n_cols
    src = src.astype(np.int64)
    dst = dst.astype(np.int64)
    if semiring == BOOLEAN:
        mask = np.uint32(0xffffffff if B >= 32 else (1 << B) - 1)
        xw = np.ascontiguousarray(x, dtype=np.uint32).reshape(n_in) & mask
        y = np.zeros(n_out, dtype=np.uint32)
        np.bitwise_or.at(y, dst, xw[src])
        return OracleResult(y, None, int(src.size))
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(n_in, B)
    if semiring == PLUS_TIMES:
        y = np.zeros((n_out, B), dtype=np.float64)
        scale = np.zeros((n_out, B), dtype=np.float64)
        contrib = np.float64(w) * x[src].astype(np.float64)
        for k in range(B):
            y[:, k] = np.bincount(dst, weights=contrib[:, k], minlength=n_out)
            scale[:, k] = np.bincount(dst, weights=np.abs(contrib[:, k]), minlength=n_out)
        return OracleResult(y, scale, int(src.size))
    # tropical: fp32 w + x, min in the total order
    contrib = (np.float32(w) + x[src]).astype(np.float32)
    key = _total_order_key(contrib)
    ykey = np.full((n_out, B), _total_order_key(np.array([np.inf], np.float32))[0], dtype=np.int32)
    for k in range(B):
        np.minimum.at(ykey[:, k], dst, key[:, k])
    u = ykey.view(np.uint32)
    back = np.where(u & np.uint32(0x80000000), u ^ np.uint32(0x7fffffff), u).astype(np.uint32)
    return OracleResult(back.view(np.float32), None, int(src.size))


def rows_product(rows, cols, n_rows: int, n_cols: int, direction: int, semiring: int,
                 x: np.ndarray, sample: np.ndarray, B: int = 1,
                 w: float | None = None) -> OracleResult:
    """Definition of section 2.2 for the listed outputs only (one pass, in C).

    ``rows``/``cols`` must be free of duplicates.  Row s of the result is the
    output ``sample[s]``.
    """
    if w is None:
        w = 1.0
    lib = _load()
    rows = np.ascontiguousarray(rows, dtype=np.uint32)
    cols = np.ascontiguousarray(cols, dtype=np.uint32)
    n_out = n_rows if direction == RIGHT else n_cols
    sample = np.asarray(sample, dtype=np.int64)
    slot = np.full(n_out, -1, dtype=np.int64)
    slot[sample] = np.arange(sample.size, dtype=np.int64)
    ns = sample.size
    if semiring == BOOLEAN:
        x = np.ascontiguousarray(x, dtype=np.uint32)
        y = np.zeros(ns, dtype=np.uint32)
        scale = None
    elif semiring == PLUS_TIMES:
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.zeros((ns, B), dtype=np.float64)
        scale = np.zeros((ns, B), dtype=np.float64)
    else:
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.zeros((ns, B), dtype=np.float32)
        scale = None
    lib.orc_rows_product(_ptr(rows), _ptr(cols), rows.size, direction, semiring,
                         ctypes.c_float(w), B, _ptr(x), _ptr(slot), ns, _ptr(y),
                         _ptr(scale) if scale is not None else None)
    return OracleResult(y, scale, 0)


def plus_times_tolerance(scale: np.ndarray) -> np.ndarray:
    """|y - y_ref| <= 1e-5 * sum_j |A_ij x_j| + 1e-6 (the stated fp32 bound)."""
    return 1e-5 * scale + 1e-6


def msbfs(rows, cols, n: int, sources, direction: int, max_levels: int | None = None) -> np.ndarray:
    """Hop distances from each source by level-synchronous search to the fixed
    point (the multi-source search of section 5.8 of "A GPU Engine for Sparse
    Matrix-Vector Products on k^2-Tree-Compressed Graphs"): level k+1 holds the
    vertices reached in one step from level k and not reached before.  RIGHT:
    vertex i is reached from j when A_ij = 1; LEFT: j is reached from i.  The
    step is a scipy sparse matrix-vector product.  Returns int32 n x B, -1 for
    vertices never reached (within max_levels)."""
    import scipy.sparse as sp
    r, c = dedup_edges(rows, cols)
    A = sp.csr_matrix((np.ones(r.size, np.int32), (r.astype(np.int64), c.astype(np.int64))), shape=(n, n))
    M = A if direction == RIGHT else A.T.tocsr()
    sources = [int(s) for s in sources]
    dist = np.full((n, len(sources)), -1, np.int32)
    for b, s in enumerate(sources):
        dist[s, b] = 0
        frontier = np.zeros(n, bool)
        frontier[s] = True
        visited = frontier.copy()
        level = 0
        while max_levels is None or level < max_levels:
            level += 1
            nxt = (M @ frontier.astype(np.int32)) > 0
            nxt &= ~visited
            if not nxt.any():
                break
            dist[nxt, b] = level
            visited |= nxt
            frontier = nxt
    return dist


def bool_product(rows_a, cols_a, rows_b, cols_b, n: int, m: int, p: int):
    """Boolean product C = A B of an n x m and an m x p Boolean matrix given as
    edge lists: C_ij = OR_k (A_ik AND B_kj), the product of two trees the pages
    name as the extension of the level-synchronous traversal (section 7 of "A
    GPU Engine for Sparse Matrix-Vector Products on k^2-Tree-Compressed
    Graphs").  A scipy sparse integer product (path counts) thresholded at 1.
    Returns the distinct non-zeros (rows, cols) sorted by (row, col)."""
    import scipy.sparse as sp
    ra, ca = dedup_edges(rows_a, cols_a)
    rb, cb = dedup_edges(rows_b, cols_b)
    A = sp.csr_matrix((np.ones(ra.size, np.int64), (ra.astype(np.int64), ca.astype(np.int64))), shape=(n, m))
    B = sp.csr_matrix((np.ones(rb.size, np.int64), (rb.astype(np.int64), cb.astype(np.int64))), shape=(m, p))
    C = (A @ B).tocoo()
    keep = C.data > 0
    r = C.row[keep].astype(np.uint32)
    c = C.col[keep].astype(np.uint32)
    order = np.lexsort((c, r))
    return r[order], c[order]


def transitive_closure(rows, cols, n: int, max_iters: int = 64):
    """A+ = A or A^2 or A^3 ... of an n x n Boolean matrix (pairs joined by a
    path of one or more edges) by repeated squaring, C <- C or C C, until C
    stops growing (section 7 of the same pages: "by repeated squaring the
    transitive closure").  Returns (rows, cols, iterations): the distinct
    non-zeros sorted by (row, col) and the number of squarings performed,
    the last of which added nothing."""
    r, c = dedup_edges(rows, cols)
    it = 0
    while it < max_iters:
        it += 1
        pr, pc = bool_product(r, c, r, c, n, n, n)
        nr, nc = dedup_edges(np.concatenate([r, pr]), np.concatenate([c, pc]))
        if nr.size == r.size:
            break
        r, c = nr, nc
    order = np.lexsort((c, r))
    return r[order], c[order], it
