"""ctypes binding of ``libk2t.so`` (``include/k2t.h``): argument marshalling only.

Every step of a product runs in the library's CUDA kernels; this module
only converts numpy arrays, torch tensors and streams into the pointers and
sizes the C ABI takes.  If the shared library is missing, every call fails
loudly: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libk2t.so")
CHECKED_LIB_PATH = os.path.join(_HERE, "libk2t_checked.so")   # same ABI, bounds-tested kernels
PROBE_LIB_PATH = os.path.join(_HERE, "libk2t_probe.so")   # benchmark instrumentation

RIGHT, LEFT = 0, 1
PLUS_TIMES, BOOLEAN, MIN_PLUS = 0, 1, 2
ENGINE_AUTO, ENGINE_FUSED, ENGINE_LEVELSYNC, ENGINE_CACHED, ENGINE_BANDED = 0, 1, 2, 3, 4
OFFSETS_DIRECTORY, OFFSETS_SCAN = 0, 1
MAX_LEVELS = 33
MAX_BATCH = 32

STATUS = {0: "K2T_OK", -1: "K2T_EINVAL", -2: "K2T_ERANGE", -3: "K2T_ENOMEM",
          -4: "K2T_ECUDA", -5: "K2T_ESTATE", -6: "K2T_EDEVICE", -7: "K2T_ETIMEOUT"}
STATUS_WAIT_TIMEOUT, STATUS_OUT_OF_RANGE = 1, 2

EXPORTED = ["k2t_default_opts", "k2t_build", "k2t_workspace_bytes", "k2t_upload", "k2t_spmv",
            "k2t_spmv_marked",
            "k2t_spmv_host", "k2t_stats_get", "k2t_level_signatures", "k2t_device_level",
            "k2t_decode", "k2t_free", "k2t_strerror", "k2t_last_cuda_error",
            "k2t_spmv_noalloc", "k2t_noalloc_scratch_limit", "k2t_msbfs",
            "k2t_msbfs_work_bytes", "k2t_bool_product", "k2t_bool_closure", "k2t_status"]


class Opts(ctypes.Structure):
    _fields_ = [("n_k4_levels", ctypes.c_uint32), ("cache_last_internal", ctypes.c_uint32),
                ("engine", ctypes.c_uint32), ("offsets", ctypes.c_uint32),
                ("host_top_max_nodes", ctypes.c_uint32), ("chunk_cap", ctypes.c_uint32),
                ("tile_m", ctypes.c_uint64), ("max_batch", ctypes.c_uint32),
                ("host_vectors", ctypes.c_uint32), ("use_graph", ctypes.c_uint32),
                ("threads", ctypes.c_uint32), ("band_rows", ctypes.c_uint32),
                ("band_cols", ctypes.c_uint32), ("heavy_terms", ctypes.c_uint32),
                ("heavy_mode", ctypes.c_uint32), ("leaf_k", ctypes.c_uint32),
                ("reserved", ctypes.c_uint32 * 3)]


class Stats(ctypes.Structure):
    _fields_ = [("n_rows", ctypes.c_uint64), ("n_cols", ctypes.c_uint64), ("nnz", ctypes.c_uint64),
                ("levels", ctypes.c_uint32), ("n_k4_levels", ctypes.c_uint32),
                ("dim_bits", ctypes.c_uint32), ("d0", ctypes.c_uint32),
                ("level_nodes", ctypes.c_uint64 * MAX_LEVELS), ("tree_bits", ctypes.c_uint64),
                ("t_bytes_device", ctypes.c_uint64), ("l_bytes_device", ctypes.c_uint64),
                ("dir_bytes", ctypes.c_uint64), ("top_bytes", ctypes.c_uint64),
                ("cached_bytes", ctypes.c_uint64), ("plan_bytes", ctypes.c_uint64),
                ("scratch_bytes", ctypes.c_uint64), ("vector_bytes", ctypes.c_uint64),
                ("workspace_bytes", ctypes.c_uint64), ("n_chunks", ctypes.c_uint64),
                ("n_steps", ctypes.c_uint64), ("engine", ctypes.c_uint32), ("offsets", ctypes.c_uint32),
                ("uploaded", ctypes.c_uint32), ("heavy_rows", ctypes.c_uint32),
                ("heavy_cols", ctypes.c_uint32), ("heavy_kib", ctypes.c_uint32),
                ("leaf_k", ctypes.c_uint32), ("heavy_fp64", ctypes.c_uint32 * 2),
                ("heavy_max_terms", ctypes.c_uint32 * 2), ("pad", ctypes.c_uint32),
                ("heavy_partials", ctypes.c_uint64 * 2)]


class K2TError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda: int = 0):
        msg = "%s failed: %s" % (fn, STATUS.get(status, str(status)))
        if cuda:
            msg += " (cuda error %d)" % cuda
        super().__init__(msg)
        self.status = status


_lib = None


def load() -> ctypes.CDLL:
    """Load the in-tree library; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libk2t.so is missing: run __graft_entry__.build() first "
                               "(there is no fallback implementation)")
        lib = ctypes.CDLL(LIB_PATH)
        P, U32, U64, I32 = ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32
        lib.k2t_default_opts.argtypes = [ctypes.POINTER(Opts)]
        lib.k2t_default_opts.restype = None
        lib.k2t_build.argtypes = [P, P, U64, U64, U64, ctypes.POINTER(Opts), ctypes.POINTER(P)]
        lib.k2t_workspace_bytes.argtypes = [P, ctypes.POINTER(U64)]
        lib.k2t_upload.argtypes = [P, P, U64, P]
        lib.k2t_spmv.argtypes = [P, I32, I32, ctypes.c_float, P, P, U32, P]
        lib.k2t_spmv_marked.argtypes = [P, I32, I32, ctypes.c_float, P, P, U32, P, P]
        lib.k2t_spmv_noalloc.argtypes = [P, I32, I32, ctypes.c_float, P, P, U32, P]
        lib.k2t_spmv_noalloc.restype = ctypes.c_int
        lib.k2t_noalloc_scratch_limit.argtypes = []
        lib.k2t_noalloc_scratch_limit.restype = U64
        lib.k2t_msbfs.argtypes = [P, I32, P, U32, P, P, U32, ctypes.POINTER(U32), P]
        lib.k2t_msbfs.restype = ctypes.c_int
        lib.k2t_msbfs_work_bytes.argtypes = [P]
        lib.k2t_msbfs_work_bytes.restype = U64
        lib.k2t_bool_product.argtypes = [P, P, ctypes.POINTER(Opts), ctypes.POINTER(P), P]
        lib.k2t_bool_product.restype = ctypes.c_int
        lib.k2t_bool_closure.argtypes = [P, ctypes.POINTER(Opts), U32, ctypes.POINTER(P), ctypes.POINTER(U32), P]
        lib.k2t_bool_closure.restype = ctypes.c_int
        lib.k2t_status.argtypes = [P, ctypes.POINTER(U32), I32, P]
        lib.k2t_status.restype = ctypes.c_int
        lib.k2t_spmv_host.argtypes = [P, I32, I32, ctypes.c_float, P, P, U32, P]
        lib.k2t_stats_get.argtypes = [P, ctypes.POINTER(Stats)]
        lib.k2t_level_signatures.argtypes = [P, U32, P, U64, ctypes.POINTER(U64)]
        lib.k2t_device_level.argtypes = [P, U32, ctypes.POINTER(P), ctypes.POINTER(P)]
        lib.k2t_decode.argtypes = [P, P, P, U64, ctypes.POINTER(U64)]
        lib.k2t_free.argtypes = [P]
        lib.k2t_free.restype = None
        lib.k2t_strerror.argtypes = [ctypes.c_int]
        lib.k2t_strerror.restype = ctypes.c_char_p
        lib.k2t_last_cuda_error.argtypes = []
        for name in ("k2t_build", "k2t_workspace_bytes", "k2t_upload", "k2t_spmv", "k2t_spmv_marked",
                     "k2t_spmv_host",
                     "k2t_stats_get", "k2t_level_signatures", "k2t_device_level", "k2t_decode",
                     "k2t_last_cuda_error"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise K2TError(fn, status, load().k2t_last_cuda_error())


def default_opts(**kw) -> Opts:
    o = Opts()
    load().k2t_default_opts(ctypes.byref(o))
    for k, v in kw.items():
        if not hasattr(o, k):
            raise AttributeError("k2t_opts has no field %r" % k)
        setattr(o, k, v)
    return o


def _stream_ptr(stream) -> int | None:
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:
            return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dev_ptr(t) -> int:
    if hasattr(t, "data_ptr"):
        if not t.is_cuda:
            raise ValueError("expected a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError("expected a contiguous tensor")
        return t.data_ptr()
    return int(t)


class Tree:
    """A built k^2-tree: ``build`` on the host, ``upload``, then ``spmv``."""

    def __init__(self, rows, cols, n_rows: int, n_cols: int, opts: Opts | None = None, **kw):
        lib = load()
        rows = np.ascontiguousarray(rows, dtype=np.uint32)
        cols = np.ascontiguousarray(cols, dtype=np.uint32)
        if rows.shape != cols.shape:
            raise ValueError("rows and cols differ in length")
        if opts is None:
            opts = default_opts(**kw)
        self.opts = opts
        self.n_rows, self.n_cols = int(n_rows), int(n_cols)
        h = ctypes.c_void_p()
        rp = rows.ctypes.data if rows.size else None
        cp = cols.ctypes.data if cols.size else None
        _check("k2t_build", lib.k2t_build(rp, cp, rows.size, self.n_rows, self.n_cols,
                                          ctypes.byref(opts), ctypes.byref(h)))
        self._h = h
        self._arena = None

    def close(self):
        if getattr(self, "_h", None):
            load().k2t_free(self._h)
            self._h = None
        self._arena = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def workspace_bytes(self) -> int:
        v = ctypes.c_uint64()
        _check("k2t_workspace_bytes", load().k2t_workspace_bytes(self._h, ctypes.byref(v)))
        return int(v.value)

    def stats(self) -> Stats:
        s = Stats()
        _check("k2t_stats_get", load().k2t_stats_get(self._h, ctypes.byref(s)))
        return s

    def upload(self, arena=None, stream=None):
        """Copy the device image into ``arena`` (a CUDA uint8 tensor of at least
        workspace_bytes) or into library-owned memory when arena is None."""
        if arena is None:
            _check("k2t_upload", load().k2t_upload(self._h, None, 0, _stream_ptr(stream)))
        else:
            nbytes = arena.numel() * arena.element_size()
            _check("k2t_upload", load().k2t_upload(self._h, _dev_ptr(arena), nbytes, _stream_ptr(stream)))
            self._arena = arena  # keep the memory alive with the tree
        return self

    def spmv(self, direction: int, semiring: int, x, y, B: int = 1, w: float = 1.0, stream=None):
        """Queue y = A x (RIGHT) or y^T = x^T A (LEFT) on device tensors."""
        _check("k2t_spmv", load().k2t_spmv(self._h, direction, semiring, ctypes.c_float(w),
                                           _dev_ptr(x), _dev_ptr(y), B, _stream_ptr(stream)))
        return y

    def spmv_marked(self, direction: int, semiring: int, x, y, B: int, w: float, stream, event_after_fill):
        """spmv that records a cudaEvent_t (handle as int) after the fill kernel."""
        _check("k2t_spmv_marked", load().k2t_spmv_marked(self._h, direction, semiring, ctypes.c_float(w),
                                                         _dev_ptr(x), _dev_ptr(y), B, _stream_ptr(stream),
                                                         event_after_fill))
        return y

    def spmv_noalloc(self, direction: int, semiring: int, x, y, B: int = 1, w: float = 1.0, stream=None):
        """Level-synchronous product with scratch in the library's static device
        array (no allocation); see k2t_spmv_noalloc in include/k2t.h."""
        _check("k2t_spmv_noalloc", load().k2t_spmv_noalloc(self._h, direction, semiring, ctypes.c_float(w),
                                                           _dev_ptr(x), _dev_ptr(y), B, _stream_ptr(stream)))
        return y

    def status(self, clear: bool = False, stream=None) -> int:
        """The tree's device status word (k2t_status): waits for the stream,
        returns the word and, with clear, resets it."""
        w = ctypes.c_uint32()
        _check("k2t_status", load().k2t_status(self._h, ctypes.byref(w), int(bool(clear)), _stream_ptr(stream)))
        return int(w.value)

    def msbfs(self, direction: int, sources, dist, work, max_levels: int = 1 << 30, stream=None) -> int:
        """Multi-source BFS (k2t_msbfs): dist (CUDA int32, n x B) and work (CUDA
        buffer of msbfs_work_bytes()) are the caller's; returns the levels run."""
        src = np.ascontiguousarray(sources, dtype=np.uint32)
        lv = ctypes.c_uint32()
        _check("k2t_msbfs", load().k2t_msbfs(self._h, direction, src.ctypes.data, src.size, _dev_ptr(dist),
                                             _dev_ptr(work), max_levels, ctypes.byref(lv), _stream_ptr(stream)))
        return int(lv.value)

    @classmethod
    def _adopt(cls, handle, n_rows: int, n_cols: int, opts: Opts) -> "Tree":
        t = cls.__new__(cls)
        t.opts = opts
        t.n_rows, t.n_cols = int(n_rows), int(n_cols)
        t._h = handle
        t._arena = None
        return t

    def bool_product(self, other: "Tree", stream=None, opts: Opts | None = None, **kw) -> "Tree":
        """Boolean C = self * other through k2t_bool_product; C is a new host
        tree built with ``opts`` (or the given option keywords)."""
        if opts is None:
            opts = default_opts(**kw)
        h = ctypes.c_void_p()
        _check("k2t_bool_product", load().k2t_bool_product(self._h, other._h, ctypes.byref(opts), ctypes.byref(h),
                                                           _stream_ptr(stream)))
        return Tree._adopt(h, self.n_rows, other.n_cols, opts)

    def bool_closure(self, max_iters: int = 64, stream=None, opts: Opts | None = None, **kw):
        """Transitive closure by repeated squaring (k2t_bool_closure); returns
        (tree, squarings run)."""
        if opts is None:
            opts = default_opts(**kw)
        h = ctypes.c_void_p()
        it = ctypes.c_uint32()
        _check("k2t_bool_closure", load().k2t_bool_closure(self._h, ctypes.byref(opts), int(max_iters),
                                                           ctypes.byref(h), ctypes.byref(it), _stream_ptr(stream)))
        return Tree._adopt(h, self.n_rows, self.n_cols, opts), int(it.value)

    def msbfs_work_bytes(self) -> int:
        return int(load().k2t_msbfs_work_bytes(self._h))

    def spmv_host(self, direction: int, semiring: int, x: np.ndarray, y: np.ndarray, B: int = 1,
                  w: float = 1.0, stream=None):
        """Product on host arrays (copies in and out inside the call)."""
        if not (x.flags["C_CONTIGUOUS"] and y.flags["C_CONTIGUOUS"]):
            raise ValueError("expected contiguous host arrays")
        _check("k2t_spmv_host", load().k2t_spmv_host(self._h, direction, semiring, ctypes.c_float(w),
                                                     x.ctypes.data, y.ctypes.data, B,
                                                     _stream_ptr(stream)))
        return y

    def level_signatures(self, level: int) -> np.ndarray:
        lib = load()
        n = ctypes.c_uint64()
        lib.k2t_level_signatures(self._h, level, None, 0, ctypes.byref(n))
        out = np.zeros(int(n.value), dtype=np.uint8)
        _check("k2t_level_signatures", lib.k2t_level_signatures(
            self._h, level, out.ctypes.data if out.size else None, out.size, ctypes.byref(n)))
        return out

    def device_level(self, level: int):
        s, d = ctypes.c_void_p(), ctypes.c_void_p()
        _check("k2t_device_level", load().k2t_device_level(self._h, level, ctypes.byref(s), ctypes.byref(d)))
        return s.value, d.value

    def decode(self):
        lib = load()
        n = ctypes.c_uint64()
        lib.k2t_decode(self._h, None, None, 0, ctypes.byref(n))
        r = np.zeros(int(n.value), dtype=np.uint32)
        c = np.zeros(int(n.value), dtype=np.uint32)
        _check("k2t_decode", lib.k2t_decode(self._h, r.ctypes.data if r.size else None,
                                            c.ctypes.data if c.size else None, r.size, ctypes.byref(n)))
        return r, c


_probe_lib = None


def probe(kind: int, x, y, n: int, m: int, stream=None):
    """One pass of a memory-system ceiling probe of the benchmark's own
    library libk2t_probe.so (kinds in csrc/probe/k2t_probe.cu)."""
    global _probe_lib
    if _probe_lib is None:
        if not os.path.exists(PROBE_LIB_PATH):
            raise RuntimeError("libk2t_probe.so is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(PROBE_LIB_PATH)
        P, U64, I32 = ctypes.c_void_p, ctypes.c_uint64, ctypes.c_int32
        lib.k2t_probe.argtypes = [I32, P, P, U64, U64, P]
        lib.k2t_probe.restype = ctypes.c_int
        _probe_lib = lib
    _check("k2t_probe", _probe_lib.k2t_probe(kind, _dev_ptr(x) if x is not None else None, _dev_ptr(y), n, m,
                                             _stream_ptr(stream)))


@dataclass
class LevelInfo:
    levels: int
    d0: int
    nodes: list


def level_info(tree: Tree) -> LevelInfo:
    s = tree.stats()
    return LevelInfo(int(s.levels), int(s.d0), [int(s.level_nodes[d]) for d in range(s.levels)])
