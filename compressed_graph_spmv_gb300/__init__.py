"""k^2-tree semiring SpMV on GB300 (sm_103a): thin Python binding of libk2t.so.

The C ABI is declared in ``include/k2t.h``; ``k2t.Tree`` wraps it.  Build the
shared library with ``compressed_graph_spmv_gb300._build.build()`` (or
``__graft_entry__.build()``).
"""
from .k2t import (BOOLEAN, ENGINE_AUTO, ENGINE_BANDED, ENGINE_CACHED, ENGINE_FUSED, ENGINE_LEVELSYNC, LEFT,
                  MIN_PLUS, OFFSETS_DIRECTORY, OFFSETS_SCAN, PLUS_TIMES, RIGHT, K2TError, Tree,
                  default_opts, load)

__all__ = ["Tree", "default_opts", "load", "K2TError", "RIGHT", "LEFT", "PLUS_TIMES", "BOOLEAN",
           "MIN_PLUS", "ENGINE_AUTO", "ENGINE_BANDED", "ENGINE_FUSED", "ENGINE_LEVELSYNC", "ENGINE_CACHED",
           "OFFSETS_DIRECTORY", "OFFSETS_SCAN"]
