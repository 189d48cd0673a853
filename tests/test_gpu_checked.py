"""The bounds-checked build (libk2t_checked.so, compiled with K2T_CHECKED):
the same C ABI, with kernels that test every leaf's outputs and inputs, the
FUSED chunks' level widths and the LEVELSYNC expand positions against the
bounds of what they address, and report a failed test in the device status
word (K2T_STATUS_OUT_OF_RANGE) instead of touching the memory.  On valid
trees no test may fire and the results must equal the oracle's, for every
engine, semiring, direction and batch shape.  This is the repository's
stand-in for a memory checker: no GPU is faulted, and nothing here feeds
invalid input to a kernel."""
import numpy as np
import pytest

import oracle
from oracle import BOOLEAN, LEFT, PLUS_TIMES, RIGHT, TROPICAL
import synth
from gpu_util import assert_match, device_product, random_x

pytestmark = pytest.mark.gpu

K = pytest.importorskip("compressed_graph_spmv_gb300.k2t")

ENGINES = [
    dict(engine=1),
    dict(engine=1, chunk_cap=4),
    dict(engine=2, offsets=0, tile_m=16),
    dict(engine=2, offsets=1, tile_m=64),
    dict(engine=3, cache_last_internal=1),
    dict(engine=4, cache_last_internal=1, band_rows=16),
    dict(engine=3, cache_last_internal=1, leaf_k=4),
    dict(engine=1, leaf_k=4),
]


@pytest.fixture(autouse=True)
def checked_library(monkeypatch):
    """Route the binding to the checked build for one test, then back."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import gc
    gc.collect()   # trees of other tests are freed by the library that made them
    monkeypatch.setattr(K, "LIB_PATH", K.CHECKED_LIB_PATH)
    monkeypatch.setattr(K, "_lib", None)
    K.load()
    yield
    gc.collect()   # trees made with the checked build are freed by it


@pytest.mark.parametrize("seed", range(4))
def test_checked_build_random_ragged(seed):
    rng = np.random.default_rng(900 + seed)
    nr = int(rng.integers(1, 900))
    nc = int(rng.integers(1, 900))
    rows, cols, _ = synth.random_small(seed, nr, nc, float(rng.choice([0.003, 0.03, 0.2])))
    ot = oracle.OracleTree(rows, cols, nr, nc)
    for kw in ENGINES:
        t = K.Tree(rows, cols, nr, nc, host_top_max_nodes=int(rng.choice([1, 16])),
                   heavy_terms=int(rng.choice([0, 4])), **kw).upload()
        for semiring in (PLUS_TIMES, BOOLEAN, TROPICAL):
            for B in (1, 3, 8, 32):
                if semiring == BOOLEAN and B not in (1, 32):
                    continue
                d = int(rng.integers(0, 2))
                n_in = nc if d == RIGHT else nr
                x = random_x(rng, semiring, n_in, B)
                ref = ot.spmv(d, semiring, x, B=B)
                got = device_product(t, d, semiring, x, B)
                assert t.status() == 0, (kw, semiring, B, d)
                assert_match(semiring, got, ref, "checked seed%d %s sr%d B%d d%d" % (seed, kw, semiring, B, d))
        t.close()


def test_checked_build_rmat_all_engines():
    n = 1 << 14
    rows, cols = synth.rmat(14, 0.57, 0.19, 0.19, 150000, 31)
    rng = np.random.default_rng(31)
    for kw in ENGINES:
        t = K.Tree(rows, cols, n, n, **kw).upload()
        for d in (RIGHT, LEFT):
            for semiring, B in ((PLUS_TIMES, 1), (PLUS_TIMES, 16), (BOOLEAN, 32), (TROPICAL, 4)):
                x = random_x(rng, semiring, n, B)
                ref = oracle.spmv_edges(rows, cols, n, n, d, semiring, x, B=B)
                got = device_product(t, d, semiring, x, B)
                assert t.status() == 0, (kw, d, semiring, B)
                assert_match(semiring, got, ref, "checked rmat %s d%d sr%d B%d" % (kw, d, semiring, B))
        t.close()
