"""GPU parity: every engine, semiring, direction and batch width against the
CPU oracle, through the C ABI, on seeded inputs spanning many chunks/tiles.
Tolerances are stated in tests/gpu_util.py."""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import BOOLEAN, LEFT, PLUS_TIMES, RIGHT, TROPICAL
import synth
from gpu_util import assert_match, device_product, random_x

pytestmark = pytest.mark.gpu

K = pytest.importorskip("compressed_graph_spmv_gb300.k2t")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

ENGINES = [
    dict(engine=1),                                   # fused, tree-only
    dict(engine=1, chunk_cap=4),                       # fused, many tiny chunks
    dict(engine=2, offsets=0, tile_m=16),              # level-sync, directory, many tiles
    dict(engine=2, offsets=1, tile_m=16),              # level-sync, scan
    dict(engine=2, offsets=0, tile_m=1 << 20, use_graph=0),
    dict(engine=3, cache_last_internal=1),             # k^2+F
    dict(engine=4, cache_last_internal=1),             # k^2+F by row band
    dict(engine=4, cache_last_internal=1, band_rows=16),
    dict(engine=3, cache_last_internal=1, leaf_k=4),   # k^2+F with 4x4 leaves (section 5.6)
    dict(engine=1, leaf_k=4),                          # tree-only with 4x4 leaves
    dict(engine=1, leaf_k=4, chunk_cap=4),
]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K.load()


def _tree(rows, cols, nr, nc, **kw):
    return K.Tree(rows, cols, nr, nc, **kw).upload()


def test_figure1_all_engines():
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "figure1.json")))
    e = np.array(g["edges_decoded"], np.uint32)
    ot = oracle.OracleTree(e[:, 0], e[:, 1], 8, 8)
    rng = np.random.default_rng(0)
    for kw in ENGINES:
        t = _tree(e[:, 0], e[:, 1], 8, 8, host_top_max_nodes=1, **kw)
        for semiring in (PLUS_TIMES, BOOLEAN, TROPICAL):
            for d in (RIGHT, LEFT):
                x = random_x(rng, semiring, 8, 3)
                ref = ot.spmv(d, semiring, x, B=3)
                assert_match(semiring, device_product(t, d, semiring, x, 3), ref, "%s sr%d d%d" % (kw, semiring, d))


@pytest.mark.parametrize("seed", range(8))
def test_random_ragged(seed):
    rng = np.random.default_rng(100 + seed)
    nr = int(rng.integers(1, 700))
    nc = int(rng.integers(1, 700))
    n_k4 = int(rng.integers(0, 3))
    rows, cols, _ = synth.random_small(seed, nr, nc, float(rng.choice([0.002, 0.02, 0.2])))
    ot = oracle.OracleTree(rows, cols, nr, nc, n_k4=n_k4)
    top = int(rng.choice([1, 16, 65536]))
    heavy = int(rng.choice([0, 3, 12]))  # small limits send most outputs to the fp64 sums
    for kw in ENGINES:
        t = _tree(rows, cols, nr, nc, n_k4_levels=n_k4, host_top_max_nodes=top, heavy_terms=heavy, **kw)
        for semiring in (PLUS_TIMES, BOOLEAN, TROPICAL):
            for B in (1, 2, 3, 4, 8, 32):
                if semiring == BOOLEAN and B not in (1, 3, 32):
                    continue
                d = int(rng.integers(0, 2))
                n_in = nc if d == RIGHT else nr
                x = random_x(rng, semiring, n_in, B)
                w = float(rng.choice([1.0, 0.5, 2.0])) if semiring != BOOLEAN else 1.0
                ref = ot.spmv(d, semiring, x, B=B, w=w)
                got = device_product(t, d, semiring, x, B, w=w)
                assert_match(semiring, got, ref, "seed%d %s h%d sr%d B%d d%d" % (seed, kw, heavy, semiring, B, d))


def _magnitude_mix(big_at_end: bool):
    """A symmetric 4096 x 4096 matrix whose rows (and columns) 5, 6, 7, 8
    hold 160, 2000, 161 and 100 non-zeros: one in column g (0, or 4095 when
    big_at_end) and the rest spread over [16, 4095).  Row 9 holds one cell,
    (9, 9), listed 300 times.  With x_g = 2^24 and every other x = 1 the exact sums
    are 2^24 + (count - 1); an fp32 sum that adds 2^24 first loses every 1
    after it, up to 1999 off against a bound of 1e-5 * (2^24 + 1999) ~ 168."""
    n = 4096
    g = n - 1 if big_at_end else 0
    rng = np.random.default_rng(77 + int(big_at_end))
    rows, cols = [], []
    for r, cnt in ((5, 160), (6, 2000), (7, 161), (8, 100)):
        others = rng.choice(np.arange(16, n - 1), size=cnt - 1, replace=False)
        c = np.concatenate([[g], others]).astype(np.uint32)
        rows.append(np.full(cnt, r, np.uint32))
        cols.append(c)
    r = np.concatenate(rows)
    c = np.concatenate(cols)
    rep = np.full(300, 9, np.uint32)
    rows = np.concatenate([r, c, rep])
    cols = np.concatenate([c, r, rep])
    x = np.ones(n, np.float32)
    x[g] = 2.0 ** 24
    return rows, cols, n, x


@pytest.mark.parametrize("big_at_end", [False, True])
def test_plus_times_bound_default_options(big_at_end):
    """Default heavy options (heavy_terms 160, bounded fp32 partial sums),
    every engine, B = 1, 4, 16, right and left: the magnitude mix of
    _magnitude_mix with the large input at the lowest column and again at
    the highest (so the order in which the atomics meet it differs) meets
    the plus-times bound on every output.  The 160-term rows stay one fp32
    sum, the longer rows are split, and the repeated pair's row (300 listed
    entries in one partial whatever the split) falls back to fp64."""
    rows, cols, n, x1 = _magnitude_mix(big_at_end)
    for kw in ENGINES:
        t = _tree(rows, cols, n, n, **kw)
        s = t.stats()
        assert (s.heavy_rows, s.heavy_cols) == (3, 3)           # rows 6, 7 and the repeated pair's row 9
        assert s.heavy_fp64[0] == 1 and s.heavy_fp64[1] == 1    # row 9 / column 9
        assert 0 < s.heavy_max_terms[0] <= 160
        for B in (1, 4, 16):
            x = np.repeat(x1[:, None], B, axis=1)
            for d in (RIGHT, LEFT):
                ref = oracle.spmv_edges(rows, cols, n, n, d, PLUS_TIMES, x, B=B)
                got = device_product(t, d, PLUS_TIMES, x, B)
                assert_match(PLUS_TIMES, got, ref, "%s B%d d%d end%d" % (kw, B, d, big_at_end))
                for r, cnt in ((5, 160), (6, 2000), (7, 161), (8, 100)):
                    exact = 2.0 ** 24 + (cnt - 1)
                    assert np.all(np.abs(got[r].astype(np.float64) - exact) <= 1e-5 * exact + 1e-6), (kw, B, d, r)


def test_tropical_signed_zero_order():
    """Tropical minima follow the IEEE total order with -0 < +0: with w = -0,
    an input of -0 contributes -0 and one of +0 contributes +0, so an output
    reaching both holds -0 (bit pattern 0x80000000); the oracle takes the
    same order, and the comparison is bit for bit."""
    n = 64
    rows = np.array([1, 1, 2, 3, 3, 4], np.uint32)
    cols = np.array([10, 11, 11, 12, 13, 10], np.uint32)
    ot = oracle.OracleTree(rows, cols, n, n)
    x = np.full((n, 2), np.inf, np.float32)
    x[10] = [-0.0, 0.0]
    x[11] = [0.0, -0.0]
    x[12] = [-0.0, -0.0]
    x[13] = [0.0, 0.0]
    for kw in ENGINES:
        t = _tree(rows, cols, n, n, host_top_max_nodes=1, **kw)
        for d in (RIGHT, LEFT):
            xd = x if d == RIGHT else np.full((n, 2), -0.0, np.float32)
            ref = ot.spmv(d, TROPICAL, xd, B=2, w=-0.0)
            got = device_product(t, d, TROPICAL, xd, 2, w=-0.0)
            assert_match(TROPICAL, got, ref, "%s d%d" % (kw, d))
            if d == RIGHT:
                assert got[1].view(np.uint32).tolist() == [0x80000000, 0x80000000]
                assert got[3].view(np.uint32).tolist() == [0x80000000, 0x80000000]
                assert got[4].view(np.uint32).tolist() == [0x80000000, 0x00000000]


@pytest.mark.parametrize("heavy_mode", [1, 0])
@pytest.mark.parametrize("heavy_terms", [0, 4])
def test_heavy_outputs_hub_cancellation(heavy_terms, heavy_mode):
    """Row 0 and column 0 hold 5000 non-zeros, more than the heavy limit
    (default 160, or 4): with x_0 = 2^24 and x_j = 1 for the other 4999, the
    sum is 2^24 + 4999.  An fp32 sum can lose each 1 against 2^24 (up to 4999
    off, far beyond the plus-times bound).  fp64 mode (1) sums exactly and
    rounds once, so it matches bit for bit, whatever the order of the atomics;
    split mode (0) keeps fp32 partial sums of at most the limit's terms and
    must meet the bound.  Outputs 1..4999 hold the single term 2^24, the rest
    zero, in both modes."""
    n = 8192
    j = np.arange(5000, dtype=np.uint32)
    rows = np.concatenate([np.zeros(5000, np.uint32), j[1:]])
    cols = np.concatenate([j, np.zeros(4999, np.uint32)])
    exact = np.float64(2 ** 24) + 4999.0
    want = np.zeros(n, np.float32)
    want[0] = np.float32(exact)
    want[1:5000] = np.float32(2 ** 24)
    tol0 = 1e-5 * exact + 1e-6
    for kw in ENGINES:
        t = _tree(rows, cols, n, n, heavy_terms=heavy_terms, heavy_mode=heavy_mode, host_top_max_nodes=16, **kw)
        s = t.stats()
        assert (s.heavy_rows, s.heavy_cols) == (1, 1)
        for B in (1, 2, 3, 4, 16):
            x = np.ones((n, B), np.float32)
            x[0] = 2.0 ** 24
            for d in (RIGHT, LEFT):
                got = device_product(t, d, PLUS_TIMES, x, B)
                if heavy_mode == 1:
                    assert np.array_equal(got, np.repeat(want[:, None], B, axis=1)), (kw, B, d, got[0])
                else:
                    assert np.array_equal(got[1:], np.repeat(want[1:, None], B, axis=1)), (kw, B, d)
                    assert np.all(np.abs(got[0].astype(np.float64) - exact) <= tol0), (kw, B, d, got[0])


@pytest.mark.parametrize("heavy_mode", [0, 1])
def test_heavy_outputs_large_hub(heavy_mode):
    """A row and a column with 2^19 non-zeros each (x ~ U(0,1)), where a
    single fp32 sum drifts to about the plus-times bound: both heavy modes
    must meet it on every cached and tree-only engine, for B = 1 and 16."""
    n = 1 << 19
    rng = np.random.default_rng(31)
    r0, c0, _ = synth.random_small(31, n, n, 2e-6)
    a = np.arange(n, dtype=np.uint32)
    rows, cols = oracle.dedup_edges(np.concatenate([r0, np.full(n, 7, np.uint32), a]),
                                    np.concatenate([c0, a, np.full(n, 11, np.uint32)]))
    for kw in (ENGINES[0], ENGINES[2], ENGINES[5], ENGINES[6], ENGINES[8], ENGINES[9]):
        t = _tree(rows, cols, n, n, heavy_mode=heavy_mode, **kw)
        assert t.stats().heavy_rows >= 1 and t.stats().heavy_cols >= 1
        for B in (1, 16):
            x = rng.random(size=(n, B), dtype=np.float32)
            for d in (RIGHT, LEFT):
                hub = 7 if d == RIGHT else 11
                sample = np.unique(np.concatenate([[hub, 0, n - 1], rng.integers(0, n, size=200)]))
                got = device_product(t, d, PLUS_TIMES, x, B)
                ref = oracle.rows_product(rows, cols, n, n, d, PLUS_TIMES, x, sample, B=B)
                assert_match(PLUS_TIMES, got[sample], ref, "%s mode%d B%d d%d" % (kw, heavy_mode, B, d))


def test_uniform_1024_plus_times():
    wl = synth.uniform_c1()
    ot = oracle.OracleTree(wl.rows, wl.cols, wl.n_rows, wl.n_cols)
    for kw in ENGINES:
        t = _tree(wl.rows, wl.cols, wl.n_rows, wl.n_cols, host_top_max_nodes=64, **kw)
        for d in (RIGHT, LEFT):
            ref = ot.spmv(d, PLUS_TIMES, wl.xs[d], B=1)
            assert_match(PLUS_TIMES, device_product(t, d, PLUS_TIMES, wl.xs[d], 1), ref, str(kw))


def test_exact_special_cases():
    rows, cols = synth.rmat(16, 0.57, 0.19, 0.19, 400000, 11)
    n = 1 << 16
    r, c = oracle.dedup_edges(rows, cols)
    for kw in ENGINES[:1] + ENGINES[2:4] + ENGINES[5:]:
        t = _tree(rows, cols, n, n, host_top_max_nodes=256, **kw)
        # x = 1: out-degree / in-degree, exact in fp32 whatever the atomic order
        y = device_product(t, RIGHT, PLUS_TIMES, np.ones((n, 1), np.float32), 1)[:, 0]
        assert np.array_equal(y, np.bincount(r, minlength=n).astype(np.float32))
        y = device_product(t, LEFT, PLUS_TIMES, np.ones((n, 1), np.float32), 1)[:, 0]
        assert np.array_equal(y, np.bincount(c, minlength=n).astype(np.float32))
        # tropical with x = 0, w = 1: 1 on non-empty rows, +inf elsewhere
        y = device_product(t, RIGHT, TROPICAL, np.zeros((n, 1), np.float32), 1, w=1.0)[:, 0]
        ne = np.zeros(n, bool)
        ne[r] = True
        assert np.all(y[ne] == 1.0) and np.all(np.isinf(y[~ne]))


def test_rmat_medium_all_semirings():
    """R-MAT 2^17, ~1M edges: O1 (edge-list definition) on every output."""
    rows, cols = synth.rmat(17, 0.57, 0.19, 0.19, 1 << 20, 12)
    n = 1 << 17
    rng = np.random.default_rng(12)
    for kw in (ENGINES[0], ENGINES[2], ENGINES[3], ENGINES[5], ENGINES[6], ENGINES[8], ENGINES[9]):
        t = _tree(rows, cols, n, n, **kw)
        for semiring, B in ((PLUS_TIMES, 1), (PLUS_TIMES, 16), (BOOLEAN, 32), (TROPICAL, 8)):
            for d in (RIGHT, LEFT):
                x = random_x(rng, semiring, n, B)
                ref = oracle.spmv_edges(rows, cols, n, n, d, semiring, x, B=B)
                assert_match(semiring, device_product(t, d, semiring, x, B), ref, "%s sr%d B%d" % (kw, semiring, B))


def test_empty_matrix_fills():
    z = np.zeros(0, np.uint32)
    for kw in ENGINES:
        t = _tree(z, z, 100, 37, **kw)
        y = device_product(t, RIGHT, TROPICAL, np.ones((37, 2), np.float32), 2)
        assert np.all(np.isinf(y))
        y = device_product(t, LEFT, PLUS_TIMES, np.ones((100, 5), np.float32), 5)
        assert np.all(y == 0)


def test_host_buffer_product():
    rows, cols = synth.rmat(12, 0.57, 0.19, 0.19, 20000, 13)
    n = 4096
    t = _tree(rows, cols, n, n, host_vectors=1, max_batch=8)
    rng = np.random.default_rng(13)
    x = rng.uniform(0, 1, size=(n, 8)).astype(np.float32)
    y = np.zeros((n, 8), np.float32)
    t.spmv_host(RIGHT, PLUS_TIMES, x, y, B=8)
    ref = oracle.spmv_edges(rows, cols, n, n, RIGHT, PLUS_TIMES, x, B=8)
    assert_match(PLUS_TIMES, y, ref, "host")
    with pytest.raises(K.K2TError):
        t.spmv_host(RIGHT, PLUS_TIMES, x, y, B=16)


def test_footprint_equals_prediction():
    import torch
    rows, cols = synth.rmat(18, 0.57, 0.19, 0.19, 4 << 20, 14)
    for kw in (dict(engine=1), dict(engine=3, cache_last_internal=1), dict(engine=2, tile_m=1 << 16),
               dict(engine=4, cache_last_internal=1)):
        t = K.Tree(rows, cols, 1 << 18, 1 << 18, **kw)
        ws = t.workspace_bytes()
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        t.upload()
        torch.cuda.synchronize()
        free1 = torch.cuda.mem_get_info()[0]
        used = free0 - free1
        # cudaMalloc rounds to 2 MiB pages
        assert abs(used - ws) <= (2 << 20), (kw, used, ws)
        t.close()
        # an arena from torch of exactly the predicted size also works
        t = K.Tree(rows, cols, 1 << 18, 1 << 18, **kw)
        arena = torch.empty(t.workspace_bytes(), dtype=torch.uint8, device="cuda")
        t.upload(arena)
        x = torch.rand(1 << 18, 1, device="cuda")
        y = torch.empty_like(x)
        t.spmv(RIGHT, PLUS_TIMES, x, y)
        torch.cuda.synchronize()


def test_argument_errors():
    import torch
    rows, cols = synth.rmat(10, 0.57, 0.19, 0.19, 3000, 15)
    t = _tree(rows, cols, 1024, 1024)
    x = torch.rand(1024 * 33, device="cuda")
    y = torch.empty(1024 * 33, device="cuda")
    with pytest.raises(K.K2TError) as e:
        t.spmv(RIGHT, PLUS_TIMES, x, y, B=33)
    assert e.value.status == -2
    lib = K.load()
    import ctypes
    assert lib.k2t_spmv(t.handle, 0, 0, ctypes.c_float(1.0), x.data_ptr() + 2, y.data_ptr(), 1, None) == -1
    assert lib.k2t_spmv(t.handle, 0, 0, ctypes.c_float(1.0), x.data_ptr(), x.data_ptr(), 1, None) == -1
    assert lib.k2t_spmv(t.handle, 3, 0, ctypes.c_float(1.0), x.data_ptr(), y.data_ptr(), 1, None) == -1
    with pytest.raises(K.K2TError) as e:
        t.upload()
    assert e.value.status == -5
