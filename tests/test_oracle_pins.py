"""Pins for the CPU oracle, against facts the pages and the mathematics fix.

The oracle (``oracle/``) is the reference every GPU result is compared with,
so it is itself checked here against things other than itself:

* the worked example of Figure 1 of "A GPU Engine for Sparse Matrix-Vector
  Products on k^2-Tree-Compressed Graphs" (``tests/golden/figure1.json``):
  the printed bitstrings T and L, fan-outs, child offsets, directory samples,
  leaf codes and origins, the rank formula of section 2.1 and the claims of
  section 3.3;
* dense brute force on small matrices (numpy matrix products, min/OR
  reductions), for every semiring, both directions and several batch widths;
* closed forms and invariants: nodes per level equal the number of distinct
  blocks, popcount of a level equals the size of the next one, popcount of
  L equals nnz, decode reproduces the edge set, left(A) = right(A^T);
* exact special cases: x = 1 gives degrees, x = e_j gives a column, tropical
  x = 0 with w = 1 gives 1 on non-empty rows and +inf elsewhere.
"""
import json
import os

import numpy as np
import pytest

import oracle
from oracle import BOOLEAN, LEFT, PLUS_TIMES, RIGHT, TROPICAL
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "figure1.json")


def _fig1():
    with open(GOLDEN) as f:
        return json.load(f)


def _edges(g):
    e = np.array(g["edges_decoded"], dtype=np.uint32)
    return e[:, 0].copy(), e[:, 1].copy()


# --- Figure 1 -----------------------------------------------------------
def test_figure1_bitstrings():
    g = _fig1()
    r, c = _edges(g)
    t = oracle.OracleTree(r, c, g["n"], g["n"])
    assert t.levels == g["levels"]
    assert t.bitstring(0) == g["T_level0"]
    assert t.bitstring(1) == "".join(g["T_level1"])
    assert t.bitstring(2) == "".join(g["L"])
    assert t.level_nodes() == [1, 4, g["level2_nodes"]]
    assert t.t_bits == 4 + 16


def test_figure1_fanouts_offsets_directory():
    g = _fig1()
    r, c = _edges(g)
    t = oracle.OracleTree(r, c, g["n"], g["n"])
    lvl1 = t.bitstring(1)
    fan = [lvl1[4 * i:4 * i + 4].count("1") for i in range(4)]
    assert fan == g["level1_fanouts"]
    off = list(np.concatenate([[0], np.cumsum(fan)[:-1]]))
    assert off == g["level1_child_offsets"]
    assert sum(fan) == g["level2_nodes"]
    # directory with S = 2: the offset of the first child of nodes 0 and 2
    assert [off[0], off[2]] == g["directory_S2_level1"]
    # node 01 finds its first child at the sample of its block + popcount(1000)
    assert g["directory_S2_level1"][0] + g["T_level1"][0].count("1") == off[1]


def test_figure1_rank_formula():
    g = _fig1()
    r, c = _edges(g)
    t = oracle.OracleTree(r, c, g["n"], g["n"])
    ex = g["rank_example"]
    assert t.rank1(ex["p"]) == ex["rank1"]
    # k^2 * rank1(T, p) (section 2.1) and the oracle's per-level formula agree
    assert 4 * t.rank1(ex["p"]) == ex["child_pos"] == t.child_pos(1, ex["p"])
    assert (ex["child_pos"] - t.t_bits) // 4 == ex["leaf_index"]


def test_figure1_decode_and_codes():
    g = _fig1()
    r, c = _edges(g)
    t = oracle.OracleTree(r, c, g["n"], g["n"])
    dr, dc = t.decode()
    assert sorted(zip(dr.tolist(), dc.tolist())) == sorted(map(tuple, g["edges_decoded"]))
    # leaf codes: parent quadrant bits then leaf quadrant bits; origin = deinterleave * 2
    for code, origin in zip(g["leaf_codes"], g["leaf_origins"]):
        rb = code[0] + code[2]
        cb = code[1] + code[3]
        assert [int(rb, 2) * 2, int(cb, 2) * 2] == origin
    # cell (3, 5): path 01 10 11 -> row bits 011, column bits 101
    p = g["cell_3_5_path"]
    assert int(p[0][0] + p[1][0] + p[2][0], 2) == 3
    assert int(p[0][1] + p[1][1] + p[2][1], 2) == 5
    assert (3, 5) in set(zip(dr.tolist(), dc.tolist()))


def test_figure1_worked_claims():
    """Section 3.3: updates per thread of the last kernel and their collisions."""
    g = _fig1()
    r, c = _edges(g)
    cells = set(map(tuple, g["edges_decoded"]))
    # thread = level-1 node = 4x4 block (r // 4, c // 4)
    per_thread = {}
    for (i, j) in cells:
        key = "%d%d" % (i // 4, j // 4)
        per_thread.setdefault(key, []).append((i, j))
    assert {k: len(v) for k, v in per_thread.items()} == g["claims"]["thread_updates"]
    ys = {k: [list(e) for e in v if e[0] == 1] for k, v in per_thread.items()}
    assert {k: v for k, v in ys.items() if v} == g["claims"]["y1_sources"]
    y6 = {k: sum(1 for e in v if e[0] == 6) for k, v in per_thread.items()}
    assert {k: v for k, v in y6.items() if v} == g["claims"]["y6_cells_per_thread"]
    # the leaf 01 10 holds the single cell (3, 5): x5 reaches y3 (right product)
    t = oracle.OracleTree(r, c, g["n"], g["n"])
    x = np.zeros((8, 1), np.float32)
    x[5] = 1.0
    y = t.spmv(RIGHT, PLUS_TIMES, x).y[:, 0]
    assert y[3] == 1.0 and y[1] == 1.0 and y.sum() == 2.0
    # leaf 5 (code 1010, origin (6, 0)) holds (6, 1): x1 reaches y6
    x = np.zeros((8, 1), np.float32)
    x[1] = 1.0
    y = t.spmv(RIGHT, PLUS_TIMES, x).y[:, 0]
    assert y[6] == 1.0 and y[5] == 1.0 and y[1] == 1.0 and y.sum() == 3.0


# --- dense brute force ----------------------------------------------------
def _key(v):
    u = np.ascontiguousarray(v, dtype=np.float32).view(np.uint32)
    return np.where(u & np.uint32(0x80000000), u ^ np.uint32(0x7fffffff), u).astype(np.uint32).view(np.int32)


def dense_product(A, direction, semiring, x, B, w):
    M = A if direction == RIGHT else A.T          # M[out, in]
    if semiring == PLUS_TIMES:
        return M.astype(np.float64) @ (np.float64(w) * x.astype(np.float64))
    if semiring == BOOLEAN:
        mask = 0xffffffff if B >= 32 else (1 << B) - 1
        y = np.zeros(M.shape[0], dtype=np.uint32)
        for b in range(32):
            if not (mask >> b) & 1:
                continue
            bit = ((x >> np.uint32(b)) & np.uint32(1)).astype(np.int64)
            hit = (M.astype(np.int64) @ bit) > 0
            y |= (hit.astype(np.uint32) << np.uint32(b))
        return y
    contrib = (np.float32(w) + x).astype(np.float32)   # (n_in, B)
    K = _key(contrib)
    inf_key = _key(np.array([np.inf], np.float32))[0]
    y = np.empty((M.shape[0], B), dtype=np.float32)
    for o in range(M.shape[0]):
        sel = K[M[o]]
        kk = sel.min(axis=0) if sel.shape[0] else np.full(B, inf_key, np.int32)
        u = kk.astype(np.int32).view(np.uint32)
        y[o] = np.where(u & np.uint32(0x80000000), u ^ np.uint32(0x7fffffff), u).astype(np.uint32).view(np.float32)
    return y


def _random_x(rng, semiring, n, B):
    if semiring == BOOLEAN:
        return rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    x = rng.uniform(-3, 3, size=(n, B)).astype(np.float32)
    if semiring == TROPICAL:
        x[rng.random(size=(n, B)) < 0.3] = np.inf
    return x


def _check_equal(semiring, got, want, scale=None):
    if semiring == PLUS_TIMES:
        tol = 1e-9 * (np.abs(want) + 1.0)
        assert np.all(np.abs(got - want) <= tol)
    else:
        assert np.array_equal(np.asarray(got).view(np.uint32), np.asarray(want).view(np.uint32))


@pytest.mark.parametrize("seed", range(16))
def test_brute_force_small(seed):
    rng = np.random.default_rng(1000 + seed)
    n_rows = int(rng.integers(1, 70))
    n_cols = int(rng.integers(1, 70))
    n_k4 = int(rng.integers(0, 3)) if max(n_rows, n_cols) > 4 else 0
    leaf_k = 4 if seed % 2 else 2
    rows, cols, _ = synth.random_small(seed, n_rows, n_cols, float(rng.choice([0.01, 0.05, 0.3])))
    A = np.zeros((n_rows, n_cols), dtype=bool)
    A[rows, cols] = True
    t = oracle.OracleTree(rows, cols, n_rows, n_cols, n_k4=n_k4, leaf_k=leaf_k)
    assert t.leaf_k == leaf_k
    for semiring in (PLUS_TIMES, BOOLEAN, TROPICAL):
        for B in (1, 3, 32):
            for direction in (RIGHT, LEFT):
                n_in = n_cols if direction == RIGHT else n_rows
                x = _random_x(rng, semiring, n_in, B)
                w = {PLUS_TIMES: 1.0, BOOLEAN: 1.0, TROPICAL: float(rng.choice([0.0, 1.0, 2.5]))}[semiring]
                if semiring == PLUS_TIMES and B == 3:
                    w = 0.75
                want = dense_product(A, direction, semiring, x, B, w)
                o2 = t.spmv(direction, semiring, x, B=B, w=w)
                o1 = oracle.spmv_edges(rows, cols, n_rows, n_cols, direction, semiring, x, B=B, w=w)
                _check_equal(semiring, o2.y, want)
                _check_equal(semiring, o1.y, want)
                assert o2.cells == int(A.sum())


# --- closed forms and invariants -----------------------------------------
def _level_side(dim_bits, n_k4, d):
    used = sum(2 if e < n_k4 else 1 for e in range(d))
    return 1 << (dim_bits - used)


@pytest.mark.parametrize("n_k4,leaf_k", [(0, 2), (1, 2), (2, 2), (0, 4), (1, 4), (2, 4)])
def test_invariants(n_k4, leaf_k):
    rows, cols, _ = synth.random_small(7 + n_k4, 300, 200, 0.01)
    t = oracle.OracleTree(rows, cols, 300, 200, n_k4=n_k4, leaf_k=leaf_k)
    # side 2^9 = 512; levels: n_k4 of k = 4, then k = 2, then the leaf level
    assert t.dim_bits == 9 and t.levels == 9 - n_k4 - (leaf_k == 4)
    assert _level_side(t.dim_bits, n_k4, t.levels - 1) == leaf_k
    bits = t.bits()
    start = t.level_start()
    nodes = t.level_nodes()
    r, c = oracle.dedup_edges(rows, cols)
    for d in range(t.levels):
        side = _level_side(t.dim_bits, n_k4, d)
        distinct = len(set(zip((r // side).tolist(), (c // side).tolist())))
        assert nodes[d] == distinct, d
        if d + 1 < t.levels:
            assert int(bits[start[d]:start[d + 1]].sum()) == nodes[d + 1]
        assert nodes[d] <= (nodes[d + 1] if d + 1 < t.levels else r.size)  # levels never shrink
    assert int(bits[start[t.levels - 1]:].sum()) == r.size          # popcount(L) = nnz
    dr, dc = t.decode()
    assert sorted(zip(dr.tolist(), dc.tolist())) == sorted(zip(r.tolist(), c.tolist()))


def test_figure1_leaf4_by_hand():
    """The Figure 1 matrix (8 x 8) with 4 x 4 leaves, derived by hand from its
    twelve cells: the root's four quadrants of side 4 are all non-empty
    (T = 1111), and each leaf lists its cells at bit 4*dr + dc:
      rows 0-3, cols 0-3: (1,1)                   -> bit 5
      rows 0-3, cols 4-7: (0,4) (1,5) (3,5)       -> bits 0, 5, 13
      rows 4-7, cols 0-3: (5,1) (5,2) (6,1) (6,2) -> bits 5, 6, 9, 10
      rows 4-7, cols 4-7: (6,6) (6,7) (7,6) (7,7) -> bits 10, 11, 14, 15"""
    g = json.load(open(GOLDEN))
    e = np.array(g["edges_decoded"], np.uint32)
    t = oracle.OracleTree(e[:, 0], e[:, 1], 8, 8, leaf_k=4)
    assert t.levels == 2 and t.level_nodes() == [1, 4]
    assert t.bitstring(0) == "1111"
    assert t.bitstring(1) == ("0000010000000000" "1000010000000100"
                              "0000011001100000" "0000000000110011")
    assert t.child_pos(0, 2) == 4 + 2 * 16  # third set bit of the root -> third leaf
    x = np.arange(1, 9, dtype=np.float32).reshape(8, 1)
    y = t.spmv(RIGHT, PLUS_TIMES, x).y[:, 0]
    # x_c = c + 1 summed over each row's columns: row 6 has 1, 2, 6, 7 -> 2+3+7+8
    assert y.tolist() == [5.0, 8.0, 0.0, 6.0, 0.0, 5.0, 20.0, 15.0]


def test_left_equals_right_of_transpose():
    rows, cols, rng = synth.random_small(21, 90, 140, 0.02)
    t = oracle.OracleTree(rows, cols, 90, 140)
    tt = oracle.OracleTree(cols, rows, 140, 90)
    for semiring in (PLUS_TIMES, BOOLEAN, TROPICAL):
        x = _random_x(rng, semiring, 90, 4)
        a = t.spmv(LEFT, semiring, x, B=4)
        b = tt.spmv(RIGHT, semiring, x, B=4)
        _check_equal(semiring, a.y, b.y)


def test_special_cases():
    rows, cols, _ = synth.random_small(33, 128, 96, 0.03)
    t = oracle.OracleTree(rows, cols, 128, 96)
    r, c = oracle.dedup_edges(rows, cols)
    # x = 1 gives out-degrees (right) and in-degrees (left), exactly
    y = t.spmv(RIGHT, PLUS_TIMES, np.ones((96, 1), np.float32)).y[:, 0]
    assert np.array_equal(y, np.bincount(r, minlength=128).astype(np.float64))
    y = t.spmv(LEFT, PLUS_TIMES, np.ones((128, 1), np.float32)).y[:, 0]
    assert np.array_equal(y, np.bincount(c, minlength=96).astype(np.float64))
    # x = e_j gives column j in every semiring
    j = int(c[0])
    col = np.zeros(128, bool)
    col[r[c == j]] = True
    e = np.zeros((96, 1), np.float32)
    e[j] = 1.0
    assert np.array_equal(t.spmv(RIGHT, PLUS_TIMES, e).y[:, 0] != 0, col)
    eb = np.zeros(96, np.uint32)
    eb[j] = 1
    assert np.array_equal(t.spmv(RIGHT, BOOLEAN, eb, B=1).y != 0, col)
    # Boolean with 32 one-hot vectors gives 32 columns at once
    js = np.unique(c)[:32]
    xb = np.zeros(96, np.uint32)
    for b, jj in enumerate(js):
        xb[jj] |= np.uint32(1 << b)
    yb = t.spmv(RIGHT, BOOLEAN, xb, B=32).y
    for b, jj in enumerate(js):
        colj = np.zeros(128, bool)
        colj[r[c == jj]] = True
        assert np.array_equal(((yb >> np.uint32(b)) & 1).astype(bool), colj)
    # tropical, x = 0 and w = 1: 1 on non-empty rows, +inf on empty ones
    yt = t.spmv(RIGHT, TROPICAL, np.zeros((96, 1), np.float32), w=1.0).y[:, 0]
    nonempty = np.zeros(128, bool)
    nonempty[r] = True
    assert np.all(yt[nonempty] == 1.0) and np.all(np.isinf(yt[~nonempty]))


def test_tropical_total_order_signed_zero():
    """Reading: min in the IEEE total order without NaN, so -0 < +0."""
    rows = np.array([0, 0, 1], np.uint32)
    cols = np.array([0, 1, 1], np.uint32)
    t = oracle.OracleTree(rows, cols, 2, 2)
    # w = -0: contributions are -0 + -0 = -0 and -0 + +0 = +0 (IEEE sums)
    x = np.array([[-0.0], [0.0]], np.float32)
    y = t.spmv(RIGHT, TROPICAL, x, w=-0.0).y[:, 0]
    assert y.view(np.uint32).tolist() == [0x80000000, 0x00000000]
    y1 = oracle.spmv_edges(rows, cols, 2, 2, RIGHT, TROPICAL, x, w=-0.0).y[:, 0]
    assert y1.view(np.uint32).tolist() == [0x80000000, 0x00000000]


def test_empty_matrix():
    rows = np.zeros(0, np.uint32)
    t = oracle.OracleTree(rows, rows, 16, 16)
    assert t.bitstring(0) == "0000" and t.level_nodes()[1:] == [0] * (t.levels - 1)
    assert np.all(t.spmv(RIGHT, PLUS_TIMES, np.ones((16, 1), np.float32)).y == 0)
    assert np.all(np.isinf(t.spmv(RIGHT, TROPICAL, np.ones((16, 2), np.float32), B=2).y))


def test_rows_product_matches_definition():
    rows, cols = synth.rmat(10, 0.57, 0.19, 0.19, 5000, 5)
    rng = np.random.default_rng(5)
    for direction in (RIGHT, LEFT):
        for semiring, B in ((PLUS_TIMES, 2), (BOOLEAN, 5), (TROPICAL, 3)):
            x = _random_x(rng, semiring, 1024, B)
            full = oracle.spmv_edges(rows, cols, 1024, 1024, direction, semiring, x, B=B)
            sample = rng.choice(1024, size=50, replace=False)
            part = oracle.rows_product(rows, cols, 1024, 1024, direction, semiring, x, sample, B=B)
            _check_equal(semiring, part.y, full.y[sample])


def test_medium_tree_matches_definition():
    """O2 (tree descent) against O1 (edge list) on a power-law graph."""
    rows, cols = synth.rmat(12, 0.57, 0.19, 0.19, 40000, 9)
    t = oracle.OracleTree(rows, cols, 4096, 4096)
    rng = np.random.default_rng(9)
    for direction in (RIGHT, LEFT):
        for semiring, B in ((PLUS_TIMES, 1), (BOOLEAN, 32), (TROPICAL, 8)):
            x = _random_x(rng, semiring, 4096, B)
            a = t.spmv(direction, semiring, x, B=B)
            b = oracle.spmv_edges(rows, cols, 4096, 4096, direction, semiring, x, B=B)
            _check_equal(semiring, a.y, b.y)
            if semiring == PLUS_TIMES:
                assert np.allclose(a.scale, b.scale)


@pytest.mark.parametrize("seed", range(3))
def test_band_parallel_descent_equals_serial(seed):
    """The multicore descent (subtrees of one level grouped into row bands for
    right products and column bands for left ones, bands shared among
    threads) gives exactly the single-thread descent's result on every
    semiring, at every band level and thread count: each output receives its
    contributions in the same order, so even the fp64 plus-times sums and
    their scales agree bit for bit, and a band never has two writers.  The
    single-thread descent is itself pinned by brute force above."""
    rng = np.random.default_rng(500 + seed)
    nr, nc = int(rng.integers(300, 2000)), int(rng.integers(300, 2000))
    rows, cols, _ = synth.random_small(50 + seed, nr, nc, 0.01)
    hub = rng.integers(0, nr)
    rows = np.concatenate([rows, np.full(nc // 2, hub, np.uint32)])
    cols = np.concatenate([cols, rng.choice(nc, nc // 2, replace=False).astype(np.uint32)])
    t = oracle.OracleTree(rows, cols, nr, nc, n_k4=seed % 2, leaf_k=4 if seed == 2 else 2)
    for semiring, B in ((PLUS_TIMES, 3), (BOOLEAN, 32), (TROPICAL, 2)):
        for d in (RIGHT, LEFT):
            n_in = nc if d == RIGHT else nr
            if semiring == BOOLEAN:
                x = rng.integers(0, 2 ** 32, size=n_in, dtype=np.uint64).astype(np.uint32)
            else:
                x = rng.uniform(-3, 3, size=(n_in, B)).astype(np.float32)
            want = t.spmv(d, semiring, x, B=B, w=0.75)
            for level in (-1, 0, 2, t.levels - 2, t.levels - 1):
                for th in (2, 5, 0):
                    got = t.spmv(d, semiring, x, B=B, w=0.75, threads=th, band_level=level)
                    assert got.cells == want.cells
                    assert np.array_equal(np.ascontiguousarray(got.y).view(np.uint8),
                                          np.ascontiguousarray(want.y).view(np.uint8)), (semiring, d, level, th)
                    if semiring == PLUS_TIMES:
                        assert np.array_equal(got.scale, want.scale)
                    assert t.threads_used >= 1
