"""Pins of the oracle's Boolean matrix product and transitive closure (no
GPU): a triple loop over dense 0/1 matrices, identities of the product, a
hand-checked path graph, and networkx's transitive closure."""
import numpy as np
import pytest

import oracle
import synth


def _dense(r, c, n, m):
    A = np.zeros((n, m), dtype=bool)
    A[r, c] = True
    return A


def _triple_loop(A, B):
    n, m = A.shape
    p = B.shape[1]
    C = np.zeros((n, p), dtype=bool)
    for i in range(n):
        for j in range(p):
            for k in range(m):
                if A[i, k] and B[k, j]:
                    C[i, j] = True
                    break
    return C


@pytest.mark.parametrize("seed", range(10))
def test_product_brute_force(seed):
    rng = np.random.default_rng(500 + seed)
    n, m, p = (int(v) for v in rng.integers(1, 13, size=3))
    ra, ca, _ = synth.random_small(seed, n, m, float(rng.choice([0.05, 0.2, 0.5])))
    rb, cb, _ = synth.random_small(seed + 100, m, p, float(rng.choice([0.05, 0.2, 0.5])))
    r, c = oracle.bool_product(ra, ca, rb, cb, n, m, p)
    want = _triple_loop(_dense(ra, ca, n, m), _dense(rb, cb, m, p))
    assert np.array_equal(_dense(r, c, n, p), want)
    assert r.size == int(want.sum())          # distinct, no repeats
    assert np.all(np.diff(r.astype(np.int64) * p + c) > 0)   # sorted by (row, col)


def test_product_identities():
    rows, cols, _ = synth.random_small(7, 60, 45, 0.05)
    eye = np.arange(60, dtype=np.uint32)
    eye45 = np.arange(45, dtype=np.uint32)
    dr, dc = oracle.dedup_edges(rows, cols)
    r, c = oracle.bool_product(eye, eye, rows, cols, 60, 60, 45)       # I A = A
    assert np.array_equal(r, dr) and np.array_equal(c, dc)
    r, c = oracle.bool_product(rows, cols, eye45, eye45, 60, 45, 45)   # A I = A
    assert np.array_equal(r, dr) and np.array_equal(c, dc)
    rb, cb, _ = synth.random_small(8, 45, 30, 0.08)
    r1, c1 = oracle.bool_product(rows, cols, rb, cb, 60, 45, 30)        # (A B)^T = B^T A^T
    r2, c2 = oracle.bool_product(cb, rb, cols, rows, 30, 45, 60)
    assert sorted(zip(r1.tolist(), c1.tolist())) == sorted(zip(c2.tolist(), r2.tolist()))


def test_path_graph_by_hand():
    # 0 -> 1 -> 2 -> 3: the square joins vertices two steps apart; the closure
    # joins i to every j > i, found after two squarings plus one that adds nothing
    r = np.array([0, 1, 2], np.uint32)
    c = np.array([1, 2, 3], np.uint32)
    pr, pc = oracle.bool_product(r, c, r, c, 4, 4, 4)
    assert list(zip(pr.tolist(), pc.tolist())) == [(0, 2), (1, 3)]
    tr, tc, it = oracle.transitive_closure(r, c, 4)
    assert list(zip(tr.tolist(), tc.tolist())) == [(0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3)]
    assert it == 3


@pytest.mark.parametrize("seed", range(4))
def test_closure_matches_networkx(seed):
    nx = pytest.importorskip("networkx")
    rows, cols, _ = synth.random_small(40 + seed, 80, 80, 0.012 + 0.004 * seed)
    G = nx.DiGraph()
    G.add_nodes_from(range(80))
    G.add_edges_from(zip(rows.tolist(), cols.tolist()))
    # paths of one or more edges: a vertex reaches itself only through a cycle
    want = set()
    for u in range(80):
        for v in nx.descendants(G, u):
            want.add((u, v))
        if any(u in nx.descendants(G, w) for w in G.successors(u)) or G.has_edge(u, u):
            want.add((u, u))
    r, c, _ = oracle.transitive_closure(rows, cols, 80)
    assert set(zip(r.tolist(), c.tolist())) == want
