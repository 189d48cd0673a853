"""Pins for the oracle's multi-source search: a hand-checked path graph and
networkx breadth-first distances on random graphs, both directions."""
import numpy as np
import pytest

import oracle
import synth


def test_path_graph_by_hand():
    # A_ij = 1 for i = j + 1: along RIGHT products, i is reached from j = i - 1
    n = 6
    rows = np.arange(1, n, dtype=np.uint32)
    cols = np.arange(0, n - 1, dtype=np.uint32)
    d = oracle.msbfs(rows, cols, n, [0, 3], oracle.RIGHT)
    assert d[:, 0].tolist() == [0, 1, 2, 3, 4, 5]
    assert d[:, 1].tolist() == [-1, -1, -1, 0, 1, 2]
    d = oracle.msbfs(rows, cols, n, [5], oracle.LEFT)
    assert d[:, 0].tolist() == [5, 4, 3, 2, 1, 0]
    d = oracle.msbfs(rows, cols, n, [0], oracle.RIGHT, max_levels=2)
    assert d[:, 0].tolist() == [0, 1, 2, -1, -1, -1]


@pytest.mark.parametrize("seed", range(4))
def test_against_networkx(seed):
    nx = pytest.importorskip("networkx")
    n = 300
    rows, cols, rng = synth.random_small(seed, n, n, 0.004)
    sources = rng.choice(n, size=5, replace=False)
    for direction in (oracle.RIGHT, oracle.LEFT):
        g = nx.DiGraph()
        g.add_nodes_from(range(n))
        for r, c in zip(rows.tolist(), cols.tolist()):
            if direction == oracle.RIGHT:
                g.add_edge(c, r)   # i = r is reached from j = c
            else:
                g.add_edge(r, c)
        d = oracle.msbfs(rows, cols, n, sources, direction)
        for b, s in enumerate(sources):
            want = np.full(n, -1, np.int32)
            for v, k in nx.single_source_shortest_path_length(g, int(s)).items():
                want[v] = k
            assert np.array_equal(d[:, b], want)
