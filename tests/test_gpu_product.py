"""GPU parity of the product of two trees (k2t_bool_product) and of the
transitive closure by repeated squaring (k2t_bool_closure) against the
oracle's definitions: the distinct non-zeros of C must match exactly."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

K = pytest.importorskip("compressed_graph_spmv_gb300.k2t")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K.load()


def _cells(tree):
    r, c = tree.decode()
    return sorted(zip(r.tolist(), c.tolist()))


def _want(r, c):
    return sorted(zip(r.tolist(), c.tolist()))


@pytest.mark.parametrize("seed", range(10))
def test_product_random_ragged(seed):
    rng = np.random.default_rng(700 + seed)
    bits = int(rng.integers(2, 10))
    lo, hi = (1 << (bits - 1)) + 1 if bits > 2 else 1, 1 << bits
    n, m, p = (int(v) for v in rng.integers(lo, hi + 1, size=3))
    dens = float(rng.choice([0.003, 0.02, 0.1]))
    ra, ca, _ = synth.random_small(seed, n, m, dens)
    rb, cb, _ = synth.random_small(seed + 50, m, p, dens)
    a = K.Tree(ra, ca, n, m, host_top_max_nodes=int(rng.choice([1, 64])))
    b = K.Tree(rb, cb, m, p)
    c = a.bool_product(b)
    assert (c.n_rows, c.n_cols) == (n, p)
    assert _cells(c) == _want(*oracle.bool_product(ra, ca, rb, cb, n, m, p)), (n, m, p)


@pytest.mark.parametrize("scale,edges", [(12, 20000), (14, 60000)])
def test_product_rmat_square_and_transpose(scale, edges):
    n = 1 << scale
    rows, cols = synth.rmat(scale, 0.57, 0.19, 0.19, edges, scale)
    a = K.Tree(rows, cols, n, n)
    at = K.Tree(cols, rows, n, n)
    assert _cells(a.bool_product(a)) == _want(*oracle.bool_product(rows, cols, rows, cols, n, n, n))
    assert _cells(a.bool_product(at)) == _want(*oracle.bool_product(rows, cols, cols, rows, n, n, n))


def test_product_large_sparse_graph():
    """2^17 vertices, local edges (targets within +-256 of the source, the
    web-like recipe), A A through many tiles and a multi-level frontier."""
    wl_r, wl_c = synth.weblike(1 << 17, lam=6.0, seed=9)
    n = 1 << 17
    a = K.Tree(wl_r, wl_c, n, n)
    assert _cells(a.bool_product(a)) == _want(*oracle.bool_product(wl_r, wl_c, wl_r, wl_c, n, n, n))


@pytest.mark.parametrize("seed", range(4))
def test_closure_random(seed):
    rows, cols, _ = synth.random_small(80 + seed, 200, 200, 0.004 + 0.002 * seed)
    a = K.Tree(rows, cols, 200, 200)
    c, it = a.bool_closure()
    r, cc, it_ref = oracle.transitive_closure(rows, cols, 200)
    assert _cells(c) == _want(r, cc)
    assert it == it_ref


def test_product_edge_cases():
    z = np.zeros(0, np.uint32)
    e = K.Tree(z, z, 64, 64)
    one = np.array([3], np.uint32)
    a = K.Tree(one, np.array([5], np.uint32), 64, 64)
    assert _cells(e.bool_product(a)) == [] and _cells(a.bool_product(e)) == []
    b = K.Tree(np.array([5], np.uint32), np.array([9], np.uint32), 64, 64)
    assert _cells(a.bool_product(b)) == [(3, 9)]
    for bad in (K.Tree(one, one, 32, 64),                       # inner sizes differ
                K.Tree(one, one, 64, 200),                       # padded sides differ
                K.Tree(one, one, 64, 64, n_k4_levels=1),         # hybrid top
                K.Tree(one, one, 64, 64, leaf_k=4, cache_last_internal=1)):
        with pytest.raises(K.K2TError) as err:
            a.bool_product(bad)
        assert err.value.status == -1
