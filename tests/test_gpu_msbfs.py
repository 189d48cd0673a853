"""GPU multi-source search (k2t_msbfs) against the oracle's level-synchronous
search: distance tables must match exactly, for both directions and several
engines, with repeated sources and a level cap."""
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


def _run(tree, direction, sources, n, max_levels=1 << 30):
    import torch
    dist = torch.empty(n * len(sources), dtype=torch.int32, device="cuda")
    work = torch.empty(tree.msbfs_work_bytes(), dtype=torch.uint8, device="cuda")
    levels = tree.msbfs(direction, sources, dist, work, max_levels=max_levels)
    torch.cuda.synchronize()
    return dist.cpu().numpy().reshape(n, len(sources)), levels


@pytest.mark.parametrize("kw", [dict(engine=1), dict(engine=2, tile_m=512),
                                dict(engine=3, cache_last_internal=1), dict(engine=4, cache_last_internal=1)])
def test_msbfs_matches_oracle(kw):
    n = 1 << 13
    rows, cols = synth.rmat(13, 0.57, 0.19, 0.19, 40000, 41)
    tree = K.Tree(rows, cols, n, n, host_top_max_nodes=64, **kw).upload()
    rng = np.random.default_rng(41)
    for direction in (K.RIGHT, K.LEFT):
        sources = rng.choice(n, size=32, replace=True)
        got, levels = _run(tree, direction, sources, n)
        want = oracle.msbfs(rows, cols, n, sources, direction)
        assert np.array_equal(got, want)
        assert levels == int(want.max()) + 1
        got, levels = _run(tree, direction, sources[:7], n, max_levels=2)
        assert np.array_equal(got, oracle.msbfs(rows, cols, n, sources[:7], direction, max_levels=2))
        assert levels == 2


def test_msbfs_errors():
    import torch
    rows, cols = synth.rmat(8, 0.57, 0.19, 0.19, 500, 42)
    tree = K.Tree(rows, cols, 256, 256).upload()
    dist = torch.empty(256 * 2, dtype=torch.int32, device="cuda")
    work = torch.empty(tree.msbfs_work_bytes(), dtype=torch.uint8, device="cuda")
    with pytest.raises(K.K2TError) as e:
        tree.msbfs(K.RIGHT, [0, 256], dist, work)
    assert e.value.status == -2
    rect = K.Tree(rows[:10] % 100, cols[:10], 100, 256).upload()
    with pytest.raises(K.K2TError) as e:
        rect.msbfs(K.RIGHT, [0], dist, work)
    assert e.value.status == -1
