"""k2t_spmv_noalloc: the level-synchronous product for callers that cannot
call cudaMalloc (a framework that owns all device memory through its own
pool, code that must not synchronise the device, a memory budget fixed in
advance).  Its frontier buffers live in a static device array of the library,
so it must give the same results as k2t_spmv on the same tree, call after
call, while the array keeps whatever the previous call left in it.

This file is named so that pytest collects it after every other test file.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_match, random_x

pytestmark = pytest.mark.gpu

K = pytest.importorskip("compressed_graph_spmv_gb300.k2t")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K.load()


def _product(tree, fn, direction, semiring, x_np, B, n_in, n_out):
    import torch
    if semiring == oracle.BOOLEAN:
        x = torch.from_numpy(x_np.view(np.int32).reshape(n_in)).cuda()
        y = torch.full((n_out,), -1, dtype=torch.int32, device="cuda")
    else:
        x = torch.from_numpy(x_np.reshape(n_in, B)).cuda()
        y = torch.full((n_out, B), float("nan"), dtype=torch.float32, device="cuda")
    getattr(tree, fn)(direction, semiring, x, y, B=B)
    torch.cuda.synchronize()
    out = y.cpu().numpy()
    return out.view(np.uint32) if semiring == oracle.BOOLEAN else out


def _scribble(offsets):
    """Run the allocation-free product on a tree of another shape (other
    graph, other tile size, other offset source), so the static array holds
    that tree's frontier coordinates and scan sums, not the ones the next
    call needs."""
    n = 1 << 13
    r, c = synth.rmat(13, 0.45, 0.15, 0.15, 60000, 5)
    other = K.Tree(r, c, n, n, engine=K.ENGINE_LEVELSYNC, offsets=1 - offsets, tile_m=64,
                   host_top_max_nodes=16).upload()
    x = np.random.default_rng(5).integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    _product(other, "spmv_noalloc", oracle.RIGHT, oracle.BOOLEAN, x, 32, n, n)


@pytest.mark.parametrize("offsets", [0, 1])
def test_noalloc_matches_spmv_twice(offsets):
    n = 1 << 14
    rows, cols = synth.rmat(14, 0.57, 0.19, 0.19, 200000, 21)
    tree = K.Tree(rows, cols, n, n, engine=K.ENGINE_LEVELSYNC, offsets=offsets, tile_m=4096,
                  host_top_max_nodes=256).upload()
    assert tree.stats().n_steps > 4
    rng = np.random.default_rng(21)
    for semiring, B in ((oracle.PLUS_TIMES, 1), (oracle.BOOLEAN, 32), (oracle.TROPICAL, 4)):
        for direction in (oracle.RIGHT, oracle.LEFT):
            x = random_x(rng, semiring, n, B)
            ref = oracle.spmv_edges(rows, cols, n, n, direction, semiring, x, B=B)
            want = _product(tree, "spmv", direction, semiring, x, B, n, n)
            for call in range(2):
                if call == 0:
                    _scribble(offsets)
                got = _product(tree, "spmv_noalloc", direction, semiring, x, B, n, n)
                if semiring == oracle.PLUS_TIMES:
                    # both within the fp32 bound of the exact product
                    assert_match(semiring, got, ref, "noalloc call %d" % call)
                    assert_match(semiring, want, ref, "spmv")
                else:
                    assert np.array_equal(got, want), "call %d" % call


def test_noalloc_limits():
    lib = K.load()
    limit = int(lib.k2t_noalloc_scratch_limit())
    assert limit == 64 << 20
    n = 1 << 20
    rows, cols = synth.rmat(20, 0.57, 0.19, 0.19, 16 << 20, 22)
    # tiles of 2^22 children: the frontier buffers exceed the static array
    big = K.Tree(rows, cols, n, n, engine=K.ENGINE_LEVELSYNC, tile_m=1 << 22).upload()
    assert big.stats().scratch_bytes > limit
    import torch
    x = torch.rand(n, 1, device="cuda")
    y = torch.empty(n, 1, device="cuda")
    with pytest.raises(K.K2TError) as e:
        big.spmv_noalloc(0, 0, x, y)
    assert e.value.status == -2
    # another engine is not served by this entry point
    fused = K.Tree(rows[:1000], cols[:1000], n, n).upload()
    assert lib.k2t_spmv_noalloc(fused.handle, 0, 0, ctypes.c_float(1.0), x.data_ptr(), y.data_ptr(), 1,
                                None) == -5
    # sizes past what the array holds are refused before any launch; a tree
    # that fits still runs after the refusal
    small = K.Tree(rows, cols, n, n, engine=K.ENGINE_LEVELSYNC, tile_m=1 << 16).upload()
    assert small.stats().scratch_bytes <= limit
    small.spmv_noalloc(0, 0, x, y)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
