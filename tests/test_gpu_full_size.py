"""GPU parity at the workloads' full sizes, in the bench's configuration:
every product of a workload is run once through the C ABI and 2048 sampled
outputs per product are compared with the oracle's definition evaluated one
output at a time (bit-exact for Boolean and tropical, the fp32 bound for
plus-times, as stated in tests/gpu_util.py).  The 1.2 G-edge workload is
generated on the host (about 80 s on 16 cores)."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_match

pytestmark = pytest.mark.gpu

K = pytest.importorskip("compressed_graph_spmv_gb300.k2t")

WORKLOADS = {
    "uniform-1024": (lambda: synth.uniform_c1(), dict(), [(0, 1), (1, 1)]),
    "rmat20": (lambda: synth.rmat_c2(), dict(), [(0, 1), (1, 1)]),
    "weblike22": (lambda: synth.weblike_c3(), dict(n_k4_levels=2), [(0, 32), (1, 32)]),
    "social24": (lambda: synth.social_c4(), dict(), [(0, 8)]),
    "rmat27": (lambda: synth.large_c5(B=16), dict(cache_last_internal=1), [(0, 1), (1, 1), (0, 16), (1, 16)]),
    # 4x4 leaves (section 5.6) on the cached engine
    "rmat20-leaf4": (lambda: synth.rmat_c2(), dict(cache_last_internal=1, leaf_k=4), [(0, 1), (1, 1)]),
    "weblike22-leaf4": (lambda: synth.weblike_c3(), dict(n_k4_levels=2, cache_last_internal=1, leaf_k=4),
                        [(0, 32), (1, 32)]),
    "social24-leaf4": (lambda: synth.social_c4(), dict(cache_last_internal=1, leaf_k=4), [(0, 8)]),
    "clustered22": (lambda: synth.clustered(), dict(cache_last_internal=1, leaf_k=2), [(0, 1), (1, 1)]),
    "clustered22-leaf4": (lambda: synth.clustered(), dict(cache_last_internal=1, leaf_k=4), [(0, 1), (1, 1)]),
    # tree-only with the automatic leaf size: 4x4 leaves on the FUSED engine
    "clustered22-fused-auto": (lambda: synth.clustered(), dict(), [(0, 1), (1, 1)]),
    "rmat20-fused-leaf4": (lambda: synth.rmat_c2(), dict(leaf_k=4), [(0, 1), (1, 1)]),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K.load()


def _vector(wl, d, B):
    x = wl.xs[d]
    if wl.semiring == synth.BOOLEAN:
        return np.ascontiguousarray(x, dtype=np.uint32)
    return np.ascontiguousarray(x[:, :B], dtype=np.float32)


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_full_size_sampled_parity(name):
    import torch
    make, opts, products = WORKLOADS[name]
    wl = make()
    tree = K.Tree(wl.rows, wl.cols, wl.n_rows, wl.n_cols, max_batch=max(b for _, b in products), **opts).upload()
    rng = np.random.default_rng(123)
    boolean = wl.semiring == synth.BOOLEAN
    for d, B in products:
        xv = _vector(wl, d, B)
        n_out = wl.n_rows if d == 0 else wl.n_cols
        if boolean:
            x = torch.from_numpy(xv.view(np.int32)).cuda()
            y = torch.empty(n_out, dtype=torch.int32, device="cuda")
        else:
            x = torch.from_numpy(xv).cuda()
            y = torch.empty(n_out, B, dtype=torch.float32, device="cuda")
        tree.spmv(d, wl.semiring, x, y, B=B, w=wl.w)
        torch.cuda.synchronize()
        got = y.cpu().numpy()
        got = got.view(np.uint32) if boolean else got
        sample = np.unique(np.concatenate([rng.integers(0, n_out, size=2040), [0, 1, n_out - 2, n_out - 1]]))
        ref = oracle.rows_product(wl.rows, wl.cols, wl.n_rows, wl.n_cols, d, wl.semiring, xv, sample, B=B, w=wl.w)
        assert_match(wl.semiring, got[sample], ref, "%s dir %d B %d" % (name, d, B))
        del x, y
    tree.close()
