"""The device status word: kernels set bits in the first word of a tree's
arena instead of trapping (bit 0: a bounded wait ran out; bit 1: a checked
build found an index out of range), and synchronising calls map a set word
to K2T_ETIMEOUT / K2T_EDEVICE until k2t_status clears it.

The failure is injected from the host: the test owns the arena (a torch
buffer passed to k2t_upload) and writes the bit into its first word.  No
kernel is made to time out and no GPU is faulted."""
import numpy as np
import pytest

import oracle
import synth
from gpu_util import assert_match

pytestmark = pytest.mark.gpu

K = pytest.importorskip("compressed_graph_spmv_gb300.k2t")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K.load()


@pytest.mark.parametrize("bit, code", [(K.STATUS_WAIT_TIMEOUT, -7), (K.STATUS_OUT_OF_RANGE, -6)])
def test_status_word_is_reported_and_cleared(bit, code):
    import torch
    n = 4096
    rows, cols = synth.rmat(12, 0.57, 0.19, 0.19, 20000, 41)
    t = K.Tree(rows, cols, n, n, host_vectors=1, max_batch=1)
    arena = torch.zeros(t.workspace_bytes(), dtype=torch.uint8, device="cuda")
    t.upload(arena)
    x = np.random.default_rng(41).uniform(0, 1, size=(n, 1)).astype(np.float32)
    y = np.zeros((n, 1), np.float32)
    ref = oracle.spmv_edges(rows, cols, n, n, oracle.RIGHT, oracle.PLUS_TIMES, x)
    t.spmv_host(oracle.RIGHT, oracle.PLUS_TIMES, x, y)
    assert t.status() == 0
    assert_match(oracle.PLUS_TIMES, y, ref, "before")
    # a kernel would have set the bit: write it into the arena's first word
    arena[0] = bit
    torch.cuda.synchronize()
    for _ in range(2):   # sticky until cleared
        with pytest.raises(K.K2TError) as e:
            t.spmv_host(oracle.RIGHT, oracle.PLUS_TIMES, x, y)
        assert e.value.status == code
        assert t.status() == bit
    # multi-source search reads the word after its first level
    sq = K.Tree(rows, cols, n, n, cache_last_internal=1)
    sq_arena = torch.zeros(sq.workspace_bytes(), dtype=torch.uint8, device="cuda")
    sq.upload(sq_arena)
    sq_arena[0] = bit
    dist = torch.empty(n, dtype=torch.int32, device="cuda")
    work = torch.empty(sq.msbfs_work_bytes(), dtype=torch.uint8, device="cuda")
    with pytest.raises(K.K2TError) as e:
        sq.msbfs(oracle.RIGHT, [int(rows[0])], dist, work, max_levels=4)
    assert e.value.status == code
    assert sq.status(clear=True) == bit and sq.status() == 0
    # clearing restores normal service
    assert t.status(clear=True) == bit
    assert t.status() == 0
    y[:] = -1.0
    t.spmv_host(oracle.RIGHT, oracle.PLUS_TIMES, x, y)
    assert_match(oracle.PLUS_TIMES, y, ref, "after clear")
