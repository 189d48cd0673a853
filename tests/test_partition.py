"""Row-band (right) / column-band (left) partition of a product over ranks.

A k^2-tree product shards without a collective per product: rank r owns the
rows [r*n/R, (r+1)*n/R) (right product) or the columns (left product), builds
the tree of its band and computes its slice of y; an iterative user would
all-gather the slices into the next x.  Checked here with two gloo ranks on
CPU: the gathered band products equal the full product, and each rank's
library-built band tree (host build, no GPU) decodes to its band's edges.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    import oracle
    import synth
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n = 1 << 11
        rows, cols = synth.rmat(11, 0.57, 0.19, 0.19, 20000, 31)
        rng = np.random.default_rng(31)
        x = rng.uniform(0, 1, size=(n, 2)).astype(np.float32)
        ok = True
        for direction in (oracle.RIGHT, oracle.LEFT):
            key = rows if direction == oracle.RIGHT else cols
            lo, hi = rank * n // world, (rank + 1) * n // world
            sel = (key >= lo) & (key < hi)
            r, c = rows[sel], cols[sel]
            if direction == oracle.RIGHT:
                t = oracle.OracleTree(r - lo, c, hi - lo, n)
                part = t.spmv(direction, oracle.PLUS_TIMES, x, B=2).y
            else:
                t = oracle.OracleTree(r, c - lo, n, hi - lo)
                part = t.spmv(direction, oracle.PLUS_TIMES, x, B=2).y
            chunks = [torch.zeros(((k + 1) * n // world - k * n // world, 2), dtype=torch.float64)
                      for k in range(world)]
            dist.all_gather(chunks, torch.from_numpy(np.ascontiguousarray(part)))
            full = torch.cat(chunks).numpy()
            ref = oracle.spmv_edges(rows, cols, n, n, direction, oracle.PLUS_TIMES, x, B=2).y
            ok &= bool(np.allclose(full, ref, rtol=1e-12, atol=1e-12))
            # the library's own host build of the band: it decodes to exactly
            # the band's distinct edges, and the bands' non-zeros add up
            from compressed_graph_spmv_gb300 import k2t as K
            if direction == oracle.RIGHT:
                band = K.Tree(r - lo, c, hi - lo, n, cache_last_internal=1)
                want = oracle.dedup_edges(r - lo, c)
            else:
                band = K.Tree(r, c - lo, n, hi - lo, cache_last_internal=1)
                want = oracle.dedup_edges(r, c - lo)
            dr, dc = band.decode()
            got = oracle.dedup_edges(dr, dc)
            ok &= bool(np.array_equal(got[0], want[0]) and np.array_equal(got[1], want[1]))
            cnt = torch.tensor([int(band.stats().nnz)], dtype=torch.int64)
            dist.all_reduce(cnt)
            ok &= int(cnt.item()) == int(oracle.dedup_edges(rows, cols)[0].size)
        q.put((rank, ok))
    finally:
        dist.destroy_process_group()


def test_band_partition_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    results = dict(q.get(timeout=5) for _ in procs)
    assert all(p.exitcode == 0 for p in procs)
    assert results == {0: True, 1: True}


def _turns_worker(rank, world, port, q):
    import sys
    import time
    import torch.distributed as dist
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        def work():
            t0 = time.time()
            time.sleep(0.3)
            return (t0, time.time())
        q.put((rank, bench.one_at_a_time(rank, world, dist.group.WORLD, work)))
    finally:
        dist.destroy_process_group()


def test_replicas_prepare_one_at_a_time():
    """bench.py's replicas generate and build in turn: rank r's turn starts
    only after rank r-1's has ended (two gloo ranks on CPU)."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_turns_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    spans = dict(q.get(timeout=5) for _ in procs)
    assert all(p.exitcode == 0 for p in procs)
    assert spans[0][1] <= spans[1][0]
