"""Host side of the library (no GPU): construction, planning, workspace, ABI.

The library's builder (path-key sort, bottom-up grouping) must produce the
same level-order bitstrings as the oracle's recursive subdivision, bit for
bit, for k = 2 and hybrid k = 4 / k = 2 trees, and decode to the edge set.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import synth

k2 = pytest.importorskip("compressed_graph_spmv_gb300")
from compressed_graph_spmv_gb300 import k2t as K  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib_bits(tree, level, n_k4, leaf_k=2):
    sig = tree.level_signatures(level)
    if level < n_k4 or (leaf_k == 4 and level == tree.stats().levels - 1):
        s16 = sig.reshape(-1, 2).astype(np.uint16)
        s16 = s16[:, 0] | (s16[:, 1] << 8)
        return np.unpackbits(s16.view(np.uint8), bitorder="little")
    return np.unpackbits(sig, bitorder="little").reshape(-1, 8)[:, :4].reshape(-1)


def _compare(rows, cols, n_rows, n_cols, n_k4=0, leaf_k=2, **kw):
    ot = oracle.OracleTree(rows, cols, n_rows, n_cols, n_k4=n_k4, leaf_k=leaf_k)
    if leaf_k == 4:
        kw = dict(kw, leaf_k=4, cache_last_internal=1)
    lt = K.Tree(rows, cols, n_rows, n_cols, n_k4_levels=n_k4, **kw)
    s = lt.stats()
    assert s.levels == ot.levels and s.dim_bits == ot.dim_bits and s.leaf_k == leaf_k
    bits = ot.bits()
    start = ot.level_start()
    for d in range(ot.levels):
        assert int(s.level_nodes[d]) == ot.level_nodes()[d]
        assert np.array_equal(_lib_bits(lt, d, n_k4, leaf_k), bits[start[d]:start[d + 1]]), d
    r, c = lt.decode()
    dr, dc = oracle.dedup_edges(rows, cols)
    assert sorted(zip(r.tolist(), c.tolist())) == sorted(zip(dr.tolist(), dc.tolist()))
    assert s.nnz == dr.size
    return lt


@pytest.mark.parametrize("seed", range(10))
def test_build_matches_oracle_random(seed):
    rng = np.random.default_rng(seed)
    n_rows = int(rng.integers(1, 300))
    n_cols = int(rng.integers(1, 300))
    n_k4 = int(rng.integers(0, 3))
    rows, cols, _ = synth.random_small(seed, n_rows, n_cols, float(rng.choice([0.001, 0.01, 0.1])))
    _compare(rows, cols, n_rows, n_cols, n_k4=n_k4)
    _compare(rows, cols, n_rows, n_cols, n_k4=n_k4, leaf_k=4)


@pytest.mark.parametrize("leaf_k", [2, 4])
def test_build_matches_oracle_rmat_threads(leaf_k):
    rows, cols = synth.rmat(14, 0.57, 0.19, 0.19, 100000, 3)
    a = _compare(rows, cols, 1 << 14, 1 << 14, leaf_k=leaf_k, threads=1)
    b = _compare(rows, cols, 1 << 14, 1 << 14, leaf_k=leaf_k, threads=7)
    for d in range(a.stats().levels):
        assert np.array_equal(a.level_signatures(d), b.level_signatures(d))


def test_build_figure1_leaf4():
    """The Figure 1 matrix with 4 x 4 leaves: two levels, root 1111, four
    16-bit leaves (the oracle's hand-derived pin), and the option errors."""
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "figure1.json")))
    e = np.array(g["edges_decoded"], np.uint32)
    t = _compare(e[:, 0], e[:, 1], 8, 8, leaf_k=4)
    s = t.stats()
    assert s.levels == 2 and s.l_bytes_device == 2 * 4 + 16
    assert t.level_signatures(1).view(np.uint16).tolist() == [1 << 5, 1 | 1 << 5 | 1 << 13,
                                                              1 << 5 | 1 << 6 | 1 << 9 | 1 << 10,
                                                              1 << 10 | 1 << 11 | 1 << 14 | 1 << 15]
    for bad in (dict(leaf_k=3, cache_last_internal=1), dict(leaf_k=4, engine=2),
                dict(leaf_k=4, engine=2, cache_last_internal=1), dict(leaf_k=4, engine=4, cache_last_internal=1)):
        with pytest.raises(K.K2TError) as err:
            K.Tree(e[:, 0], e[:, 1], 8, 8, **bad)
        assert err.value.status == -1, bad
    # the tree-only FUSED engine takes 4x4 leaves as well
    for ok in (dict(leaf_k=4), dict(leaf_k=4, engine=1)):
        assert K.Tree(e[:, 0], e[:, 1], 8, 8, **ok).stats().leaf_k == 4


def test_automatic_leaf_size():
    """leaf_k 0 (the default) picks 4x4 leaves when the 2x2 leaves would hold
    at least 1.75 non-zeros on average, on the engines that have them (FUSED,
    CACHED); the tree then equals the one built with leaf_k 4 explicitly."""
    wl = synth.clustered(scale=12, block=16, per_row=8, seed=3)    # 2x2 leaves hold ~2.1 non-zeros
    r, c = wl.rows, wl.cols
    n = 1 << 12
    for kw in (dict(), dict(cache_last_internal=1)):
        auto = K.Tree(r, c, n, n, **kw)
        four = K.Tree(r, c, n, n, leaf_k=4, **kw)
        assert auto.stats().leaf_k == 4 and auto.opts.leaf_k == 0
        for d in range(four.stats().levels):
            assert np.array_equal(auto.level_signatures(d), four.level_signatures(d))
    assert K.Tree(r, c, n, n, engine=2).stats().leaf_k == 2          # LEVELSYNC: 2x2 only
    assert K.Tree(r, c, n, n, leaf_k=2).stats().leaf_k == 2
    rr, cc = synth.rmat(12, 0.57, 0.19, 0.19, 30000, 4)               # ~1.03 per 2x2 leaf
    assert K.Tree(rr, cc, n, n).stats().leaf_k == 2


def test_build_figure1_and_top_level():
    import json
    g = json.load(open(os.path.join(ROOT, "tests", "golden", "figure1.json")))
    e = np.array(g["edges_decoded"], np.uint32)
    t = _compare(e[:, 0], e[:, 1], 8, 8)
    s = t.stats()
    # the deepest level with at most 2^16 nodes is the last internal one (3.4)
    assert s.d0 == 1


def test_empty_and_degenerate():
    z = np.zeros(0, np.uint32)
    t = K.Tree(z, z, 5, 3)
    s = t.stats()
    assert s.nnz == 0 and s.level_nodes[0] == 1 and s.dim_bits == 3
    assert t.level_signatures(0).tolist() == [0]
    one = np.array([0], np.uint32)
    _compare(one, one, 1, 1)
    _compare(np.array([3], np.uint32), np.array([0], np.uint32), 4, 1)


def test_errors():
    r = np.array([0, 5], np.uint32)
    c = np.array([0, 1], np.uint32)
    with pytest.raises(K.K2TError) as e:
        K.Tree(r, c, 5, 5)
    assert e.value.status == -2  # ERANGE
    with pytest.raises(K.K2TError) as e:
        K.Tree(r, c, 0, 5)
    assert e.value.status == -1
    with pytest.raises(K.K2TError) as e:
        K.Tree(r, c, 8, 8, engine=3, cache_last_internal=0)
    assert e.value.status == -1
    with pytest.raises(K.K2TError) as e:
        K.Tree(r, c, 8, 8, max_batch=33)
    assert e.value.status == -2
    with pytest.raises(K.K2TError) as e:
        K.Tree(r, c, 8, 8, chunk_cap=5000)
    with pytest.raises(K.K2TError) as e:
        K.Tree(r, c, 8, 8, chunk_cap=3)
    assert e.value.status == -1
    t = K.Tree(r, c, 8, 8)
    lib = K.load()
    # products before upload are out of order; no GPU needed to see that
    assert lib.k2t_spmv(t.handle, 0, 0, ctypes.c_float(1.0), 16, 32, 1, None) == -5
    assert lib.k2t_spmv(None, 0, 0, ctypes.c_float(1.0), 16, 32, 1, None) == -1
    assert lib.k2t_strerror(-3) == b"out of memory"


def _layout_parts(s):
    """Sum of the parts the statistics list; the heavy outputs' tables and
    sums are given in KiB (rounded up), so the sum may exceed the exact bytes
    by under 1 KiB."""
    return (s.t_bytes_device + s.l_bytes_device + s.dir_bytes + s.top_bytes + s.cached_bytes +
            s.plan_bytes + s.scratch_bytes + s.vector_bytes + 1024 * s.heavy_kib)


@pytest.mark.parametrize("engine", [1, 2, 3, 4])
def test_workspace_accounting(engine):
    rows, cols = synth.rmat(12, 0.57, 0.19, 0.19, 30000, 4)
    t = K.Tree(rows, cols, 4096, 4096, engine=engine, cache_last_internal=int(engine >= 3),
               host_vectors=1, max_batch=4, tile_m=4096, chunk_cap=512, host_top_max_nodes=64)
    s = t.stats()
    ws = t.workspace_bytes()
    assert ws == s.workspace_bytes
    parts = _layout_parts(s)
    # every part is placed at a 256-byte boundary: the total exceeds the sum of
    # the parts by the alignment padding only (plus the 64-byte status word)
    nparts = 4 * s.levels + 20
    assert parts - 1024 <= ws <= parts + 256 * nparts + 256
    assert s.vector_bytes == 2 * 4096 * 4 * 4
    if engine == 1:
        assert s.n_chunks > 1 and s.plan_bytes > 0 and s.scratch_bytes == 0
    if engine == 2:
        assert s.n_steps > 1 and s.scratch_bytes > 0
    if engine == 3:
        assert s.cached_bytes == 8 * s.level_nodes[s.levels - 2] + 16
    if engine == 4:
        n2 = s.level_nodes[s.levels - 2]
        assert s.cached_bytes == (8 * n2 + 16) + (4 * n2 + 16) + ((n2 + 1) // 2 + 16)


def test_options_struct_matches_header():
    """The binding's k2t_opts mirrors the header: defaults round-trip."""
    o = K.default_opts()
    assert o.band_rows == 4096 and o.chunk_cap == 256 and o.tile_m == 1 << 20 and o.max_batch == 32
    assert o.heavy_terms == 160 and o.leaf_k == 0
    # sizes and field offsets as a C compiler lays the header's structs out
    import subprocess
    import tempfile
    probe = "\n".join([
        "#include <stddef.h>", "#include <stdio.h>", "#include \"k2t.h\"",
        "int main(void) {",
        "  printf(\"%zu %zu %zu %zu %zu\\n\", sizeof(k2t_opts), sizeof(k2t_stats),",
        "         offsetof(k2t_opts, leaf_k), offsetof(k2t_stats, leaf_k), offsetof(k2t_stats, heavy_partials));",
        "  return 0; }"])
    with tempfile.TemporaryDirectory() as d:
        src, exe = os.path.join(d, "p.c"), os.path.join(d, "p")
        with open(src, "w") as f:
            f.write(probe)
        subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), src, "-o", exe], check=True)
        got = [int(v) for v in subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split()]
    assert got == [ctypes.sizeof(K.Opts), ctypes.sizeof(K.Stats), K.Opts.leaf_k.offset, K.Stats.leaf_k.offset,
                   K.Stats.heavy_partials.offset]
    with pytest.raises(K.K2TError):
        K.Tree(np.zeros(1, np.uint32), np.zeros(1, np.uint32), 8, 8, engine=4, cache_last_internal=1,
               band_rows=100)


def test_banded_layout():
    rows, cols = synth.rmat(12, 0.57, 0.19, 0.19, 30000, 8)
    a = K.Tree(rows, cols, 4096, 4096, engine=4, cache_last_internal=1, band_rows=64)
    b = K.Tree(rows, cols, 4096, 4096, engine=3, cache_last_internal=1)
    sa, sb = a.stats(), b.stats()
    assert sa.engine == 4 and sb.engine == 3
    assert sa.plan_bytes > 0 and sa.level_nodes[sa.levels - 2] == sb.level_nodes[sb.levels - 2]


def test_chunk_plan_covers_every_node():
    """Fused plan: chunks are whole subtrees; together they cover each level
    below the host-expanded top exactly once, in level order."""
    rows, cols = synth.rmat(13, 0.57, 0.19, 0.19, 60000, 6)
    for cap in (4, 7, 256, 512):
        t = K.Tree(rows, cols, 8192, 8192, engine=1, chunk_cap=cap)
        h = t.handle
        s = t.stats()
        # read the chunk table through the host copy in the planner's layout
        stride = 2 + 2 * (s.levels - s.d0)
        assert s.plan_bytes >= s.n_chunks * stride * 4


def test_library_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "k2t.h")).read()
    declared = set(re.findall(r"\b(k2t_[a-z_]+)\s*\(", header))
    lib = K.load()
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(K.EXPORTED)
    # the bounds-checked build exports the same ABI
    import ctypes
    checked = ctypes.CDLL(K.CHECKED_LIB_PATH)
    for name in declared:
        assert hasattr(checked, name), name


def test_libraries_export_only_the_c_api():
    """Both builds export the declared calls and no k2t C++ symbol (hidden
    visibility), so the two can be loaded into one process without their
    template instances and function-local state binding to each other."""
    import shutil
    import subprocess
    nm = shutil.which("nm")
    if nm is None:
        pytest.skip("nm not installed")
    for path in (K.LIB_PATH, K.CHECKED_LIB_PATH):
        out = subprocess.run([nm, "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
        names = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
        assert set(K.EXPORTED) <= names, path
        assert not [n for n in names if "3k2t" in n], path   # no mangled k2t:: symbol


@pytest.mark.parametrize("heavy_terms", [0, 5, 30, 0xFFFFFFFF])
def test_heavy_outputs_stats(heavy_terms):
    """Heavy outputs are those with more than heavy_terms non-zeros in the
    input list (0 selects the default 160).  Per direction with any, their
    tables take one word per heavy output (the list) and one record word per
    output up to the last heavy one (padded for a 16-byte read); the sums
    take, for the direction with more, rows of max_batch fp32
    words: 2^bits partial sums per heavy output, or two rows of fp64 slot for
    an output summed in fp64."""
    rng = np.random.default_rng(21)
    nr, nc = 300, 200
    rows, cols, _ = synth.random_small(3, nr, nc, 0.05)
    hub_r = np.full(150, 7, np.uint32)
    hub_c = rng.integers(0, nc, size=150).astype(np.uint32)
    rows = np.concatenate([rows, hub_r, rng.integers(0, nr, size=120).astype(np.uint32)])
    cols = np.concatenate([cols, hub_c, np.full(120, 11, np.uint32)])
    t = K.Tree(rows, cols, nr, nc, heavy_terms=heavy_terms, max_batch=4)
    s = t.stats()
    lim = 160 if heavy_terms == 0 else heavy_terms
    cr, cc = np.bincount(rows, minlength=nr), np.bincount(cols, minlength=nc)
    hr = int((cr > lim).sum()) if rows.size > lim else 0
    hc = int((cc > lim).sum()) if rows.size > lim else 0
    assert (s.heavy_rows, s.heavy_cols) == (hr, hc)
    if heavy_terms == 5:
        assert hr > 1 and hc > 1
    if heavy_terms == 30:
        assert hr >= 1 and hc >= 1
    if heavy_terms == 0:
        assert hr == 1 and hc == 0   # the 150-entry hub row, with the random entries of row 7
    tables = 0
    acc_rows = 0
    for d, (h, cnt) in enumerate(((hr, cr), (hc, cc))):
        if h:
            last = int(np.nonzero(cnt > lim)[0].max())
            hdir = ((last + 1 + 3) // 4 * 4 + 4) * 4
            tables += 4 * h + hdir
            acc_rows = max(acc_rows, int(s.heavy_partials[d]) + 2 * int(s.heavy_fp64[d]))
    want = tables + acc_rows * 4 * 4
    assert s.heavy_kib == (want + 1023) // 1024
    if hr:
        # every heavy output is split into at least two partial sums of at most
        # the limit's terms, or (when one run of 32 inputs already holds more)
        # summed in fp64
        assert s.heavy_partials[0] >= 2 * (hr - s.heavy_fp64[0])
        assert s.heavy_max_terms[0] <= lim and (s.heavy_max_terms[0] > 0 or s.heavy_fp64[0] == hr)
    base = K.Tree(rows, cols, nr, nc, heavy_terms=0xFFFFFFFF, max_batch=4).workspace_bytes()
    assert want <= t.workspace_bytes() - base <= want + 6 * 256
    f64 = K.Tree(rows, cols, nr, nc, heavy_terms=heavy_terms, heavy_mode=1, max_batch=4).stats()
    assert list(f64.heavy_partials) == [0, 0] and list(f64.heavy_fp64) == [hr, hc]
    assert f64.heavy_kib == (tables + 2 * max(hr, hc) * 4 * 4 + 1023) // 1024   # fp64 mode: two rows each
    with pytest.raises(K.K2TError):
        K.Tree(rows, cols, nr, nc, heavy_mode=2)


def test_product_argument_errors_on_host():
    """k2t_bool_product / k2t_bool_closure reject mismatched or unsupported
    trees before touching the device (no GPU needed)."""
    lib = K.load()
    import ctypes
    one = np.array([3], np.uint32)
    a = K.Tree(one, one, 64, 64)
    out = ctypes.c_void_p()
    it = ctypes.c_uint32()
    o = K.default_opts()
    for bad in (K.Tree(one, one, 32, 64),                    # inner sizes differ
                K.Tree(one, one, 64, 200),                    # padded sides differ
                K.Tree(one, one, 64, 64, n_k4_levels=1),      # hybrid top
                K.Tree(one, one, 64, 64, leaf_k=4, cache_last_internal=1)):
        assert lib.k2t_bool_product(a.handle, bad.handle, ctypes.byref(o), ctypes.byref(out), None) == -1
        assert not out.value
    assert lib.k2t_bool_product(None, a.handle, ctypes.byref(o), ctypes.byref(out), None) == -1
    rect = K.Tree(one, one, 64, 32)
    assert lib.k2t_bool_closure(rect.handle, ctypes.byref(o), 8, ctypes.byref(out), ctypes.byref(it), None) == -1
    assert lib.k2t_bool_closure(a.handle, ctypes.byref(o), 8, ctypes.byref(out), None, None) == -1


def test_bench_traffic_follows_device_sources(monkeypatch):
    """roofline.traffic is reported only for the workload the capture was
    taken on (traffic does not scale with the edges) and only while the
    device sources match the digest of that capture."""
    import bench
    table = bench.MEASURED_TRAFFIC
    monkeypatch.setitem(table, "digest", bench.device_digest())
    monkeypatch.setitem(table, "workload", "rmat27-bfs-1200M")
    monkeypatch.setitem(table, "nnz", 4000)
    monkeypatch.setitem(table, "bytes", {"right B=1": 123000})
    assert bench.measured_traffic("rmat27-bfs-1200M", 4000, "right B=1")[0] == 123000
    assert bench.measured_traffic("rmat27-bfs-1200M", 4000, "left B=1")[0] is None
    assert bench.measured_traffic("rmat24-bfs-150M", 1000, "right B=1")[0] is None
    assert bench.measured_traffic("weblike22", 4000, "right B=1")[0] is None
    monkeypatch.setitem(table, "digest", "0" * 64)
    assert bench.measured_traffic("rmat27-bfs-1200M", 4000, "right B=1")[0] is None


def test_clustered_generator_shape():
    """synth.clustered: every row holds exactly per_row distinct columns, all
    inside its own block-aligned window (block-diagonal), seeded."""
    wl = synth.clustered(scale=12, block=16, per_row=8, seed=3)
    n = 1 << 12
    assert wl.rows.size == 8 * n and wl.n_rows == n == wl.n_cols
    assert np.all(wl.cols // 16 == wl.rows // 16)
    r, c = oracle.dedup_edges(wl.rows, wl.cols)
    assert r.size == wl.rows.size                                   # distinct per row
    assert np.array_equal(np.bincount(r, minlength=n), np.full(n, 8))
    again = synth.clustered(scale=12, block=16, per_row=8, seed=3)
    assert np.array_equal(again.cols, wl.cols)


@pytest.mark.parametrize("leaf_k", [2, 4])
def test_largest_side(leaf_k):
    """n = 2^32 (the largest side): 32 levels (31 with 4x4 leaves), cells at
    the four corners and near the middle decode back, and match the oracle's
    tree bit for bit."""
    top = (1 << 32) - 1
    rows = np.array([0, top, 0, top, 1 << 31, 12345], np.uint32)
    cols = np.array([0, 0, top, top, (1 << 31) - 1, 1 << 30], np.uint32)
    t = _compare(rows, cols, 1 << 32, 1 << 32, leaf_k=leaf_k)
    s = t.stats()
    assert s.dim_bits == 32 and s.levels == 32 - (leaf_k == 4) and s.nnz == 6
    with pytest.raises(K.K2TError) as e:
        K.Tree(rows, cols, (1 << 32) + 1, 4)
    assert e.value.status == -2


def test_device_digest_ignores_comments_only():
    """The digest keying roofline.traffic changes with code, not with comments
    or layout."""
    import bench
    a = bench._code_only("int f(int x) { // add one\n  return x + 1; /* done */ }\n")
    b = bench._code_only("int f(int x)\n{\n    return x + 1;\n}")
    c = bench._code_only("int f(int x) { return x + 2; }")
    assert a == b != c


@pytest.mark.parametrize("leaf_k", [2, 4])
def test_heavy_outputs_bounded_partials(leaf_k):
    """Plus-times outputs with more than heavy_terms non-zeros (counted over
    the input list) are heavy, and the builder splits each into fp32 partial
    sums that receive at most heavy_terms terms: the largest count it found
    is at most the limit, and the partials number at least the heavy terms
    divided by the limit."""
    rows, cols = synth.rmat(14, 0.57, 0.19, 0.19, 400000, 21)
    n = 1 << 14
    kw = dict(cache_last_internal=1, leaf_k=4) if leaf_k == 4 else {}
    for limit in (160, 40):
        t = K.Tree(rows, cols, n, n, heavy_terms=limit, **kw)
        s = t.stats()
        for d, ids in ((0, rows), (1, cols)):
            cnt = np.bincount(ids, minlength=n)
            heavy = cnt > limit
            assert (s.heavy_rows, s.heavy_cols)[d] == int(heavy.sum())
            assert s.heavy_fp64[d] == 0
            assert 0 < s.heavy_max_terms[d] <= limit
            assert s.heavy_partials[d] >= int(cnt[heavy].sum()) / limit
    # fp64 mode: every heavy output has an fp64 slot and no partial sums
    t = K.Tree(rows, cols, n, n, heavy_mode=1, **kw)
    s = t.stats()
    assert s.heavy_fp64[0] == s.heavy_rows > 0 and s.heavy_partials[0] == 0
    # no heavy outputs at all
    s = K.Tree(rows, cols, n, n, heavy_terms=0xffffffff, **kw).stats()
    assert s.heavy_rows == s.heavy_cols == 0 and s.heavy_kib == 0


def test_status_needs_upload():
    """k2t_status on a tree that was never uploaded is out of order (no GPU
    call is made)."""
    rows, cols = synth.rmat(8, 0.57, 0.19, 0.19, 500, 42)
    t = K.Tree(rows, cols, 256, 256)
    with pytest.raises(K.K2TError) as e:
        t.status()
    assert e.value.status == -5
    assert K.load().k2t_strerror(-7) == b"device-side wait ran out"


def test_bench_oracle_sample_takes_whole_random_bands():
    """The CPU baseline's sample: every non-zero of the chosen 2^band_bits-row
    bands and nothing else, bands drawn uniformly (not the leading hub rows),
    about the target edge count."""
    import bench
    wl = synth.rmat_c2(scale=14, edges_per_vertex=8, seed=3)
    r, c, desc = bench.oracle_sample(wl, 20000, band_bits=6, seed=17)
    bands = np.unique(r >> 6)
    rows_in = np.isin(wl.rows >> 6, bands)
    assert r.size == int(rows_in.sum())                      # whole bands
    assert set(zip(r.tolist(), c.tolist())) == set(zip(wl.rows[rows_in].tolist(), wl.cols[rows_in].tolist()))
    assert 20000 <= r.size <= 20000 + int(np.bincount(wl.rows >> 6).max())
    nb = (wl.n_rows + 63) >> 6
    assert bands.max() > nb // 2 and bands.min() < nb // 2   # spread over the id range
    assert "random row bands" in desc


def test_bench_algorithmic_bytes_formula():
    """A product's algorithmic bytes: the tree parts its engine reads, x read
    once (4 bytes a vector entry) and y read and written once (8 bytes);
    Boolean vectors take one word whatever B."""
    import bench
    rows, cols = synth.rmat(10, 0.57, 0.19, 0.19, 6000, 4)
    s = K.Tree(rows, cols, 1024, 768 + 256, cache_last_internal=1).stats()
    tree = s.t_bytes_device + s.l_bytes_device + s.dir_bytes + s.top_bytes + s.cached_bytes + s.plan_bytes
    assert bench.algorithmic_bytes(s, synth.PLUS_TIMES, 0, 16) == tree + 4 * s.n_cols * 16 + 8 * s.n_rows * 16
    assert bench.algorithmic_bytes(s, synth.BOOLEAN, 1, 32) == tree + 4 * s.n_rows + 8 * s.n_cols
