"""Benchmark: edges/s of k^2-tree semiring SpMV (right and left) on one GB300,
with the achieved HBM bandwidth of the product kernel against the measured
peak, an end-to-end figure through host buffers, and the CPU oracle timed
on a bounded sample of the same workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one pass of the hot path over the workload: the right and the
left product (for the large R-MAT workload also the 16-vector batch), each
a fill of y plus the product kernel.  Inputs are resident in HBM when the
timed region starts; L2 is flushed between steps when the working set is
smaller than four times L2.  Under torchrun every rank runs an independent
replica (no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import resource
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "edges/s per k²-tree SpMV (right & left) on 1 GB300; achieved HBM GB/s vs peak"


# --- workloads ----------------------------------------------------------------
def make_workload(name: str):
    """(Workload, library options, list of (dir, B) products per step)."""
    if name == "uniform-1024":
        wl = synth.uniform_c1()
        return wl, dict(), [(0, 1), (1, 1)]
    if name == "uniform20":
        wl = synth.uniform_large()
        return wl, dict(), [(0, 1), (1, 1)]
    if name == "rmat20":
        wl = synth.rmat_c2()
        return wl, dict(), [(0, 1), (1, 1)]
    if name == "weblike22":
        wl = synth.weblike_c3()
        return wl, dict(n_k4_levels=2), [(0, 32), (1, 32)]
    if name == "social24":
        wl = synth.social_c4()
        return wl, dict(), [(0, 8)]
    if name == "clustered22":
        wl = synth.clustered()
        return wl, dict(cache_last_internal=1), [(0, 1), (1, 1)]
    if name.startswith("rmat27"):
        wl = synth.large_c5(B=16)
        return wl, dict(cache_last_internal=1), [(0, 1), (1, 1), (0, 16), (1, 16)]
    if name.startswith("rmat"):   # rmatS: the large recipe at a smaller scale (tests, profiles)
        scale = int(name[4:])
        wl = synth.large_c5(scale=scale, edges=int(1.2e9 * (1 << scale) / (1 << 27)), B=16)
        return wl, dict(cache_last_internal=1), [(0, 1), (1, 1), (0, 16), (1, 16)]
    raise SystemExit("unknown workload %r" % name)


def vector(wl, direction, B):
    x = wl.xs[direction]
    if wl.semiring == synth.BOOLEAN:
        return np.ascontiguousarray(x, dtype=np.uint32)
    return np.ascontiguousarray(x[:, :B], dtype=np.float32)


# --- clocks -------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


class RawEvents:
    """CUDA runtime events through ctypes: the library records one of them
    itself (k2t_spmv_marked), which torch.cuda.Event cannot observe."""

    def __init__(self):
        import ctypes
        import ctypes.util
        lib = None
        for name in ("libcudart.so.13", "libcudart.so", ctypes.util.find_library("cudart")):
            if not name:
                continue
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None:
            raise RuntimeError("libcudart not found")
        self.c = ctypes
        self.lib = lib
        lib.cudaEventCreate.argtypes = [ctypes.POINTER(ctypes.c_void_p)]
        lib.cudaEventRecord.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
        lib.cudaEventElapsedTime.argtypes = [ctypes.POINTER(ctypes.c_float), ctypes.c_void_p, ctypes.c_void_p]
        lib.cudaEventDestroy.argtypes = [ctypes.c_void_p]

    def create(self):
        h = self.c.c_void_p()
        if self.lib.cudaEventCreate(self.c.byref(h)) != 0:
            raise RuntimeError("cudaEventCreate failed")
        return h.value

    def record(self, ev, stream_handle):
        if self.lib.cudaEventRecord(ev, stream_handle) != 0:
            raise RuntimeError("cudaEventRecord failed")

    def ms(self, a, b):
        v = self.c.c_float()
        if self.lib.cudaEventElapsedTime(self.c.byref(v), a, b) != 0:
            raise RuntimeError("cudaEventElapsedTime failed")
        return float(v.value)

    def destroy(self, ev):
        self.lib.cudaEventDestroy(ev)


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


# --- measured DRAM traffic ---------------------------------------------------------
# dram__bytes_read.sum + dram__bytes_write.sum per launch of the product kernel,
# captured by ncu on the full-size workload itself (these three metrics take one
# pass, so the capture replays nothing):
#   python bench.py --steps 2 --warmup 1 --no-cpu-baseline --no-parity --no-ceilings
#   ncu --metrics gpu__time_duration.sum,dram__bytes_read.sum,dram__bytes_write.sum \
#       --clock-control none -k regex:cached_block -s 4 -c 4 --csv --log-file dram27.csv <same command>
# Traffic does not grow in proportion to the edges (on the same recipe at 2^24
# the B = 16 launches move 1.3-1.6x their algorithmic bytes, at 2^27 2.6-3.1x:
# the rows of x and y in flight outgrow L2), so the numbers serve only the
# workload they were taken on.  They hold only for the device sources they were
# taken on: "digest" is the SHA-256 of those sources, and any later change to
# them makes roofline.traffic null until a new capture.
MEASURED_TRAFFIC = {"digest": "29cd9dc78fb44eed3a99cc4c72481beab5da7ce65b2fefeab8ea747b938da3ad",
                    "workload": "rmat27-bfs-1200M", "nnz": 1200000000,
                    "bytes": {"right B=1": 16156469760, "left B=1": 18788308992,
                              "right B=16": 95999932672, "left B=16": 112268192256}}


def _code_only(text: str) -> str:
    """C/C++/CUDA source without comments and with whitespace runs collapsed
    (the sources hold no string literal containing a comment marker)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def device_digest() -> str:
    """SHA-256 of the device sources' code (comments and layout ignored)."""
    import hashlib
    csrc = os.path.join(ROOT, "compressed_graph_spmv_gb300", "csrc")
    h = hashlib.sha256()
    paths = [os.path.join(csrc, n) for n in sorted(os.listdir(csrc)) if n.endswith((".cu", ".cuh", ".h", ".cpp"))]
    for path in paths + [os.path.join(ROOT, "include", "k2t.h")]:
        with open(path) as f:
            h.update(os.path.basename(path).encode() + b"\0" + _code_only(f.read()).encode())
    return h.hexdigest()


def measured_traffic(wl_name: str, nnz: int, product: str):
    """(bytes per launch, source) for a product of the captured workload;
    (None, why) for any other workload or device code."""
    t = MEASURED_TRAFFIC
    if not t["digest"] or product not in t["bytes"]:
        return None, "no capture recorded"
    if wl_name != t["workload"] or nnz != t["nnz"]:
        return None, "captured on %s only (traffic does not scale with the edges)" % t["workload"]
    if t["digest"] != device_digest():
        return None, "device code changed since the capture"
    return int(t["bytes"][product]), "ncu dram__bytes_read.sum + dram__bytes_write.sum on %s" % t["workload"]


# --- byte accounting ------------------------------------------------------------
def algorithmic_bytes(stats, semiring, direction, B):
    """Bytes a product kernel must move: the tree parts it reads, x once, y
    read and written once (the count of the pages' Table 4)."""
    tree = (stats.t_bytes_device + stats.l_bytes_device + stats.dir_bytes + stats.top_bytes +
            stats.cached_bytes + stats.plan_bytes)
    n_in = stats.n_cols if direction == 0 else stats.n_rows
    n_out = stats.n_rows if direction == 0 else stats.n_cols
    width = 1 if semiring == synth.BOOLEAN else B
    return int(tree + 4 * n_in * width + 8 * n_out * width)


# --- parity on sampled outputs --------------------------------------------------
def parity_sample(wl, got: dict, n_sample: int = 2048, seed: int = 99):
    """Compare sampled outputs of every timed product with the oracle's
    edge-list definition (section 2.2), bit-exact or within the fp32 bound."""
    import oracle
    rng = np.random.default_rng(seed)
    checked, bad = 0, 0
    for (d, B), y in got.items():
        n_out = wl.n_rows if d == 0 else wl.n_cols
        sample = np.unique(rng.integers(0, n_out, size=n_sample))
        ref = oracle.rows_product(wl.rows, wl.cols, wl.n_rows, wl.n_cols, d, wl.semiring,
                                  vector(wl, d, B), sample, B=B, w=wl.w)
        if wl.semiring == synth.PLUS_TIMES:
            err = np.abs(y[sample].astype(np.float64) - ref.y)
            bad += int((~(err <= oracle.plus_times_tolerance(ref.scale))).sum())
        else:
            g = np.ascontiguousarray(y[sample]).view(np.uint32)
            bad += int((g != np.ascontiguousarray(ref.y).view(np.uint32)).sum())
        checked += int(ref.y.size)
    return {"checked_entries": checked, "mismatches": bad, "ok": bad == 0,
            "against": "oracle edge-list definition on sampled outputs"}


# --- CPU oracle on a bounded sample ------------------------------------------------
def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or platform.machine()


def oracle_sample(wl, target_edges: int, band_bits: int = 10, seed: int = 17):
    """Edges of uniformly random aligned row bands of 2^band_bits rows, drawn
    until about target_edges are kept.  Inside a band every non-zero of its
    rows is kept, so the subtrees below the band's level have the full
    matrix's shape there; the bands spread over the whole id range, so the
    sample mixes hub rows and sparse rows as the matrix does."""
    m = wl.rows.size
    if m <= target_edges:
        return wl.rows, wl.cols, "all %d edges" % m
    nb = max(1, (wl.n_rows + (1 << band_bits) - 1) >> band_bits)
    per_band = np.bincount(wl.rows >> band_bits, minlength=nb)
    order = np.random.default_rng(seed).permutation(nb)
    take = int(np.searchsorted(np.cumsum(per_band[order]), target_edges)) + 1
    keep = np.zeros(nb, bool)
    keep[order[:take]] = True
    sel = keep[wl.rows >> band_bits]
    return wl.rows[sel], wl.cols[sel], ("%d random row bands of %d rows (of %d): %d of %d edges"
                                        % (take, 1 << band_bits, nb, int(sel.sum()), m))


def time_oracle(wl, products, target_edges: int, steps: int = 1, warmup: int = 0, threads: int = 1):
    """The oracle's rank-based recursive descent over the sample, right and
    left, single-threaded (threads 1) or shared among host threads by row /
    column bands (threads 0: one per core); returns (edges/s, description,
    per-step seconds, units per step, threads used)."""
    import oracle
    r, c, desc = oracle_sample(wl, target_edges)
    t = oracle.OracleTree(r, c, wl.n_rows, wl.n_cols, n_k4=0)
    m = int(oracle.dedup_edges(r, c)[0].size)
    times = []
    for it in range(warmup + steps):
        t0 = time.perf_counter()
        units = 0
        for (d, B) in products:
            t.spmv(d, wl.semiring, vector(wl, d, B), B=B, w=wl.w, threads=threads)
            units += m * B
        dt = time.perf_counter() - t0
        if it >= warmup:
            times.append(dt)
    return units / statistics.median(times), desc, times, units, t.threads_used


def run_reference(args):
    """The reference arm: the oracle's descent on all host cores (row / column
    bands), on a bounded sample of the workload, as edges/s."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    wl, _, products = make_workload(args.workload)
    if args.products:
        products = [tuple(int(v) for v in p.split(":")) for p in args.products.split(",")]
    eps, desc, times, units, used = time_oracle(wl, products, args.oracle_edges, steps=args.steps,
                                                warmup=args.warmup, threads=0)
    total = sum(times)
    value = units * len(times) / total
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": "edges/s", "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": dtype_name(wl), "data": "synthetic",
           "config": {"workload": wl.name, "nnz": int(wl.rows.size), "n": int(wl.n_rows),
                      "products": [list(p) for p in products], "parallelism": "host threads"},
           "cpu_baseline": {"value": value, "unit": "edges/s", "cores": used, "threads": used,
                            "kind": "oracle", "cpu_model": cpu_model(), "sample": desc},
           "e2e": {"value": value, "unit": "edges/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))


def dtype_name(wl):
    return "u32" if wl.semiring == synth.BOOLEAN else "f32"


def one_at_a_time(rank: int, world: int, group, fn):
    """Run fn on every rank, one rank after the other (rank 0 first), with a
    barrier of `group` between turns; returns this rank's result."""
    import torch.distributed as dist
    out = None
    for turn in range(world):
        if turn == rank:
            out = fn()
        if group is not None:
            dist.barrier(group=group)
    return out


# --- the GPU arm ------------------------------------------------------------------
def run_ours(args):
    import torch
    import compressed_graph_spmv_gb300 as k2t
    from compressed_graph_spmv_gb300 import k2t as K

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # Replicas generate and build in turn (a CPU-side barrier with a long
    # timeout between turns): a builder's host peak (about 70 GB on the 1.2G
    # edge graph) is then paid by one rank at a time.
    turns = None
    if world > 1:
        import datetime
        turns = dist.new_group(backend="gloo", timeout=datetime.timedelta(hours=3))

    def prepare():
        t_gen = time.perf_counter()
        wl, wopts, products = make_workload(args.workload)
        if args.products:
            products = [tuple(int(v) for v in p.split(":")) for p in args.products.split(",")]
        t_gen = time.perf_counter() - t_gen
        max_b = max(B for _, B in products)
        opts = dict(wopts, host_vectors=1, max_batch=max_b)
        if args.engine is not None:
            opts["engine"] = args.engine
            opts["cache_last_internal"] = int(args.engine in (3, 4))
        for kv in args.opt:
            k, v = kv.split("=", 1)
            opts[k] = int(v, 0)
        t_build = time.perf_counter()
        tree = K.Tree(wl.rows, wl.cols, wl.n_rows, wl.n_cols, **opts)
        t_build = time.perf_counter() - t_build
        return wl, products, opts, tree, t_gen, t_build

    wl, products, opts, tree, t_gen, t_build = one_at_a_time(rank, world, turns, prepare)
    st = tree.stats()
    ws = tree.workspace_bytes()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    tree.upload()
    torch.cuda.synchronize()
    footprint = free0 - torch.cuda.mem_get_info()[0]

    boolean = wl.semiring == synth.BOOLEAN
    dev_x, dev_y = {}, {}
    for (d, B) in products:
        xv = vector(wl, d, B)
        n_out = wl.n_rows if d == 0 else wl.n_cols
        if boolean:
            dev_x[(d, B)] = torch.from_numpy(xv.view(np.int32)).cuda()
            dev_y[(d, B)] = torch.empty(n_out, dtype=torch.int32, device="cuda")
        else:
            dev_x[(d, B)] = torch.from_numpy(xv).cuda()
            dev_y[(d, B)] = torch.empty(n_out, B, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    m = int(st.nnz)

    def product(p, ev=None):
        d, B = p
        if ev is None:
            tree.spmv(d, wl.semiring, dev_x[p], dev_y[p], B=B, w=wl.w, stream=stream)
        else:
            tree.spmv_marked(d, wl.semiring, dev_x[p], dev_y[p], B, wl.w, stream, ev)

    # parity of every timed product on sampled outputs, before timing
    for p in products:
        product(p)
    torch.cuda.synchronize()
    got = {p: (dev_y[p].cpu().numpy().view(np.uint32) if boolean else dev_y[p].cpu().numpy()) for p in products}
    parity = parity_sample(wl, got) if not args.no_parity else {"skipped": True}

    # L2 flush between steps unless the working set dwarfs L2
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    work_bytes = max(algorithmic_bytes(st, wl.semiring, d, B) for d, B in products)
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda") if work_bytes < 4 * l2 else None

    for _ in range(args.warmup):
        for p in products:
            product(p)
        if flush is not None:
            flush.add_(1.0)
    torch.cuda.synchronize()

    nprod = len(products)
    rev = RawEvents()
    sh = stream.cuda_stream
    evs = [[(rev.create(), rev.create(), rev.create()) for _ in products] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for s in range(args.steps):
        for i, p in enumerate(products):
            e0, e1, e2 = evs[s][i]
            rev.record(e0, sh)
            product(p, e1)
            rev.record(e2, sh)
        if flush is not None:
            flush.add_(1.0)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    clk = clocks.stop()

    prod_ms = np.array([[rev.ms(evs[s][i][0], evs[s][i][2]) for i in range(nprod)] for s in range(args.steps)])
    main_ms = np.array([[rev.ms(evs[s][i][1], evs[s][i][2]) for i in range(nprod)] for s in range(args.steps)])
    for row in evs:
        for trip in row:
            for e in trip:
                rev.destroy(e)
    step_ms = prod_ms.sum(axis=1)
    total_s = float(step_ms.sum()) / 1e3
    if dist:
        tt = torch.tensor([total_s], device="cuda")
        dist.all_reduce(tt, op=dist.ReduceOp.MAX)
        total_s = float(tt.item())
    units_per_step = sum(m * B for _, B in products)
    value = units_per_step * args.steps * world / total_s

    # roofline of the dominant kernel (the product kernel with the largest time)
    per_kernel = []
    for i, (d, B) in enumerate(products):
        avg = float(main_ms[:, i].mean()) / 1e3
        byt = algorithmic_bytes(st, wl.semiring, d, B)
        q1, med, q3 = (float(v) for v in np.percentile(main_ms[:, i], [25, 50, 75]))
        per_kernel.append({"product": "%s B=%d" % ("right" if d == 0 else "left", B), "avg_ms": avg * 1e3,
                           "median_ms": med, "iqr_ms": q3 - q1,
                           "leaves_per_s": float(st.level_nodes[st.levels - 1]) / avg,
                           "fill_ms": float((prod_ms[:, i] - main_ms[:, i]).mean()),
                           "algorithmic_bytes": byt, "achieved_gbs": byt / avg / 1e9,
                           "edges_per_s": m * B / avg})
    # warm and cold times of each product (fill + kernel): warm right after
    # the same product, cold right after writing a buffer of twice L2
    flush2 = flush if flush is not None else torch.empty(2 * l2 // 4 + 1024, dtype=torch.float32, device="cuda")
    for i, p in enumerate(products):
        warm, cold = [], []
        for _ in range(3):
            for kind in ("cold", "warm"):
                if kind == "cold":
                    flush2.add_(1.0)
                e0, e1 = rev.create(), rev.create()
                rev.record(e0, sh)
                product(p)
                rev.record(e1, sh)
                torch.cuda.synchronize()
                (cold if kind == "cold" else warm).append(rev.ms(e0, e1))
                rev.destroy(e0)
                rev.destroy(e1)
        per_kernel[i]["warm_ms"] = float(np.median(warm))
        per_kernel[i]["cold_ms"] = float(np.median(cold))
    if flush is None:
        del flush2
    dom = max(range(nprod), key=lambda i: per_kernel[i]["avg_ms"])
    peak, peak_kind = measured_peak()
    ach = per_kernel[dom]["achieved_gbs"]
    traffic, traffic_src = measured_traffic(wl.name, m, per_kernel[dom]["product"])
    roofline = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                "traffic": traffic, "traffic_source": traffic_src, "peak_source": peak_kind,
                "kernel": per_kernel[dom]["product"],
                "bytes_per_launch": per_kernel[dom]["algorithmic_bytes"]}

    # The single-vector leaf step's own bound: a leaf costs one scattered gather
    # (its two inputs) and about one scattered reduction.  Their rates on this
    # GPU, measured now with L2-resident arrays (the probe library), allow
    # 1 / (1/gather + 1/reduction) leaves per second.
    b1 = [k for k, (d, B) in zip(per_kernel, products) if B == 1 and wl.semiring != synth.BOOLEAN]
    scatter_model = None
    if b1 and not args.no_ceilings:
        ceil = measure_ceilings(rev, stream, [("l2_resident_16MB", 1 << 22)])["l2_resident_16MB"]
        g, r = ceil["gather8_Gops"] * 1e9, ceil["red_scattered_Gops"] * 1e9
        ceil_lps = 1.0 / (1.0 / g + 1.0 / r)
        best = max(k["leaves_per_s"] for k in b1)
        scatter_model = {"model": "1 scattered gather + 1 scattered reduction per leaf, L2-resident rates",
                         "gather_per_s": g, "reduction_per_s": r, "measured": "this run",
                         "ceiling_leaves_per_s": ceil_lps, "achieved_leaves_per_s": best,
                         "frac": best / ceil_lps}

    # end to end through the C ABI with host buffers (copies inside the timed region)
    # pinned staging: one input and one output buffer per batch width, filled
    # with each product's x before its timed call
    hx, hy, hbuf = {}, {}, {}
    for p in products:
        d, B = p
        n_in = wl.n_cols if d == 0 else wl.n_rows
        n_out = wl.n_rows if d == 0 else wl.n_cols
        if B not in hbuf:
            words = (max(wl.n_rows, wl.n_cols)) * (1 if boolean else B)
            dt = torch.int32 if boolean else torch.float32
            hbuf[B] = (torch.empty(words, dtype=dt).pin_memory().numpy(),
                       torch.empty(words, dtype=dt).pin_memory().numpy())
        bx, by = hbuf[B]
        width = 1 if boolean else B
        hx[p] = bx[:n_in * width].reshape((n_in,) if boolean else (n_in, B))
        hy[p] = by[:n_out * width].reshape((n_out,) if boolean else (n_out, B))
    h2d = sum(hx[p].nbytes for p in products)
    d2h = sum(hy[p].nbytes for p in products)

    def stage_x(p):
        xv = vector(wl, p[0], p[1])
        np.copyto(hx[p], xv.view(np.int32) if boolean else xv)
    e2e_steps = max(1, min(args.steps, 5))
    for p in products:
        stage_x(p)
        tree.spmv_host(p[0], wl.semiring, hx[p], hy[p], B=p[1], w=wl.w)
    e2e_s = 0.0
    for _ in range(e2e_steps):
        for p in products:
            stage_x(p)  # host-side preparation of the input, outside the timed call
            t0 = time.perf_counter()
            tree.spmv_host(p[0], wl.semiring, hx[p], hy[p], B=p[1], w=wl.w)
            e2e_s += time.perf_counter() - t0
    e2e_s /= e2e_steps
    e2e = {"value": units_per_step * world / e2e_s, "unit": "edges/s",
           "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": e2e_steps}

    base_launches = 2 if st.engine != k2t.ENGINE_LEVELSYNC else 1 + int(st.n_steps) * (3 if st.offsets else 1)
    # plus-times products of a direction with heavy outputs add the zeroing of
    # their sums and the final rounding pass
    launches_per_step = sum(base_launches + (2 if wl.semiring == synth.PLUS_TIMES and
                                             (st.heavy_rows if d == 0 else st.heavy_cols) else 0)
                            for d, _ in products)
    out = {"metric": METRIC, "value": value, "unit": "edges/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": float(step_ms.mean()), "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(wl), "data": "synthetic",
           "config": {"workload": wl.name, "nnz": m, "n": wl.n_rows, "levels": int(st.levels), "d0": int(st.d0),
                      "options": {k: v for k, v in opts.items() if k not in ("host_vectors", "max_batch")},
                      "engine": ["auto", "fused", "levelsync", "cached", "banded"][int(st.engine)],
                      "products": [list(p) for p in products],
                      "l2": "flushed between steps" if flush is not None else "inputs larger than L2",
                      "parallelism": "replicas" if world > 1 else "single"},
           "roofline": roofline, "scatter_bound": scatter_model, "kernels": per_kernel,
           "e2e": e2e, "gpu_launches": launches_per_step * args.steps, "clocks": clk,
           "parity": parity,
           "footprint": {"predicted_bytes": ws, "measured_bytes": int(footprint),
                         "host_vector_staging_bytes": int(st.vector_bytes),
                         "product_bytes": int(ws - st.vector_bytes),
                         "tree_bits_per_edge": st.tree_bits / max(1, m),
                         "heavy_outputs": {"rows": int(st.heavy_rows), "cols": int(st.heavy_cols),
                                           "fp32_partial_sums": [int(v) for v in st.heavy_partials],
                                           "fp64_outputs": [int(v) for v in st.heavy_fp64],
                                           "most_terms_per_fp32_sum": [int(v) for v in st.heavy_max_terms],
                                           "table_and_sum_bytes": int(st.heavy_kib) * 1024}},
           "wall_ms_per_step": 1e3 * wall / args.steps,
           "host_seconds": {"generate": t_gen, "build": t_build},
           "host_peak_rss_gb": resource.getrusage(resource.RUSAGE_SELF).ru_maxrss / 1e6}
    if rank == 0 and not args.no_cpu_baseline:
        eps1, desc, _, _, _ = time_oracle(wl, products, args.oracle_edges)
        epsn, _, _, _, used = time_oracle(wl, products, args.oracle_edges, threads=0)
        out["cpu_baseline"] = {"value": epsn, "unit": "edges/s", "cores": used, "threads": used, "kind": "oracle",
                               "cpu_model": cpu_model(), "sample": desc,
                               "single_thread": {"value": eps1, "unit": "edges/s", "cores": 1}}
    if rank == 0:
        print(json.dumps(out))
    if dist:
        dist.destroy_process_group()


def measure_ceilings(rev, stream, sizes):
    """Rates of the leaf step's memory patterns on this GPU (section 5.6
    analogue), from the probe library: per array size, copy GB/s and
    scattered gathers / reductions in G operations per second."""
    import torch
    from compressed_graph_spmv_gb300 import k2t as K
    sh = stream.cuda_stream
    out = {}
    for label, n in sizes:
        x = torch.rand(n, device="cuda")
        y = torch.zeros(n, device="cuda")
        res = {}
        for kind, name, m in ((0, "copy_GBps", n), (1, "gather4_Gops", 1 << 28), (2, "gather8_Gops", 1 << 28),
                              (3, "red_consecutive_Gops", 1 << 28), (4, "red_scattered_Gops", 1 << 28),
                              (5, "smem_red_fp32_Gops", 1 << 30), (6, "smem_red_fp64_Gops", 1 << 30)):
            for _ in range(2):
                K.probe(kind, x, y, n, m, stream=stream)
            e0, e1 = rev.create(), rev.create()
            rev.record(e0, sh)
            for _ in range(5):
                K.probe(kind, x, y, n, m, stream=stream)
            rev.record(e1, sh)
            torch.cuda.synchronize()
            ms = rev.ms(e0, e1) / 5
            rev.destroy(e0)
            rev.destroy(e1)
            res[name] = (8.0 * n / (ms * 1e6)) if kind == 0 else (m / (ms * 1e6))
        out[label] = res
        del x, y
    return out


def run_ceilings(args):
    """Rates of the leaf step's memory patterns on this GPU (section 5.6 analogue)."""
    import torch
    out = {"kind": "ceilings"}
    out.update(measure_ceilings(RawEvents(), torch.cuda.current_stream(),
                                [("l2_resident_16MB", 1 << 22), ("hbm_2GB", 1 << 29)]))
    print(json.dumps(out))


def run_msbfs(args):
    """Multi-source search to the fixed point on the workload's graph (section
    5.8 analogue): B sources, both directions, cached engine."""
    import torch
    from compressed_graph_spmv_gb300 import k2t as K
    import oracle
    wl, wopts, _ = make_workload(args.workload)
    n = wl.n_rows
    B = args.bfs_sources
    tree = K.Tree(wl.rows, wl.cols, n, wl.n_cols, **dict(wopts, cache_last_internal=1))
    tree.upload()
    rng = np.random.default_rng(7)
    sources = rng.choice(n, size=B, replace=False)
    dist = torch.empty(n * B, dtype=torch.int32, device="cuda")
    work = torch.empty(tree.msbfs_work_bytes(), dtype=torch.uint8, device="cuda")
    out = {"kind": "msbfs", "workload": wl.name, "sources": B, "nnz": int(tree.stats().nnz)}
    for d, name in ((K.RIGHT, "right"), (K.LEFT, "left")):
        tree.msbfs(d, sources, dist, work, max_levels=args.bfs_levels)  # warm-up
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        levels = tree.msbfs(d, sources, dist, work, max_levels=args.bfs_levels)
        torch.cuda.synchronize()
        sec = time.perf_counter() - t0
        got = dist.cpu().numpy().reshape(n, B)
        res = {"levels": levels, "seconds": sec, "reached": int((got >= 0).sum())}
        if not args.no_parity:
            check = list(range(min(B, 2)))
            want = oracle.msbfs(wl.rows, wl.cols, n, sources[check], d, max_levels=args.bfs_levels)
            res["parity_sources_checked"] = len(check)
            res["parity_ok"] = bool(np.array_equal(got[:, check], want))
        out[name] = res
    print(json.dumps(out))


def run_bool_product(args):
    """Boolean product of two trees, C = A A (section 7 analogue), on a local
    web-like graph (n = 2^scale, Poisson(6) out-degree, targets within +-256
    w.p. 0.8): the whole k2t_bool_product call (device pair descent, records
    to the host, C's build) timed on the host clock, then the oracle's scipy
    product of the edge lists for the same C."""
    import torch
    from compressed_graph_spmv_gb300 import k2t as K
    import oracle
    scale = args.bool_product
    n = 1 << scale
    rows, cols = synth.weblike(n, lam=6.0, seed=5)
    a = K.Tree(rows, cols, n, n)
    a.bool_product(a).close()   # warm-up (context, allocations)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    c = a.bool_product(a)
    sec = time.perf_counter() - t0
    st = c.stats()
    out = {"kind": "bool_product", "workload": "local%d (weblike n=2^%d, lam 6)" % (scale, scale),
           "nnz_a": int(a.stats().nnz), "nnz_c": int(st.nnz), "seconds": sec,
           "c_nonzeros_per_s": st.nnz / sec}
    t0 = time.perf_counter()
    r, cc = oracle.bool_product(rows, cols, rows, cols, n, n, n)
    out["oracle_seconds"] = time.perf_counter() - t0
    if not args.no_parity:
        gr, gc = c.decode()
        order = np.lexsort((gc, gr))
        out["parity_ok"] = bool(np.array_equal(gr[order], r) and np.array_equal(gc[order], cc))
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="rmat27")
    ap.add_argument("--engine", type=int, default=None)
    ap.add_argument("--opt", action="append", default=[],
                    help="library option override, e.g. --opt tile_m=65536 (repeatable)")
    ap.add_argument("--products", default=None,
                    help="override the products of a step, e.g. 0:1,1:1 (direction:batch)")
    ap.add_argument("--oracle-edges", type=int, default=4_000_000)
    ap.add_argument("--no-parity", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ceilings", action="store_true", help="skip the in-run scattered-access probe")
    ap.add_argument("--ceilings", action="store_true", help="measure the leaf step's memory ceilings and exit")
    ap.add_argument("--msbfs", action="store_true", help="time a multi-source search on the workload and exit")
    ap.add_argument("--bfs-sources", type=int, default=16)
    ap.add_argument("--bfs-levels", type=int, default=32)
    ap.add_argument("--bool-product", type=int, default=0, metavar="SCALE",
                    help="time the Boolean product A A of a 2^SCALE local graph and exit")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.ceilings:
        run_ceilings(args)
    elif args.msbfs:
        run_msbfs(args)
    elif args.bool_product:
        run_bool_product(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
