"""Benchmark of the GB300 multi-column embedding front end.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload inference|inference-onehot|training|sequences-mean|
                            sequences-padded|dynamic|dynamic-small|tiny]

One JSON line on rank 0.  Default workload: the 1000-column inference forward
(700 hash-mod + 300 bucketize columns, batch 512, dims 8..64, bags 1..20).
A step is one pass of the workload's hot path over one batch:
  inference            the fused forward (inference-onehot: the same
                       columns with one value per bag, batch 4096);
  training, sequences  forward + backward (sort, run reduction) + Adagrad;
  dynamic              hash lookup-or-insert + forward + backward/Adagrad +
                       expiry sweep (one step of the 50-step stream).
Inputs are resident in HBM before timing; L2 is flushed (a write of twice its
size) between timed steps, outside the per-step CUDA events.

value         pooled rows gathered per second (valid IDs whose row was read)
roofline      the forward kernel: its algorithmic bytes per launch / its mean
              event time, against the measured HBM copy bandwidth;
              roofline_backward: the same for the whole backward call
gather_ceiling the rate random row gathers of the workload's row sizes reach
              on this GPU (measured beside the run), for reference
e2e           the same metric through the C ABI with pinned HOST buffers: H2D of
              the step's inputs, the step, D2H of the pooled output
cpu_baseline  the CPU oracle on a bounded sample of the workload: forward
              workloads on all host cores (columns split over threads, the
              one-thread rate beside it), the others on one thread
--impl reference  times that oracle alone (the reference arm of this build).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_lookup_gb300 import synth  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM = 6800.0
TRAIN_WORKLOADS = ("training", "sequences-mean", "sequences-padded", "tiny")


def peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=0):
        self.samples = []
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                self.samples.append(parts)

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        res = {"sm_mhz": None, "sm_max_mhz": None, "reasons": []}
        if not self.samples:
            return res

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(s[1]) for s in self.samples if num(s[1]) is not None]
        mx = [num(s[2]) for s in self.samples if num(s[2]) is not None]
        res["sm_mhz"] = statistics.median(sm) if sm else None
        res["sm_max_mhz"] = max(mx) if mx else None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for k, v in zip(names, s[5:9]):
                if v.strip().lower() in ("active", "1"):
                    reasons.add(k)
        res["reasons"] = sorted(reasons)
        res["samples"] = len(self.samples)
        return res


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def sync_ranks(torch):
    """Barrier across the replicas (nothing to do for one process)."""
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        torch.distributed.barrier()


def aggregate_ranks(torch, ms_step, rows_per_step, device):
    """Whole-job throughput of N replicas: every rank's rows over the slowest
    rank's step time.  Returns (max ms per step, rows per second)."""
    world = 1
    t = torch.tensor([float(ms_step)], dtype=torch.float64, device=device)
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        world = torch.distributed.get_world_size()
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    ms = float(t.item())
    return ms, rows_per_step * world / (ms / 1e3)


def make_workload(name, columns=None):
    if name == "inference":
        if columns:
            return synth.inference(n_cat=columns * 7 // 10, n_num=columns - columns * 7 // 10)
        return synth.inference()
    if name == "inference-onehot":
        # the inference columns with one value per bag, at batch 4096
        if columns:
            return synth.inference(n_cat=columns * 7 // 10, n_num=columns - columns * 7 // 10, B=4096,
                                   one_hot=True)
        return synth.inference(B=4096, one_hot=True)
    if name == "training":
        return synth.training(C=columns) if columns else synth.training()
    if name == "sequences-mean":
        return synth.sequences(mode="mean", C=columns or 20)
    if name == "sequences-padded":
        return synth.sequences(mode="padded", C=columns or 20)
    if name == "tiny":
        return synth.tiny()
    if name == "dynamic":
        return synth.dynamic(C=columns) if columns else synth.dynamic()
    if name == "dynamic-small":
        # profiling size: 10 columns over a 2^24-slot table with 2^22 rows
        return synth.dynamic(C=columns or 10, num_slots=1 << 24, row_capacity=1 << 22)
    raise SystemExit("unknown workload %s" % name)


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

ELEM_BYTES = {"f32": 4, "bf16": 2, "f16": 2, "i8": 1}


def row_bytes(c, table_dtype="f32"):
    """Bytes one gathered row reads: its elements, plus the row's scale for int8."""
    return ELEM_BYTES[table_dtype] * c.dim + (4 if table_dtype == "i8" else 0)


def forward_bytes(w, valid_per_col, table_dtype="f32"):
    """Per column: the offsets, the values, the boundaries, one row read per
    valid value and one output row per bag (padded columns: pad_len rows)."""
    total = 0
    for c, o, nv in zip(w.columns, w.offsets, valid_per_col):
        n = int(o[-1])
        e = 4 if c.transform == "bucketize" else 8
        nb = 0 if c.boundaries is None else c.boundaries.size
        total += (w.B + 1) * 4 + n * e + 4 * nb + nv * row_bytes(c, table_dtype)
        total += w.B * 4 * c.dim * (c.pad_len if c.pooling == "padded" else 1)
    return total


def backward_bytes(w, n_contrib, valid_per_col, n_unique, dim):
    """The recorded (row, source) pairs read once (8 B), one sort round trip
    (16 B), one gradient row gathered per valid contribution, and the read +
    write of weight and accumulator rows of every unique row."""
    grad = sum(nv * 4 * c.dim for c, nv in zip(w.columns, valid_per_col))
    return n_contrib * 8 + n_contrib * 16 + grad + n_unique * 16 * dim


def forward_bytes_compulsory(w, stats, table_dtype="f32"):
    """forward_bytes with each table's distinct rows read once instead of
    once per occurrence: the least a forward must move however skewed its
    ids are (the rest can come from caches)."""
    total = 0
    dims = {}
    for c, o in zip(w.columns, w.offsets):
        n = int(o[-1])
        e = 4 if c.transform == "bucketize" else 8
        nb = 0 if c.boundaries is None else c.boundaries.size
        total += (w.B + 1) * 4 + n * e + 4 * nb
        total += w.B * 4 * c.dim * (c.pad_len if c.pooling == "padded" else 1)
        dims[c.table] = c
    for t, u in stats["unique_per_table"].items():
        total += u * row_bytes(dims[t], table_dtype)
    return total


def backward_bytes_compulsory(w, n_contrib, stats, n_unique, dim):
    """backward_bytes with the upstream gradient read once (each bag's
    gradient row of a pooled column once, every padded position once)
    instead of once per contribution."""
    grad = 0
    for c, nv, ne in zip(w.columns, stats["valid"], stats["nonempty_bags"]):
        grad += (nv if c.pooling == "padded" else ne) * 4 * c.dim
    return n_contrib * 8 + n_contrib * 16 + grad + n_unique * 16 * dim


# ---------------------------------------------------------------------------
# timing harness
# ---------------------------------------------------------------------------

def timed_steps(torch, steps, stream, flush, body):
    """Run `steps` steps; body(i, marks) records events around its parts in
    the dict `marks` (name -> (start, end)).  L2 is flushed before each step
    outside the events.  Returns per-part lists of milliseconds and the wall
    time of the loop."""
    recs = []
    sync_ranks(torch)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        flush.fill_(float(i))
        marks = {}
        body(i, marks)
        recs.append(marks)
    torch.cuda.synchronize()
    sync_ranks(torch)
    wall = time.perf_counter() - t0
    out = {}
    for marks in recs:
        for k, (a, b) in marks.items():
            out.setdefault(k, []).append(a.elapsed_time(b))
    return out, wall


def event_pair(torch):
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def row_sizes_mix(w, valid_per_col, table_dtype="f32"):
    """Rows gathered per row size (rounded up to the 16 B the calibration
    kernel moves per lane)."""
    mix = {}
    for c, nv in zip(w.columns, valid_per_col):
        b = (row_bytes(c, table_dtype) + 15) // 16 * 16
        mix[b] = mix.get(b, 0) + nv
    return mix


def calibrate_gather_rate(sl, dim, table_bytes=8 << 30, n=1 << 25, reps=5, seed=0):
    """GB/s of random row gathers of `dim` floats over a table of table_bytes
    (larger than L2), timed with CUDA events on the current stream."""
    import torch
    rows = max(1, table_bytes // (dim * 4))
    table = torch.zeros((rows, dim), dtype=torch.float32, device="cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    idx = torch.randint(0, rows, (n,), generator=g, device="cuda", dtype=torch.int64).to(torch.int32)
    sink = torch.zeros(1, device="cuda")
    sl.emb_calibrate_gather(table, rows, dim, idx, n, sink)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        sl.emb_calibrate_gather(table, rows, dim, idx, n, sink)
    b.record()
    b.synchronize()
    ms = a.elapsed_time(b) / reps
    del table, idx
    return n * dim * 4 / (ms / 1e3) / 1e9


def gather_ceiling(torch, sl, mix, dev, budget_bytes=8 << 30):
    """Random-row gather rate of this GPU for the workload's row sizes: one
    gather-only pass per row size over a table larger than L2 (the library's
    calibration kernel), combined by the workload's row counts."""
    out = {}
    total_rows = sum(mix.values())
    if not total_rows or not hasattr(sl, "emb_calibrate_gather"):
        return None
    t_sum = 0.0
    for nbytes, rows in sorted(mix.items()):
        gbs = calibrate_gather_rate(sl, nbytes // 4, table_bytes=min(budget_bytes, 8 << 30))
        out[str(nbytes)] = round(gbs, 1)
        t_sum += rows * nbytes / (gbs * 1e9)
    bytes_total = sum(r * b for b, r in mix.items())
    return {"per_row_bytes_gbs": out, "mix_gbs": bytes_total / t_sum / 1e9}


# ---------------------------------------------------------------------------
# CPU oracle samples
# ---------------------------------------------------------------------------

def cpu_forward_sample(w, tables_dev, budget_s=12.0, table_dtype="f32", scales_dev=None):
    """The oracle forward (one thread) on whole columns in order until about
    budget_s of CPU work."""
    import oracle
    t_used, rows_done, cols_done = 0.0, 0, 0
    for ci, c in enumerate(w.columns):
        tab = synth.table_host(tables_dev[c.table])
        sc = None if scales_dev is None or scales_dev[c.table] is None else scales_dev[c.table].cpu().numpy()
        spec = synth.ColumnSpec(c.transform, c.pooling, c.num_rows, c.dim, 0, boundaries=c.boundaries,
                                default=c.default, pad_len=c.pad_len)
        t0 = time.perf_counter()
        _, _, rows = oracle.forward([spec], w.B, [w.offsets[ci]], [w.values[ci]], [tab], want_rows=True,
                                    table_dtypes=[table_dtype], row_scales=[sc])
        t_used += time.perf_counter() - t0
        rows_done += int((rows[0] >= 0).sum())
        cols_done += 1
        if t_used > budget_s:
            break
    sample = "%d of %d columns, all %d bags each (%d rows gathered), oracle forward, 1 thread" % (
        cols_done, len(w.columns), w.B, rows_done)
    return rows_done / t_used, sample


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_forward_sample_threads(w, tables_dev, threads, budget_s=2.0, table_dtype="f32", scales_dev=None,
                               host_bytes=8 << 30):
    """The oracle forward on all host cores: columns split over `threads`
    threads (each oracle call runs in C without the interpreter lock) on the
    first columns whose host tables fit in host_bytes, repeated until about
    budget_s of wall time; the tables are copied to the host beforehand."""
    import concurrent.futures as cf
    import oracle
    work, held = [], 0
    for ci, c in enumerate(w.columns):
        tab = synth.table_host(tables_dev[c.table])
        if work and held + tab.nbytes > host_bytes:
            break
        held += tab.nbytes
        sc = None if scales_dev is None or scales_dev[c.table] is None else scales_dev[c.table].cpu().numpy()
        spec = synth.ColumnSpec(c.transform, c.pooling, c.num_rows, c.dim, 0, boundaries=c.boundaries,
                                default=c.default, pad_len=c.pad_len)
        work.append((spec, ci, tab, sc))

    def one(item):
        spec, ci, tab, sc = item
        _, _, rows = oracle.forward([spec], w.B, [w.offsets[ci]], [w.values[ci]], [tab], want_rows=True,
                                    table_dtypes=[table_dtype], row_scales=[sc])
        return int((rows[0] >= 0).sum())

    rows_done, passes, wall = 0, 0, 0.0
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        while wall < budget_s:
            t0 = time.perf_counter()
            rows_done += sum(ex.map(one, work))
            wall += time.perf_counter() - t0
            passes += 1
    sample = "%d of %d columns, all %d bags each, %d passes (%d rows gathered), oracle forward, " \
        "columns split over %d threads" % (len(work), len(w.columns), w.B, passes, rows_done, threads)
    return rows_done / wall, sample


def cpu_forward_baseline(w, tables_dev, table_dtype="f32", scales_dev=None, budget_s=12.0):
    """cpu_baseline of the forward workloads: the oracle on all host cores,
    with its one-thread rate beside it."""
    rate1, sample1 = cpu_forward_sample(w, tables_dev, budget_s=budget_s, table_dtype=table_dtype,
                                        scales_dev=scales_dev)
    n = host_cores()
    if n <= 1:
        return {"value": rate1, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": sample1}
    # about budget_s of CPU work in all on n cores
    rate, sample = cpu_forward_sample_threads(w, tables_dev, n, budget_s=max(1.0, budget_s / n),
                                              table_dtype=table_dtype, scales_dev=scales_dev)
    return {"value": rate, "unit": "rows/s", "cores": n, "kind": "oracle", "sample": sample,
            "one_core": {"value": rate1, "sample": sample1}}


def cpu_train_sample(w, tables_dev, G_dev, budget_s=12.0):
    """The oracle forward + backward/Adagrad (one thread) on whole columns in
    order until about budget_s of CPU work (host copies of their tables)."""
    import oracle
    t_used, rows_done, cols_done = 0.0, 0, 0
    col0 = 0
    G = None
    for ci, c in enumerate(w.columns):
        if c.pooling == "padded":
            gs = synth.make_grad((w.B, c.pad_len, c.dim), 900 + ci, "cpu").numpy()
            g = None
        else:
            if G is None:
                G = G_dev.cpu().numpy() if G_dev is not None else None
            g = G[:, col0:col0 + c.dim] if G is not None else None
            gs = None
        W = tables_dev[c.table].cpu().numpy()
        A = np.zeros_like(W)
        spec = synth.ColumnSpec(c.transform, c.pooling, c.num_rows, c.dim, 0, boundaries=c.boundaries,
                                default=c.default, pad_len=c.pad_len)
        t0 = time.perf_counter()
        _, _, rows = oracle.forward([spec], w.B, [w.offsets[ci]], [w.values[ci]], [W], want_rows=True)
        oracle.backward_adagrad([spec], w.B, [w.offsets[ci]], [w.values[ci]],
                                np.ascontiguousarray(g) if g is not None else None, [gs] if gs is not None else None,
                                [W], [A], w.lr, w.eps)
        t_used += time.perf_counter() - t0
        rows_done += int((rows[0] >= 0).sum())
        cols_done += 1
        if c.pooling != "padded":
            col0 += c.dim
        if t_used > budget_s:
            break
    sample = "%d of %d columns, all %d bags each (%d rows gathered), oracle forward + backward + Adagrad, " \
             "1 thread" % (cols_done, len(w.columns), w.B, rows_done)
    return rows_done / t_used, sample


def cpu_dynamic_sample(w, budget_s=12.0):
    """The oracle hash step + forward + backward/Adagrad (one thread) on the
    first steps of the dynamic stream, scaled down to 10 columns."""
    import oracle
    ex = w.extra
    C = min(10, len(w.columns))
    cap = ex["row_capacity"]
    dim = w.columns[0].dim
    oh = oracle.Hash(cap, dim, ex["threshold"], ex["init_seed"], ex["init_scale"])
    cols = [synth.ColumnSpec("rows_given", "sum", cap, dim, 0) for _ in range(C)]
    t_used, rows_done, steps = 0.0, 0, 0
    for t in range(ex["steps"]):
        offs, keys = synth.dynamic_keys(w.seed, t, C, w.B, ex["alpha"], ex["key_bits"])
        tids = np.concatenate([np.full(k.size, c, np.int32) for c, k in enumerate(keys)])
        allk = np.concatenate(keys)
        G = synth.make_grad((w.B, C * dim), 500 + t, "cpu").numpy()
        t0 = time.perf_counter()
        rows, _ = oh.lookup_or_insert(tids, allk, t)
        vals, pos = [], 0
        for o in offs:
            vals.append(rows[pos:pos + int(o[-1])])
            pos += int(o[-1])
        oracle.forward(cols, w.B, offs, vals, [oh.W])
        oracle.backward_adagrad(cols, w.B, offs, vals, G, None, [oh.W], [oh.acc], w.lr, w.eps)
        oh.evict(t, ex["ttl"])
        t_used += time.perf_counter() - t0
        rows_done += int((rows >= 0).sum())
        steps += 1
        if t_used > budget_s:
            break
    return rows_done / max(t_used, 1e-9), "%d steps of the stream with %d of %d columns (%d rows gathered), " \
        "oracle hash + forward + backward + Adagrad + expiry, 1 thread" % (steps, C, len(w.columns), rows_done)


# ---------------------------------------------------------------------------
# reference arm: the oracle alone
# ---------------------------------------------------------------------------

class HostTables:
    """Host copies of a workload's tables, drawn on first use (the same seeded
    values the device tables hold), so that a sample touching a few columns
    does not draw all of them."""

    def __init__(self, w, table_dtype="f32"):
        self.w = w
        self.dtype = table_dtype
        self.cache = {}
        self.scales = _HostScales(self)

    def _get(self, t):
        if t not in self.cache:
            self.cache[t] = synth.lowp_table(synth.make_table(self.w.tables[t], "cpu"), self.dtype)
        return self.cache[t]

    def __getitem__(self, t):
        return self._get(t)[0]


class _HostScales:
    """Per-row scales of HostTables' int8 tables, by table index."""

    def __init__(self, host):
        self.host = host

    def __getitem__(self, t):
        return self.host._get(t)[1]


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    if args.table_dtype != "f32" and (is_training(args) or args.workload.startswith("dynamic")):
        raise SystemExit("low-precision tables are read-only: forward workloads only")
    w = make_workload(args.workload, args.columns)
    per = max(2.0, 20.0 / max(1, args.steps + args.warmup))
    vals = []
    tables = HostTables(w, args.table_dtype)
    G = None
    if is_training(args):
        width = sum(c.dim for c in w.columns if c.pooling != "padded")
        G = synth.make_grad((w.B, max(width, 1)), 77, "cpu")[:, :width] if width else None
    # forward workloads run on all host cores (columns split over threads),
    # the others on one
    threads = host_cores() if not (args.workload.startswith("dynamic") or is_training(args)) else 1
    for i in range(args.warmup + args.steps):
        if args.workload.startswith("dynamic"):
            rate, sample = cpu_dynamic_sample(w, budget_s=per)
        else:
            if is_training(args):
                rate, sample = cpu_train_sample(w, tables, G, budget_s=per)
            elif threads > 1:
                rate, sample = cpu_forward_sample_threads(w, tables, threads, budget_s=max(0.5, per / threads),
                                                          table_dtype=args.table_dtype, scales_dev=tables.scales,
                                                          host_bytes=2 << 30)
            else:
                rate, sample = cpu_forward_sample(w, tables, budget_s=per, table_dtype=args.table_dtype,
                                                  scales_dev=tables.scales)
        if i >= args.warmup:
            vals.append(rate)
    v = statistics.mean(vals)
    # one whole step of the workload at the sampled rate
    if args.workload.startswith("dynamic"):
        per_step = w.B * len(w.columns) * 2.5   # mean bag length of U{0..5}
    else:
        per_step = sum(int(o[-1]) for o in w.offsets)
    line = {"impl": "reference", "metric": metric_name(args.workload, args.forward_only), "value": v,
            "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per_step / v * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 accumulate / f32 storage", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.B, "columns": len(w.columns), "table_dtype": args.table_dtype,
                       "l2": "host run (no GPU)",
                       "parallelism": "%d host core%s" % (threads, "s" if threads > 1 else "")},
            "cpu_baseline": {"value": v, "unit": "rows/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) from
# ncu captures of the full-size launches, one pass each (the capture
# commands are kept with their summaries).  An entry holds while the sources its kernels are
# built from still hash as they did at the capture (KERNEL_SOURCES); once
# they change, the bench reports the traffic as null until it is captured
# again.
KERNEL_SOURCES = {
    "k_forward": ("forward.cu", "common.cuh", "plan.cuh"),
    "backward": ("backward.cu", "radix.cuh", "update.cuh", "common.cuh", "plan.cuh"),
}
TRAFFIC = {
    ("inference", "k_forward"): {"bytes": 493.89e6 + 48.25e6, "src": "a6316c726612c0d0",
                                 "source": "ncu, 1 pass, the full-size launch"},
    ("inference-onehot", "k_forward"): {"bytes": 446.35e6 + 461.28e6, "src": "a6316c726612c0d0",
                                        "source": "ncu, 1 pass, the full-size launch"},
    ("training", "k_forward"): {"bytes": 2888.51e6 + 775.99e6, "src": "a6316c726612c0d0",
                                "source": "ncu, 1 pass, the full-size launch"},
    ("sequences-mean", "k_forward"): {"bytes": 2345.59e6 + 118.51e6, "src": "a6316c726612c0d0",
                                      "source": "ncu, 1 pass, the full-size launch"},
    ("sequences-padded", "k_forward"): {"bytes": 2118.57e6 + 10536.77e6, "src": "a6316c726612c0d0",
                                        "source": "ncu, 1 pass, the full-size launch"},
    ("dynamic", "k_forward"): {"bytes": 73.23e6 + 188.18e6, "src": "a6316c726612c0d0",
                               "source": "ncu, 1 pass, the full-size launch"},
    # the whole backward call: digit histogram, four radix passes, run
    # reduction with Adagrad, fixup
    ("training", "backward"): {"bytes": 12855822848, "src": "1f6e971f78c704da",
                               "source": "ncu, 1 pass, each launch of one full-size call"},
    ("sequences-mean", "backward"): {"bytes": 8857675264, "src": "1f6e971f78c704da",
                                     "source": "ncu, 1 pass, each launch of one full-size call"},
    ("sequences-padded", "backward"): {"bytes": 14028081920, "src": "1f6e971f78c704da",
                                       "source": "ncu, 1 pass, each launch of one full-size call"},
}


def kernel_src_hash(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sparse_lookup_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_for(workload, kernel):
    """{"bytes": DRAM bytes per launch, "source": capture} or None."""
    e = TRAFFIC.get((workload, kernel))
    if e is None or kernel not in KERNEL_SOURCES or e["src"] != kernel_src_hash(kernel):
        return None
    return {"bytes": e["bytes"], "source": e["source"]}


def is_training(args):
    return args.workload in TRAIN_WORKLOADS and not getattr(args, "forward_only", False)


def metric_name(workload, forward_only=False):
    if workload in TRAIN_WORKLOADS and not forward_only:
        return "pooled rows gathered/sec (fwd+bwd+update)"
    if workload.startswith("dynamic"):
        return "pooled rows gathered/sec (hash+fwd+bwd+update+expiry)"
    return "pooled rows gathered/sec (forward)"


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def roofline_obj(nbytes, nbytes_comp, ms, peak, peak_kind, traffic, **extra):
    """HBM roofline of one launch (or call): occurrence-counted bytes (every
    gathered occurrence's row) and compulsory bytes (each distinct row once)
    over its mean event time, against the measured copy bandwidth."""
    ach = nbytes / (ms / 1e3) / 1e9
    achc = nbytes_comp / (ms / 1e3) / 1e9
    out = {"bound": "hbm", "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
           "traffic": traffic.get("bytes") if traffic else None,
           "bytes_per_launch": nbytes, "launch_ms": ms,
           "bytes_compulsory": nbytes_comp, "achieved_compulsory": achc, "frac_compulsory": achc / peak,
           "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs, copy burst)"}
    if traffic:
        out["traffic_dram_gbs"] = traffic["bytes"] / (ms / 1e3) / 1e9
        out["traffic_source"] = traffic["source"]
    out.update(extra)
    return out


def training_leg(torch, sl, args, dev, stream, flush, peak, peak_kind):
    """The fwd + bwd + Adagrad half of the metric, in the same run as the
    forward line: the 200-column training workload (batch 8192, dim 64,
    Zipf(1.1) ids, 3% out of range), device-timed steps with L2 flushed
    between them."""
    import argparse as _ap
    import gc
    w = synth.training()
    a2 = _ap.Namespace(**vars(args))
    a2.steps, a2.warmup, a2.backward, a2.table_dtype = args.training_steps, 3, "sort", "f32"
    res = bench_plan(torch, sl, w, a2, dev, stream, flush, train=True, leg_only=True)
    fw = statistics.mean(res["times"]["fwd"])
    bw = statistics.mean(res["times"]["bwd"])
    out = {"workload": w.name, "columns": len(w.columns), "batch": w.B, "dtype": "f32",
           "ids_per_step": res["config"]["ids_per_step"],
           "rows_gathered_per_step": res["rows_per_step"],
           "distinct_rows_per_step": res["config"]["distinct_rows_per_step"],
           "unique_rows_per_step": res["config"]["unique_rows_per_step"],
           "steps": a2.steps, "warmup": a2.warmup,
           "fwd_ms": fw, "bwd_ms": bw, "step_ms": res["ms_step"],
           "rows_per_s": res["rows_per_step"] / (res["ms_step"] / 1e3),
           "roofline": roofline_obj(res["fbytes"], res["fbytes_compulsory"], fw, peak, peak_kind,
                                    traffic_for("training", "k_forward"), kernel="k_forward"),
           "roofline_backward": roofline_obj(res["bbytes"], res["bbytes_compulsory"], bw, peak, peak_kind,
                                             traffic_for("training", "backward"),
                                             kernels="digit histogram, radix passes, run reduction + Adagrad, "
                                                     "fixup"),
           "gpu_launches": res["launches"], "clocks": res["clocks"],
           "l2": "flushed between steps (2x L2 write, outside events)"}
    del res, w
    gc.collect()
    torch.cuda.empty_cache()
    return out


def run_ours(args):
    import gc
    import torch
    import sparse_lookup_gb300 as sl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = "cuda"
    stream = torch.cuda.current_stream()
    w = make_workload(args.workload, args.columns)
    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(int(2 * l2 // 4), dtype=torch.float32, device=dev)
    if args.workload.startswith("dynamic"):
        res = bench_dynamic(torch, sl, w, args, dev, stream, flush)
    else:
        res = bench_plan(torch, sl, w, args, dev, stream, flush, train=is_training(args))

    clocks = res.pop("clocks")
    ms_step, value = aggregate_ranks(torch, res["ms_step"], res["rows_per_step"], dev)
    _, res["e2e"]["value"] = aggregate_ranks(torch, res["e2e_ms"], res["rows_per_step"], dev)
    peak, peak_kind = peaks()
    fw_ms = statistics.mean(res["times"]["fwd"])
    wl = w.name if args.table_dtype == "f32" else "%s-%s" % (w.name, args.table_dtype)
    line = {
        "metric": metric_name(args.workload, args.forward_only),
        "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": dict(res["config"], workload=w.name, batch=w.B, columns=len(w.columns),
                       l2=("not flushed: steps pipelined; the table's slots and rows exceed L2"
                           if getattr(args, "pipeline", False) else
                           "flushed between steps (2x L2 write, outside events)"),
                       parallelism="replicas" if world > 1 else "1 GPU"),
        "roofline": roofline_obj(res["fbytes"], res.get("fbytes_compulsory", res["fbytes"]), fw_ms, peak, peak_kind,
                                 traffic_for(wl, "k_forward"), kernel="k_forward"),
        "step_ms": {k: statistics.mean(v) for k, v in res["times"].items()},
        "e2e": res["e2e"],
        "gpu_launches": res["launches"],
        "clocks": clocks,
        "cpu_baseline": res.get("cpu"),
        "wall_s_timed": res["wall"],
    }
    if "bbytes" in res:
        b_ms = statistics.mean(res["times"]["bwd"])
        line["roofline_backward"] = roofline_obj(
            res["bbytes"], res["bbytes_compulsory"], b_ms, peak, peak_kind,
            traffic_for(wl, "backward") if args.backward == "sort" else None,
            kernels=("row bitmap, slot compaction, warp-merged atomics, Adagrad pass" if args.backward == "atomic"
                     else "digit histogram, radix passes, run reduction + Adagrad, fixup"))
    if res.get("ceiling"):
        line["gather_ceiling"] = res["ceiling"]
        if "row_bytes" in res:
            # row bytes alone against the rate of row gathers alone
            line["gather_ceiling"]["frac_rows"] = res["row_bytes"] / (fw_ms / 1e3) / 1e9 / res["ceiling"]["mix_gbs"]
    del res
    gc.collect()
    torch.cuda.empty_cache()
    if args.workload == "inference" and args.table_dtype == "f32" and not args.no_training_leg and args.columns is None:
        line["training"] = training_leg(torch, sl, args, dev, stream, flush, peak, peak_kind)
        line["gpu_launches"] += line["training"]["gpu_launches"]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def row_stats(w, rows_dbg, n_ids):
    """From the library's transformed rows: valid (read) values per column,
    distinct rows read per table, and bags with at least one valid value per
    column.  Values past a padded column's pad_len (or a pooled column's
    max_len) are not read."""
    r = rows_dbg.cpu().numpy()
    valid, nonempty, per_table = [], [], {}
    pos = {0: 0, 1: n_ids}
    for c, o in zip(w.columns, w.offsets):
        s = 1 if c.transform == "bucketize" else 0
        n = int(o[-1])
        rr = r[pos[s]:pos[s] + n]
        pos[s] += n
        o64 = np.asarray(o, np.int64)
        bag = np.repeat(np.arange(w.B), np.diff(o64))
        keep = rr >= 0
        cut = c.pad_len if c.pooling == "padded" else int(getattr(c, "max_len", 0) or 0)
        if cut > 0 and n:
            keep &= (np.arange(n) - o64[bag]) < cut
        valid.append(int(keep.sum()))
        nonempty.append(int(np.count_nonzero(np.bincount(bag[keep], minlength=w.B))) if n else 0)
        per_table.setdefault(c.table, []).append(rr[keep])
    uniq = {t: int(np.unique(np.concatenate(v)).size) for t, v in per_table.items()}
    return {"valid": valid, "nonempty_bags": nonempty, "unique_per_table": uniq}


def valid_counts(w, rows_dbg, n_ids):
    return row_stats(w, rows_dbg, n_ids)["valid"]


def bench_plan(torch, sl, w, args, dev, stream, flush, train, leg_only=False):
    """Time the workload's steps (forward, and for training plans backward +
    Adagrad).  leg_only: only the device-timed steps (no end-to-end leg, graph,
    gather ceiling or CPU baseline)."""
    tables = [None if t is None else synth.make_table(t, dev) for t in w.tables]
    accs = [None if t is None else torch.zeros_like(t) for t in tables] if train else None
    ids_h, id_off_h, fv_h, f_off_h = synth.jagged(w)
    n_ids, n_f = ids_h.size, fv_h.size
    has_id, has_f = id_off_h.size > 1, f_off_h.size > 1
    ids = torch.from_numpy(ids_h).to(dev) if has_id else None
    id_off = torch.from_numpy(id_off_h).to(dev) if has_id else None
    fv = torch.from_numpy(fv_h).to(dev) if has_f else None
    f_off = torch.from_numpy(f_off_h).to(dev) if has_f else None
    n_all = n_ids + n_f
    dt = args.table_dtype
    scales = None
    if dt != "f32":
        if train:
            raise SystemExit("low-precision tables are read-only: forward workloads only")
        conv = [None if t is None else synth.lowp_table(t, dt) for t in tables]
        tables = [None if x is None else x[0] for x in conv]
        scales = [None if x is None else x[1] for x in conv]
        del conv
    plan = sl.Plan(w.columns, tables, accs, max_batch=w.B, max_ids=max(n_all, 1) if train else 0, training=train,
                   backward=args.backward if train else "sort", row_scales=scales)

    rows_dbg = torch.empty(max(n_all, 1), dtype=torch.int64, device=dev)
    out, seq = plan.forward(w.B, ids, id_off, fv, f_off, rows_dbg=rows_dbg)
    torch.cuda.synchronize()
    if plan.device_status() != 0:
        raise SystemExit("device status after the forward")
    stats = row_stats(w, rows_dbg, n_ids)
    valid = stats["valid"]
    del rows_dbg
    rows_per_step = sum(valid)
    fbytes = forward_bytes(w, valid, dt)
    res = {"rows_per_step": rows_per_step, "fbytes": fbytes,
           "fbytes_compulsory": forward_bytes_compulsory(w, stats, dt),
           "row_bytes": sum(nv * row_bytes(c, dt) for c, nv in zip(w.columns, valid)),
           "config": {"ids_per_step": n_all, "rows_gathered_per_step": rows_per_step, "table_dtype": dt,
                      "distinct_rows_per_step": int(sum(stats["unique_per_table"].values()))}}
    G = Gseq = None
    if train:
        width = plan.out_width
        G = synth.make_grad((w.B, max(width, 1)), 77, dev)[:, :width].contiguous() if width else None
        Gseq = synth.make_grad((w.B * plan.seq_per_bag,), 78, dev) if plan.seq_per_bag else None
        dbg = plan.backward_update(G, Gseq, w.lr, w.eps, debug=True)
        torch.cuda.synchronize()
        n_unique = int(dbg["row"].numel())
        del dbg
        res["bbytes"] = backward_bytes(w, n_all, valid, n_unique, max(c.dim for c in w.columns))
        res["bbytes_compulsory"] = backward_bytes_compulsory(w, n_all, stats, n_unique,
                                                             max(c.dim for c in w.columns))
        res["config"]["unique_rows_per_step"] = n_unique
        res["config"]["backward"] = args.backward

    def body(i, marks):
        a, b = event_pair(torch)
        a.record(stream)
        plan.forward(w.B, ids, id_off, fv, f_off, out=out, seq_out=seq)
        b.record(stream)
        marks["fwd"] = (a, b)
        if train:
            c, d = event_pair(torch)
            c.record(stream)
            plan.backward_update(G, Gseq, w.lr, w.eps)
            d.record(stream)
            marks["bwd"] = (c, d)
        marks["step"] = (a, d if train else b)

    for _ in range(max(3, args.warmup)):
        body(0, {})
    torch.cuda.synchronize()
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    time.sleep(0.3)
    times, wall = timed_steps(torch, args.steps, stream, flush, body)
    res["clocks"] = clk.stop()
    res["times"] = {k: v for k, v in times.items() if k != "step"}
    res["ms_step"] = statistics.mean(times["step"])
    res["wall"] = wall
    bwd_launches = 0
    if train:
        # sort: histogram, passes, run reduction, fixup; atomic: mark, count,
        # scan, emit, scatter, update
        bwd_launches = 6 if args.backward == "atomic" else 3 + plan_sort_passes(plan)
    res["launches"] = args.steps * (1 + bwd_launches)
    if plan.device_status() != 0:
        raise SystemExit("device status after the timed steps")
    if leg_only:
        return res

    # end to end through the C ABI with pinned host buffers
    host = [(torch.from_numpy(x).pin_memory(), d) for x, d in ((ids_h, ids), (id_off_h, id_off), (fv_h, fv),
                                                              (f_off_h, f_off)) if d is not None]
    # upstream gradients come from the caller too; the step's result read back
    # is the forward output (pooled and, for padded columns, unpooled)
    g_host = G.cpu().pin_memory() if G is not None else None
    gs_host = Gseq.cpu().pin_memory() if Gseq is not None else None
    out_p = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    seq_p = torch.empty(seq.shape, dtype=seq.dtype).pin_memory() if seq is not None else None
    h2d = sum(x.numel() * x.element_size() for x, _ in host) + sum(
        x.numel() * 4 for x in (g_host, gs_host) if x is not None)
    d2h = sum(x.numel() * x.element_size() for x in (out_p, seq_p) if x is not None)

    def e2e_body(i, marks):
        a, b = event_pair(torch)
        a.record(stream)
        for src, dst in host:
            dst.copy_(src, non_blocking=True)
        if g_host is not None:
            G.copy_(g_host, non_blocking=True)
        if gs_host is not None:
            Gseq.copy_(gs_host, non_blocking=True)
        plan.forward(w.B, ids, id_off, fv, f_off, out=out, seq_out=seq)
        out_p.copy_(out, non_blocking=True)
        if seq_p is not None:
            seq_p.copy_(seq, non_blocking=True)
        if train:
            plan.backward_update(G, Gseq, w.lr, w.eps)
        b.record(stream)
        marks["e2e"] = (a, b)

    for _ in range(3):
        e2e_body(0, {})
    et, _ = timed_steps(torch, args.steps, stream, flush, e2e_body)
    res["e2e_ms"] = statistics.mean(et["e2e"])
    res["e2e"] = {"value": rows_per_step / (res["e2e_ms"] / 1e3), "unit": "rows/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "mode": "one step at a time: H2D, step, D2H in order on one stream"}
    # The same steps streamed: the next step's inputs copied in and the last
    # step's output copied out beside this step's kernels (double buffers,
    # three streams).  Needs a second set of the step's device buffers; for
    # steps whose copies are tiny (under 1 MB) there is nothing to overlap
    # and the one-step-at-a-time figure stands.
    extra = h2d + d2h
    if (1 << 20) <= extra < (8 << 30):
        ms = e2e_pipelined(torch, plan, w, args.steps, stream, flush, host, (G, g_host), (Gseq, gs_host),
                           (out, out_p), (seq, seq_p), train, (ids, id_off, fv, f_off))
        serial = res["e2e"]
        res["e2e"] = {"value": rows_per_step / (ms / 1e3), "unit": "rows/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "mode": "streamed: step i+1's H2D and step i-1's D2H beside step i (double buffers, "
                              "three streams, L2 flushed before each step inside the timed region)",
                      "one_step_at_a_time": {"value": serial["value"], "ms_per_step": res["e2e_ms"]},
                      "ms_per_step": ms}
        res["e2e_ms"] = ms
    if args.graph:
        # whole steps captured in a CUDA graph (up to 100 steps per graph, so
        # that one graph launch from the host covers many steps) and replayed
        # back to back: the steps without per-launch host cost (L2 not flushed
        # between steps)
        per = min(args.graph, 100)
        reps = max(1, args.graph // per)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="relaxed"):
            for _ in range(per):
                plan.forward(w.B, ids, id_off, fv, f_off, out=out, seq_out=seq)
                if train:
                    plan.backward_update(G, Gseq, w.lr, w.eps)
        g.replay()
        torch.cuda.synchronize()
        a, b = event_pair(torch)
        a.record(stream)
        for _ in range(reps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        us = a.elapsed_time(b) * 1e3 / (reps * per)
        res["config"]["graph"] = {"steps": reps * per, "steps_per_graph": per, "us_per_step": us,
                                  "rows_per_s": rows_per_step / (us * 1e-6),
                                  "l2": "not flushed between steps"}
        if plan.device_status() != 0:
            raise SystemExit("device status after the graph replays")
    res["ceiling"] = gather_ceiling(torch, sl, row_sizes_mix(w, valid, dt), dev) if not args.no_ceiling else None
    if not args.no_cpu_baseline and dist_env()[0] == 0:
        if train:
            rate, sample = cpu_train_sample(w, tables, G, budget_s=12.0)
            res["cpu"] = {"value": rate, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": sample}
        else:
            res["cpu"] = cpu_forward_baseline(w, tables, table_dtype=dt, scales_dev=scales)
    return res


def e2e_pipelined(torch, plan, w, steps, comp, flush, host, g_pair, gs_pair, out_pair, seq_pair, train,
                  dev_inputs):
    """Mean ms per step of `steps` whole steps through the public calls with
    every step's inputs copied in from pinned host memory and its pooled
    output copied back: inputs of step i+1 on one stream, the step's kernels
    on `comp`, the output of step i-1 on a third, so the copies overlap the
    kernels.  Two sets of device buffers alternate; a step waits for the
    copy-in of its own inputs, and a buffer is refilled only after the step
    that used it (kernels and copy-out) is done."""
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ids, id_off, fv, f_off = dev_inputs
    names = [d for _, d in host]
    bufs = [names, [torch.empty_like(d) for d in names]]
    G, g_host = g_pair
    Gseq, gs_host = gs_pair
    out, out_p = out_pair
    seq, seq_p = seq_pair
    Gb = [G, torch.empty_like(G) if G is not None else None]
    Gsb = [Gseq, torch.empty_like(Gseq) if Gseq is not None else None]
    outb = [out, torch.empty_like(out)]
    seqb = [seq, torch.empty_like(seq) if seq is not None else None]
    outp = [out_p, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
    seqp = [seq_p, torch.empty(seq.shape, dtype=seq.dtype).pin_memory() if seq is not None else None]

    slot = {id(d): k for k, d in enumerate(names)}

    def dev_of(b, t):
        # device input t (ids, offsets, values, offsets) of buffer set b
        return None if t is None else bufs[b][slot[id(t)]]

    def run(k):
        ev_in = [torch.cuda.Event() for _ in range(k)]
        ev_fwd = [torch.cuda.Event() for _ in range(k)]
        ev_done = [torch.cuda.Event() for _ in range(k)]
        ev_out = [torch.cuda.Event() for _ in range(k)]
        a, b_ = event_pair(torch)
        torch.cuda.synchronize()
        a.record(s_in)
        for i in range(k):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev_done[i - 2])
            with torch.cuda.stream(s_in):
                for (src, _), dst in zip(host, bufs[b]):
                    dst.copy_(src, non_blocking=True)
                if g_host is not None:
                    Gb[b].copy_(g_host, non_blocking=True)
                if gs_host is not None:
                    Gsb[b].copy_(gs_host, non_blocking=True)
            ev_in[i].record(s_in)
            comp.wait_event(ev_in[i])
            if i >= 2:
                comp.wait_event(ev_out[i - 2])
            flush.fill_(float(i))
            plan.forward(w.B, dev_of(b, ids), dev_of(b, id_off), dev_of(b, fv), dev_of(b, f_off), out=outb[b],
                         seq_out=seqb[b], stream=comp)
            ev_fwd[i].record(comp)
            if train:
                plan.backward_update(Gb[b], Gsb[b], w.lr, w.eps, stream=comp)
            s_out.wait_event(ev_fwd[i])
            with torch.cuda.stream(s_out):
                outp[b].copy_(outb[b], non_blocking=True)
                if seqp[b] is not None:
                    seqp[b].copy_(seqb[b], non_blocking=True)
            ev_out[i].record(s_out)
            ev_done[i].record(comp)
        s_out.wait_event(ev_done[k - 1])
        b_.record(s_out)
        torch.cuda.synchronize()
        return a.elapsed_time(b_) / k

    run(3)
    ms = run(steps)
    if plan.device_status() != 0:
        raise SystemExit("device status after the streamed steps")
    return ms


def plan_sort_passes(plan):
    """Radix passes of the backward: 8 bits of the global row key per pass."""
    tables = {}
    for c in plan.columns:
        tables[c.table] = int(c.num_rows)
    bits = max(1, int(sum(tables.values())).bit_length())
    return (bits + 7) // 8


def bench_dynamic(torch, sl, w, args, dev, stream, flush):
    ex = w.extra
    C, B = len(w.columns), w.B
    dim = w.columns[0].dim
    nsteps = max(3, args.warmup) + args.steps * (2 if args.pipeline else 1)
    # every step's keys resident on the device before timing
    batches = []
    max_n = 0
    for t in range(nsteps):
        offs, keys = synth.dynamic_keys(w.seed, t, C, B, ex["alpha"], ex["key_bits"])
        tids = np.concatenate([np.full(k.size, c, np.int32) for c, k in enumerate(keys)])
        allk = np.concatenate(keys)
        lens = np.concatenate([np.diff(o) for o in offs])
        off = np.zeros(lens.size + 1, np.int32)
        np.cumsum(lens, out=off[1:])
        batches.append((torch.from_numpy(tids).to(dev), torch.from_numpy(allk).to(dev), torch.from_numpy(off).to(dev),
                        tids, allk, off))
        max_n = max(max_n, allk.size)
    ht = sl.HashTable(ex["num_slots"], ex["row_capacity"], dim, ex["threshold"], ex["max_probes"],
                      ex["init_seed"], ex["init_scale"], max_n)
    plan = sl.Plan(w.columns, [ht.weight], [ht.acc], max_batch=B, max_ids=max_n, training=True,
                   backward=args.backward)
    out = torch.empty((B, plan.out_width), device=dev)
    G = synth.make_grad((B, plan.out_width), 77, dev)
    rows = torch.empty(max_n, dtype=torch.int64, device=dev)
    state = {"t": 0, "rows": 0}

    def body(i, marks):
        t = state["t"]
        tids, keys, off = batches[t][:3]
        n = keys.numel()
        a, b = event_pair(torch)
        c, d = event_pair(torch)
        e, f = event_pair(torch)
        a.record(stream)
        ht.lookup_or_insert(tids, keys, t, rows_out=rows[:n])
        b.record(stream)
        plan.forward(B, rows[:n], off, None, None, out=out)
        c.record(stream)
        plan.backward_update(G, None, w.lr, w.eps)
        d.record(stream)
        ht.evict_expired(t, ex["ttl"])
        e.record(stream)
        marks["hash"] = (a, b)
        marks["fwd"] = (b, c)
        marks["bwd"] = (c, d)
        marks["evict"] = (d, e)
        marks["step"] = (a, e)
        state["t"] = t + 1

    # the first call meets a cold table (every key new); reported beside the
    # steady-state steps, not inside them
    warm = []
    for _ in range(max(3, args.warmup)):
        m = {}
        body(0, m)
        warm.append(m)
    torch.cuda.synchronize()
    first_step = {k: warm[0][k][0].elapsed_time(warm[0][k][1]) for k in ("hash", "fwd", "bwd", "evict", "step")}
    clk = ClockSampler(torch.cuda.current_device())
    clk.start()
    time.sleep(0.3)
    t_first = state["t"]
    if args.pipeline:
        times, wall = pipelined_steps(torch, ht, plan, batches, state, w, args, stream, G, out)
    else:
        times, wall = timed_steps(torch, args.steps, stream, flush, body)
    clocks = clk.stop()
    # valid rows and bytes, from the library's own rows of the last timed step
    n_last = batches[state["t"] - 1][1].numel()
    r = (state["rows_last"] if "rows_last" in state else rows[:n_last]).cpu().numpy()
    valid = int((r >= 0).sum())
    width = plan.out_width
    fbytes = (C * (B + 1) * 4 + n_last * 8 + valid * 4 * dim + B * 4 * width)
    res = {"rows_per_step": valid, "fbytes": fbytes, "clocks": clocks,
           "times": {k: v for k, v in times.items() if k != "step"},
           "ms_step": statistics.mean(times["step"] if "step" in times else times["pipelined_step"]), "wall": wall,
           "config": {"ids_per_step": n_last, "rows_gathered_per_step": valid, "num_slots": ex["num_slots"],
                      "row_capacity": ex["row_capacity"], "threshold": ex["threshold"], "ttl": ex["ttl"],
                      "stream_steps_timed": [t_first, state["t"] - 1],
                      "cold_first_step_ms": first_step, "backward": args.backward,
                      "pipeline": bool(args.pipeline),
                      "sequential_unflushed_ms": state.get("sequential_unflushed_ms")},
           "launches": args.steps * (16 + 1 + (6 if args.backward == "atomic" else 3 + plan_sort_passes(plan))
                                     + 1)}
    if ht.device_status() not in (0, 5) or plan.device_status() != 0:
        raise SystemExit("device status after the timed steps")

    # end to end: keys, table ids and offsets from pinned host memory
    hb = [(torch.from_numpy(x).pin_memory(), d) for x, d in ((batches[0][3], batches[0][0]),
                                                            (batches[0][4], batches[0][1]),
                                                            (batches[0][5], batches[0][2]))]
    out_p = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x, _ in hb)

    def e2e_body(i, marks):
        a, b = event_pair(torch)
        a.record(stream)
        for src, dst in hb:
            dst.copy_(src, non_blocking=True)
        t = state["t"]
        n = batches[0][1].numel()
        ht.lookup_or_insert(batches[0][0], batches[0][1], t, rows_out=rows[:n])
        plan.forward(B, rows[:n], batches[0][2], None, None, out=out)
        out_p.copy_(out, non_blocking=True)
        plan.backward_update(G, None, w.lr, w.eps)
        ht.evict_expired(t, ex["ttl"])
        b.record(stream)
        marks["e2e"] = (a, b)
        state["t"] = t + 1

    et, _ = timed_steps(torch, min(args.steps, 5), stream, flush, e2e_body)
    res["e2e_ms"] = statistics.mean(et["e2e"])
    res["e2e"] = {"value": valid / (res["e2e_ms"] / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": out_p.numel() * 4,
                  "mode": "one step at a time: H2D, step, D2H in order on one stream"}
    # the same steps streamed (the keys of step i+1 copied in and the pooled
    # output of step i copied out beside the step's kernels)
    ms = e2e_dynamic_streamed(torch, ht, plan, w, min(args.steps, 5), stream, flush, hb, rows, out, out_p, G,
                              state)
    serial = res["e2e"]
    res["e2e"] = {"value": valid / (ms / 1e3), "unit": "rows/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": out_p.numel() * 4,
                  "mode": "streamed: step i+1's keys in and step i's pooled output out beside the step's kernels "
                          "(double buffers, three streams, L2 flushed before each step inside the timed region)",
                  "one_step_at_a_time": {"value": serial["value"], "ms_per_step": res["e2e_ms"]},
                  "ms_per_step": ms}
    res["e2e_ms"] = ms
    res["ceiling"] = gather_ceiling(torch, sl, {dim * 4: valid}, dev) if not args.no_ceiling else None
    if not args.no_cpu_baseline and dist_env()[0] == 0:
        rate, sample = cpu_dynamic_sample(w, budget_s=12.0)
        res["cpu"] = {"value": rate, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": sample}
    return res


def e2e_dynamic_streamed(torch, ht, plan, w, steps, comp, flush, hb, rows, out, out_p, G, state):
    """Mean ms per dynamic-table step through the public calls, every step's
    keys, table ids and offsets copied in from pinned host memory and its
    pooled output copied back, the copies on their own streams beside the
    kernels (two sets of device buffers; a set is refilled only after the
    step that used it is done)."""
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    B, ttl = w.B, w.extra["ttl"]
    bufs = [[d for _, d in hb], [torch.empty_like(d) for _, d in hb]]
    outb = [out, torch.empty_like(out)]
    outp = [out_p, torch.empty(out.shape, dtype=out.dtype).pin_memory()]
    n = hb[1][1].numel()

    def run(k):
        ev_in = [torch.cuda.Event() for _ in range(k)]
        ev_fwd = [torch.cuda.Event() for _ in range(k)]
        ev_done = [torch.cuda.Event() for _ in range(k)]
        ev_out = [torch.cuda.Event() for _ in range(k)]
        a, b_ = event_pair(torch)
        torch.cuda.synchronize()
        a.record(s_in)
        for i in range(k):
            b = i % 2
            if i >= 2:
                s_in.wait_event(ev_done[i - 2])
            with torch.cuda.stream(s_in):
                for (src, _), dst in zip(hb, bufs[b]):
                    dst.copy_(src, non_blocking=True)
            ev_in[i].record(s_in)
            comp.wait_event(ev_in[i])
            if i >= 2:
                comp.wait_event(ev_out[i - 2])
            flush.fill_(float(i))
            t = state["t"]
            tids, keys, off = bufs[b]
            ht.lookup_or_insert(tids, keys, t, rows_out=rows[:n], stream=comp)
            plan.forward(B, rows[:n], off, None, None, out=outb[b], stream=comp)
            ev_fwd[i].record(comp)
            s_out.wait_event(ev_fwd[i])
            with torch.cuda.stream(s_out):
                outp[b].copy_(outb[b], non_blocking=True)
            ev_out[i].record(s_out)
            plan.backward_update(G, None, w.lr, w.eps, stream=comp)
            ht.evict_expired(t, ttl, stream=comp)
            ev_done[i].record(comp)
            state["t"] = t + 1
        s_out.wait_event(ev_done[k - 1])
        b_.record(s_out)
        torch.cuda.synchronize()
        return a.elapsed_time(b_) / k

    run(2)
    ms = run(steps)
    if ht.device_status() not in (0, 5) or plan.device_status() != 0:
        raise SystemExit("device status after the streamed steps")
    return ms


def pipelined_steps(torch, ht, plan, batches, state, w, args, stream, G, out):
    """K dynamic-table steps through DynamicPipeline: the lookup of step t+1
    and the expiry of step t on a low-priority stream beside step t's
    backward.  Steps overlap, so L2 is not flushed between them (the table's
    slots and rows are larger than L2); the time is the whole window / K,
    pipeline fill and drain included."""
    from sparse_lookup_gb300.pipeline import DynamicPipeline
    B = w.B
    max_n = max(b[1].numel() for b in batches)
    ttl = w.extra["ttl"]
    k = args.steps
    # the same steps in order on one stream, unflushed, for comparison
    rows = torch.empty(max_n, dtype=torch.int64, device=out.device)
    t0 = state["t"]
    torch.cuda.synchronize()
    a, b = event_pair(torch)
    a.record(stream)
    for t in range(t0, t0 + k):
        tids, keys, off = batches[t][:3]
        n = keys.numel()
        ht.lookup_or_insert(tids, keys, t, rows_out=rows[:n])
        plan.forward(B, rows[:n], off, None, None, out=out)
        plan.backward_update(G, None, w.lr, w.eps)
        ht.evict_expired(t, ttl)
    b.record(stream)
    torch.cuda.synchronize()
    state["sequential_unflushed_ms"] = a.elapsed_time(b) / k
    pipe = DynamicPipeline(ht, plan, ttl, B, max_n)
    t0 = t0 + k
    sync_ranks(torch)
    torch.cuda.synchronize()
    a, b = event_pair(torch)
    wall0 = time.perf_counter()
    a.record(stream)
    pipe.prefetch(t0, batches[t0][0], batches[t0][1])
    fwd = []
    for t in range(t0, t0 + k):
        fwd.append(event_pair(torch))
        pipe.forward(t, batches[t][2], out, events=fwd[-1])
        if t + 1 < t0 + k:
            pipe.prefetch(t + 1, batches[t + 1][0], batches[t + 1][1])
        pipe.backward(G, w.lr, w.eps)
    pipe.finish()
    b.record(stream)
    torch.cuda.synchronize()
    sync_ranks(torch)
    wall = time.perf_counter() - wall0
    state["t"] = t0 + k
    # the library's rows of the last step, for the valid-row count
    n_last = batches[t0 + k - 1][1].numel()
    state["rows_last"] = pipe.rows[(t0 + k - 1) % 2][:n_last]
    return {"pipelined_step": [a.elapsed_time(b) / k] * k, "fwd": [x.elapsed_time(y) for x, y in fwd]}, wall


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="inference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ceiling", action="store_true")
    ap.add_argument("--columns", type=int, default=None, help="number of columns (smaller profiling cases)")
    ap.add_argument("--forward-only", action="store_true",
                    help="training workloads: time the forward alone (inference over the same inputs)")
    ap.add_argument("--table-dtype", default="f32", choices=["f32", "bf16", "f16", "i8"],
                    help="forward workloads: store the tables as bf16, fp16 or int8 with per-row scales")
    ap.add_argument("--pipeline", action="store_true",
                    help="dynamic workload: pipelined steps (next lookup beside this backward)")
    ap.add_argument("--backward", default="sort", choices=["sort", "atomic"],
                    help="training workloads: the sort-based backward or the atomic one")
    ap.add_argument("--no-training-leg", action="store_true",
                    help="inference workload: skip the training (fwd + bwd + Adagrad) leg of the line")
    ap.add_argument("--training-steps", type=int, default=10,
                    help="timed steps of the training leg")
    ap.add_argument("--graph", type=int, default=0,
                    help="also time this many steps captured in CUDA graphs of up to 100 steps, replayed back to back")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
