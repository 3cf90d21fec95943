"""Benchmark of the GB300 multi-column embedding front end.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload inference|training|sequences-mean|sequences-padded|dynamic|tiny]

One JSON line on rank 0.  Default workload: the 1000-column inference
forward (700 hash-mod + 300 bucketize columns, batch 512).  A step is one
fused forward over one batch (training workloads: forward + backward +
Adagrad).  Inputs are resident in HBM before timing; L2 is flushed (a write of
twice its size) between timed steps, outside the per-step CUDA events.

value    pooled rows gathered per second (valid IDs whose row was read)
roofline algorithmic bytes of the dominant kernel per launch / its mean event
         time, against the measured HBM copy bandwidth
e2e      the same metric through the C ABI with pinned HOST inputs: H2D of the
         step's IDs and offsets, the forward, D2H of the pooled output
cpu_baseline the CPU oracle on a bounded sample of the same workload
--impl reference  times the CPU oracle (the reference arm of this build).
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


def make_workload(name, columns=None):
    if name == "inference":
        if columns:
            return synth.inference(n_cat=columns * 7 // 10, n_num=columns - columns * 7 // 10)
        return synth.inference()
    if name == "training":
        return synth.training()
    if name == "sequences-mean":
        return synth.sequences(mode="mean")
    if name == "sequences-padded":
        return synth.sequences(mode="padded")
    if name == "tiny":
        return synth.tiny()
    raise SystemExit("unknown workload %s" % name)


def forward_bytes(w, rows_valid_per_col):
    """Algorithmic bytes of one forward: per column the offsets, the values,
    the boundaries, one row read per valid value and one output row write per
    bag (padded columns: pad_len rows per bag)."""
    total = 0
    for c, o, nv in zip(w.columns, w.offsets, rows_valid_per_col):
        n = int(o[-1])
        e = 4 if c.transform == "bucketize" else 8
        nb = 0 if c.boundaries is None else c.boundaries.size
        total += (w.B + 1) * 4 + n * e + 4 * nb + nv * 4 * c.dim
        total += w.B * 4 * c.dim * (c.pad_len if c.pooling == "padded" else 1)
    return total


def cpu_oracle_rate(w, tables_dev, budget_s=12.0):
    """The oracle (single thread) on a bounded sample: whole columns, in
    order, until about budget_s of CPU work.  Returns (rows/s, sample text)."""
    import oracle
    t_used, rows_done, cols_done = 0.0, 0, 0
    for ci, c in enumerate(w.columns):
        tab = tables_dev[c.table].cpu().numpy()
        spec = synth.ColumnSpec(c.transform, c.pooling, c.num_rows, c.dim, 0, boundaries=c.boundaries,
                                default=c.default, pad_len=c.pad_len)
        t0 = time.perf_counter()
        _, _, rows = oracle.forward([spec], w.B, [w.offsets[ci]], [w.values[ci]], [tab], want_rows=True)
        t_used += time.perf_counter() - t0
        rows_done += int((rows[0] >= 0).sum())
        cols_done += 1
        if t_used > budget_s:
            break
    sample = "%d of %d columns, all %d bags each (%d rows gathered), oracle forward, 1 thread" % (
        cols_done, len(w.columns), w.B, rows_done)
    return rows_done / t_used, sample, cols_done


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import torch
    w = make_workload(args.workload)
    dev = "cpu"
    tables = [None if t is None else synth.make_table(t, dev) for t in w.tables]
    times, rows = [], 0
    for i in range(args.warmup + args.steps):
        rate, sample, _ = cpu_oracle_rate(w, tables, budget_s=max(2.0, 20.0 / max(1, args.steps + args.warmup)))
        if i >= args.warmup:
            times.append(rate)
    v = statistics.mean(times)
    line = {"impl": "reference", "metric": "pooled rows gathered/sec (forward)", "value": v, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "f32", "data": "synthetic", "config": {"workload": w.name, "batch": w.B,
                                                            "columns": len(w.columns)},
            "cpu_baseline": {"value": v, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    import sparse_lookup_gb300 as sl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = "cuda"
    w = make_workload(args.workload, args.columns)
    tables = [None if t is None else synth.make_table(t, dev) for t in w.tables]
    ids_h, id_off_h, fv_h, f_off_h = synth.jagged(w)
    n_ids, n_f = ids_h.size, fv_h.size
    ids = torch.from_numpy(ids_h).to(dev) if n_ids or id_off_h.size > 1 else None
    id_off = torch.from_numpy(id_off_h).to(dev) if id_off_h.size > 1 else None
    fv = torch.from_numpy(fv_h).to(dev) if f_off_h.size > 1 else None
    f_off = torch.from_numpy(f_off_h).to(dev) if f_off_h.size > 1 else None
    plan = sl.Plan(w.columns, tables, None, max_batch=w.B)
    stream = torch.cuda.current_stream()

    # one untimed call to count the valid rows (from the library's own rows)
    rows_dbg = torch.empty(n_ids + n_f, dtype=torch.int64, device=dev)
    out, seq = plan.forward(w.B, ids, id_off, fv, f_off, rows_dbg=rows_dbg)
    torch.cuda.synchronize()
    st = plan.device_status()
    if st != 0:
        raise SystemExit("device status %d" % st)
    r = rows_dbg.cpu().numpy()
    valid_per_col, pos = [], {0: 0, 1: n_ids}
    for c, o in zip(w.columns, w.offsets):
        s = 1 if c.transform == "bucketize" else 0
        n = int(o[-1])
        valid_per_col.append(int((r[pos[s]:pos[s] + n] >= 0).sum()))
        pos[s] += n
    del rows_dbg
    rows_per_step = sum(valid_per_col)
    fbytes = forward_bytes(w, valid_per_col)

    l2 = torch.cuda.get_device_properties(local).L2_cache_size
    flush = torch.empty(int(2 * l2 // 4), dtype=torch.float32, device=dev)

    def step():
        plan.forward(w.B, ids, id_off, fv, f_off, out=out, seq_out=seq)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clk = ClockSampler(local)
    clk.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(float(i))
        evs[i][0].record(stream)
        step()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        torch.distributed.barrier()
    clocks = clk.stop()
    ms = [a.elapsed_time(b) for a, b in evs]
    ms_step = statistics.mean(ms)
    if world > 1:
        t = torch.tensor([ms_step], device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms_step = float(t.item())
    value = rows_per_step * world / (ms_step / 1e3)
    achieved = fbytes / (ms_step / 1e3) / 1e9
    peak, peak_kind = peaks()

    # end to end through the C ABI with pinned host buffers
    ids_p = torch.from_numpy(ids_h).pin_memory() if ids is not None else None
    id_off_p = torch.from_numpy(id_off_h).pin_memory() if id_off is not None else None
    fv_p = torch.from_numpy(fv_h).pin_memory() if fv is not None else None
    f_off_p = torch.from_numpy(f_off_h).pin_memory() if f_off is not None else None
    out_p = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(x.numel() * x.element_size() for x in (ids_p, id_off_p, fv_p, f_off_p) if x is not None)
    d2h = out_p.numel() * out_p.element_size()

    def e2e_step():
        for src, dst in ((ids_p, ids), (id_off_p, id_off), (fv_p, fv), (f_off_p, f_off)):
            if src is not None:
                dst.copy_(src, non_blocking=True)
        step()
        out_p.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e_ms = []
    for i in range(args.steps):
        flush.fill_(float(i))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e_ms.append(a.elapsed_time(b))
    e2e_value = rows_per_step * world / (statistics.mean(e_ms) / 1e3)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        rate, sample, _ = cpu_oracle_rate(w, tables, budget_s=12.0)
        cpu = {"value": rate, "unit": "rows/s", "cores": 1, "kind": "oracle", "sample": sample}

    line = {
        "metric": "pooled rows gathered/sec (forward)",
        "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak" if world > 1 else "none",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.B, "columns": len(w.columns), "ids_per_step": n_ids + n_f,
                   "rows_gathered_per_step": rows_per_step, "l2": "flushed between steps (2x L2 write, outside events)",
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": None, "kernel": "k_forward",
                     "bytes_per_launch": fbytes, "peak_source": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)"},
        "e2e": {"value": e2e_value, "unit": "rows/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
        "wall_s_timed": t_wall,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="inference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--columns", type=int, default=None, help="inference: number of columns (profiling)")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
