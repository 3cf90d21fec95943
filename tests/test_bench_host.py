"""Host-side parts of the benchmark that need no GPU: the CPU baseline of the
forward workloads (the oracle run on one thread, and on all host cores with
columns split over threads) and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    sys.path.insert(0, ROOT)
    from oracle import build as obuild
    obuild.build()
    import bench as b
    return b


def _small(seed=3):
    from sparse_lookup_gb300 import synth
    return synth.random_small(seed, C=6, B=40, train=False, allow_padded=False)


def test_threaded_oracle_counts_the_same_rows(bench):
    """Columns split over threads gather exactly the rows one thread does, in
    whole passes over the sampled columns."""
    w = _small()
    tables = bench.HostTables(w)
    rate1, sample1 = bench.cpu_forward_sample(w, tables, budget_s=0.2)
    rate4, sample4 = bench.cpu_forward_sample_threads(w, tables, 4, budget_s=0.2)
    assert rate1 > 0 and rate4 > 0
    one_pass = int(sample1.split("(")[1].split()[0])
    passes = int(sample4.split(" passes")[0].split()[-1])
    rows = int(sample4.split("(")[1].split()[0])
    assert "6 of 6 columns" in sample1 and "6 of 6 columns" in sample4
    assert rows == passes * one_pass


def test_threaded_oracle_respects_the_host_memory_bound(bench):
    """Only the first columns whose tables fit in host_bytes are sampled
    (always at least one)."""
    w = _small(4)
    tables = bench.HostTables(w)
    _, sample = bench.cpu_forward_sample_threads(w, tables, 2, budget_s=0.05, host_bytes=1)
    assert sample.startswith("1 of 6 columns")


def test_forward_baseline_reports_cores_and_one_core_rate(bench, monkeypatch):
    w = _small(5)
    tables = bench.HostTables(w)
    monkeypatch.setattr(bench, "host_cores", lambda: 3)
    cb = bench.cpu_forward_baseline(w, tables, budget_s=0.3)
    assert cb["kind"] == "oracle" and cb["unit"] == "rows/s" and cb["cores"] == 3
    assert cb["value"] > 0 and cb["one_core"]["value"] > 0
    assert "split over 3 threads" in cb["sample"]
    monkeypatch.setattr(bench, "host_cores", lambda: 1)
    cb1 = bench.cpu_forward_baseline(w, tables, budget_s=0.3)
    assert cb1["cores"] == 1 and "one_core" not in cb1


def test_reference_arm_line():
    """`bench.py --impl reference` prints one JSON line with the contract's
    keys, timing the oracle on the host (no GPU needed)."""
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny", "--steps", "1", "--warmup", "1"], capture_output=True, text=True, timeout=300,
                       cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "cpu_baseline", "e2e", "config"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def _rows_dbg(w):
    """The transformed row of every value as the library reports it (rows of
    values past a cut included), from the oracle, laid out id stream first."""
    import numpy as np
    import torch

    import oracle
    tabs = [None if t is None else np.zeros((t.num_rows, t.dim), np.float32) for t in w.tables]
    _, _, rows = oracle.forward(w.columns, w.B, w.offsets, w.values, tabs, want_rows=True)
    ids = [r for c, r in zip(w.columns, rows) if c.transform != "bucketize"]
    fvs = [r for c, r in zip(w.columns, rows) if c.transform == "bucketize"]
    n_ids = int(sum(r.size for r in ids))
    flat = np.concatenate([np.asarray(r, np.int64) for r in ids + fvs]) if ids or fvs else np.zeros(0, np.int64)
    return torch.from_numpy(flat), n_ids, rows


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_row_statistics_and_compulsory_bytes_by_brute_force(bench, seed):
    """The valid values, non-empty bags and distinct rows per table that the
    compulsory byte counts rest on, and the counts themselves, against a
    value-by-value count (padded cuts, truncation, dropped ids, shared
    tables)."""
    from sparse_lookup_gb300 import synth
    w = synth.random_small(seed, C=8, B=30, train=True, allow_weights=False)
    rows_dbg, n_ids, rows = _rows_dbg(w)
    st = bench.row_stats(w, rows_dbg, n_ids)
    valid, nonempty, seen = [], [], {}
    for c, o, r in zip(w.columns, w.offsets, rows):
        cut = c.pad_len if c.pooling == "padded" else int(c.max_len or 0)
        nv, bags = 0, set()
        for b in range(w.B):
            for p in range(int(o[b]), int(o[b + 1])):
                if r[p] >= 0 and (cut == 0 or p - int(o[b]) < cut):
                    nv += 1
                    bags.add(b)
                    seen.setdefault(c.table, set()).add(int(r[p]))
        valid.append(nv)
        nonempty.append(len(bags))
    assert st["valid"] == valid
    assert st["nonempty_bags"] == nonempty
    assert st["unique_per_table"] == {t: len(s) for t, s in seen.items()}

    fixed = 0
    for c, o in zip(w.columns, w.offsets):
        n = int(o[-1])
        per_value = 4 if c.transform == "bucketize" else 8
        nb = 0 if c.boundaries is None else c.boundaries.size
        out_rows = w.B * (c.pad_len if c.pooling == "padded" else 1)
        fixed += (w.B + 1) * 4 + n * per_value + 4 * nb + out_rows * c.dim * 4
    dim_of = {c.table: c.dim for c in w.columns}
    rows_once = sum(len(s) * dim_of[t] * 4 for t, s in seen.items())
    assert bench.forward_bytes_compulsory(w, st) == fixed + rows_once
    rows_each = sum(nv * c.dim * 4 for c, nv in zip(w.columns, valid))
    assert bench.forward_bytes(w, valid) == fixed + rows_each

    n_contrib = int(rows_dbg.numel())
    n_unique = sum(len(s) for s in seen.values())
    dmax = max(c.dim for c in w.columns)
    grad_once = sum((nv if c.pooling == "padded" else ne) * c.dim * 4
                    for c, nv, ne in zip(w.columns, valid, nonempty))
    assert bench.backward_bytes_compulsory(w, n_contrib, st, n_unique, dmax) == \
        n_contrib * 24 + grad_once + n_unique * 16 * dmax


def test_traffic_entry_holds_only_for_the_sources_it_was_captured_from(bench, monkeypatch):
    """A DRAM traffic figure is reported only while the kernel sources hash as
    they did at its capture; any other hash turns it into null."""
    key = next(iter(bench.TRAFFIC))
    entry = bench.TRAFFIC[key]
    monkeypatch.setattr(bench, "kernel_src_hash", lambda kernel: entry["src"])
    assert bench.traffic_for(*key)["bytes"] == entry["bytes"]
    monkeypatch.setattr(bench, "kernel_src_hash", lambda kernel: "0" * 16)
    assert bench.traffic_for(*key) is None
    assert bench.traffic_for("no-such-workload", "k_forward") is None


def test_roofline_fractions(bench):
    """Achieved bandwidth and fractions of one launch from bytes and time."""
    r = bench.roofline_obj(6.0e9, 3.0e9, 2.0, 6000.0, "measured", {"bytes": 4.5e9, "source": "a capture"})
    assert r["achieved"] == pytest.approx(3000.0) and r["frac"] == pytest.approx(0.5)
    assert r["achieved_compulsory"] == pytest.approx(1500.0) and r["frac_compulsory"] == pytest.approx(0.25)
    assert r["traffic"] == 4.5e9 and r["traffic_dram_gbs"] == pytest.approx(2250.0)
    assert bench.roofline_obj(1.0, 1.0, 1.0, 1.0, "measured", None)["traffic"] is None
