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
