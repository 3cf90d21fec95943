"""GPU parity of the collision-free dynamic table (lookup-or-insert with the
frequency filter, deterministic row assignment, expiry) against the oracle,
through the C ABI."""
import numpy as np
import pytest

import oracle
import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import build as slbuild
from sparse_lookup_gb300 import synth

from helpers import DynamicRun, assert_close, compare_hash_maps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    slbuild.build()
    sl.lib()


def lookup(ht, tids, keys, step):
    import torch
    r = ht.lookup_or_insert(torch.tensor(tids, dtype=torch.int32, device="cuda"),
                            torch.tensor(keys, dtype=torch.int64, device="cuda"), step)
    torch.cuda.synchronize()
    return r.cpu().numpy().tolist(), ht.device_status()


def test_hand_traced_scenario():
    """The same scenario the oracle is pinned on (threshold 3, ttl 2, 3 rows)."""
    ht = sl.HashTable(1024, 3, 4, 3, 64, 42, 0.5, 64)
    A, B_, C, D, E, F_, G_, H = 100, 50, 7, 8, 30, 20, 9, 10
    assert lookup(ht, [0] * 6, [A, A, B_, B_, B_, C], 0) == ([-1, -1, 0, 0, 0, -1], 0)
    assert lookup(ht, [0] * 3, [A, C, D], 1) == ([1, -1, -1], 0)
    ex = ht.export()
    assert dict(zip(ex["key"].tolist(), ex["count"].tolist())) == {A: -1, B_: -1, C: 2, D: 1}
    ht.evict_expired(3, 2)
    ht.evict_expired(4, 2)
    assert len(ht.export()["key"]) == 0
    assert lookup(ht, [0] * 6, [E, E, E, F_, F_, F_], 5) == ([1, 1, 1, 0, 0, 0], 0)
    assert lookup(ht, [0] * 6, [G_, G_, G_, H, H, H], 6) == ([2, 2, 2, -1, -1, -1], 5)
    assert lookup(ht, [0], [H], 7) == ([-1], 5)
    ht.evict_expired(8, 2)
    assert lookup(ht, [0], [H], 8) == ([0], 0)
    # admitted rows are initialised exactly as the oracle does
    w = ht.weight.cpu().numpy()
    for row, key in ((0, H), (1, E), (2, G_)):
        want = [oracle.hash_init_value(42, 0, key, d, 0.5) for d in range(4)]
        assert w[row].tolist() == want


@pytest.mark.parametrize("seed,thr,ttl,cap", [(1, 3, 4, 40), (2, 1, 0, 500), (3, 2, 3, 5000), (4, 5, 8, 200)])
def test_random_streams_match_oracle(seed, thr, ttl, cap):
    rng = np.random.default_rng(seed)
    ht = sl.HashTable(1 << 12, cap, 8, thr, 256, seed, 0.1, 3000)
    oh = oracle.Hash(cap, 8, thr, seed, 0.1)
    for step in range(30):
        n = int(rng.integers(0, 3000))
        keys = synth.zipf(rng, 400, 1.1, n)
        tids = rng.integers(0, 4, n).astype(np.int32)
        got, st = lookup(ht, tids, keys, step) if n else ([], 0)
        want, st_o = oh.lookup_or_insert(tids, keys, step)
        assert got == want.tolist(), "step %d" % step
        assert (st == 5) == (st_o == oracle.ERR_FULL), (st, st_o)
        ht.evict_expired(step, ttl)
        oh.evict(step, ttl)
        compare_hash_maps(ht.export(), oh.export(), "step %d" % step)
        ex = oh.export()
        adm = ex["row"] >= 0
        w = ht.weight.cpu().numpy()
        assert np.array_equal(w[ex["row"][adm]], oh.W[ex["row"][adm]]), "initial rows"


@pytest.mark.parametrize("seed", [11, 12])
def test_irregular_calls_match_oracle(seed):
    """Expiry stays exact when lookups repeat a step, skip steps, or are not
    followed by an expiry, and when ttl changes from call to call or exceeds
    the window of touch lists (those cases fall back to full sweeps).  The
    row pool never fills here: a repeated step does not re-list keys a full
    pool left without a row (calls are told apart by their step)."""
    rng = np.random.default_rng(seed)
    cap = 4000
    ht = sl.HashTable(1 << 12, cap, 8, 2, 256, seed, 0.1, 2000)
    oh = oracle.Hash(cap, 8, 2, seed, 0.1)
    step = 0
    for it in range(60):
        step += int(rng.choice([0, 1, 1, 1, 2, 5]))
        for _ in range(int(rng.choice([1, 1, 2]))):
            n = int(rng.integers(1, 2000))
            keys = synth.zipf(rng, 300, 1.1, n)
            tids = rng.integers(0, 3, n).astype(np.int32)
            got, st = lookup(ht, tids, keys, step)
            want, st_o = oh.lookup_or_insert(tids, keys, step)
            assert st == 0 and st_o == 0, (st, st_o)
            assert got == want.tolist(), "iteration %d" % it
        if rng.random() < 0.8:
            ttl = int(rng.choice([0, 1, 3, 10, 14, 20, 40]))
            ht.evict_expired(step, ttl)
            oh.evict(step, ttl)
            compare_hash_maps(ht.export(), oh.export(), "iteration %d" % it)


def test_probe_limit_is_reported_not_hung():
    ht = sl.HashTable(1024, 4096, 4, 1, 2, 1, 0.1, 5000)
    keys = np.arange(5000, dtype=np.int64) * 7919
    got, st = lookup(ht, np.zeros(5000, np.int32), keys, 0)
    assert st == 6
    assert sum(r >= 0 for r in got) <= 1024


def test_keys_outside_the_range_are_rejected_on_the_device():
    ht = sl.HashTable(1024, 16, 4, 1, 16, 1, 0.1, 16)
    got, st = lookup(ht, [0, 1 << 15, 2, -1], [5, 5, 1 << 48, 5], 0)
    assert st == 1
    assert got == [0, -1, -1, -1]


def test_dynamic_training_loop_small():
    """lookup -> forward -> backward/Adagrad -> evict for 20 steps of a scaled
    dynamic workload; rows bit-exact, pooled output and the row pool within
    1e-5 rel / 1e-6 abs of the oracle."""
    run = DynamicRun(C=8, B=512, steps=20, num_slots=1 << 16, cap=1 << 13, ttl=4, key_bits=20)
    for t in range(run.steps):
        r = run.step(t, check=True)
        assert r["status"][0] in (0, 5) and r["status"][1] == 0, r["status"]
        g, o = r["rows"]
        assert np.array_equal(g, o), "rows step %d" % t
        assert_close(*r["out"], what="pooled step %d" % t)
    adm = run.oh.export()
    rows = adm["row"][adm["row"] >= 0]
    assert_close(run.ht.weight.cpu().numpy()[rows], run.oh.W[rows], "row pool weights", rtol=1e-4, atol=1e-5)
