"""Failure handling that faults, traps and hangs no GPU: a bounded device wait
made to run out on purpose is reported (EMB_ERR_TIMEOUT latched, the sort's
fail word raised) and the kernels that would consume the incomplete sort do
nothing; device allocations made to fail on the host (an armed hook, no real
exhaustion) make every create call return EMB_ERR_OOM with nothing leaked."""
import numpy as np
import pytest

import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import build as slbuild
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.synth import ColumnSpec, TableSpec

pytestmark = pytest.mark.gpu

OOM = 3
TIMEOUT = 8


@pytest.fixture(scope="module", autouse=True)
def built():
    slbuild.build()
    sl.lib()


@pytest.fixture(autouse=True)
def disarm():
    yield
    sl.emb_debug_fail_alloc(-1)


def _settled_live_allocations():
    # plans and tables of earlier tests that are no longer referenced are
    # freed now, not by a garbage collection in the middle of the count
    import gc
    gc.collect()
    return sl.emb_debug_live_allocations()


def test_sort_wait_that_runs_out_is_reported_and_its_output_unused():
    r = sl.emb_selftest_sort_timeout()
    assert r["status"] == 0, r
    assert r["latched"] == TIMEOUT, r
    assert r["fail_word"] != 0, r
    assert r["table_untouched"], r
    assert 0.0 < r["wait_ms"] < 60000.0, r
    # the context is still usable afterwards
    import torch
    x = torch.arange(10, device="cuda")
    assert int(x.sum()) == 45


def _plan_args(training):
    import torch
    cols = [ColumnSpec("identity", "sum", 100, 8, 0), ColumnSpec("hash_mod", "mean", 50, 16, 1),
            ColumnSpec("bucketize", "padded", 4, 4, 2, boundaries=np.array([-1.0, 0.0, 1.0], np.float32),
                       pad_len=3)]
    tabs = [synth.make_table(TableSpec(c.num_rows, c.dim, 7 + i), "cuda") for i, c in enumerate(cols)]
    accs = [torch.zeros_like(t) for t in tabs] if training else None
    return cols, tabs, accs


@pytest.mark.parametrize("training,backward", [(False, "sort"), (True, "sort"), (True, "atomic")])
def test_every_plan_allocation_failure_returns_oom_and_leaks_nothing(training, backward):
    cols, tabs, accs = _plan_args(training)
    base = _settled_live_allocations()
    failures = 0
    for k in range(200):
        sl.emb_debug_fail_alloc(k)
        try:
            plan = sl.Plan(cols, tabs, accs, max_batch=32, max_ids=512, training=training, backward=backward)
        except sl.EmbError as e:
            assert e.status == OOM, (k, e.status)
            assert sl.emb_debug_live_allocations() == base, "allocation %d: leaked" % k
            failures += 1
            continue
        sl.emb_debug_fail_alloc(-1)
        # the first k allocations succeeded and there is no k-th: the plan works
        assert sl.emb_debug_live_allocations()[0] > base[0]
        plan.close()
        assert sl.emb_debug_live_allocations() == base
        break
    else:
        pytest.fail("the plan never got all its allocations")
    # one failure per allocation site reached: 7 for any plan, the training
    # workspace adds 14 more, the atomic backward's 7 more
    assert failures == (7 if not training else 21 if backward == "sort" else 28), failures


def test_every_hash_allocation_failure_returns_oom_and_leaks_nothing():
    base = _settled_live_allocations()
    failures = 0
    for k in range(100):
        sl.emb_debug_fail_alloc(k)
        try:
            ht = sl.HashTable(1 << 12, 1 << 10, 8, 2, 64, 1, 0.01, 4096)
        except sl.EmbError as e:
            assert e.status == OOM, (k, e.status)
            assert sl.emb_debug_live_allocations() == base, "allocation %d: leaked" % k
            failures += 1
            continue
        sl.emb_debug_fail_alloc(-1)
        ht.close()
        assert sl.emb_debug_live_allocations() == base
        break
    else:
        pytest.fail("the table never got all its allocations")
    assert failures == 16, failures   # one per allocation of the table
