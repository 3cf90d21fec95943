"""The allocation-free sparse Adagrad entry point, checked against the
plan-based path (emb_forward + emb_backward_update) on the same inputs and
against the CPU oracle's backward + Adagrad (one identity column, one value
per bag) at 1e-5 rel / 1e-6 abs, on two calls in a row.

Some callers cannot call cudaMalloc (a framework that owns all device memory
through its own pool, a serving process that forbids allocation after
start-up, a plugin handed only pointers); emb_sparse_adagrad_noalloc serves
them from a fixed scratch area inside the library.  This file is collected
last so that a run stopping at the first failure has run everything else."""
import numpy as np
import pytest

import oracle
import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import build as slbuild
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.synth import ColumnSpec, TableSpec

from helpers import Taint, assert_close, check_rows, excluded_cap

pytestmark = pytest.mark.gpu

MAX_N = 1 << 18


@pytest.fixture(scope="module", autouse=True)
def built():
    slbuild.build()
    sl.lib()


def _inputs(n, num_rows, dim, seed):
    rng = np.random.default_rng(seed)
    rows = synth.scatter_ranks(synth.zipf(rng, num_rows, 1.1, n), num_rows)
    bad = rng.random(n) < 0.03
    rows[bad] = np.where(rng.random(int(bad.sum())) < 0.5, -1, num_rows + 3)
    return rows.astype(np.int64)


def _oracle_step(rows_h, grads_h, W, A, num_rows, dim, lr=0.01, eps=1e-10):
    """The oracle's backward + Adagrad of one call (one identity column, each
    contribution its own bag) on the touched rows of host tables W / A (both
    updated in place).  Returns (touched rows, oracle result, rows before)."""
    n = rows_h.size
    col = ColumnSpec("identity", "sum", num_rows, dim, 0)
    touched = np.unique(rows_h[(rows_h >= 0) & (rows_h < num_rows)])
    W0, A0 = W[touched].copy(), A[touched].copy()
    Wr, Ar = W0.copy(), A0.copy()
    ref = oracle.backward_rows([col], n, [np.arange(n + 1, dtype=np.int32)], [rows_h], grads_h, None,
                               (np.zeros(touched.size, np.int32), touched), Wr, Ar, lr, eps)
    W[touched], A[touched] = Wr, Ar
    return touched, ref, W0, A0, Wr, Ar


@pytest.mark.parametrize("n,num_rows,dim", [(1000, 50, 8), (20000, 3000, 64), (MAX_N, 100000, 128),
                                            (5000, 700, 256), (3, 10, 4), (40000, (1 << 24) + 5, 4)])
def test_noalloc_matches_plan_path_and_oracle_two_calls(n, num_rows, dim):
    """Two calls in a row; the last case needs four sort passes (rows above
    2^24)."""
    import torch
    rows_h = _inputs(n, num_rows, dim, seed=n + dim)
    rows = torch.from_numpy(rows_h).cuda()
    W0 = synth.make_table(TableSpec(num_rows, dim, 5), "cuda")
    Wa, Aa = W0.clone(), torch.zeros_like(W0)
    Wb, Ab = W0.clone(), torch.zeros_like(W0)
    Wo, Ao = W0.cpu().numpy(), np.zeros((num_rows, dim), np.float32)
    # plan path: one identity column, one value per bag, grad_out row = the value's gradient
    col = ColumnSpec("identity", "sum", num_rows, dim, 0)
    plan = sl.Plan([col], [Wa], [Aa], max_batch=n, max_ids=n, training=True)
    offs = torch.arange(n + 1, dtype=torch.int32, device="cuda")
    excluded, checked = 0, 0
    taint = Taint(dim)   # elements whose weights differ after an ill-conditioned step
    for step in range(2):
        grads = synth.make_grad((n, dim), 100 + step, "cuda")
        plan.forward(n, rows, offs, None, None)
        plan.backward_update(grads, None, 0.01, 1e-10)
        sl.emb_sparse_adagrad_noalloc(rows, n, grads, Wb, Ab, num_rows, dim, 0.01, 1e-10)
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert sl.emb_noalloc_get_device_status() == 0
        assert_close(Wb.cpu().numpy(), Wa.cpu().numpy(), "weights after call %d" % (step + 1))
        assert_close(Ab.cpu().numpy(), Aa.cpu().numpy(), "accumulators after call %d" % (step + 1))
        # the oracle, from the state the first call left on its own side
        touched, ref, W0r, A0r, Wr, Ar = _oracle_step(rows_h, grads.cpu().numpy(), Wo, Ao, num_rows, dim)
        idx = torch.from_numpy(touched).cuda()
        before = taint.get(touched)
        e, m, _, outside = check_rows(ref["grad"], ref["absgrad"], ref["count"], ref["grad"], W0r, A0r,
                                      Wb[idx].cpu().numpy(), Ab[idx].cpu().numpy(), Wr, Ar, 0.01, 1e-10,
                                      tainted=before, what="call %d" % (step + 1))
        taint.set(touched, outside)
        excluded += e
        checked += m
    assert excluded <= excluded_cap(checked), (excluded, checked)
    assert not np.array_equal(Wb.cpu().numpy(), W0.cpu().numpy())


def test_noalloc_empty_call_changes_nothing():
    import torch
    W = synth.make_table(TableSpec(64, 8, 5), "cuda")
    A = torch.zeros_like(W)
    W0 = W.clone()
    rows = torch.zeros(1, dtype=torch.int64, device="cuda")
    grads = torch.zeros((1, 8), device="cuda")
    sl.emb_sparse_adagrad_noalloc(rows, 0, grads, W, A, 64, 8, 0.01, 1e-10)
    torch.cuda.synchronize()
    assert sl.emb_noalloc_get_device_status() == 0
    assert torch.equal(W, W0) and not A.any()


def test_noalloc_rejects_sizes_beyond_the_maximum():
    import torch
    W = torch.zeros((10, 8), device="cuda")
    A = torch.zeros_like(W)
    rows = torch.zeros(MAX_N + 1, dtype=torch.int64, device="cuda")
    grads = torch.zeros((MAX_N + 1, 8), device="cuda")
    with pytest.raises(sl.EmbError) as e:
        sl.emb_sparse_adagrad_noalloc(rows, MAX_N + 1, grads, W, A, 10, 8, 0.01, 1e-10)
    assert e.value.status == 2
    with pytest.raises(sl.EmbError) as e:
        sl.emb_sparse_adagrad_noalloc(rows, 4, grads, torch.zeros((10, 260), device="cuda"),
                                      torch.zeros((10, 260), device="cuda"), 10, 260, 0.01, 1e-10)
    assert e.value.status == 2
