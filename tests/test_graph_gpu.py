"""The forward and the training step captured in a CUDA graph and replayed:
the forward's tile-ticket counter resets itself at the end of every launch,
the backward's scratch is cleared by memset nodes, so replays give the same
results as eager calls (checked against the oracle)."""
import numpy as np
import pytest

import oracle
import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.synth import ColumnSpec, TableSpec, Workload

from helpers import Materialized, assert_close

pytestmark = pytest.mark.gpu


def long_bag_workload(seed=5):
    """Mean bag length well above 64: the forward runs its persistent schedule."""
    rng = np.random.default_rng(seed)
    B = 96
    lens = rng.integers(60, 400, B)
    lens[rng.random(B) < 0.1] = 0
    n = int(lens.sum())
    cols = [ColumnSpec("identity", "mean", 3000, 32, 0), ColumnSpec("hash_mod", "sum", 3000, 64, 1)]
    vals = [rng.integers(-5, 3005, n).astype(np.int64), rng.integers(-2 ** 63, 2 ** 63 - 1, n, dtype=np.int64)]
    off = synth.bag_offsets(lens)
    return Workload("graph", B, cols, [TableSpec(3000, 32, 11), TableSpec(3000, 64, 12)], [off, off], vals,
                    lr=0.05)


def test_forward_graph_replays_match_oracle():
    import torch
    w = long_bag_workload()
    m = Materialized(w, "cuda")
    plan = sl.Plan(w.columns, m.tables, None, max_batch=w.B)
    out = torch.empty((w.B, plan.out_width), device="cuda")
    plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off, out=out)   # eager first
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off, out=out)
    ref, _ = oracle.forward(w.columns, w.B, w.offsets, w.values, m.host_tables())
    for r in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert plan.device_status() == 0
        assert_close(out.cpu().numpy(), ref, "replay %d" % r)
    out.zero_()
    plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off, out=out)   # eager after the replays
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, "eager after replays")


def test_training_step_graph_replays_match_oracle():
    import torch
    w = long_bag_workload(6)
    m = Materialized(w, "cuda", with_acc=True, acc_init=0.1)
    W = m.host_tables()
    A = [a.cpu().numpy() for a in m.accs]
    plan = sl.Plan(w.columns, m.tables, m.accs, max_batch=w.B, max_ids=m.n_ids + m.n_f, training=True)
    out = torch.empty((w.B, plan.out_width), device="cuda")
    G = synth.make_grad((w.B, plan.out_width), 31, "cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off, out=out)
        plan.backward_update(G, None, w.lr, w.eps)
    Gh = G.cpu().numpy()
    for r in range(2):
        g.replay()
        oracle.backward_adagrad(w.columns, w.B, w.offsets, w.values, Gh, None, W, A, w.lr, w.eps)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    for t in range(len(W)):
        assert_close(m.tables[t].cpu().numpy(), W[t], "weights of table %d after two replays" % t)
        assert_close(m.accs[t].cpu().numpy(), A[t], "accumulators of table %d after two replays" % t)
