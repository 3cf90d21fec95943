"""Parity at the full sizes the benchmark times, in its launch configuration:
the 200-column training step, the 20-column sequence workload (mean and
padded), and 50 steps of the dynamic hash-table stream.

Every output is checked.  The tables are too large to copy to the host at
once, so the oracle runs one column at a time (each of these workloads gives
every column a table of its own): the column's table is copied to the host
for its forward; for its backward the table's initial values are drawn
again from their seed on the device and the touched rows gathered, so the
oracle's backward restricted to those rows (orc_backward_rows) starts from
the same rows the library updated.  Unique rows and counts of the whole step
are bit-exact; every pooled output, every padded copy (bit-exact), every
touched row's aggregated gradient, weights and accumulator are compared.
"""
import dataclasses
import gc

import numpy as np
import pytest

import oracle
from helpers import (Materialized, assert_close, assert_close_skip, check_rows, compare_hash_maps, excluded_cap,
                     pooled_slices, seq_slices, DynamicRun)
from sparse_lookup_gb300 import synth

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def _free():
    import torch
    gc.collect()
    torch.cuda.empty_cache()


def _full_training_step(w):
    """Forward + backward/Adagrad of workload w at full size, every output
    checked against the oracle column by column."""
    import torch
    import sparse_lookup_gb300 as sl
    assert len({c.table for c in w.columns}) == len(w.columns), "one table per column"
    m = Materialized(w, "cuda", with_acc=True, acc_init=0.0)
    plan = sl.Plan(w.columns, m.tables, m.accs, max_batch=w.B, max_ids=m.n_ids + m.n_f, training=True)
    out, seq = plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    psl, _ = pooled_slices(w.columns)
    ssl, _ = seq_slices(w.columns, w.B)
    o = out.cpu().numpy() if out is not None and out.numel() else None

    # forward: every pooled element and every padded copy, one column at a time
    for c, col in enumerate(w.columns):
        spec = dataclasses.replace(col, table=0)
        ref, rseq = oracle.forward([spec], w.B, [w.offsets[c]], [w.values[c]], [m.tables[col.table].cpu().numpy()])
        if col.pooling == "padded":
            start, shape = ssl[c]
            got = seq[start:start + int(np.prod(shape))].cpu().numpy().reshape(shape)
            assert np.array_equal(got, rseq[0]), "padded column %d" % c   # a copy: bit-exact
        else:
            off, d = psl[c]
            assert_close(o[:, off:off + d], ref, "column %d" % c)
    del o

    width = plan.out_width
    G = synth.make_grad((w.B, max(width, 1)), 77, "cuda")[:, :width].contiguous() if width else None
    Gseq = synth.make_grad((w.B * plan.seq_per_bag,), 78, "cuda") if plan.seq_per_bag else None
    dbg = plan.backward_update(G, Gseq, w.lr, w.eps, debug=True)
    torch.cuda.synchronize()
    assert plan.device_status() == 0

    # unique rows and counts of the whole step: bit-exact
    u = oracle.unique_counts(w.columns, w.B, w.offsets, w.values)
    col_table = plan.info["col_table"]
    t2s = {}
    for c, t in zip(w.columns, col_table):
        t2s.setdefault(int(t), c.table)
    gt = np.array([t2s[int(t)] for t in dbg["table"].cpu().numpy()], np.int64)
    assert np.array_equal(gt, u["table"]), "unique tables"
    assert np.array_equal(dbg["row"].cpu().numpy(), u["row"]), "unique rows"
    assert np.array_equal(dbg["count"].cpu().numpy().astype(np.int64), u["count"]), "counts"

    # every touched row, one column (= table) at a time
    G_h = G.cpu().numpy() if G is not None else None
    flat = Gseq.cpu().numpy() if Gseq is not None else None
    excluded, total = 0, 0
    for c, col in enumerate(w.columns):
        sel = np.flatnonzero(u["table"] == col.table)
        if not sel.size:
            continue
        rows = u["row"][sel]
        idx = torch.from_numpy(rows).cuda()
        W0 = synth.make_table(w.tables[col.table], "cuda")[idx].cpu().numpy()
        A0 = np.zeros_like(W0)
        Wg = m.tables[col.table][idx].cpu().numpy()
        Ag = m.accs[col.table][idx].cpu().numpy()
        g = dbg["grad"][torch.from_numpy(sel).cuda(), :col.dim].cpu().numpy()
        spec = dataclasses.replace(col, table=0)
        if col.pooling == "padded":
            start, shape = ssl[c]
            Gc, Gs = None, [flat[start:start + int(np.prod(shape))].reshape(shape)]
        else:
            off, d = psl[c]
            Gc, Gs = np.ascontiguousarray(G_h[:, off:off + d]), None
        Wr, Ar = W0.copy(), A0.copy()
        ref = oracle.backward_rows([spec], w.B, [w.offsets[c]], [w.values[c]], Gc, Gs,
                                   (np.zeros(rows.size, np.int32), rows), Wr, Ar, w.lr, w.eps)
        assert np.array_equal(ref["count"], u["count"][sel]), "counts of column %d" % c
        e, n, _, _ = check_rows(ref["grad"], ref["absgrad"], ref["count"], g, W0, A0, Wg, Ag, Wr, Ar, w.lr, w.eps,
                             what="column %d" % c)
        excluded += e
        total += n
        del W0, Wg, Ag
    dims = {col.table: col.dim for col in w.columns}
    tabs, n_per = np.unique(u["table"], return_counts=True)
    assert total == int(sum(dims[int(t)] * int(k) for t, k in zip(tabs, n_per))), "every touched element checked"
    assert excluded <= excluded_cap(total), (excluded, total)
    print("excluded %d of %d updated elements" % (excluded, total))
    del m, plan, out, seq, G, Gseq, dbg
    _free()


def test_training_workload_full_size():
    """200 identity columns, batch 8192, Zipf(1.1) ids, 3% out of range."""
    _full_training_step(synth.training())


def test_sequence_workload_mean_full_size():
    """20 columns, batch 1024, sequences of 200-1000 ids, mean pooling."""
    _full_training_step(synth.sequences(mode="mean"))


def test_sequence_workload_padded_full_size():
    """20 columns, batch 1024, unpooled [1024, 1000, 128] per column."""
    _full_training_step(synth.sequences(mode="padded"))


def test_dynamic_stream_full_size():
    """100 columns over one 2^27-slot table, batch 16384, 50 steps of
    lookup-or-insert -> forward -> backward/Adagrad -> expiry: rows bit-exact
    every step, hash maps bit-exact every tenth step, every step's pooled
    output within 1e-5 rel / 1e-6 abs of the oracle's forward over the rows
    the library read, and every touched row's gradient, weights and
    accumulator within 1e-5 rel / 1e-6 abs of the free-running oracle
    (exclusions: elements the fp32 sum leaves ill-conditioned, counted); the
    row pool at the end too."""
    w = synth.dynamic()
    ex = w.extra
    run = DynamicRun(C=len(w.columns), B=w.B, steps=ex["steps"], num_slots=ex["num_slots"], cap=ex["row_capacity"],
                     dim=w.columns[0].dim, thr=ex["threshold"], ttl=ex["ttl"], seed=w.seed, alpha=ex["alpha"],
                     key_bits=ex["key_bits"], lr=w.lr, max_probes=ex["max_probes"])
    for t in range(run.steps):
        r = run.step(t)
        assert r["status"][0] in (0, 5) and r["status"][1] == 0, r["status"]
        g, o = r["rows"]
        assert np.array_equal(g, o), "rows step %d" % t
        assert_close_skip(*r["out"], what="pooled step %d" % t)
        if t % 10 == 9:
            compare_hash_maps(run.ht.export(), run.oh.export(), "step %d" % t)
    run.pool.check_pool(run.ht.weight, run.ht.acc)
    print("excluded %d of %d updated elements" % (run.excluded, run.checked))
    del run
    _free()
