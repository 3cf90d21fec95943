"""Shared test plumbing: materialise seeded workloads on the device, run the
oracle on the same inputs, compare with the tolerance the parity bar states
(fp32: |gpu - ref| <= 1e-6 + 1e-5 |ref|; integers bit-exact)."""
import numpy as np

import oracle
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.synth import ColumnSpec, TableSpec, Workload

RTOL = 1e-5
ATOL = 1e-6


def assert_close(got, ref, what="", rtol=RTOL, atol=ATOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    both_nan = np.isnan(got) & np.isnan(ref)
    bad = ~both_nan & ~(np.abs(got - ref) <= atol + rtol * np.abs(ref))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d elements out of tolerance, e.g. %s got %s ref %s" % (
            what, int(bad.sum()), bad.size, idx.tolist(), got[bad][:5].tolist(), ref[bad][:5].tolist()))


class Materialized:
    """A workload's tables and jagged inputs on a device."""

    def __init__(self, w, device="cuda", with_acc=False, acc_init=0.0):
        import torch
        self.w = w
        self.device = device
        self.tables = []
        for spec in w.tables:
            self.tables.append(None if spec is None else synth.make_table(spec, device))
        self.accs = None
        if with_acc:
            self.accs = [None if t is None else torch.full_like(t, acc_init) for t in self.tables]
        ids, id_off, fv, f_off = synth.jagged(w)
        self.ids_h, self.id_off_h, self.fv_h, self.f_off_h = ids, id_off, fv, f_off
        n_id_cols = sum(1 for c in w.columns if c.transform != "bucketize")
        n_f_cols = len(w.columns) - n_id_cols
        self.ids = torch.from_numpy(ids).to(device) if n_id_cols else None
        self.id_off = torch.from_numpy(id_off).to(device) if n_id_cols else None
        self.fv = torch.from_numpy(fv).to(device) if n_f_cols else None
        self.f_off = torch.from_numpy(f_off).to(device) if n_f_cols else None
        self.n_ids = ids.size
        self.n_f = fv.size
        idw, fw = synth.jagged_weights(w)
        self.idw = torch.from_numpy(idw).to(device) if idw is not None and n_id_cols else None
        self.fw = torch.from_numpy(fw).to(device) if fw is not None and n_f_cols else None

    def host_tables(self):
        return [None if t is None else t.cpu().numpy() for t in self.tables]

    def rows_dbg_split(self, rows_dbg):
        """Per-column slices of the library's rows_dbg output."""
        r = rows_dbg.cpu().numpy()
        out, pos = [], {0: 0, 1: self.n_ids}
        for c, o in zip(self.w.columns, self.w.offsets):
            st = 1 if c.transform == "bucketize" else 0
            n = int(o[-1])
            out.append(r[pos[st]:pos[st] + n])
            pos[st] += n
        return out


def pooled_slices(columns):
    """Float offset and dim of each pooled column inside an output row."""
    off, res = 0, []
    for c in columns:
        if c.pooling == "padded":
            res.append(None)
        else:
            res.append((off, c.dim))
            off += c.dim
    return res, off


def seq_slices(columns, B):
    """(start, shape) of each padded column inside the concatenated seq_out."""
    off, res = 0, []
    for c in columns:
        if c.pooling == "padded":
            n = B * c.pad_len * c.dim
            res.append((off, (B, c.pad_len, c.dim)))
            off += n
        else:
            res.append(None)
    return res, off


def oracle_sampled_forward(w, tables_dev, bags):
    """Oracle forward of a sample of (column, bag) pairs of a large workload:
    for each sampled bag, a one-bag problem on a compact table holding only
    the rows that bag touches (rows are remapped; the pooled result is the
    same).  Returns {(c, b): pooled vector} for pooled columns."""
    import torch
    res = {}
    for c, b in bags:
        col = w.columns[c]
        o = w.offsets[c]
        vals = w.values[c][o[b]:o[b + 1]]
        rows = oracle.column_rows(col, vals)
        valid = rows[rows >= 0]
        uniq, inv = np.unique(valid, return_inverse=True)
        sub = tables_dev[col.table][torch.from_numpy(uniq).to(tables_dev[col.table].device)].cpu().numpy() \
            if uniq.size else np.zeros((1, col.dim), np.float32)
        ids = np.full(rows.shape, -1, np.int64)
        ids[rows >= 0] = inv
        spec = synth.ColumnSpec("identity", col.pooling, max(int(uniq.size), 1), col.dim, 0,
                                default=col.default, pad_len=col.pad_len)
        out, seq = oracle.forward([spec], 1, [np.array([0, ids.size], np.int32)], [ids], [sub])
        res[(c, b)] = seq[0][0] if col.pooling == "padded" else out[0]
    return res


U32 = 2.0 ** -24


def gamma(k):
    """Higham's gamma_k = k u / (1 - k u) for fp32 (u = 2^-24): any order of
    summing k terms errs by at most gamma_{k-1} * sum|terms|."""
    ku = np.asarray(k, np.float64) * U32
    return ku / (1.0 - ku)


class TrainStep:
    """One forward + backward/Adagrad step of a workload on the device through
    the C ABI, and the oracle's result for the same inputs."""

    def __init__(self, w, acc_init=0.0, grad_seed=77, device="cuda", backward="sort"):
        import torch
        import sparse_lookup_gb300 as sl
        self.w = w
        m = Materialized(w, device, with_acc=True, acc_init=acc_init)
        self.m = m
        self.W0 = m.host_tables()
        self.A0 = [None if a is None else a.cpu().numpy() for a in m.accs]
        n = m.n_ids + m.n_f
        self.plan = sl.Plan(w.columns, m.tables, m.accs, max_batch=max(w.B, 1), max_ids=max(n, 1), training=True,
                            backward=backward)
        self.out, self.seq = self.plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off, id_weights=m.idw,
                                               f_weights=m.fw)
        width = self.plan.out_width
        self.G = synth.make_grad((w.B, max(width, 1)), grad_seed, device)[:, :width].contiguous()
        self.Gseq = None
        if self.plan.seq_per_bag:
            self.Gseq = synth.make_grad((w.B * self.plan.seq_per_bag,), grad_seed + 1, device)
        self.dbg = self.plan.backward_update(self.G if width else None, self.Gseq, w.lr, w.eps, debug=True)
        torch.cuda.synchronize()
        self.status = self.plan.device_status()
        self.info = self.plan.info

    def again(self, grad_seed):
        """Another step on the same plan and inputs with a new upstream
        gradient, from the tables as the previous step left them."""
        import torch
        w, m = self.w, self.m
        self.W0 = m.host_tables()
        self.A0 = [None if a is None else a.cpu().numpy() for a in m.accs]
        self.out, self.seq = self.plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off, id_weights=m.idw,
                                               f_weights=m.fw)
        width = self.plan.out_width
        self.G = synth.make_grad((w.B, max(width, 1)), grad_seed, "cuda")[:, :width].contiguous()
        if self.plan.seq_per_bag:
            self.Gseq = synth.make_grad((w.B * self.plan.seq_per_bag,), grad_seed + 1, "cuda")
        self.dbg = self.plan.backward_update(self.G if width else None, self.Gseq, w.lr, w.eps, debug=True)
        torch.cuda.synchronize()
        self.status = self.plan.device_status()
        return self

    def oracle(self):
        w = self.w
        G = self.G.cpu().numpy()
        gseq = None
        if self.Gseq is not None:
            s = self.Gseq.cpu().numpy()
            sl_, _ = seq_slices(w.columns, w.B)
            gseq = [None if sp is None else s[sp[0]:sp[0] + int(np.prod(sp[1]))].reshape(sp[1]) for sp in sl_]
        Wr = [None if t is None else t.copy() for t in self.W0]
        Ar = [None if t is None else t.copy() for t in self.A0]
        nt = len(Wr)
        dummy = np.zeros((1, 1), np.float32)
        Wl = [Wr[i] if Wr[i] is not None else dummy for i in range(nt)]
        Al = [Ar[i] if Ar[i] is not None else dummy for i in range(nt)]
        ref = oracle.backward_adagrad(w.columns, w.B, w.offsets, w.values, G, gseq, Wl, Al, w.lr, w.eps,
                                      weights=w.weights)
        # magnitudes for the summation-error bound: the same aggregation of |G|
        Wd = [np.zeros_like(x) for x in Wl]
        Ad = [np.zeros_like(x) for x in Al]
        absg = oracle.backward_adagrad(w.columns, w.B, w.offsets, w.values, np.abs(G),
                                       None if gseq is None else [None if g is None else np.abs(g) for g in gseq],
                                       Wd, Ad, w.lr, w.eps,
                                       weights=None if w.weights is None else [np.abs(x) for x in w.weights])
        return ref, absg, Wl, Al

    def gpu_table_to_spec(self):
        """GPU table index (first appearance of a weight pointer) -> spec table id."""
        out = {}
        for c, t in zip(self.w.columns, self.info["col_table"]):
            out.setdefault(t, c.table)
        return out


# Exclusions the parity bar allows: elements whose Adagrad step fp32 summation
# cannot determine (see check_rows), at most this fraction of the elements
# checked, with a floor of 16 for small problems (one cancelling pair of bags
# repeats its element in every row the two bags share).
MAX_EXCLUDED_FRAC = 1e-6
MIN_EXCLUDED_CAP = 16


def excluded_cap(total):
    return max(MIN_EXCLUDED_CAP, MAX_EXCLUDED_FRAC * total)


def check_rows(gr, absg, count, g_gpu, w0, a0, w_gpu, a_gpu, w_ref, a_ref, lr, eps, tainted=None, what="rows"):
    """Touched rows of one step, vectorised ([n, dim] arrays, count [n]).

    The aggregated gradient must lie within 1e-5 rel / 1e-6 abs of the
    oracle's fp64 sum, or within the probabilistic bound of fp32 summation
    (Higham & Mary, 2019): lambda sqrt(k) u sum|x| with lambda = 8 and k =
    count + 1 (the mean scale's own rounding adds at most u sum|x|, inside
    it).  The updated weight must lie within 1e-5 / 1e-6 unless its step is
    ill-conditioned at that bound: the first Adagrad step from acc = 0 has
    dW/dg = lr eps / g^2, and a sum whose sign fp32 cannot determine flips
    the step ("ambiguous").  `tainted` marks elements that were ambiguous in
    an earlier step of the same run (their weights may differ by that step's
    flip ever since).  The accumulator must lie within 1e-5 / 1e-6 or within
    the error the gradient bound implies (g^2 is sign-blind: no exclusion).
    Returns (excluded, checked, ambiguous mask, outside mask): excluded =
    the elements outside the weight tolerance (the outside mask), all of them
    ambiguous or tainted."""
    gr = np.asarray(gr, np.float64)
    absg = np.asarray(absg, np.float64)
    k = np.asarray(count, np.float64).reshape(-1, *([1] * (gr.ndim - 1))) + 1.0
    pbnd = 8.0 * np.sqrt(k) * U32 * absg + 1e-30
    err = np.abs(np.asarray(g_gpu, np.float64) - gr)
    ok = (err <= ATOL + RTOL * np.abs(gr)) | (err <= pbnd)
    if not ok.all():
        i = np.argwhere(~ok)[:4]
        raise AssertionError("%s: aggregated gradient outside the bound at %s: err %s bound %s" % (
            what, i.tolist(), err[~ok][:4], pbnd[~ok][:4]))
    a0 = np.asarray(a0, np.float64)
    w0 = np.asarray(w0, np.float64)

    def step(gg):
        return w0 - lr * gg / (np.sqrt(a0 + gg * gg) + eps)
    spread = np.abs(step(gr + pbnd) - step(gr - pbnd))
    amb = spread > ATOL + RTOL * np.abs(step(gr))
    skip = amb if tainted is None else (amb | np.asarray(tainted, bool))
    wr = np.asarray(w_ref, np.float64)
    errw = np.abs(np.asarray(w_gpu, np.float64) - wr)
    within = errw <= ATOL + RTOL * np.abs(wr)
    okw = within | skip
    if not okw.all():
        i = np.argwhere(~okw)[:4]
        raise AssertionError("%s: weights outside the tolerance at %s: %s vs %s" % (
            what, i.tolist(), np.asarray(w_gpu)[~okw][:4], wr[~okw][:4]))
    ar = np.asarray(a_ref, np.float64)
    abound = 2 * np.abs(gr) * pbnd + pbnd * pbnd + 4 * U32 * np.abs(ar)
    erra = np.abs(np.asarray(a_gpu, np.float64) - ar)
    oka = (erra <= ATOL + RTOL * np.abs(ar)) | (erra <= abound)
    if not oka.all():
        i = np.argwhere(~oka)[:4]
        raise AssertionError("%s: accumulators outside the bound at %s: %s vs %s" % (
            what, i.tolist(), np.asarray(a_gpu)[~oka][:4], ar[~oka][:4]))
    return int((~within).sum()), int(gr.size), amb, ~within


def check_row_update(key, gr, absg, count, g_gpu, w0, a0, w_gpu, a_gpu, w_ref, a_ref, lr, eps):
    """check_rows for one row.  Returns (excluded, checked)."""
    e, n, _, _ = check_rows(np.asarray(gr)[None], np.asarray(absg)[None], [count], np.asarray(g_gpu)[None],
                         np.asarray(w0)[None], np.asarray(a0)[None], np.asarray(w_gpu)[None],
                         np.asarray(a_gpu)[None], np.asarray(w_ref)[None], np.asarray(a_ref)[None], lr, eps,
                         what="row %s" % (key,))
    return e, n


def check_train_step(ts):
    """Bit-exact unique rows and counts; every touched row checked by
    check_rows; untouched rows unchanged.  Returns the number of elements
    outside the tolerance (all ill-conditioned), which must stay within
    excluded_cap of the updated elements."""
    assert ts.status == 0, "device status %d" % ts.status
    ref, absg, Wr, Ar = ts.oracle()
    n = len(ref["row"])
    d = ts.dbg
    assert int(d["row"].numel()) == n, (int(d["row"].numel()), n)
    t2s = ts.gpu_table_to_spec()
    gt = np.array([t2s[int(t)] for t in d["table"].cpu().numpy()], np.int64)
    assert np.array_equal(gt, ref["table"]), "unique tables"
    assert np.array_equal(d["row"].cpu().numpy(), ref["row"]), "unique rows"
    assert np.array_equal(d["count"].cpu().numpy().astype(np.int64), ref["count"]), "counts"
    g = d["grad"].cpu().numpy()
    excluded, total = 0, 0
    dims = {c.table: c.dim for c in ts.w.columns}
    for t_gpu, t_spec in t2s.items():
        Wg = ts.m.tables[t_spec].cpu().numpy()
        Ag = ts.m.accs[t_spec].cpu().numpy()
        W0 = ts.W0[t_spec]
        A0 = ts.A0[t_spec]
        sel = np.flatnonzero(ref["table"] == t_spec)
        rows = ref["row"][sel]
        touched = np.zeros(W0.shape[0], bool)
        touched[rows] = True
        assert np.array_equal(Wg[~touched], W0[~touched]), "untouched rows changed"
        assert np.array_equal(Ag[~touched], A0[~touched]), "untouched accumulators changed"
        if not sel.size:
            continue
        dim = dims[t_spec]
        gr = np.stack([ref["grad"][i] for i in sel])
        ab = np.stack([absg["grad"][i] for i in sel])
        e, m, _, _ = check_rows(gr, ab, ref["count"][sel], g[sel, :dim], W0[rows], A0[rows], Wg[rows], Ag[rows],
                             Wr[t_spec][rows], Ar[t_spec][rows], ts.w.lr, ts.w.eps, what="table %d" % t_spec)
        excluded += e
        total += m
    assert excluded <= excluded_cap(total), (excluded, total)
    return excluded


def compare_hash_maps(gpu, ref, what=""):
    """Exported maps must be identical as (tid, key) -> row maps, with equal
    counts while counting and equal last_seen."""
    assert np.array_equal(gpu["tid"], ref["tid"].astype(np.int32)), what + " tids"
    assert np.array_equal(gpu["key"], ref["key"]), what + " keys"
    assert np.array_equal(gpu["row"], ref["row"]), what + " rows"
    counting = ref["row"] < 0
    assert np.array_equal(gpu["count"][counting], ref["count"][counting].astype(np.int32)), what + " counts"
    assert np.array_equal(gpu["last_seen"], ref["last_seen"]), what + " last_seen"


class Taint:
    """Elements (row, d) of a row pool whose weight may differ between the
    library and the oracle because an earlier step was ill-conditioned there
    (check_rows' ambiguous mask), kept sparse: sorted rows with a [dim] mask
    each.  A row handed out again starts clean (both sides write the same
    initial values)."""

    def __init__(self, dim):
        self.dim = dim
        self.rows = np.zeros(0, np.int64)
        self.mask = np.zeros((0, dim), bool)

    def get(self, rows):
        rows = np.asarray(rows, np.int64)
        out = np.zeros((rows.size, self.dim), bool)
        if self.rows.size and rows.size:
            pos = np.minimum(np.searchsorted(self.rows, rows), self.rows.size - 1)
            hit = self.rows[pos] == rows
            out[hit] = self.mask[pos[hit]]
        return out

    def set(self, rows, mask):
        rows = np.asarray(rows, np.int64)
        keep = ~np.isin(self.rows, rows)
        on = mask.any(axis=1)
        r = np.concatenate([self.rows[keep], rows[on]])
        m = np.concatenate([self.mask[keep], mask[on]])
        order = np.argsort(r, kind="stable")
        self.rows, self.mask = r[order], m[order]

    def clear(self, rows):
        rows = np.asarray(rows, np.int64)
        keep = ~np.isin(self.rows, rows)
        self.rows, self.mask = self.rows[keep], self.mask[keep]

    def count(self):
        return int(self.mask.sum())


class OraclePool:
    """The oracle's side of the dynamic-table loop, free-running on its own
    row pool: per step the lookup, the pooled output (with the output
    elements that read a tainted weight marked), and the backward + Adagrad
    of every touched row (orc_backward_rows: the gradient, its magnitude sum
    and the updated rows, written back into the pool).  The ambiguous
    elements of each step join the taint."""

    def __init__(self, cap, dim, thr, seed, cols, B, lr, eps):
        self.oh = oracle.Hash(cap, dim, thr, seed, 0.01)
        self.cols, self.B, self.lr, self.eps = cols, B, lr, eps
        self.dim = dim
        self.taint = Taint(dim)

    def step(self, tids, keys, t, offs, G, ttl, want_out=True):
        oh = self.oh
        rows_o, st = oh.lookup_or_insert(tids, keys, t)
        self.taint.clear(oh.last_admitted())
        vals, pos = [], 0
        for o in offs:
            n = int(o[-1])
            vals.append(rows_o[pos:pos + n])
            pos += n
        res = dict(rows=rows_o, status=st)
        if want_out:
            out = oracle.forward(self.cols, self.B, offs, vals, [oh.W])[0]
            skip = np.zeros(out.shape, bool)
            if self.taint.rows.size:
                psl, _ = pooled_slices(self.cols)
                for c, (o, v) in enumerate(zip(offs, vals)):
                    tv = self.taint.get(np.where(v >= 0, v, -1))
                    hit = np.flatnonzero(tv.any(axis=1) & (v >= 0))
                    if hit.size:
                        bag = np.searchsorted(np.asarray(o, np.int64), hit, side="right") - 1
                        off, d = psl[c]
                        for b, i in zip(bag, hit):
                            skip[b, off:off + d] |= tv[i]
            res["out"], res["out_skip"] = out, skip
        touched = np.unique(rows_o[rows_o >= 0])
        W0 = np.ascontiguousarray(oh.W[touched])
        A0 = np.ascontiguousarray(oh.acc[touched])
        Wr, Ar = W0.copy(), A0.copy()
        ref = oracle.backward_rows(self.cols, self.B, offs, vals, G, None,
                                   (np.zeros(touched.size, np.int32), touched), Wr, Ar, self.lr, self.eps)
        oh.W[touched] = Wr
        oh.acc[touched] = Ar
        tainted = self.taint.get(touched)
        # which elements fp32 summation leaves ill-conditioned this step
        amb = check_rows(ref["grad"], ref["absgrad"], ref["count"], ref["grad"], W0, A0, Wr, Ar, Wr, Ar,
                         self.lr, self.eps)[2]
        # (a caller that sees the library's rows may narrow this taint to
        # the elements that do differ)
        self.taint.set(touched, tainted | amb)
        oh.evict(t, ttl)
        res.update(touched=touched, W0=W0, A0=A0, Wr=Wr, Ar=Ar, ref=ref, tainted=tainted)
        return res

    def check_pool(self, weight, acc, what="row pool"):
        """Every live row of the library's pool against the oracle's: within
        1e-5 rel / 1e-6 abs except tainted elements (counted).  Returns
        (excluded, checked)."""
        import torch
        adm = self.oh.export()
        live = np.sort(adm["row"][adm["row"] >= 0])
        if not live.size:
            return 0, 0
        idx = torch.from_numpy(live).to(weight.device)
        Wg = weight[idx].cpu().numpy().astype(np.float64)
        Ag = acc[idx].cpu().numpy().astype(np.float64)
        Wo = self.oh.W[live].astype(np.float64)
        Ao = self.oh.acc[live].astype(np.float64)
        tainted = self.taint.get(live)
        within = np.abs(Wg - Wo) <= ATOL + RTOL * np.abs(Wo)
        assert (within | tainted).all(), "%s: weights outside the tolerance, untainted" % what
        assert (np.abs(Ag - Ao) <= ATOL + RTOL * np.abs(Ao)).all(), "%s: accumulators" % what
        excluded = int((~within).sum())
        assert excluded <= excluded_cap(Wg.size), (excluded, Wg.size)
        return excluded, Wg.size


class DynamicRun:
    """The dynamic-table training loop through the C ABI -- per step:
    hash_lookup_or_insert -> emb_forward (rows_given columns over the table's
    row pool) -> emb_backward_update -> hash_evict_expired -- next to the
    oracle doing the same on its own row pool (OraclePool).  Each step
    compares the rows bit-exactly, the pooled output with the oracle's
    forward over the rows the library read (so the forward's arithmetic
    alone is under test, with no exclusion), and every touched row's
    aggregated gradient, weights and accumulator with the free-running
    oracle at 1e-5 rel / 1e-6 abs; the only elements allowed outside are
    those the fp32 sum leaves ill-conditioned in that step or an earlier one
    (counted, capped)."""

    def __init__(self, C, B, steps, num_slots, cap, dim=32, thr=3, ttl=10, seed=1005, alpha=1.2, key_bits=34,
                 max_len=5, lr=0.01, max_probes=128):
        import sparse_lookup_gb300 as sl
        self.C, self.B, self.steps, self.ttl, self.lr = C, B, steps, ttl, lr
        self.eps = 1e-10
        self.seed, self.alpha, self.key_bits, self.max_len = seed, alpha, key_bits, max_len
        self.dim = dim
        max_keys = C * B * max_len
        self.ht = sl.HashTable(num_slots, cap, dim, thr, max_probes, seed, 0.01, max_keys)
        self.cols = [synth.ColumnSpec("rows_given", "sum", cap, dim, 0) for _ in range(C)]
        self.pool = OraclePool(cap, dim, thr, seed, self.cols, B, lr, self.eps)
        self.oh = self.pool.oh
        self.plan = sl.Plan(self.cols, [self.ht.weight], [self.ht.acc], max_batch=B, max_ids=max_keys,
                            training=True)
        self.excluded = 0
        self.checked = 0

    def step(self, t, check_out=True, check_update=True):
        """One step on both sides; returns dict(status, rows (gpu, oracle),
        out (gpu, oracle, skip mask) when check_out).  With check_update the
        touched rows are compared here (failures raise)."""
        import torch
        offs, keys = synth.dynamic_keys(self.seed, t, self.C, self.B, self.alpha, self.key_bits, self.max_len)
        tids = np.concatenate([np.full(k.size, c, np.int32) for c, k in enumerate(keys)])
        allk = np.concatenate(keys)
        rows = self.ht.lookup_or_insert(torch.from_numpy(tids).cuda(), torch.from_numpy(allk).cuda(), t)
        ids_off = np.concatenate([[0], np.cumsum(np.concatenate([np.diff(o) for o in offs]))]).astype(np.int32)
        out, _ = self.plan.forward(self.B, rows, torch.from_numpy(ids_off).cuda(), None, None)
        torch.cuda.synchronize()
        rows_g = rows.cpu().numpy()
        if check_out:
            # the rows this forward read, as the library held them before the
            # backward: the oracle's forward over the same values tests the
            # forward's arithmetic alone, with no exclusion
            read = np.unique(rows_g[rows_g >= 0])
            W_read = self.ht.weight[torch.from_numpy(read).cuda()].cpu().numpy()
        G = synth.make_grad((self.B, self.plan.out_width), 500 + t, "cuda")
        dbg = self.plan.backward_update(G, None, self.lr, self.eps, debug=check_update)
        self.ht.evict_expired(t, self.ttl)
        torch.cuda.synchronize()
        st_h, st_p = self.ht.device_status(), self.plan.device_status()
        o = self.pool.step(tids, allk, t, offs, G.cpu().numpy(), self.ttl, want_out=False)
        res = dict(status=(st_h, st_p, o["status"]), rows=(rows_g, o["rows"]))
        if check_out:
            vals, pos = [], 0
            for off in offs:
                m = int(off[-1])
                v = rows_g[pos:pos + m]
                vals.append(np.where(v >= 0, np.searchsorted(read, v), -1).astype(np.int64))
                pos += m
            cols = [synth.ColumnSpec("rows_given", "sum", max(int(read.size), 1), self.dim, 0) for _ in self.cols]
            tab = W_read if read.size else np.zeros((1, self.dim), np.float32)
            ref = oracle.forward(cols, self.B, offs, vals, [tab])[0]
            res["out"] = (out.cpu().numpy(), ref, np.zeros(ref.shape, bool))
        if check_update:
            touched = o["touched"]
            assert np.array_equal(dbg["row"].cpu().numpy(), touched), "unique rows step %d" % t
            assert np.array_equal(dbg["count"].cpu().numpy().astype(np.int64), o["ref"]["count"]), \
                "counts step %d" % t
            idx = torch.from_numpy(touched).cuda()
            Wg = self.ht.weight[idx].cpu().numpy()
            Ag = self.ht.acc[idx].cpu().numpy()
            g = dbg["grad"][:, :self.dim].cpu().numpy()
            ref = o["ref"]
            e, m, _, outside = check_rows(ref["grad"], ref["absgrad"], ref["count"], g, o["W0"], o["A0"], Wg, Ag,
                                          o["Wr"], o["Ar"], self.lr, self.eps, tainted=o["tainted"],
                                          what="step %d" % t)
            # the taint follows the elements that differ, not all that might
            self.pool.taint.set(touched, outside)
            self.excluded += e
            self.checked += m
            assert self.excluded <= excluded_cap(self.checked), (self.excluded, self.checked)
        return res


def assert_close_skip(got, ref, skip, what=""):
    """assert_close on the elements not marked in `skip`; returns how many
    were skipped."""
    keep = ~np.asarray(skip, bool)
    assert_close(np.asarray(got)[keep], np.asarray(ref)[keep], what)
    return int((~keep).sum())


def padded_pieces_case(case):
    """Plans with padded columns longer than the whole-warp threshold (their
    bags are copied in pieces of positions): "ids-only" (a stream of only
    such columns, pad lengths 130 / 777 / 300 / 1000, dims 8 / 128 / 36 /
    200), "fvals-only" (a bucketized one alone in its stream), "mixed" (beside
    pooled columns in both streams) and "static" (bags of a few values)."""
    rng = np.random.default_rng({"ids-only": 11, "fvals-only": 12, "mixed": 13, "static": 14}[case])
    B = 50
    bnd = np.sort(rng.normal(size=60)).astype(np.float32)

    def lens(hi):
        x = rng.integers(0, hi, B)
        x[::9] = 0
        return x

    def ids(n, rows):
        return rng.integers(-5, rows + 5, n).astype(np.int64)

    cols, tabs, offs, vals = [], [], [], []

    def add(col, tab, ln, v):
        cols.append(col)
        tabs.append(tab)
        offs.append(synth.bag_offsets(ln))
        vals.append(v)

    if case == "ids-only":
        # the id stream holds only long padded columns: pieces do all of it
        for k, (pad, dim) in enumerate(((130, 8), (777, 128), (300, 36), (1000, 200))):
            ln = lens(pad + 200)
            add(ColumnSpec("identity" if k != 2 else "hash_mod", "padded", 900, dim, k, pad_len=pad),
                TableSpec(900, dim, 30 + k), ln,
                ids(int(ln.sum()), 900) if k != 2 else rng.integers(-2 ** 63, 2 ** 63 - 1, int(ln.sum()),
                                                                    dtype=np.int64))
    elif case == "fvals-only":
        # the value stream holds one long padded column, the id stream pools
        ln = lens(1300)
        add(ColumnSpec("bucketize", "padded", 61, 200, 0, boundaries=bnd, pad_len=1000), TableSpec(61, 200, 40),
            ln, rng.normal(size=int(ln.sum())).astype(np.float32))
        ln = lens(40)
        add(ColumnSpec("identity", "sum", 500, 64, 1), TableSpec(500, 64, 41), ln, ids(int(ln.sum()), 500))
    elif case == "mixed":
        # long padded columns beside pooled ones in both streams
        for k, (pool, pad) in enumerate((("padded", 300), ("sum", 0), ("mean", 0), ("padded", 1000))):
            ln = lens(1200)
            add(ColumnSpec("identity", pool, 700, 64, k, pad_len=pad), TableSpec(700, 64, 50 + k), ln,
                ids(int(ln.sum()), 700))
        ln = lens(400)
        add(ColumnSpec("bucketize", "padded", 61, 32, 4, boundaries=bnd, pad_len=130), TableSpec(61, 32, 54), ln,
            rng.normal(size=int(ln.sum())).astype(np.float32))
    else:
        # bags of a few values under a long pad: a launch of one tile per warp
        for k, pad in enumerate((300, 1000)):
            ln = lens(6)
            add(ColumnSpec("identity", "padded", 400, 16, k, pad_len=pad), TableSpec(400, 16, 60 + k), ln,
                ids(int(ln.sum()), 400))
    return Workload("padded-" + case, B, cols, tabs, offs, vals, lr=0.01)


def long_pooled_case(case):
    """Plans with long pooled bags (129 to 5000 values) beside short and empty
    ones, whose launches take the dynamic schedule: "sum-mean" (both poolings,
    dims 8 / 64 / 128), "weighted" (value weights on SUM columns), "fvals"
    (bucketized values), "truncated" (max_len 150 and 1000) and "wide" (rows
    of 200 floats)."""
    rng = np.random.default_rng({"sum-mean": 21, "weighted": 22, "fvals": 23, "truncated": 24, "wide": 25}[case])
    B = 48
    bnd = np.sort(rng.normal(size=40)).astype(np.float32)

    def lens():
        x = np.where(rng.random(B) < 0.6, rng.integers(129, 5000, B), rng.integers(0, 20, B))
        x[::11] = 0
        return x

    cols, tabs, offs, vals = [], [], [], []
    dims = {"sum-mean": (8, 64, 128), "weighted": (32, 64), "fvals": (16, 64), "truncated": (64, 128),
            "wide": (200, 36)}[case]
    for k, dim in enumerate(dims):
        ln = lens()
        n = int(ln.sum())
        pool = "mean" if k % 2 else "sum"
        if case == "weighted":
            pool = "sum"
        if case == "fvals" and k == 0:
            cols.append(ColumnSpec("bucketize", pool, bnd.size + 1, dim, k, boundaries=bnd))
            tabs.append(TableSpec(bnd.size + 1, dim, 70 + k))
            vals.append(rng.normal(size=n).astype(np.float32))
        else:
            rows = 3000
            cols.append(ColumnSpec("identity", pool, rows, dim, k,
                                   max_len=(150, 1000)[k] if case == "truncated" else 0))
            tabs.append(TableSpec(rows, dim, 70 + k))
            vals.append(rng.integers(-5, rows + 5, n).astype(np.int64))
        offs.append(synth.bag_offsets(ln))
    w = Workload("long-" + case, B, cols, tabs, offs, vals, lr=0.01)
    if case == "weighted":
        w.weights = [rng.uniform(-1.0, 2.0, int(o[-1])).astype(np.float32) for o in offs]
    return w
