"""Shared test plumbing: materialise seeded workloads on the device, run the
oracle on the same inputs, compare with the tolerance the parity bar states
(fp32: |gpu - ref| <= 1e-6 + 1e-5 |ref|; integers bit-exact)."""
import numpy as np

import oracle
from sparse_lookup_gb300 import synth

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


def check_row_update(key, gr, absg, count, g_gpu, w0, a0, w_gpu, a_gpu, w_ref, a_ref, lr, eps):
    """One touched row: the aggregated gradient within the fp32 summation
    bound of the oracle's fp64 sum; the updated weights within 1e-5 rel /
    1e-6 abs except elements that fp32 summation leaves ill-conditioned (the
    first Adagrad step from acc = 0 has dW/dg = lr eps / g^2, and a sign fp32
    does not determine flips the step); the accumulator within the bound the
    gradient error implies.  Returns (elements outside the tolerance, all of
    them ill-conditioned; elements checked)."""
    gr = np.asarray(gr, np.float64)
    absg = np.asarray(absg, np.float64)
    k = int(count) + 1
    bnd = gamma(k) * absg + 1e-30
    err = np.abs(np.asarray(g_gpu, np.float64) - gr)
    ok = (err <= ATOL + RTOL * np.abs(gr)) | (err <= bnd)
    assert ok.all(), "aggregated gradient of row %s: err %s bound %s" % (key, err[~ok][:4], bnd[~ok][:4])
    # probabilistic bound (Higham & Mary, 2019): lambda sqrt(k) u sum|x|,
    # used only to decide which weights fp32 leaves ill-conditioned
    pbnd = np.minimum(bnd, 8.0 * np.sqrt(k) * U32 * absg) + 1e-30
    a0 = np.asarray(a0, np.float64)
    w0 = np.asarray(w0, np.float64)
    step = lambda gg: w0 - lr * gg / (np.sqrt(a0 + gg * gg) + eps)
    spread = np.abs(step(gr + pbnd) - step(gr - pbnd))
    amb = spread > ATOL + RTOL * np.abs(step(gr))
    wr = np.asarray(w_ref, np.float64)
    errw = np.abs(np.asarray(w_gpu, np.float64) - wr)
    within = errw <= ATOL + RTOL * np.abs(wr)
    okw = within | amb
    assert okw.all(), "weights of row %s: %s vs %s" % (key, np.asarray(w_gpu)[~okw][:4], wr[~okw][:4])
    ar = np.asarray(a_ref, np.float64)
    abound = 2 * np.abs(gr) * pbnd + pbnd * pbnd + 4 * U32 * np.abs(ar)
    erra = np.abs(np.asarray(a_gpu, np.float64) - ar)
    oka = (erra <= ATOL + RTOL * np.abs(ar)) | (erra <= abound) | amb
    assert oka.all(), "accumulator of row %s: %s vs %s" % (key, np.asarray(a_gpu)[~oka][:4], ar[~oka][:4])
    return int((amb & ~within).sum()), gr.size


def check_train_step(ts, max_ambiguous_frac=1e-5):
    """Bit-exact unique rows and counts; every touched row checked by
    check_row_update; untouched rows unchanged.  Returns the number of
    elements outside the tolerance (all ill-conditioned), which must stay
    below max(16, 1e-5 of the updated elements): one cancelling pair of bags
    repeats its element in every row the two bags share."""
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
    index = {(int(ref["table"][i]), int(ref["row"][i])): i for i in range(n)}
    for t_gpu, t_spec in t2s.items():
        Wg = ts.m.tables[t_spec].cpu().numpy()
        Ag = ts.m.accs[t_spec].cpu().numpy()
        W0 = ts.W0[t_spec]
        touched = np.zeros(W0.shape[0], bool)
        sel = ref["table"] == t_spec
        touched[ref["row"][sel]] = True
        assert np.array_equal(Wg[~touched], W0[~touched]), "untouched rows changed"
        assert np.array_equal(Ag[~touched], ts.A0[t_spec][~touched]), "untouched accumulators changed"
        dim = dims[t_spec]
        for r in ref["row"][sel]:
            i = index[(t_spec, int(r))]
            e, m = check_row_update((t_spec, int(r)), ref["grad"][i], absg["grad"][i], ref["count"][i],
                                    g[i, :dim], W0[r], ts.A0[t_spec][r], Wg[r], Ag[r], Wr[t_spec][r],
                                    Ar[t_spec][r], ts.w.lr, ts.w.eps)
            excluded += e
            total += m
    assert excluded <= max(16, max_ambiguous_frac * total), (excluded, total)
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


class DynamicRun:
    """The dynamic-table training loop through the C ABI -- per step:
    hash_lookup_or_insert -> emb_forward (rows_given columns over the table's
    row pool) -> emb_backward_update -> hash_evict_expired -- next to the
    oracle doing the same on the host."""

    def __init__(self, C, B, steps, num_slots, cap, dim=32, thr=3, ttl=10, seed=1005, alpha=1.2, key_bits=34,
                 max_len=5, lr=0.01, max_probes=128, check_every=1):
        import torch
        import sparse_lookup_gb300 as sl
        self.C, self.B, self.steps, self.ttl, self.lr = C, B, steps, ttl, lr
        self.seed, self.alpha, self.key_bits, self.max_len = seed, alpha, key_bits, max_len
        self.check_every = check_every
        max_keys = C * B * max_len
        self.ht = sl.HashTable(num_slots, cap, dim, thr, max_probes, seed, 0.01, max_keys)
        self.oh = oracle.Hash(cap, dim, thr, seed, 0.01)
        self.cols = [synth.ColumnSpec("rows_given", "sum", cap, dim, 0) for _ in range(C)]
        self.plan = sl.Plan(self.cols, [self.ht.weight], [self.ht.acc], max_batch=B, max_ids=max_keys,
                            training=True)

    def step(self, t, check, check_out=None):
        """One step; check: return the rows of both sides; check_out (default:
        check): also the pooled outputs of both sides."""
        check_out = check if check_out is None else check_out
        import torch
        offs, keys = synth.dynamic_keys(self.seed, t, self.C, self.B, self.alpha, self.key_bits, self.max_len)
        tids = np.concatenate([np.full(k.size, c, np.int32) for c, k in enumerate(keys)])
        allk = np.concatenate(keys)
        rows = self.ht.lookup_or_insert(torch.from_numpy(tids).cuda(), torch.from_numpy(allk).cuda(), t)
        ids_off = np.concatenate([[0], np.cumsum(np.concatenate([np.diff(o) for o in offs]))]).astype(np.int32)
        out, _ = self.plan.forward(self.B, rows, torch.from_numpy(ids_off).cuda(), None, None)
        G = synth.make_grad((self.B, self.plan.out_width), 500 + t, "cuda")
        self.plan.backward_update(G, None, self.lr, 1e-10)
        self.ht.evict_expired(t, self.ttl)
        torch.cuda.synchronize()
        st_h, st_p = self.ht.device_status(), self.plan.device_status()
        # oracle
        rows_o, st_o = self.oh.lookup_or_insert(tids, allk, t)
        res = dict(status=(st_h, st_p, st_o))
        vals = []
        pos = 0
        for o in offs:
            n = int(o[-1])
            vals.append(rows_o[pos:pos + n])
            pos += n
        if check:
            res["rows"] = (rows.cpu().numpy(), rows_o)
        if check_out:
            res["out"] = (out.cpu().numpy(), oracle.forward(self.cols, self.B, offs, vals, [self.oh.W])[0])
        oracle.backward_adagrad(self.cols, self.B, offs, vals, G.cpu().numpy(), None, [self.oh.W], [self.oh.acc],
                                self.lr, 1e-10)
        self.oh.evict(t, self.ttl)
        return res
