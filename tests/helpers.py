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
