"""CPU oracle of the multi-column embedding front end: a thin ctypes wrapper
around oracle.c (plain C, fp64 accumulation, single thread).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the
cpu_baseline / reference legs of bench.py may import this package.  The
product library (sparse_lookup_gb300) never imports it, and this package
imports nothing from there: the two share no code.

Columns are described by any object with the attributes ``transform``
('identity', 'hash_mod', 'bucketize', 'rows_given'), ``pooling`` ('sum',
'mean', 'padded'), ``num_rows``, ``dim``, ``table`` (physical table index),
``boundaries`` (float32 array or None), ``default`` (float32 [dim] or None)
and ``pad_len``.  Each function names the page passage it follows; the
definitions themselves are restated in oracle.c.
"""
import ctypes
from ctypes import c_int32, c_int64, c_uint32, c_uint64, c_float, c_void_p, POINTER

import numpy as np

from . import build as _build

TRANSFORM = {"identity": 0, "hash_mod": 1, "bucketize": 2, "rows_given": 3}
POOLING = {"sum": 0, "mean": 1, "padded": 2}

OK, ERR_ARG, ERR_OOM, ERR_FULL = 0, 1, 3, 5


class _Col(ctypes.Structure):
    _fields_ = [
        ("transform", c_int32),
        ("pooling", c_int32),
        ("num_rows", c_int64),
        ("dim", c_int32),
        ("table", c_int32),
        ("boundaries", c_void_p),
        ("num_boundaries", c_int32),
        ("pad_len", c_int32),
        ("default_vec", c_void_p),
        ("out_col", c_int64),
        ("max_len", c_int32),
        ("reserved", c_int32),
        ("weights", c_void_p),
        ("table_dtype", c_int32),
        ("reserved2", c_int32),
        ("row_scale", c_void_p),
    ]


TABLE_DTYPE = {"f32": 0, "bf16": 1, "f16": 2, "i8": 3}
_TABLE_NP = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16, "i8": np.int8}


_lib = None


def lib():
    """Load (building first if needed) liboracle.so."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_splitmix64.restype = c_uint64
        L.orc_splitmix64.argtypes = [c_uint64]
        L.orc_column_rows.restype = c_int32
        L.orc_column_rows.argtypes = [POINTER(_Col), c_int64, c_void_p, c_void_p, c_void_p]
        L.orc_forward.restype = c_int32
        L.orc_forward.argtypes = [POINTER(_Col), c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                  c_void_p, c_void_p, c_int64, c_void_p, c_void_p]
        L.orc_backward_adagrad.restype = c_int32
        L.orc_backward_adagrad.argtypes = [POINTER(_Col), c_int32, c_int32, c_void_p, c_void_p,
                                           c_void_p, c_void_p, c_int64, c_void_p, c_void_p,
                                           c_void_p, c_float, c_float, c_int64, POINTER(c_int64),
                                           c_void_p, c_void_p, c_void_p, c_void_p, c_int64]
        L.orc_backward_rows.restype = c_int32
        L.orc_backward_rows.argtypes = [POINTER(_Col), c_int32, c_int32, c_void_p, c_void_p, c_void_p,
                                        c_void_p, c_int64, c_void_p, c_int64, c_void_p, c_void_p,
                                        c_void_p, c_void_p, c_int32, c_float, c_float, c_void_p,
                                        c_void_p, c_void_p]
        L.orc_hash_init_value.restype = c_float
        L.orc_hash_init_value.argtypes = [c_uint64, c_int32, c_int64, c_int32, c_float]
        L.orc_hash_create.restype = c_void_p
        L.orc_hash_create.argtypes = [c_int64, c_int32, c_int32, c_uint64, c_float, c_void_p, c_void_p]
        L.orc_hash_destroy.restype = None
        L.orc_hash_destroy.argtypes = [c_void_p]
        L.orc_hash_lookup_or_insert.restype = c_int32
        L.orc_hash_lookup_or_insert.argtypes = [c_void_p, c_void_p, c_void_p, c_int64, c_uint32, c_void_p]
        L.orc_hash_evict.restype = c_int64
        L.orc_hash_evict.argtypes = [c_void_p, c_uint32, c_uint32]
        L.orc_hash_export.restype = c_int64
        L.orc_hash_export.argtypes = [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64]
        L.orc_hash_last_admitted.restype = c_int64
        L.orc_hash_last_admitted.argtypes = [c_void_p, c_void_p, c_int64]
        for f in ("orc_hash_size", "orc_hash_bump", "orc_hash_free_count"):
            getattr(L, f).restype = c_int64
            getattr(L, f).argtypes = [c_void_p]
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _ptr_array(arrs):
    """Host array of pointers (NULL for None) plus the arrays it keeps alive."""
    arr = (c_void_p * max(1, len(arrs)))()
    for i, a in enumerate(arrs):
        arr[i] = None if a is None else a.ctypes.data
    return arr


def _cols(cols, weights=None, table_dtypes=None, row_scales=None):
    """ctypes column array; pooled columns get consecutive out_col offsets;
    weights: optional per-column fp32 value weights (None entries: none);
    table_dtypes / row_scales: optional per physical table storage type
    ("f32", "bf16", "f16", "i8") and int8 row scales.
    Returns (array, keep-alive list, pooled width)."""
    arr = (_Col * max(1, len(cols)))()
    keep = []
    off = 0
    for i, c in enumerate(cols):
        wts = None if weights is None or weights[i] is None else np.ascontiguousarray(weights[i], np.float32)
        keep.append(wts)
        arr[i].weights = None if wts is None else wts.ctypes.data
        bnd = None if getattr(c, "boundaries", None) is None else np.ascontiguousarray(c.boundaries, np.float32)
        dft = None if getattr(c, "default", None) is None else np.ascontiguousarray(c.default, np.float32)
        keep += [bnd, dft]
        arr[i].transform = TRANSFORM[c.transform]
        arr[i].pooling = POOLING[c.pooling]
        arr[i].num_rows = int(c.num_rows)
        arr[i].dim = int(c.dim)
        arr[i].table = int(c.table)
        arr[i].boundaries = None if bnd is None else bnd.ctypes.data
        arr[i].num_boundaries = 0 if bnd is None else int(bnd.size)
        arr[i].pad_len = int(getattr(c, "pad_len", 0) or 0)
        arr[i].default_vec = None if dft is None else dft.ctypes.data
        arr[i].out_col = off if c.pooling != "padded" else 0
        arr[i].max_len = int(getattr(c, "max_len", 0) or 0)
        dt = "f32" if table_dtypes is None else table_dtypes[c.table]
        arr[i].table_dtype = TABLE_DTYPE[dt]
        if dt == "i8":
            sc = np.ascontiguousarray(row_scales[c.table], np.float32)
            keep.append(sc)
            arr[i].row_scale = sc.ctypes.data
        if c.pooling != "padded":
            off += int(c.dim)
    return arr, keep, off


def _values(cols, values):
    ids, fv = [], []
    for c, v in zip(cols, values):
        if c.transform == "bucketize":
            ids.append(None)
            fv.append(np.ascontiguousarray(v, np.float32))
        else:
            ids.append(np.ascontiguousarray(v, np.int64))
            fv.append(None)
    return ids, fv


def splitmix64(x: int) -> int:
    """One SplitMix64 output with state = x (hash transform, RecIS §3.1)."""
    return int(lib().orc_splitmix64(c_uint64(x & 0xFFFFFFFFFFFFFFFF)))


def column_rows(col, values) -> np.ndarray:
    """Transformed and safety-checked row per value (-1 = dropped).
    RecIS §3.1 transforms; RECom "Why this problem is worth solving" guards."""
    arr, keep, _ = _cols([col])
    n = len(values)
    ids, fv = _values([col], [values])
    out = np.empty(max(n, 1), np.int64)
    st = lib().orc_column_rows(arr, n, _ptr(ids[0]), _ptr(fv[0]), _ptr(out))
    if st != OK:
        raise ValueError("oracle column_rows failed: %d" % st)
    return out[:n]


def forward(cols, B, offsets, values, tables, want_rows=False, weights=None, table_dtypes=None,
            row_scales=None):
    """Pooled output [B, sum(dim of pooled cols)] (fp32), padded outputs
    (list, None for pooled columns) and optionally the rows per column.
    weights: optional per-column value weights, used by SUM columns.
    table_dtypes: optional storage type per physical table ("f32", "bf16" or
    "f16" as uint16 bit patterns, "i8" with row_scales[t] per row).
    RecIS §3.2 Algorithm 1 (forward); RECom guards and default fill."""
    arr, keep, width = _cols(cols, weights, table_dtypes, row_scales)
    C = len(cols)
    offs = [np.ascontiguousarray(o, np.int32) for o in offsets]
    ids, fv = _values(cols, values)
    tabs = [np.ascontiguousarray(t, _TABLE_NP["f32" if table_dtypes is None else table_dtypes[i]])
            for i, t in enumerate(tables)]
    out = np.zeros((B, max(width, 1)), np.float32)
    seq = [np.zeros((B, c.pad_len, c.dim), np.float32) if c.pooling == "padded" else None for c in cols]
    rows = [np.empty(max(int(o[B]), 1), np.int64) for o in offs] if want_rows else None
    st = lib().orc_forward(arr, C, B, _ptr_array(offs), _ptr_array(ids), _ptr_array(fv),
                           _ptr_array(tabs), _ptr(out), out.shape[1], _ptr_array(seq),
                           _ptr_array(rows) if rows is not None else None)
    if st != OK:
        raise ValueError("oracle forward failed: %d" % st)
    out = out[:, :width]
    if want_rows:
        rows = [r[: int(o[B])] for r, o in zip(rows, offs)]
        return out, seq, rows
    return out, seq


def backward_adagrad(cols, B, offsets, values, G, Gseq, W, acc, lr, eps, weights=None):
    """Backward + sparse Adagrad (RecIS §3.2 Algorithm 1 backward semantics,
    Figure 3 local reduce-ID; Adagrad as in torch.optim.Adagrad).
    W, acc: lists of float32 host tables per physical table, updated in place.
    Returns dict(table, row, count, grad) over unique rows, ascending by
    (table, row); grad is a list of float32 [dim] arrays.  weights: optional
    per-column value weights (SUM columns pass w_r G to their rows)."""
    arr, keep, width = _cols(cols, weights)
    C = len(cols)
    offs = [np.ascontiguousarray(o, np.int32) for o in offsets]
    ids, fv = _values(cols, values)
    G = np.ascontiguousarray(G, np.float32) if G is not None else np.zeros((B, 1), np.float32)
    gs = [None if g is None else np.ascontiguousarray(g, np.float32) for g in (Gseq or [None] * C)]
    for w, a in zip(W, acc):
        assert w.dtype == np.float32 and w.flags.c_contiguous
        assert a.dtype == np.float32 and a.flags.c_contiguous
    total = int(sum(int(o[B]) for o in offs))
    cap = max(total, 1)
    maxdim = max([int(c.dim) for c in cols] + [1])
    u_table = np.empty(cap, np.int32)
    u_row = np.empty(cap, np.int64)
    u_count = np.empty(cap, np.int64)
    u_grad = np.empty(cap * maxdim, np.float32)
    nu = c_int64(0)
    st = lib().orc_backward_adagrad(arr, C, B, _ptr_array(offs), _ptr_array(ids), _ptr_array(fv),
                                    _ptr(G), G.shape[1], _ptr_array(gs), _ptr_array(W),
                                    _ptr_array(acc), c_float(lr), c_float(eps), cap,
                                    ctypes.byref(nu), _ptr(u_table), _ptr(u_row), _ptr(u_count),
                                    _ptr(u_grad), u_grad.size)
    if st != OK:
        raise ValueError("oracle backward failed: %d" % st)
    n = nu.value
    dims = {int(c.table): int(c.dim) for c in cols}
    grads, pos = [], 0
    for i in range(n):
        d = dims[int(u_table[i])]
        grads.append(u_grad[pos:pos + d].copy())
        pos += d
    return dict(table=u_table[:n].copy(), row=u_row[:n].copy(), count=u_count[:n].copy(), grad=grads)


def backward_rows(cols, B, offsets, values, G, Gseq, targets, W_rows, acc_rows, lr, eps, weights=None):
    """The backward + Adagrad of backward_adagrad restricted to chosen rows,
    for tables too large to copy to the host.  targets: (table, row) pairs,
    or a tuple of two arrays (tables int32, rows int64);
    W_rows / acc_rows: float32 [n_targets, dim] host copies of those rows
    before the step, updated in place.  Each target's gradient is summed in
    the same order as backward_adagrad sums it.  Returns dict(table, row,
    count, grad [n, dim] fp32, absgrad [n, dim] fp64: sum of |scale * G|),
    ascending by (table, row) (W_rows / acc_rows must follow that order)."""
    arr, keep, width = _cols(cols, weights)
    C = len(cols)
    offs = [np.ascontiguousarray(o, np.int32) for o in offsets]
    ids, fv = _values(cols, values)
    G = np.ascontiguousarray(G, np.float32) if G is not None else np.zeros((B, 1), np.float32)
    gs = [None if g is None else np.ascontiguousarray(g, np.float32) for g in (Gseq or [None] * C)]
    if isinstance(targets, tuple) and len(targets) == 2 and isinstance(targets[0], np.ndarray):
        t_table = np.ascontiguousarray(targets[0], np.int32)
        t_row = np.ascontiguousarray(targets[1], np.int64)
    else:
        t_table = np.ascontiguousarray([t for t, _ in targets], np.int32)
        t_row = np.ascontiguousarray([r for _, r in targets], np.int64)
    order = np.lexsort((t_row, t_table))
    assert np.array_equal(order, np.arange(t_row.size)), "targets must ascend by (table, row)"
    assert W_rows.dtype == np.float32 and W_rows.flags.c_contiguous and W_rows.shape == acc_rows.shape
    assert acc_rows.dtype == np.float32 and acc_rows.flags.c_contiguous
    n, ld = W_rows.shape
    count = np.zeros(max(n, 1), np.int64)
    grad = np.zeros((max(n, 1), ld), np.float32)
    absg = np.zeros((max(n, 1), ld), np.float64)
    st = lib().orc_backward_rows(arr, C, B, _ptr_array(offs), _ptr_array(ids), _ptr_array(fv), _ptr(G),
                                 G.shape[1], _ptr_array(gs), n, _ptr(t_table), _ptr(t_row), _ptr(W_rows),
                                 _ptr(acc_rows), ld, c_float(lr), c_float(eps), _ptr(count), _ptr(grad),
                                 _ptr(absg))
    if st != OK:
        raise ValueError("oracle backward_rows failed: %d" % st)
    return dict(table=t_table, row=t_row, count=count[:n], grad=grad[:n], absgrad=absg[:n])


def unique_counts(cols, B, offsets, values):
    """Distinct (table, row) pairs that receive a gradient, ascending, with
    the number of contributions each (RecIS §3.2 Figure 3, local reduce-ID
    with counts): the valid rows of every column (padded columns: the first
    pad_len values of a bag), counted by numpy.unique."""
    keys = []
    for c, o, v in zip(cols, offsets, values):
        rows = column_rows(c, v)
        o = np.asarray(o, np.int64)
        valid = rows >= 0
        cut = c.pad_len if c.pooling == "padded" else int(getattr(c, "max_len", 0) or 0)
        if cut > 0:
            bag = np.repeat(np.arange(B), np.diff(o))
            valid &= (np.arange(rows.size) - o[bag]) < cut
        keys.append(np.int64(c.table) * (np.int64(1) << 40) + rows[valid])
    allk = np.concatenate(keys) if keys else np.zeros(0, np.int64)
    u, cnt = np.unique(allk, return_counts=True)
    return dict(table=(u >> 40).astype(np.int64), row=u & ((np.int64(1) << 40) - 1), count=cnt.astype(np.int64))


def hash_init_value(seed, tid, key, d, init_scale):
    """Initial value of element d of a newly admitted key's row."""
    return float(lib().orc_hash_init_value(c_uint64(seed & 0xFFFFFFFFFFFFFFFF), tid, key, d,
                                           c_float(init_scale)))


class Hash:
    """Collision-free dynamic table with frequency filter and expiry
    (Monolith §2.1 "Tabel Hash"); host row pool W/acc owned by this object."""

    def __init__(self, row_capacity, dim, threshold, seed, init_scale):
        self.W = np.zeros((row_capacity, dim), np.float32)
        self.acc = np.zeros((row_capacity, dim), np.float32)
        self.dim = dim
        self._h = lib().orc_hash_create(row_capacity, dim, threshold, c_uint64(seed),
                                        c_float(init_scale), _ptr(self.W), _ptr(self.acc))
        if not self._h:
            raise ValueError("oracle hash_create failed")

    def close(self):
        if self._h:
            lib().orc_hash_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def lookup_or_insert(self, tids, keys, step):
        tids = np.ascontiguousarray(tids, np.int32)
        keys = np.ascontiguousarray(keys, np.int64)
        n = keys.size
        rows = np.empty(max(n, 1), np.int64)
        st = lib().orc_hash_lookup_or_insert(self._h, _ptr(tids), _ptr(keys), n, step, _ptr(rows))
        return rows[:n], st

    def evict(self, now, ttl):
        return int(lib().orc_hash_evict(self._h, now, ttl))

    def size(self):
        return int(lib().orc_hash_size(self._h))

    def bump(self):
        return int(lib().orc_hash_bump(self._h))

    def free_count(self):
        return int(lib().orc_hash_free_count(self._h))

    def last_admitted(self):
        """Rows the last lookup_or_insert handed out (and initialised), in
        admission order."""
        n = int(lib().orc_hash_last_admitted(self._h, None, 0))
        out = np.empty(max(n, 1), np.int64)
        lib().orc_hash_last_admitted(self._h, _ptr(out), n)
        return out[:n]

    def export(self):
        """All live entries as a dict of arrays sorted by (tid, key)."""
        n = int(lib().orc_hash_export(self._h, None, None, None, None, None, 0))
        m = max(n, 1)
        t = np.empty(m, np.int32)
        k = np.empty(m, np.int64)
        r = np.empty(m, np.int64)
        c = np.empty(m, np.int64)
        s = np.empty(m, np.uint32)
        lib().orc_hash_export(self._h, _ptr(t), _ptr(k), _ptr(r), _ptr(c), _ptr(s), n)
        order = np.lexsort((k[:n], t[:n]))
        return dict(tid=t[:n][order], key=k[:n][order], row=r[:n][order],
                    count=c[:n][order], last_seen=s[:n][order])
