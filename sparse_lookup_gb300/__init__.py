"""sparse_lookup_gb300 -- GB300-native multi-column embedding front end.

Thin Python binding over the C ABI of libsparse_lookup.so (include/emb.h).
Every function here only marshals arguments: tensors become raw device
pointers, column specs become emb_column_desc structs.  All compute runs in
the library's CUDA kernels; there is no CPU fallback.  If the library has not
been built, every call raises.

Raw entry points keep their C names (emb_plan_create, emb_forward,
emb_backward_update, hash_lookup_or_insert, hash_evict_expired, ...); the
``Plan`` and ``HashTable`` classes wrap them for callers that hold PyTorch
tensors.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int32, c_int64, c_uint32, c_uint64, c_void_p

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsparse_lookup.so")

STATUS = {
    0: "EMB_OK", 1: "EMB_ERR_INVALID_ARG", 2: "EMB_ERR_UNSUPPORTED", 3: "EMB_ERR_OOM",
    4: "EMB_ERR_CUDA", 5: "EMB_ERR_TABLE_FULL", 6: "EMB_ERR_PROBE_LIMIT",
    7: "EMB_ERR_BAD_INDEX", 8: "EMB_ERR_TIMEOUT",
}
TRANSFORM = {"identity": 0, "hash_mod": 1, "bucketize": 2, "rows_given": 3}
TABLE_DTYPE = {"float32": 0, "bfloat16": 1, "float16": 2, "int8": 3}   # torch dtype name -> emb_table_dtype
POOLING = {"sum": 0, "mean": 1, "padded": 2}
PLAN_TRAINING = 1
PLAN_ATOMIC_BACKWARD = 2


class EmbError(RuntimeError):
    def __init__(self, status, where):
        self.status = int(status)
        super().__init__("%s: %s" % (where, STATUS.get(self.status, str(status))))


class EmbColumnDesc(ctypes.Structure):
    _fields_ = [
        ("transform", c_int32),
        ("pooling", c_int32),
        ("num_rows", c_int64),
        ("dim", c_int32),
        ("pad_len", c_int32),
        ("boundaries", c_void_p),
        ("num_boundaries", c_int32),
        ("max_len", c_int32),
        ("weight", c_void_p),
        ("adagrad_acc", c_void_p),
        ("default_vec", c_void_p),
        ("table_dtype", c_int32),
        ("reserved", c_int32),
        ("row_scale", c_void_p),
    ]


class EmbBackwardDebug(ctypes.Structure):
    _fields_ = [
        ("n_unique", c_void_p),
        ("uniq_table", c_void_p),
        ("uniq_row", c_void_p),
        ("counts", c_void_p),
        ("agg_grad", c_void_p),
    ]


_lib = None

# name -> (restype, argtypes)
_SIGS = {
    "emb_plan_create": (c_int32, [POINTER(EmbColumnDesc), c_int32, c_int32, c_int64, c_uint32, POINTER(c_void_p)]),
    "emb_plan_destroy": (c_int32, [c_void_p]),
    "emb_plan_info": (c_int32, [c_void_p, POINTER(c_int64), POINTER(c_int64), POINTER(c_int32), c_void_p,
                                POINTER(c_int64)]),
    "emb_forward": (c_int32, [c_void_p, c_int32, c_void_p, c_void_p, c_void_p, c_int64, c_void_p, c_void_p,
                              c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_void_p]),
    "emb_backward_update": (c_int32, [c_void_p, c_void_p, c_void_p, c_float, c_float, c_void_p,
                                      POINTER(EmbBackwardDebug)]),
    "emb_get_device_status": (c_int32, [c_void_p, c_void_p]),
    "hash_create": (c_int32, [c_int64, c_int64, c_int32, c_int32, c_int32, c_uint64, c_float, c_int64,
                              POINTER(c_void_p)]),
    "hash_rows": (c_int32, [c_void_p, POINTER(c_void_p), POINTER(c_void_p)]),
    "hash_lookup_or_insert": (c_int32, [c_void_p, c_void_p, c_void_p, c_int64, c_uint32, c_void_p, c_void_p]),
    "hash_evict_expired": (c_int32, [c_void_p, c_uint32, c_uint32, c_void_p, c_void_p]),
    "hash_import": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64, c_void_p]),
    "hash_export": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_int64,
                              POINTER(c_int64), c_void_p]),
    "hash_get_device_status": (c_int32, [c_void_p, c_void_p]),
    "hash_destroy": (c_int32, [c_void_p]),
    "emb_sparse_adagrad_noalloc": (c_int32, [c_void_p, c_int64, c_void_p, c_void_p, c_void_p, c_int64, c_int32,
                                             c_float, c_float, c_void_p]),
    "emb_calibrate_gather": (c_int32, [c_void_p, c_int64, c_int32, c_void_p, c_int64, c_void_p, c_void_p]),
    "emb_selftest_hash_mod": (c_int32, [c_void_p, c_int64, c_int64, c_void_p]),
    "emb_noalloc_get_device_status": (c_int32, [c_void_p]),
    "emb_selftest_sort_timeout": (c_int32, [c_void_p, c_void_p, c_void_p, c_void_p]),
    "emb_debug_fail_alloc": (c_int32, [c_int64]),
    "emb_debug_live_allocations": (c_int32, [c_void_p, c_void_p]),
    "emb_version": (c_char_p, []),
}

EXPORTED = tuple(_SIGS)


def lib():
    """The loaded CUDA library.  Raises if it was not built: there is no
    fallback path."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libsparse_lookup.so is missing: run __graft_entry__.build() "
                               "(nvcc, sm_103a) first; there is no CPU fallback")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status, where):
    if status != 0:
        raise EmbError(status, where)


def ptr(x):
    """Raw pointer of a tensor / ndarray / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError("cannot take a pointer of %r" % type(x))


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------------------
# raw C names
# ---------------------------------------------------------------------------

def emb_plan_create(descs, max_batch, max_ids, flags):
    arr = (EmbColumnDesc * len(descs))(*descs)
    h = c_void_p()
    _check(lib().emb_plan_create(arr, len(descs), max_batch, max_ids, flags, ctypes.byref(h)), "emb_plan_create")
    return h.value


def emb_plan_destroy(plan):
    _check(lib().emb_plan_destroy(plan), "emb_plan_destroy")


def emb_plan_info(plan, n_cols):
    w, s, t, ws = c_int64(), c_int64(), c_int32(), c_int64()
    ct = (c_int32 * max(1, n_cols))()
    _check(lib().emb_plan_info(plan, ctypes.byref(w), ctypes.byref(s), ctypes.byref(t), ct, ctypes.byref(ws)),
           "emb_plan_info")
    return dict(out_width=w.value, seq_floats_per_bag=s.value, n_tables=t.value,
                col_table=list(ct)[:n_cols], workspace_bytes=ws.value)


def emb_forward(plan, batch, ids, id_offsets, id_weights, n_ids, fvals, f_offsets, f_weights, n_fvals, out,
                seq_out, rows_dbg=None, stream=None):
    _check(lib().emb_forward(plan, batch, ptr(ids), ptr(id_offsets), ptr(id_weights), n_ids, ptr(fvals),
                             ptr(f_offsets), ptr(f_weights), n_fvals, ptr(out), ptr(seq_out), ptr(rows_dbg),
                             _stream(stream)), "emb_forward")


def emb_backward_update(plan, grad_out, grad_seq, lr, eps, stream=None, dbg=None):
    _check(lib().emb_backward_update(plan, ptr(grad_out), ptr(grad_seq), lr, eps, _stream(stream),
                                     ctypes.byref(dbg) if dbg is not None else None), "emb_backward_update")


def emb_get_device_status(plan, stream=None):
    return int(lib().emb_get_device_status(plan, _stream(stream)))


def hash_create(num_slots, row_capacity, dim, admit_threshold, max_probes, init_seed, init_scale,
                max_keys_per_call):
    h = c_void_p()
    _check(lib().hash_create(num_slots, row_capacity, dim, admit_threshold, max_probes,
                             init_seed & 0xFFFFFFFFFFFFFFFF, init_scale, max_keys_per_call, ctypes.byref(h)),
           "hash_create")
    return h.value


def hash_rows(h):
    w, a = c_void_p(), c_void_p()
    _check(lib().hash_rows(h, ctypes.byref(w), ctypes.byref(a)), "hash_rows")
    return w.value, a.value


def hash_lookup_or_insert(h, table_ids, keys, n, step, rows_out, stream=None):
    _check(lib().hash_lookup_or_insert(h, ptr(table_ids), ptr(keys), n, step, ptr(rows_out), _stream(stream)),
           "hash_lookup_or_insert")


def hash_evict_expired(h, now, ttl, stream=None, n_evicted_dev=None):
    _check(lib().hash_evict_expired(h, now, ttl, _stream(stream), ptr(n_evicted_dev)), "hash_evict_expired")


def hash_export(h, tids, keys, rows, counts, last_seen, cap, stream=None):
    n = c_int64()
    _check(lib().hash_export(h, ptr(tids), ptr(keys), ptr(rows), ptr(counts), ptr(last_seen), cap,
                             ctypes.byref(n), _stream(stream)), "hash_export")
    return n.value


def hash_import(h, tids, keys, rows, counts, last_seen, n, stream=None):
    _check(lib().hash_import(h, ptr(tids), ptr(keys), ptr(rows), ptr(counts), ptr(last_seen), n, _stream(stream)),
           "hash_import")


def hash_get_device_status(h, stream=None):
    return int(lib().hash_get_device_status(h, _stream(stream)))


def hash_destroy(h):
    _check(lib().hash_destroy(h), "hash_destroy")


def emb_sparse_adagrad_noalloc(rows, n, grads, weight, acc, num_rows, dim, lr, eps, stream=None):
    """One sparse Adagrad step on one table with no allocation (fixed scratch
    inside the library; n <= 2^18, dim <= 256)."""
    _check(lib().emb_sparse_adagrad_noalloc(ptr(rows), n, ptr(grads), ptr(weight), ptr(acc), num_rows, dim, lr,
                                            eps, _stream(stream)), "emb_sparse_adagrad_noalloc")


def emb_noalloc_get_device_status(stream=None):
    """Latched device status of emb_sparse_adagrad_noalloc calls (cleared)."""
    return int(lib().emb_noalloc_get_device_status(_stream(stream)))


def emb_selftest_sort_timeout():
    """Runs the sort's bounded-wait self test; returns dict(status, latched,
    fail_word, table_untouched, wait_ms)."""
    latched, fail = ctypes.c_uint32(0), ctypes.c_uint32(0)
    untouched, ms = ctypes.c_int32(0), ctypes.c_float(0.0)
    st = lib().emb_selftest_sort_timeout(ctypes.byref(latched), ctypes.byref(fail), ctypes.byref(untouched),
                                         ctypes.byref(ms))
    return dict(status=int(st), latched=latched.value, fail_word=fail.value, table_untouched=bool(untouched.value),
                wait_ms=ms.value)


def emb_debug_fail_alloc(after):
    _check(lib().emb_debug_fail_alloc(after), "emb_debug_fail_alloc")


def emb_debug_live_allocations():
    """(count, bytes) of the device allocations the library's handles hold."""
    c, b = ctypes.c_int64(0), ctypes.c_int64(0)
    _check(lib().emb_debug_live_allocations(ctypes.byref(c), ctypes.byref(b)), "emb_debug_live_allocations")
    return c.value, b.value


def emb_calibrate_gather(table, num_rows, dim, row_idx, n, sink, stream=None):
    _check(lib().emb_calibrate_gather(ptr(table), num_rows, dim, ptr(row_idx), n, ptr(sink), _stream(stream)),
           "emb_calibrate_gather")


def emb_selftest_hash_mod(ids, num_rows):
    import numpy as np
    ids = np.ascontiguousarray(ids, np.int64)
    out = np.empty(max(ids.size, 1), np.int64)
    _check(lib().emb_selftest_hash_mod(ptr(ids), ids.size, num_rows, ptr(out)), "emb_selftest_hash_mod")
    return out[: ids.size]


def emb_version():
    return lib().emb_version().decode()


# ---------------------------------------------------------------------------
# tensor-level wrappers (marshalling only)
# ---------------------------------------------------------------------------

class Plan:
    """A plan over columns described by objects with the attributes
    transform, pooling, num_rows, dim, table, boundaries, default, pad_len
    (e.g. synth.ColumnSpec).  ``weights[t]`` / ``accs[t]`` are the device
    tables of physical table t.  The device copies of boundaries and default
    vectors are owned here and live as long as the plan.  backward: "sort"
    (radix sort + run reduction, deterministic) or "atomic" (warp merge +
    atomics into a compact gradient).  A table's storage type follows its
    tensor's dtype (float32, bfloat16, float16, or int8 with
    ``row_scales[t]``, fp32 per row); low-precision tables are for inference
    plans."""

    def __init__(self, columns, weights, accs=None, max_batch=1, max_ids=0, training=False, device="cuda",
                 backward="sort", row_scales=None):
        import torch
        self.columns = list(columns)
        self.training = training
        self._keep = []
        descs = []
        for c in self.columns:
            d = EmbColumnDesc()
            d.transform = TRANSFORM[c.transform]
            d.pooling = POOLING[c.pooling]
            d.num_rows = int(c.num_rows)
            d.dim = int(c.dim)
            d.pad_len = int(getattr(c, "pad_len", 0) or 0)
            d.max_len = int(getattr(c, "max_len", 0) or 0) if c.pooling != "padded" else 0
            if getattr(c, "boundaries", None) is not None:
                b = torch.as_tensor(c.boundaries, dtype=torch.float32).to(device).contiguous()
                self._keep.append(b)
                d.boundaries = b.data_ptr()
                d.num_boundaries = int(b.numel())
            if getattr(c, "default", None) is not None:
                v = torch.as_tensor(c.default, dtype=torch.float32).to(device).contiguous()
                self._keep.append(v)
                d.default_vec = v.data_ptr()
            tw = weights[c.table]
            d.weight = tw.data_ptr()
            d.table_dtype = TABLE_DTYPE[str(tw.dtype).replace("torch.", "")]
            if d.table_dtype == TABLE_DTYPE["int8"]:
                d.row_scale = row_scales[c.table].data_ptr()
            if accs is not None:
                d.adagrad_acc = accs[c.table].data_ptr()
            descs.append(d)
        if backward not in ("sort", "atomic"):
            raise ValueError("backward: 'sort' or 'atomic'")
        flags = (PLAN_TRAINING if training else 0) | (PLAN_ATOMIC_BACKWARD if backward == "atomic" else 0)
        self.backward = backward
        self.handle = emb_plan_create(descs, max_batch, max_ids, flags)
        self.info = emb_plan_info(self.handle, len(descs))
        self.out_width = self.info["out_width"]
        self.seq_per_bag = self.info["seq_floats_per_bag"]
        self.max_dim = max(int(c.dim) for c in self.columns)
        self.max_ids = max_ids

    def close(self):
        if getattr(self, "handle", None):
            emb_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, batch, ids, id_offsets, fvals, f_offsets, out=None, seq_out=None, rows_dbg=None,
                stream=None, id_weights=None, f_weights=None):
        import torch
        dev = id_offsets.device if id_offsets is not None else f_offsets.device
        if out is None:
            out = torch.empty((batch, self.out_width), dtype=torch.float32, device=dev)
        if seq_out is None and self.seq_per_bag:
            seq_out = torch.empty((batch * self.seq_per_bag,), dtype=torch.float32, device=dev)
        n_ids = 0 if ids is None else ids.numel()
        n_f = 0 if fvals is None else fvals.numel()
        for wt, vals in ((id_weights, ids), (f_weights, fvals)):
            if wt is not None and (vals is None or wt.numel() != vals.numel() or wt.dtype != torch.float32):
                raise ValueError("value weights: one float32 per value of their stream")
        emb_forward(self.handle, batch, ids, id_offsets, id_weights, n_ids, fvals, f_offsets, f_weights, n_f,
                    out, seq_out, rows_dbg, stream)
        return out, seq_out

    def backward_update(self, grad_out, grad_seq, lr, eps, stream=None, debug=False):
        import torch
        if not debug:
            emb_backward_update(self.handle, grad_out, grad_seq, lr, eps, stream)
            return None
        dev = grad_out.device if grad_out is not None else grad_seq.device
        cap = max(self.max_ids, 1)
        t = dict(n_unique=torch.zeros(1, dtype=torch.int64, device=dev),
                 uniq_table=torch.empty(cap, dtype=torch.int32, device=dev),
                 uniq_row=torch.empty(cap, dtype=torch.int64, device=dev),
                 counts=torch.empty(cap, dtype=torch.int32, device=dev),
                 agg_grad=torch.zeros((cap, self.max_dim), dtype=torch.float32, device=dev))
        dbg = EmbBackwardDebug(*[t[k].data_ptr() for k in ("n_unique", "uniq_table", "uniq_row", "counts",
                                                           "agg_grad")])
        emb_backward_update(self.handle, grad_out, grad_seq, lr, eps, stream, dbg)
        n = int(t["n_unique"].item())
        return dict(table=t["uniq_table"][:n], row=t["uniq_row"][:n], count=t["counts"][:n],
                    grad=t["agg_grad"][:n])

    def device_status(self, stream=None):
        return emb_get_device_status(self.handle, stream)


class HashTable:
    """Collision-free dynamic table on the device (hash_* entry points).
    ``weight`` / ``acc`` are torch views of the row pool owned by the table."""

    def __init__(self, num_slots, row_capacity, dim, admit_threshold, max_probes, init_seed, init_scale,
                 max_keys_per_call):
        import torch
        self.dim = dim
        self.row_capacity = row_capacity
        self.handle = hash_create(num_slots, row_capacity, dim, admit_threshold, max_probes, init_seed,
                                  init_scale, max_keys_per_call)
        w, a = hash_rows(self.handle)
        self.weight_ptr, self.acc_ptr = w, a
        self.weight = _device_view(w, (row_capacity, dim))
        self.acc = _device_view(a, (row_capacity, dim))

    def lookup_or_insert(self, table_ids, keys, step, rows_out=None, stream=None):
        import torch
        n = keys.numel()
        if rows_out is None:
            rows_out = torch.empty(n, dtype=torch.int64, device=keys.device)
        hash_lookup_or_insert(self.handle, table_ids, keys, n, step, rows_out, stream)
        return rows_out

    def evict_expired(self, now, ttl, stream=None, n_evicted=None):
        hash_evict_expired(self.handle, now, ttl, stream, n_evicted)

    def export(self, cap=None, stream=None):
        """All live entries as host numpy arrays sorted by (tid, key)."""
        import numpy as np
        import torch
        n = hash_export(self.handle, None, None, None, None, None, 0, stream)
        cap = n if cap is None else cap
        dev = "cuda"
        t = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
        k = torch.empty(max(cap, 1), dtype=torch.int64, device=dev)
        r = torch.empty(max(cap, 1), dtype=torch.int64, device=dev)
        c = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
        s = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
        n = hash_export(self.handle, t, k, r, c, s, cap, stream)
        m = min(n, cap)
        t, k, r, c = [x[:m].cpu().numpy() for x in (t, k, r, c)]
        s = s[:m].cpu().numpy().view(np.uint32)
        order = np.lexsort((k, t))
        return dict(tid=t[order], key=k[order], row=r[order], count=c[order], last_seen=s[order])

    def import_entries(self, snap, stream=None):
        """Restore the entries of a snapshot (a dict as export() returns:
        host arrays tid, key, row, count, last_seen); the row pool is the
        caller's to restore through .weight / .acc."""
        import numpy as np
        import torch
        n = int(len(snap["key"]))
        dev = "cuda"
        t = torch.from_numpy(np.ascontiguousarray(snap["tid"], np.int32)).to(dev)
        k = torch.from_numpy(np.ascontiguousarray(snap["key"], np.int64)).to(dev)
        r = torch.from_numpy(np.ascontiguousarray(snap["row"], np.int64)).to(dev)
        cnt = np.where(np.asarray(snap["row"]) >= 0, 0, np.asarray(snap["count"]))
        c = torch.from_numpy(np.ascontiguousarray(cnt, np.int32)).to(dev)
        s = torch.from_numpy(np.ascontiguousarray(snap["last_seen"], np.uint32).view(np.int32)).to(dev)
        hash_import(self.handle, t, k, r, c, s, n, stream)

    def device_status(self, stream=None):
        return hash_get_device_status(self.handle, stream)

    def close(self):
        if getattr(self, "handle", None):
            hash_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _device_view(ptr_value, shape):
    """A torch float32 tensor viewing library-owned device memory (no copy)."""
    import torch

    class _Holder:
        pass

    h = _Holder()
    h.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": "<f4", "data": (ptr_value, False),
                                  "version": 2, "strides": None}
    return torch.as_tensor(h, device="cuda")
