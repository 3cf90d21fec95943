"""Seeded synthetic inputs for the multi-column embedding front end.

This module only draws inputs: column descriptions, CSR bags, IDs, feature
values, bucket boundaries, tables and upstream gradients.  It holds none of
the method's arithmetic (no hashing into rows, no bucketizing, no pooling, no
optimizer), so both the CUDA path and the CPU oracle may take their inputs
from it.

Workloads (seed = 1000 + workload index, sub-seeded per column):
  tiny        8 hash-mod columns, B=64, 1000 rows x dim 16, bags U{0..5},
              IDs U[0, 2^40), sum pooling, one training step, lr 0.01.
  inference   700 hash-mod + 300 bucketize columns, B=512; rows log-uniform
              1e3..1e6; 10..100 boundaries from sorted N(0,1) draws; values
              N(0,1); dims U{8,16,32,64}; bags U{1..20} with 5% forced empty;
              sum/mean per column by a seeded coin; forward only.
  training    200 identity columns, B=8192, rows log-uniform 1e5..1e7, dim 64,
              bags U{1..50}, IDs bounded-Zipf(1.1) scattered by a bijection,
              3% out-of-range IDs; sum pooling; forward + backward + Adagrad.
  sequences   20 identity columns, B=1024, lengths U{200..1000}, 1e7 rows,
              dim 128, Zipf(1.05); mean pooling, or padded unpooled [B,1000,128].
  dynamic     100 columns over one hash table, B=16384, bags U{0..5}, keys
              Zipf(1.2) over 2^34 scattered by an odd multiplier; dim 32;
              admission threshold 3, expiry after 10 idle steps; 50 steps.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GOLDEN_RATIO = (1.0 + 5.0 ** 0.5) / 2.0


@dataclass
class ColumnSpec:
    transform: str                 # 'identity' | 'hash_mod' | 'bucketize' | 'rows_given'
    pooling: str                   # 'sum' | 'mean' | 'padded'
    num_rows: int
    dim: int
    table: int                     # physical table index (columns may share one)
    boundaries: np.ndarray | None = None
    default: np.ndarray | None = None
    pad_len: int = 0
    max_len: int = 0               # sum / mean: pool only a bag's first max_len values (0 = all)


@dataclass
class TableSpec:
    num_rows: int
    dim: int
    seed: int
    std: float = 0.01


@dataclass
class Workload:
    name: str
    B: int
    columns: list
    tables: list
    offsets: list                  # per column int32 [B+1], relative to its values
    values: list                   # per column int64 (ids) or float32 (bucketize)
    lr: float = 0.01
    eps: float = 1e-10
    train: bool = False
    seed: int = 0
    extra: dict = field(default_factory=dict)
    weights: list | None = None    # per column fp32 value weights (weighted SUM bags), or None

    @property
    def n_values(self) -> int:
        return int(sum(int(o[-1]) for o in self.offsets))


# --------------------------------------------------------------------------
# distributions
# --------------------------------------------------------------------------

def _h_integral(x, q):
    """Integral of t^-q from 1 to x (q != 1 handled through expm1/log)."""
    lx = np.log(x)
    t = (1.0 - q) * lx
    small = np.abs(t) < 1e-8
    ratio = np.where(small, 1.0 + 0.5 * t, np.expm1(np.where(small, 1.0, t)) / np.where(small, 1.0, t))
    return ratio * lx


def _h_integral_inv(u, q):
    t = np.maximum(u * (1.0 - q), -1.0)
    small = np.abs(t) < 1e-8
    ratio = np.where(small, 1.0 - 0.5 * t, np.log1p(np.where(small, 0.0, t)) / np.where(small, 1.0, t))
    return np.exp(ratio * u)


def zipf(rng: np.random.Generator, n: int, alpha: float, size: int) -> np.ndarray:
    """Bounded Zipf ranks k in [1, n], P(k) proportional to k^-alpha, drawn by
    rejection-inversion (Hoermann & Derflinger, 1996).  Vectorised: rejected
    draws are redrawn until every slot is accepted."""
    q = float(alpha)
    h = lambda x: np.exp(-q * np.log(x))
    hx1 = float(_h_integral(np.float64(1.5), q)) - 1.0
    hn = float(_h_integral(np.float64(n + 0.5), q))
    s = 2.0 - float(_h_integral_inv(_h_integral(np.float64(2.5), q) - h(np.float64(2.0)), q))
    out = np.empty(size, np.int64)
    todo = np.arange(size)
    while todo.size:
        u = hn + rng.random(todo.size) * (hx1 - hn)
        x = _h_integral_inv(u, q)
        k = np.clip(np.floor(x + 0.5), 1, n)
        ok = (k - x <= s) | (u >= _h_integral(k + 0.5, q) - h(k))
        out[todo[ok]] = k[ok].astype(np.int64)
        todo = todo[~ok]
    return out


def _is_prime(p: int) -> bool:
    if p < 2:
        return False
    if p % 2 == 0:
        return p == 2
    r = int(math.isqrt(p))
    f = 3
    while f <= r:
        if p % f == 0:
            return False
        f += 2
    return True


def scatter_prime(n: int) -> int:
    """Smallest prime above n / golden ratio that is coprime with n."""
    p = int(n / GOLDEN_RATIO) + 1
    while not (_is_prime(p) and math.gcd(p, n) == 1):
        p += 1
    return p


def scatter_ranks(k: np.ndarray, n: int) -> np.ndarray:
    """Map Zipf ranks 1..n to rows by the bijection (k-1)*p mod n, so that hot
    ranks are not adjacent in memory."""
    p = scatter_prime(n)
    return ((k - 1) * np.int64(p)) % np.int64(n)


def log_uniform_int(rng, lo, hi, size):
    return np.rint(np.exp(rng.uniform(np.log(lo), np.log(hi), size))).astype(np.int64)


def bag_offsets(lengths: np.ndarray) -> np.ndarray:
    off = np.zeros(lengths.size + 1, np.int64)
    np.cumsum(lengths, out=off[1:])
    assert off[-1] < 2 ** 31
    return off.astype(np.int32)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

def tiny(seed: int = 1001) -> Workload:
    rng = np.random.default_rng(seed)
    C, B = 8, 64
    cols, tabs, offs, vals = [], [], [], []
    for c in range(C):
        r = np.random.default_rng([seed, c])
        cols.append(ColumnSpec("hash_mod", "sum", 1000, 16, c))
        tabs.append(TableSpec(1000, 16, seed * 1000 + c))
        lens = r.integers(0, 6, B)
        offs.append(bag_offsets(lens))
        vals.append(r.integers(0, 2 ** 40, int(lens.sum()), dtype=np.int64))
    del rng
    return Workload("tiny", B, cols, tabs, offs, vals, lr=0.01, train=True, seed=seed)


def inference(seed: int = 1002, n_cat: int = 700, n_num: int = 300, B: int = 512,
              one_hot: bool = False) -> Workload:
    """one_hot: every bag holds exactly one value (the same columns)."""
    cols, tabs, offs, vals = [], [], [], []
    coin = np.random.default_rng([seed, 99])
    for c in range(n_cat + n_num):
        r = np.random.default_rng([seed, c])
        dim = int(r.choice([8, 16, 32, 64]))
        pooling = "sum" if coin.random() < 0.5 else "mean"
        lens = r.integers(1, 21, B)
        lens[r.random(B) < 0.05] = 0
        if one_hot:
            lens = np.ones(B, np.int64)
        n = int(lens.sum())
        if c < n_cat:
            rows = int(log_uniform_int(r, 1e3, 1e6, 1)[0])
            cols.append(ColumnSpec("hash_mod", pooling, rows, dim, c))
            vals.append(r.integers(-2 ** 63, 2 ** 63 - 1, n, dtype=np.int64, endpoint=True))
        else:
            nb = int(r.integers(10, 101))
            bnd = np.unique(np.sort(r.standard_normal(nb).astype(np.float32)))
            rows = int(bnd.size) + 1
            cols.append(ColumnSpec("bucketize", pooling, rows, dim, c, boundaries=bnd))
            vals.append(r.standard_normal(n).astype(np.float32))
        tabs.append(TableSpec(rows, dim, seed * 10000 + c))
        offs.append(bag_offsets(lens))
    return Workload("inference-onehot" if one_hot else "inference", B, cols, tabs, offs, vals, train=False,
                    seed=seed)


def training(seed: int = 1003, C: int = 200, B: int = 8192, rows_lo: float = 1e5,
             rows_hi: float = 1e7, dim: int = 64, max_len: int = 50, alpha: float = 1.1,
             p_oor: float = 0.03) -> Workload:
    cols, tabs, offs, vals = [], [], [], []
    for c in range(C):
        r = np.random.default_rng([seed, c])
        rows = int(log_uniform_int(r, rows_lo, rows_hi, 1)[0])
        lens = r.integers(1, max_len + 1, B)
        n = int(lens.sum())
        ids = scatter_ranks(zipf(r, rows, alpha, n), rows)
        bad = r.random(n) < p_oor
        nb = int(bad.sum())
        low = r.random(nb) < 0.5
        off_range = r.integers(0, rows, nb)
        ids[bad] = np.where(low, -1 - off_range, rows + off_range)
        cols.append(ColumnSpec("identity", "sum", rows, dim, c))
        tabs.append(TableSpec(rows, dim, seed * 10000 + c))
        offs.append(bag_offsets(lens))
        vals.append(ids.astype(np.int64))
    return Workload("training", B, cols, tabs, offs, vals, lr=0.01, train=True, seed=seed)


def sequences(seed: int = 1004, mode: str = "mean", C: int = 20, B: int = 1024,
              rows: int = 10 ** 7, dim: int = 128, len_lo: int = 200, len_hi: int = 1000,
              pad_len: int = 1000, alpha: float = 1.05) -> Workload:
    assert mode in ("mean", "padded")
    cols, tabs, offs, vals = [], [], [], []
    for c in range(C):
        r = np.random.default_rng([seed, c])
        lens = r.integers(len_lo, len_hi + 1, B)
        n = int(lens.sum())
        ids = scatter_ranks(zipf(r, rows, alpha, n), rows)
        cols.append(ColumnSpec("identity", mode, rows, dim, c, pad_len=pad_len if mode == "padded" else 0))
        tabs.append(TableSpec(rows, dim, seed * 10000 + c))
        offs.append(bag_offsets(lens))
        vals.append(ids.astype(np.int64))
    return Workload("sequences-" + mode, B, cols, tabs, offs, vals, lr=0.01, train=True, seed=seed)


KEY_MULT = np.uint64(0x9E3779B97F4A7C15)


def dynamic_keys(seed: int, step: int, C: int = 100, B: int = 16384, alpha: float = 1.2,
                 key_bits: int = 34, max_len: int = 5):
    """One step of the dynamic-table stream: per column CSR offsets and raw
    int64 keys (Zipf ranks scattered over 2^key_bits by an odd multiplier,
    which is a bijection modulo a power of two).  Returns (offsets, keys)."""
    offs, keys = [], []
    mask = np.uint64((1 << key_bits) - 1)
    for c in range(C):
        r = np.random.default_rng([seed, step, c])
        lens = r.integers(0, max_len + 1, B)
        n = int(lens.sum())
        k = zipf(r, 1 << key_bits, alpha, n).astype(np.uint64)
        with np.errstate(over="ignore"):
            kk = ((k - np.uint64(1)) * KEY_MULT) & mask
        offs.append(bag_offsets(lens))
        keys.append(kk.astype(np.int64))
    return offs, keys


def dynamic(seed: int = 1005, C: int = 100, B: int = 16384, dim: int = 32, steps: int = 50,
            num_slots: int = 1 << 27, row_capacity: int = 1 << 25, threshold: int = 3,
            ttl: int = 10, key_bits: int = 34, alpha: float = 1.2) -> Workload:
    cols = [ColumnSpec("rows_given", "sum", row_capacity, dim, 0) for _ in range(C)]
    w = Workload("dynamic", B, cols, [TableSpec(row_capacity, dim, seed)], [], [], lr=0.01,
                 train=True, seed=seed)
    w.extra = dict(num_slots=num_slots, row_capacity=row_capacity, threshold=threshold, ttl=ttl,
                   steps=steps, key_bits=key_bits, alpha=alpha, max_probes=128,
                   init_seed=seed, init_scale=0.01)
    return w


def onehot_small(seed: int, C: int = 6, B: int | None = None, weighted: bool = False) -> Workload:
    """Columns whose bags hold one value each, with runs broken here and
    there by an empty bag or a bag of 2-3 values (sometimes cut back to one
    by max_len), over every transform and pooling and dims up to 256."""
    r = np.random.default_rng([seed, 17])
    B = int(r.integers(200, 1500)) if B is None else B
    cols, tabs, offs, vals = [], [], [], []
    for c in range(C):
        kind = str(r.choice(["identity", "hash_mod", "bucketize"]))
        dim = int(r.choice([4, 8, 16, 32, 64, 128, 200, 256]))
        pooling = str(r.choice(["sum", "mean", "sum", "mean", "padded"]))
        lens = np.ones(B, np.int64)
        breaks = r.random(B) < float(r.choice([0.0, 0.002, 0.02]))
        lens[breaks] = r.choice(np.array([0, 2, 3]), int(breaks.sum()))
        n = int(lens.sum())
        bnd = None
        if kind == "bucketize":
            bnd = np.unique(np.sort(r.standard_normal(int(r.integers(1, 60))).astype(np.float32)))
            rows = int(bnd.size) + 1
            v = r.standard_normal(n).astype(np.float32)
            v[r.random(n) < 0.02] = np.nan
        else:
            rows = int(r.integers(1, 5000))
            if kind == "identity":
                v = r.integers(-3, rows + 3, n, dtype=np.int64)
            else:
                v = r.integers(-2 ** 63, 2 ** 63 - 1, n, dtype=np.int64, endpoint=True)
        default = r.standard_normal(dim).astype(np.float32) if r.random() < 0.4 else None
        pad = int(r.integers(1, 4)) if pooling == "padded" else 0
        trunc = 1 if pooling != "padded" and r.random() < 0.3 else 0
        cols.append(ColumnSpec(kind, pooling, rows, dim, c, boundaries=bnd, default=default, pad_len=pad,
                               max_len=trunc))
        tabs.append(TableSpec(rows, dim, seed * 1000 + 500 + c))
        offs.append(bag_offsets(lens))
        vals.append(v)
    wts = [r.uniform(-1.0, 2.0, int(o[-1])).astype(np.float32) for o in offs] if weighted else None
    return Workload("onehot%d" % seed, B, cols, tabs, offs, vals, lr=0.05, seed=seed, weights=wts)


def random_small(seed: int, C: int | None = None, B: int | None = None, train: bool = True,
                 dims=(4, 8, 12, 16, 32, 64, 128), allow_padded: bool = True,
                 shared_tables: bool = True, allow_trunc: bool = True,
                 allow_weights: bool = True) -> Workload:
    """Small mixed plans for parity tests: every transform and pooling, dims
    that are not powers of two, empty bags, long bags, out-of-range and
    extreme int64 IDs, NaN/inf feature values, defaults, shared tables,
    truncated bags, value weights (used by SUM columns)."""
    r = np.random.default_rng([seed, 7])
    rt = np.random.default_rng([seed, 8])   # sequence truncation, drawn apart from the rest
    C = int(r.integers(1, 12)) if C is None else C
    B = int(r.integers(1, 70)) if B is None else B
    cols, tabs, offs, vals = [], [], [], []
    for c in range(C):
        kind = r.choice(["identity", "hash_mod", "bucketize", "identity", "hash_mod"])
        dim = int(r.choice(dims))
        pooling = str(r.choice(["sum", "mean", "padded"] if allow_padded else ["sum", "mean"]))
        lens = r.integers(0, int(r.choice([3, 8, 40, 300])), B)
        lens[r.random(B) < 0.1] = 0
        n = int(lens.sum())
        bnd = None
        if kind == "bucketize":
            nb = int(r.integers(1, 40))
            bnd = np.unique(np.sort(r.standard_normal(nb).astype(np.float32)))
            rows = int(bnd.size) + 1
            v = r.standard_normal(n).astype(np.float32)
            special = r.random(n)
            v[special < 0.02] = np.nan
            v[(special >= 0.02) & (special < 0.04)] = np.inf
            v[(special >= 0.04) & (special < 0.06)] = -np.inf
            if n and bnd.size:
                pick = r.random(n) < 0.05
                v[pick] = bnd[r.integers(0, bnd.size, int(pick.sum()))]
        else:
            rows = int(r.integers(1, 3000))
            if kind == "identity":
                v = r.integers(-5, rows + 5, n, dtype=np.int64)
                ext = r.random(n) < 0.02
                v[ext] = r.choice(np.array([-2 ** 63, 2 ** 63 - 1, -1, rows, rows - 1], np.int64),
                                  int(ext.sum()))
            else:
                v = r.integers(-2 ** 63, 2 ** 63 - 1, n, dtype=np.int64, endpoint=True)
        table = c
        if shared_tables and c > 0 and kind != "bucketize" and r.random() < 0.25:
            prev = [i for i, pc in enumerate(cols) if pc.transform != "bucketize"]
            if prev:
                j = int(r.choice(prev))
                table, rows, dim = cols[j].table, cols[j].num_rows, cols[j].dim
                if kind == "identity":
                    v = r.integers(-5, rows + 5, n, dtype=np.int64)
        default = r.standard_normal(dim).astype(np.float32) if r.random() < 0.3 else None
        pad = int(r.integers(1, 50)) if pooling == "padded" else 0
        trunc = int(rt.integers(1, 25)) if allow_trunc and pooling != "padded" and rt.random() < 0.3 else 0
        cols.append(ColumnSpec(str(kind), pooling, rows, dim, table, boundaries=bnd,
                               default=default, pad_len=pad, max_len=trunc))
        if table == c:
            tabs.append(TableSpec(rows, dim, seed * 1000 + c))
        else:
            tabs.append(None)
        offs.append(bag_offsets(lens))
        vals.append(v)
    wts = None
    if allow_weights and rt.random() < 0.3:
        wts = [rt.uniform(-1.0, 2.0, int(o[-1])).astype(np.float32) for o in offs]
    return Workload("random%d" % seed, B, cols, tabs, offs, vals, lr=0.05, train=train, seed=seed, weights=wts)


def random_many_bags(seed: int, B: int = 4096, C: int = 96, train: bool = True) -> Workload:
    """Mixed plans with many short bags (mean length about 4), large enough
    that a launch tiles its streams by bags on a 152-SM GPU: every transform
    and pooling (padded columns with short pad_len), dims 4..128, empty bags,
    rare long bags of 129..400 values, columns of one-value bags, truncated
    bags, shared tables, value weights on some plans."""
    r = np.random.default_rng([seed, 17])
    cols, tabs, offs, vals = [], [], [], []
    for c in range(C):
        kind = str(r.choice(["identity", "hash_mod", "bucketize", "hash_mod"]))
        dim = int(r.choice((4, 8, 12, 16, 32, 64, 128)))
        pooling = str(r.choice(["sum", "mean", "sum", "mean", "padded"]))
        if r.random() < 0.1:
            lens = np.ones(B, np.int64)
            lens[r.random(B) < 0.02] = 0
        else:
            lens = r.integers(0, 9, B)
            lens[r.random(B) < 0.1] = 0
            long = r.random(B) < 0.002
            lens[long] = r.integers(129, 401, int(long.sum()))
        n = int(lens.sum())
        bnd = None
        if kind == "bucketize":
            bnd = np.unique(np.sort(r.standard_normal(int(r.integers(1, 60))).astype(np.float32)))
            rows = int(bnd.size) + 1
            v = r.standard_normal(n).astype(np.float32)
            v[r.random(n) < 0.02] = np.nan
        else:
            rows = int(r.integers(1, 50000))
            if kind == "identity":
                v = r.integers(-3, rows + 3, n, dtype=np.int64)
            else:
                v = r.integers(-2 ** 63, 2 ** 63 - 1, n, dtype=np.int64, endpoint=True)
        table = c
        if c > 0 and kind != "bucketize" and r.random() < 0.15:
            prev = [i for i, pc in enumerate(cols) if pc.transform != "bucketize"]
            if prev:
                j = int(r.choice(prev))
                table, rows, dim = cols[j].table, cols[j].num_rows, cols[j].dim
                if kind == "identity":
                    v = r.integers(-3, rows + 3, n, dtype=np.int64)
        default = r.standard_normal(dim).astype(np.float32) if r.random() < 0.2 else None
        pad = int(r.integers(1, 13)) if pooling == "padded" else 0
        trunc = int(r.integers(1, 6)) if pooling != "padded" and r.random() < 0.15 else 0
        cols.append(ColumnSpec(kind, pooling, rows, dim, table, boundaries=bnd, default=default, pad_len=pad,
                               max_len=trunc))
        tabs.append(TableSpec(rows, dim, seed * 1000 + 500 + c) if table == c else None)
        offs.append(bag_offsets(lens))
        vals.append(v)
    wts = None
    if r.random() < 0.5:
        wts = [r.uniform(-1.0, 2.0, int(o[-1])).astype(np.float32) for o in offs]
    return Workload("many_bags%d" % seed, B, cols, tabs, offs, vals, lr=0.05, train=train, seed=seed,
                    weights=wts)


# --------------------------------------------------------------------------
# materialisation helpers (inputs only)
# --------------------------------------------------------------------------

def make_table(spec: TableSpec, device="cpu"):
    """fp32 [num_rows, dim] table drawn N(0, std^2) from a seeded generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(spec.seed))
    t = torch.empty((spec.num_rows, spec.dim), dtype=torch.float32, device=device)
    t.normal_(0.0, spec.std, generator=g)
    return t


def lowp_table(t, dtype: str):
    """A copy of fp32 table t stored as "bf16" / "f16" (round to nearest
    even), or "i8" with a per-row symmetric scale (max |row| / 127, 1 for an
    all-zero row; q = round(x / scale) in [-127, 127]).  Returns (table,
    row scales or None)."""
    import torch
    if dtype == "f32":
        return t, None
    if dtype == "bf16":
        return t.to(torch.bfloat16), None
    if dtype == "f16":
        return t.to(torch.float16), None
    if dtype == "i8":
        amax = t.abs().amax(dim=1)
        scale = torch.where(amax > 0, amax / 127.0, torch.ones_like(amax)).to(torch.float32).contiguous()
        q = torch.round(t / scale[:, None]).clamp_(-127, 127).to(torch.int8).contiguous()
        return q, scale
    raise ValueError("table dtype %r" % dtype)


def table_host(t):
    """Host copy of a (possibly low-precision) table as the oracle reads it:
    float32, uint16 bit patterns for bf16 / f16, int8."""
    import torch
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def make_grad(shape, seed: int, device="cpu"):
    """Upstream gradient N(0, 1) from a seeded generator."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.empty(shape, dtype=torch.float32, device=device)
    t.normal_(0.0, 1.0, generator=g)
    return t


def jagged(w: Workload):
    """Concatenate the per-column inputs into the two jagged streams the
    library takes: int64 values of the non-bucketize columns and fp32 values
    of the bucketize columns, each with one CSR offsets array over its
    (column, bag) segments in column order.  Returns numpy arrays
    (ids, id_offsets, fvals, f_offsets)."""
    id_cols = [i for i, c in enumerate(w.columns) if c.transform != "bucketize"]
    f_cols = [i for i, c in enumerate(w.columns) if c.transform == "bucketize"]

    def stream(idx, dtype):
        parts, segs, base = [], [np.zeros(1, np.int64)], 0
        for i in idx:
            o = w.offsets[i].astype(np.int64)
            parts.append(np.asarray(w.values[i], dtype))
            segs.append(base + o[1:])
            base += int(o[-1])
        vals = np.concatenate(parts) if parts else np.zeros(0, dtype)
        off = np.concatenate(segs)
        assert off[-1] < 2 ** 31
        return vals, off.astype(np.int32)

    ids, id_off = stream(id_cols, np.int64)
    fv, f_off = stream(f_cols, np.float32)
    return ids, id_off, fv, f_off


def jagged_weights(w: Workload):
    """The value weights laid out like jagged()'s two streams, or (None, None)
    for an unweighted workload."""
    if w.weights is None:
        return None, None
    out = []
    for want in (False, True):
        parts = [np.asarray(w.weights[i], np.float32) for i, c in enumerate(w.columns)
                 if (c.transform == "bucketize") == want]
        out.append(np.concatenate(parts) if parts else np.zeros(0, np.float32))
    return out[0], out[1]
