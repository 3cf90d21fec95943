"""GPU parity of the forward over tables stored as bf16, fp16 and int8 with
a per-row scale (fp32 pooling) against the oracle, which decodes the stored
elements itself: rows bit-exact, padded copies bit-exact, pooled outputs
within tolerance."""
import numpy as np
import pytest

import oracle
import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import build as slbuild
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.synth import ColumnSpec, TableSpec, Workload

from helpers import Materialized, assert_close, seq_slices

pytestmark = pytest.mark.gpu

NAMES = {"f32": "float32", "bf16": "bfloat16", "f16": "float16", "i8": "int8"}


@pytest.fixture(scope="module", autouse=True)
def built():
    slbuild.build()
    sl.lib()


def run_lowp(w, dtypes):
    """Forward of workload w with physical table t stored as dtypes[t];
    compared with the oracle on the stored elements."""
    import torch
    m = Materialized(w, "cuda")
    tabs, scales = [], []
    for t, tab in enumerate(m.tables):
        if tab is None:
            tabs.append(None), scales.append(None)
            continue
        q, sc = synth.lowp_table(tab, dtypes[t])
        tabs.append(q), scales.append(sc)
    n = m.n_ids + m.n_f
    plan = sl.Plan(w.columns, tabs, None, max_batch=max(w.B, 1), row_scales=scales)
    rows_dbg = torch.full((max(n, 1),), -7, dtype=torch.int64, device="cuda")
    out, seq = plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off, rows_dbg=rows_dbg, id_weights=m.idw,
                            f_weights=m.fw)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    host = [np.zeros((1, 4), np.float32) if q is None else synth.table_host(q) for q in tabs]
    hs = [None if s is None else s.cpu().numpy() for s in scales]
    dts = [dtypes[t] if tabs[t] is not None else "f32" for t in range(len(tabs))]
    ref_out, ref_seq, ref_rows = oracle.forward(w.columns, w.B, w.offsets, w.values, host, want_rows=True,
                                                weights=w.weights, table_dtypes=dts, row_scales=hs)
    for c, (got, ref) in enumerate(zip(m.rows_dbg_split(rows_dbg), ref_rows)):
        assert np.array_equal(got, ref), "rows of column %d" % c
    if ref_out.shape[1]:
        assert_close(out.cpu().numpy(), ref_out, "pooled output")
    sl_, _ = seq_slices(w.columns, w.B)
    if seq is not None:
        s = seq.cpu().numpy()
        for c, sp in enumerate(sl_):
            if sp is not None:
                start, shape = sp
                got = s[start:start + int(np.prod(shape))].reshape(shape)
                assert np.array_equal(got, ref_seq[c]), "padded column %d" % c


@pytest.mark.parametrize("seed", range(16))
def test_random_plans(seed):
    """Every transform and pooling, weights, truncation, shared tables; the
    tables of one plan cycle through the four storage types."""
    w = synth.random_small(500 + seed, train=False)
    kinds = ["bf16", "f16", "i8", "f32"]
    run_lowp(w, [kinds[(seed + t) % 4] for t in range(len(w.tables))])


@pytest.mark.parametrize("dt", ["bf16", "f16", "i8"])
def test_long_one_value_and_wide_rows(dt):
    """Long bags (whole-warp pooling), runs of one-value bags (copy path) and
    dims up to 256 (two float4 per lane)."""
    rng = np.random.default_rng(7)
    B = 300
    lens = np.where(rng.random(B) < 0.3, rng.integers(129, 700, B), rng.integers(0, 12, B))
    n = int(lens.sum())
    cols = [ColumnSpec("hash_mod", "mean", 4000, 64, 0), ColumnSpec("identity", "sum", 4000, 256, 1),
            ColumnSpec("identity", "padded", 4000, 200, 2, pad_len=150)]
    vals = [rng.integers(-2 ** 63, 2 ** 63 - 1, n, dtype=np.int64), rng.integers(-5, 4005, n).astype(np.int64),
            rng.integers(-5, 4005, n).astype(np.int64)]
    off = synth.bag_offsets(lens)
    w = Workload("lp", B, cols, [TableSpec(4000, 64, 1), TableSpec(4000, 256, 2), TableSpec(4000, 200, 3)],
                 [off] * 3, vals)
    run_lowp(w, [dt, dt, dt])
    run_lowp(synth.onehot_small(9, weighted=True), [dt] * 6)


def test_training_plan_rejects_low_precision_tables():
    import torch
    w = synth.tiny()
    m = Materialized(w, "cuda", with_acc=True)
    tabs = [None if t is None else t.to(torch.bfloat16) for t in m.tables]
    with pytest.raises(sl.EmbError) as e:
        sl.Plan(w.columns, tabs, m.accs, max_batch=w.B, max_ids=m.n_ids + m.n_f + 1, training=True)
    assert e.value.status == 2
