"""GPU parity of the fused forward (transform, guard, gather, pool / padded
copy, default fill) against the CPU oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import build as slbuild
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.synth import ColumnSpec, TableSpec, Workload

from helpers import Materialized, assert_close, long_pooled_case, padded_pieces_case, pooled_slices, seq_slices

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    slbuild.build()
    sl.lib()


def run_forward(w, training=False):
    import torch
    m = Materialized(w, "cuda", with_acc=training)
    plan = sl.Plan(w.columns, m.tables, m.accs, max_batch=max(w.B, 1),
                   max_ids=max(m.n_ids + m.n_f, 1), training=training)
    rows_dbg = torch.full((max(m.n_ids + m.n_f, 1),), -7, dtype=torch.int64, device="cuda")
    out, seq = plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off, rows_dbg=rows_dbg, id_weights=m.idw,
                            f_weights=m.fw)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    return m, plan, out, seq, rows_dbg


def check_full(w, m, out, seq, rows_dbg):
    tabs = m.host_tables()
    ref_out, ref_seq, ref_rows = oracle.forward(w.columns, w.B, w.offsets, w.values, tabs, want_rows=True,
                                                weights=w.weights)
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


def test_tiny_workload():
    w = synth.tiny()
    m, plan, out, seq, rows = run_forward(w)
    check_full(w, m, out, seq, rows)


@pytest.mark.parametrize("seed", range(40))
def test_random_small_plans(seed):
    w = synth.random_small(seed)
    m, plan, out, seq, rows = run_forward(w)
    check_full(w, m, out, seq, rows)


@pytest.mark.parametrize("seed,B,C", [(0, 4096, 96), (1, 3000, 128), (2, 4096, 96), (3, 3000, 128)])
def test_many_short_bags(seed, B, C):
    """Launches with more tiles than a GB300 holds warps, whose short-bag
    streams are cut into runs of 32-bag chunks instead of value tiles: dealt
    column by column, widest rows first, where the tiles split the batch
    evenly (B 4096); tiles across column ends where they do not (B 3000).
    Long, empty and one-value bags, padded and truncated columns, weights,
    shared tables."""
    w = synth.random_many_bags(seed, B, C)
    m, plan, out, seq, rows = run_forward(w)
    check_full(w, m, out, seq, rows)


@pytest.mark.parametrize("seed", range(12))
def test_one_value_bags(seed):
    """Runs of one-value bags (copied without pooling, up to 256 bags per
    warp chunk) broken by empty and longer bags at random places; half the
    plans weighted."""
    w = synth.onehot_small(seed, weighted=seed % 2 == 1)
    m, plan, out, seq, rows = run_forward(w)
    check_full(w, m, out, seq, rows)


@pytest.mark.parametrize("dim", [4, 12, 20, 36, 60, 124, 128, 132, 200, 256])
def test_every_dim_class(dim):
    """Lane-group widths 1..32 and the two-float4-per-lane path (dim > 128)."""
    rng = np.random.default_rng(dim)
    B = 37
    lens = rng.integers(0, 300, B)
    lens[::7] = 0
    n = int(lens.sum())
    cols = [ColumnSpec("identity", "sum", 700, dim, 0), ColumnSpec("identity", "mean", 700, dim, 0),
            ColumnSpec("identity", "padded", 700, dim, 0, pad_len=150)]
    ids = rng.integers(-10, 710, n).astype(np.int64)
    off = synth.bag_offsets(lens)
    w = Workload("dims", B, cols, [TableSpec(700, dim, 5)], [off] * 3, [ids] * 3)
    m, plan, out, seq, rows = run_forward(w)
    check_full(w, m, out, seq, rows)


def test_long_bags_take_the_cta_path():
    """Bags of 129..5000 values (cooperative pooling) next to short ones."""
    rng = np.random.default_rng(2)
    B = 64
    lens = np.where(rng.random(B) < 0.5, rng.integers(129, 5000, B), rng.integers(0, 20, B))
    n = int(lens.sum())
    cols = [ColumnSpec("hash_mod", "mean", 5000, 64, 0), ColumnSpec("identity", "sum", 5000, 128, 1)]
    vals = [rng.integers(-2 ** 63, 2 ** 63 - 1, n, dtype=np.int64), rng.integers(-5, 5005, n).astype(np.int64)]
    off = synth.bag_offsets(lens)
    w = Workload("long", B, cols, [TableSpec(5000, 64, 1), TableSpec(5000, 128, 2)], [off, off], vals)
    m, plan, out, seq, rows = run_forward(w)
    check_full(w, m, out, seq, rows)


@pytest.mark.parametrize("case", ["ids-only", "fvals-only", "mixed", "static"])
def test_long_padded_bags_copied_in_pieces(case):
    """Padded columns longer than the whole-warp threshold are copied in
    pieces of positions, dealt as tiles of their own: pad lengths 130 (a
    piece past the end), 300, 777 and 1000 (pieces with ragged ends), bags
    from empty to past pad_len (their cut values recorded by the last
    piece), a stream of only such columns (no value tiles at all), one that
    mixes them with pooled columns, and bags so short that the launch takes
    one tile per warp."""
    w = padded_pieces_case(case)
    m, plan, out, seq, rows = run_forward(w)
    check_full(w, m, out, seq, rows)


@pytest.mark.parametrize("case", ["sum-mean", "weighted", "fvals", "truncated", "wide"])
def test_long_pooled_bags_in_training_plans(case):
    """Training plans (which record every value for the backward) with long
    pooled bags under the dynamic schedule: bags of 129 to 5000 values beside
    short and empty ones, sum and mean, value weights, bucketized values,
    truncation and rows of 200 floats.  A second launch into a fresh output
    gives the same bits."""
    import torch
    w = long_pooled_case(case)
    m, plan, out, seq, rows = run_forward(w, training=True)
    check_full(w, m, out, seq, rows)
    fresh = torch.full_like(out, float("nan"))
    plan.forward(w.B, m.ids, m.id_off, m.fv, m.f_off, out=fresh, id_weights=m.idw, f_weights=m.fw)
    torch.cuda.synchronize()
    assert plan.device_status() == 0
    assert torch.equal(fresh, out)


def test_all_bags_empty_and_defaults():
    B = 9
    dft = np.arange(8, dtype=np.float32) - 3.5
    cols = [ColumnSpec("identity", "sum", 10, 8, 0, default=dft), ColumnSpec("identity", "mean", 10, 8, 0),
            ColumnSpec("bucketize", "sum", 3, 8, 1, boundaries=np.array([0.0, 1.0], np.float32), default=dft)]
    off0 = np.zeros(B + 1, np.int32)
    off1 = synth.bag_offsets(np.full(B, 2))
    vals = [np.zeros(0, np.int64), np.full(2 * B, 99, np.int64), np.zeros(0, np.float32)]
    w = Workload("empty", B, cols, [TableSpec(10, 8, 1), TableSpec(3, 8, 2)], [off0, off1, off0], vals)
    m, plan, out, seq, rows = run_forward(w)
    o = out.cpu().numpy()
    assert np.array_equal(o[:, 0:8], np.tile(dft, (B, 1)))
    assert np.array_equal(o[:, 8:16], np.zeros((B, 8), np.float32))
    assert np.array_equal(o[:, 16:24], np.tile(dft, (B, 1)))
    check_full(w, m, out, seq, rows)


def test_zero_batch_is_a_no_op():
    import torch
    w = synth.tiny()
    m = Materialized(w, "cuda")
    plan = sl.Plan(w.columns, m.tables, None, max_batch=w.B)
    out = torch.empty((0, plan.out_width), device="cuda")
    sl.emb_forward(plan.handle, 0, m.ids, torch.zeros(1, dtype=torch.int32, device="cuda"), None, 0, None, None,
                   None, 0, out, None)
    torch.cuda.synchronize()
    assert plan.device_status() == 0


def test_bad_offsets_are_clamped_and_reported():
    """Offsets past the end of the values are clamped on the device (no
    out-of-bounds read) and latch EMB_ERR_BAD_INDEX."""
    import torch
    w = synth.tiny()
    m = Materialized(w, "cuda")
    plan = sl.Plan(w.columns, m.tables, None, max_batch=w.B)
    off = m.id_off.clone()
    off[5] = m.n_ids + 1000
    plan.forward(w.B, m.ids, off, None, None)
    torch.cuda.synchronize()
    assert plan.device_status() == 7
    assert plan.device_status() == 0


def test_training_plan_forward_matches_inference_plan():
    w = synth.random_small(3, allow_padded=True)
    _, _, out_i, seq_i, _ = run_forward(w, training=False)
    _, _, out_t, seq_t, _ = run_forward(w, training=True)
    assert np.array_equal(out_i.cpu().numpy(), out_t.cpu().numpy())
    if seq_i is not None:
        assert np.array_equal(seq_i.cpu().numpy(), seq_t.cpu().numpy())


def test_deterministic():
    w = synth.random_small(8)
    a = run_forward(w)[2].cpu().numpy()
    b = run_forward(w)[2].cpu().numpy()
    assert np.array_equal(a, b)


@pytest.mark.slow
def test_inference_workload_full_size_every_output():
    """1000-column inference workload at full size, in the launch
    configuration the forward benchmark times: every transformed row
    bit-exact and every pooled output element (512 x 30k) within 1e-5 rel /
    1e-6 abs of the oracle, which runs on chunks of columns whose tables are
    copied to the host a chunk at a time."""
    import dataclasses
    w = synth.inference()
    m, plan, out, seq, rows_dbg = run_forward(w)
    got_rows = m.rows_dbg_split(rows_dbg)
    for c in range(0, len(w.columns)):
        ref = oracle.column_rows(w.columns[c], w.values[c])
        assert np.array_equal(got_rows[c], ref), c
    psl, _ = pooled_slices(w.columns)
    o = out.cpu().numpy()
    checked = 0

    def run_chunk(chunk):
        specs = [dataclasses.replace(w.columns[c], table=j) for j, c in enumerate(chunk)]
        tabs = [m.tables[w.columns[c].table].cpu().numpy() for c in chunk]
        ref, _ = oracle.forward(specs, w.B, [w.offsets[c] for c in chunk], [w.values[c] for c in chunk], tabs)
        pos = 0
        for c in chunk:
            off, d = psl[c]
            assert_close(o[:, off:off + d], ref[:, pos:pos + d], "column %d" % c)
            pos += d
        return sum(w.columns[c].dim for c in chunk) * w.B

    chunk, held = [], 0
    for c, col in enumerate(w.columns):
        nbytes = col.num_rows * col.dim * 4
        if chunk and held + nbytes > (1 << 30):
            checked += run_chunk(chunk)
            chunk, held = [], 0
        chunk.append(c)
        held += nbytes
    if chunk:
        checked += run_chunk(chunk)
    assert checked == o.size
