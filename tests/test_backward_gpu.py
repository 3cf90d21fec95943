"""GPU parity of the backward (radix sort, unique rows and counts, segmented
gradient reduction) and the fused sparse Adagrad update, through the C ABI."""
import numpy as np
import pytest

import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import build as slbuild
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.synth import ColumnSpec, TableSpec, Workload

import oracle
from helpers import TrainStep, assert_close, check_train_step, padded_pieces_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    slbuild.build()
    sl.lib()


def test_tiny_training_step():
    check_train_step(TrainStep(synth.tiny()))


@pytest.mark.parametrize("seed", range(30))
def test_random_small_plans(seed):
    check_train_step(TrainStep(synth.random_small(100 + seed)))


@pytest.mark.parametrize("seed,B,C", [(4, 4096, 96), (5, 3000, 128)])
def test_many_short_bags_training_step(seed, B, C):
    """A training step over a forward whose short-bag streams tile by runs of
    32-bag chunks (the records it writes feed the backward)."""
    check_train_step(TrainStep(synth.random_many_bags(seed, B, C)))


def test_well_conditioned_accumulator_start():
    """acc0 = 0.1: no first-step sign sensitivity, nothing excluded."""
    assert check_train_step(TrainStep(synth.random_small(7), acc_init=0.1)) == 0


def test_hot_row_spans_many_ctas():
    """One row receives 300k contributions (runs cut by many CTA boundaries),
    next to a uniform spread."""
    rng = np.random.default_rng(4)
    B = 3000
    lens = rng.integers(50, 150, B)
    n = int(lens.sum())
    ids = rng.integers(0, 5000, n).astype(np.int64)
    ids[rng.random(n) < 0.9] = 1234
    for dim in (8, 64, 200):
        cols = [ColumnSpec("identity", "sum", 5000, dim, 0), ColumnSpec("identity", "mean", 5000, dim, 1)]
        w = Workload("hot", B, cols, [TableSpec(5000, dim, 3), TableSpec(5000, dim, 4)],
                     [synth.bag_offsets(lens)] * 2, [ids, ids], lr=0.01)
        check_train_step(TrainStep(w))


@pytest.mark.parametrize("rows", [(1 << 24) + 3, 40_000_000, (1 << 27) - 2000])
def test_keys_of_25_to_27_bits_sort_in_three_passes(rows):
    """Row keys of 25, 26 and 27 bits (three passes of 9-bit digits, the
    last digit's top bits unused at 25 and 26), two tables, hot rows that
    span many CTAs beside rows near the top of the key range; enough
    contributions for several sort tiles."""
    rng = np.random.default_rng(rows % 1000)
    B = 2048
    lens = rng.integers(1, 30, B)
    n = int(lens.sum())
    small = 1000
    ids = rng.integers(rows - 5000, rows, n).astype(np.int64)
    ids[rng.random(n) < 0.3] = rows - 7
    ids2 = rng.integers(0, small, n).astype(np.int64)
    cols = [ColumnSpec("identity", "sum", rows, 4, 0), ColumnSpec("identity", "mean", small, 4, 1)]
    w = Workload("wide-keys", B, cols, [TableSpec(rows, 4, 11), TableSpec(small, 4, 12)],
                 [synth.bag_offsets(lens)] * 2, [ids, ids2], lr=0.01)
    check_train_step(TrainStep(w))


def test_padded_and_mean_sequences_small():
    w = synth.sequences(seed=5, mode="padded", C=3, B=40, rows=3000, dim=128, len_lo=50, len_hi=300,
                        pad_len=200)
    check_train_step(TrainStep(w))
    w = synth.sequences(seed=6, mode="mean", C=3, B=40, rows=3000, dim=128, len_lo=50, len_hi=300)
    check_train_step(TrainStep(w))


@pytest.mark.parametrize("case", ["ids-only", "fvals-only", "mixed", "static"])
def test_long_padded_pieces_training_step(case):
    """Forward + backward + Adagrad of plans whose long padded bags are
    copied in pieces: every position's gradient reaches its row once, cut
    values and zero positions none."""
    check_train_step(TrainStep(padded_pieces_case(case)))


def test_truncated_sequences():
    """Sequence truncation: long bags cut to their first 150 values (still
    pooled by the whole warp) and to their first 40 (short-bag path), sum and
    mean, forward + backward against the oracle; the cut values get no
    gradient."""
    from dataclasses import replace
    for mode, cut in (("mean", 150), ("mean", 40)):
        w = synth.sequences(seed=7, mode=mode, C=3, B=40, rows=3000, dim=128, len_lo=50, len_hi=400)
        w.columns = [replace(c, max_len=cut, pooling=p) for c, p in zip(w.columns, ("mean", "sum", "mean"))]
        ts = TrainStep(w)
        check_train_step(ts)
        ref, _, rows = oracle.forward(w.columns, w.B, w.offsets, w.values, ts.W0, want_rows=True)
        assert_close(ts.out.cpu().numpy(), ref, "pooled, max_len %d" % cut)


def _weigh(w, seed):
    rng = np.random.default_rng(seed)
    w.weights = [rng.uniform(-1.0, 2.0, int(o[-1])).astype(np.float32) for o in w.offsets]
    return w


@pytest.mark.parametrize("seed", range(12))
def test_weighted_random_small_plans(seed):
    """Value weights on every column of a random plan (both streams; SUM
    columns use them, MEAN and padded ones ignore them): pooled output and
    training step against the oracle."""
    w = _weigh(synth.random_small(300 + seed), seed)
    ts = TrainStep(w)
    check_train_step(ts)
    ref, _ = oracle.forward(w.columns, w.B, w.offsets, w.values, ts.W0, weights=w.weights)
    if ref.shape[1]:
        assert_close(ts.out.cpu().numpy(), ref, "weighted pooled output")


@pytest.mark.parametrize("dim", [8, 128, 200])
def test_weighted_long_and_short_bags(dim):
    """Weighted SUM bags of 50-400 values (short bags pooled by lane groups,
    long ones by the whole warp) beside an unweighted MEAN column of the
    same stream."""
    from dataclasses import replace
    w = synth.sequences(seed=8, mode="mean", C=3, B=40, rows=3000, dim=dim, len_lo=50, len_hi=400)
    w.columns = [replace(c, pooling=p) for c, p in zip(w.columns, ("sum", "mean", "sum"))]
    _weigh(w, dim)
    ts = TrainStep(w)
    check_train_step(ts)
    ref, _ = oracle.forward(w.columns, w.B, w.offsets, w.values, ts.W0, weights=w.weights)
    assert_close(ts.out.cpu().numpy(), ref, "weighted pooled output")


@pytest.mark.parametrize("seed", range(6))
def test_one_value_bags(seed):
    """Training step over runs of one-value bags (records written by the
    copy path), half the plans weighted."""
    check_train_step(TrainStep(synth.onehot_small(50 + seed, weighted=seed % 2 == 0)))


def test_shared_table_columns_merge():
    rng = np.random.default_rng(9)
    B = 500
    cols = [ColumnSpec("rows_given", "sum", 2000, 32, 0) for _ in range(6)]
    offs, vals = [], []
    for c in range(6):
        lens = rng.integers(0, 6, B)
        offs.append(synth.bag_offsets(lens))
        v = rng.integers(-1, 2000, int(lens.sum())).astype(np.int64)
        vals.append(v)
    w = Workload("shared", B, cols, [TableSpec(2000, 32, 1)], offs, vals, lr=0.01)
    check_train_step(TrainStep(w))


def test_deterministic_updates():
    a = TrainStep(synth.random_small(21))
    b = TrainStep(synth.random_small(21))
    for t in range(len(a.m.tables)):
        if a.m.tables[t] is None:
            continue
        assert np.array_equal(a.m.tables[t].cpu().numpy(), b.m.tables[t].cpu().numpy())
        assert np.array_equal(a.m.accs[t].cpu().numpy(), b.m.accs[t].cpu().numpy())


def test_backward_without_forward_is_rejected():
    import torch
    w = synth.tiny()
    from helpers import Materialized
    m = Materialized(w, "cuda", with_acc=True)
    plan = sl.Plan(w.columns, m.tables, m.accs, max_batch=w.B, max_ids=m.n_ids, training=True)
    g = torch.zeros((w.B, plan.out_width), device="cuda")
    with pytest.raises(sl.EmbError) as e:
        plan.backward_update(g, None, 0.01, 1e-10)
    assert e.value.status == 1


def test_empty_batch_backward():
    import torch
    w = Workload("empty", 5, [ColumnSpec("identity", "sum", 10, 8, 0)], [TableSpec(10, 8, 1)],
                 [np.zeros(6, np.int32)], [np.zeros(0, np.int64)])
    ts = TrainStep(w)
    assert ts.status == 0
    assert int(ts.dbg["row"].numel()) == 0
