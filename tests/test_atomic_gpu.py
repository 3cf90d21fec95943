"""GPU parity of the atomic backward (warp merge of equal rows + vector
atomics into a compact gradient, RecIS §3.2 Algorithm 1 backward) against
the oracle, through the C ABI: unique rows and counts bit-exact, gradients
within the fp32 summation bound (the order of the atomics is not fixed)."""
import numpy as np
import pytest

import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import build as slbuild
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.synth import ColumnSpec, TableSpec, Workload

from helpers import TrainStep, check_train_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    slbuild.build()
    sl.lib()


@pytest.mark.parametrize("seed", range(20))
def test_random_small_plans(seed):
    check_train_step(TrainStep(synth.random_small(100 + seed), backward="atomic"))


def test_second_step_starts_clean():
    """The compact gradient, the counts and the bitmap are left clear: a
    second and third step on the same plan match the oracle from the state
    the previous step left."""
    ts = TrainStep(synth.random_small(17), backward="atomic")
    check_train_step(ts)
    check_train_step(ts.again(91))
    check_train_step(ts.again(92))


def test_hot_row_spans_many_warps():
    """One row receives 300k contributions (merged per warp, then atomics from
    thousands of warps), next to a uniform spread."""
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
        check_train_step(TrainStep(w, backward="atomic"))


def test_padded_mean_weighted_and_one_value_bags():
    w = synth.sequences(seed=5, mode="padded", C=3, B=40, rows=3000, dim=128, len_lo=50, len_hi=300,
                        pad_len=200)
    check_train_step(TrainStep(w, backward="atomic"))
    w = synth.sequences(seed=6, mode="mean", C=3, B=40, rows=3000, dim=128, len_lo=50, len_hi=300)
    check_train_step(TrainStep(w, backward="atomic"))
    check_train_step(TrainStep(synth.onehot_small(3, weighted=True), backward="atomic"))


def test_same_rows_as_the_sorted_backward():
    """Both backward kinds touch the same rows and leave the same tables up
    to fp32 summation order."""
    a = TrainStep(synth.random_small(33), backward="sort")
    b = TrainStep(synth.random_small(33), backward="atomic")
    for k in ("table", "row", "count"):
        assert np.array_equal(a.dbg[k].cpu().numpy(), b.dbg[k].cpu().numpy()), k
    ga, gb = a.dbg["grad"].cpu().numpy(), b.dbg["grad"].cpu().numpy()
    assert np.allclose(ga, gb, rtol=1e-5, atol=1e-6)


def test_empty_batch():
    w = Workload("empty", 5, [ColumnSpec("identity", "sum", 10, 8, 0)], [TableSpec(10, 8, 1)],
                 [np.zeros(6, np.int32)], [np.zeros(0, np.int64)])
    ts = TrainStep(w, backward="atomic")
    assert ts.status == 0
    assert int(ts.dbg["row"].numel()) == 0
