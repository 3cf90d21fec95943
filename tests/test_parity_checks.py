"""The parity checkers the GPU tests use, run on the CPU with the oracle on
both sides: the restricted backward of the dynamic-table loop reproduces the
plain in-order loop bit for bit, and check_rows accepts exactly what the
fp32 summation bound allows -- a dropped contribution or a flipped weight
step where the sign of the sum is certain fails, a flip where it is not
passes and is counted.  CPU only."""
import numpy as np
import pytest

import oracle
from helpers import OraclePool, Taint, check_rows, excluded_cap
from sparse_lookup_gb300 import synth


def _dyn_inputs(t, C, B, dim):
    offs, keys = synth.dynamic_keys(1005, t, C, B, 1.2, 20, 5)
    tids = np.concatenate([np.full(k.size, c, np.int32) for c, k in enumerate(keys)])
    G = synth.make_grad((B, C * dim), 500 + t, "cpu").numpy()
    return offs, tids, np.concatenate(keys), G


def test_oracle_pool_equals_the_plain_in_order_loop():
    C, B, cap, dim, ttl = 4, 256, 1 << 12, 8, 3
    cols = [synth.ColumnSpec("rows_given", "sum", cap, dim, 0) for _ in range(C)]
    pool = OraclePool(cap, dim, 3, 1005, cols, B, 0.01, 1e-10)
    oh = oracle.Hash(cap, dim, 3, 1005, 0.01)
    for t in range(8):
        offs, tids, keys, G = _dyn_inputs(t, C, B, dim)
        o = pool.step(tids, keys, t, offs, G, ttl)
        rows, _ = oh.lookup_or_insert(tids, keys, t)
        vals, pos = [], 0
        for off in offs:
            n = int(off[-1])
            vals.append(rows[pos:pos + n])
            pos += n
        out = oracle.forward(cols, B, offs, vals, [oh.W])[0]
        oracle.backward_adagrad(cols, B, offs, vals, G, None, [oh.W], [oh.acc], 0.01, 1e-10)
        oh.evict(t, ttl)
        assert np.array_equal(o["rows"], rows)
        assert np.array_equal(o["out"], out)
        assert np.array_equal(pool.oh.W, oh.W) and np.array_equal(pool.oh.acc, oh.acc)


def test_taint_set_get_clear():
    tt = Taint(4)
    tt.set(np.array([5, 2]), np.array([[0, 1, 0, 0], [0, 0, 0, 0]], bool))
    assert tt.rows.tolist() == [5]
    tt.set(np.array([3]), np.array([[1, 0, 0, 1]], bool))
    assert tt.rows.tolist() == [3, 5]
    got = tt.get(np.array([1, 3, 5, 9]))
    assert got.tolist() == [[0, 0, 0, 0], [1, 0, 0, 1], [0, 1, 0, 0], [0, 0, 0, 0]]
    tt.clear(np.array([3]))
    assert tt.rows.tolist() == [5] and tt.count() == 1


def _one_row_case(seed, k):
    """k contributions of N(0,1) to one row of 64 elements: the oracle's fp64
    sum, magnitude sum, and an fp32 sum in contribution order."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((k, 64)).astype(np.float32)
    g64 = x.astype(np.float64).sum(axis=0)
    g32 = np.zeros(64, np.float32)
    for r in x:
        g32 = (g32 + r).astype(np.float32)
    return x, g64, np.abs(x.astype(np.float64)).sum(axis=0), g32


def _adagrad32(w, a, g, lr=0.01, eps=1e-10):
    a2 = (a + g * g).astype(np.float32)
    return (w - (lr * g) / (np.sqrt(a2) + eps)).astype(np.float32), a2


def test_check_rows_accepts_an_fp32_order_and_catches_a_dropped_contribution():
    x, g64, ab, g32 = _one_row_case(1, 40)
    w0 = np.full(64, 0.02, np.float32)
    a0 = np.zeros(64, np.float32)
    w_ref, a_ref = _adagrad32(w0, a0, g64.astype(np.float32))
    w_got, a_got = _adagrad32(w0, a0, g32)
    e, n, _, _ = check_rows(g64[None], ab[None], [40], g32[None], w0[None], a0[None], w_got[None], a_got[None],
                         w_ref[None], a_ref[None], 0.01, 1e-10)
    assert n == 64 and e <= excluded_cap(n)
    dropped = (g32 - x[7]).astype(np.float32)     # one contribution lost
    w_bad, a_bad = _adagrad32(w0, a0, dropped)
    with pytest.raises(AssertionError, match="aggregated gradient"):
        check_rows(g64[None], ab[None], [40], dropped[None], w0[None], a0[None], w_bad[None], a_bad[None],
                   w_ref[None], a_ref[None], 0.01, 1e-10)


def test_check_rows_excludes_only_sign_ambiguous_flips():
    # element 0: a sum that cancels to below the fp32 bound (its sign is not
    # determined), element 1: a clearly positive sum
    k = 2
    ab = np.array([[1.0, 1.0]])
    g64 = np.array([[1e-9, 0.5]])
    w0 = np.array([[0.02, 0.02]], np.float32)
    a0 = np.zeros((1, 2), np.float32)
    w_ref, a_ref = _adagrad32(w0, a0, g64.astype(np.float32))
    flip0 = np.array([[-1e-9, 0.5]], np.float32)
    w_got, a_got = _adagrad32(w0, a0, flip0)
    e, n, amb, out = check_rows(g64, ab, [k], flip0, w0, a0, w_got, a_got, w_ref, a_ref, 0.01, 1e-10)
    assert amb.tolist() == [[True, False]] and e == 1 and out.tolist() == [[True, False]]
    # the same flip of the weight step on element 1 is an error
    w_bad = w_ref.copy()
    w_bad[0, 1] = w_ref[0, 1] + 0.02
    with pytest.raises(AssertionError, match="weights"):
        check_rows(g64, ab, [k], g64.astype(np.float32), w0, a0, w_bad, a_ref, w_ref, a_ref, 0.01, 1e-10)
    # a tainted element (ambiguous in an earlier step) may differ too
    e, _, _, _ = check_rows(g64, ab, [k], g64.astype(np.float32), w0, a0, w_bad, a_ref, w_ref, a_ref, 0.01, 1e-10,
                         tainted=np.array([[False, True]]))
    assert e == 1
