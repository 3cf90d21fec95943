"""Pins of the CPU oracle against facts that do not come from the oracle
itself: published known answers, library routines the definition reduces to
(numpy.searchsorted, torch.nn.functional.embedding_bag and its autograd,
torch.optim.Adagrad), hand-worked examples, closed forms and invariants.
CPU only."""
import os

import numpy as np
import pytest

import oracle
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.synth import ColumnSpec

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MASK = (1 << 64) - 1


def _golden(name):
    out = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line)
    return out


# ---------------------------------------------------------------- transform

def test_splitmix64_published_seed0_sequence():
    """Hash transform = one SplitMix64 output with state = ID; the outputs for
    ID = i * gamma are the published seed-0 sequence."""
    for line in _golden("splitmix64_seed0.txt"):
        i, state, out = line.split()
        assert int(state, 16) == (int(i) * 0x9E3779B97F4A7C15) & MASK
        assert oracle.splitmix64(int(state, 16)) == int(out, 16)


def test_hash_mod_is_unsigned_modulo_of_the_hash():
    rng = np.random.default_rng(0)
    ids = rng.integers(-2 ** 63, 2 ** 63 - 1, 500, dtype=np.int64, endpoint=True)
    ids[:4] = [-2 ** 63, -1, 0, 2 ** 63 - 1]
    for rows in (1, 2, 3, 1000, 999_983, 2 ** 31 - 1, 2 ** 40 + 7):
        col = ColumnSpec("hash_mod", "sum", rows, 4, 0)
        got = oracle.column_rows(col, ids)
        want = [oracle.splitmix64(int(x) & MASK) % rows for x in ids]
        assert got.tolist() == want
        assert got.min() >= 0 and got.max() < rows


def test_bucketize_matches_searchsorted_right():
    """row = #{j : bnd[j] <= x}: numpy.searchsorted(side='right') for every
    ordered x; a value equal to a boundary goes to the upper bucket."""
    rng = np.random.default_rng(1)
    for nb in (1, 2, 10, 100):
        bnd = np.unique(rng.standard_normal(nb).astype(np.float32))
        x = rng.standard_normal(2000).astype(np.float32)
        x[:bnd.size] = bnd
        x[-3:] = [np.inf, -np.inf, np.float32(bnd[-1]) + np.float32(1e-6)]
        col = ColumnSpec("bucketize", "sum", bnd.size + 1, 4, 0, boundaries=bnd)
        got = oracle.column_rows(col, x)
        assert got.tolist() == np.searchsorted(bnd, x, side="right").tolist()
        assert got[x == np.inf].tolist() == [bnd.size]
        assert got[x == -np.inf].tolist() == [0]


def test_bucketize_nan_goes_to_bucket_zero():
    bnd = np.array([-1.0, 0.0, 2.0], np.float32)
    col = ColumnSpec("bucketize", "sum", 4, 4, 0, boundaries=bnd)
    assert oracle.column_rows(col, np.array([np.nan, -np.nan], np.float32)).tolist() == [0, 0]


def test_identity_safety_drops_out_of_range():
    col = ColumnSpec("identity", "sum", 10, 4, 0)
    ids = np.array([0, 9, 10, -1, -2 ** 63, 2 ** 63 - 1, 5], np.int64)
    assert oracle.column_rows(col, ids).tolist() == [0, 9, -1, -1, -1, -1, 5]
    col = ColumnSpec("rows_given", "sum", 10, 4, 0)
    assert oracle.column_rows(col, np.array([-1, 3, 11], np.int64)).tolist() == [-1, 3, -1]


# ------------------------------------------------------------------ forward

def _hand_table():
    return np.array([[1, 2], [3, 4], [10, 20], [-5, 0.5]], np.float32)


def test_forward_hand_worked_example():
    """Three bags typed by hand: [0, 2], [], [1, 1, 7(out of range), -1]."""
    E = _hand_table()
    off = np.array([0, 2, 2, 6], np.int32)
    ids = np.array([0, 2, 1, 1, 7, -1], np.int64)
    dft = np.array([0.25, -0.75], np.float32)
    cols = [ColumnSpec("identity", "sum", 4, 2, 0),
            ColumnSpec("identity", "mean", 4, 2, 0, default=dft)]
    out, _, rows = oracle.forward(cols, 3, [off, off], [ids, ids], [E], want_rows=True)
    assert out.tolist() == [[11, 22, 5.5, 11],
                            [0, 0, 0.25, -0.75],
                            [6, 8, 3, 4]]
    assert rows[0].tolist() == [0, 2, 1, 1, -1, -1]


def test_forward_padded_hand_worked_example():
    E = _hand_table()
    off = np.array([0, 3, 3, 5], np.int32)
    ids = np.array([3, 9, 1, 2, 0], np.int64)
    cols = [ColumnSpec("identity", "padded", 4, 2, 0, pad_len=2)]
    out, seq = oracle.forward(cols, 3, [off], [ids], [E])
    assert out.shape == (3, 0)
    assert seq[0].tolist() == [[[-5, 0.5], [0, 0]],
                               [[0, 0], [0, 0]],
                               [[10, 20], [1, 2]]]


def _tables(w):
    return [None if t is None else synth.make_table(t).numpy() for t in w.tables]


def test_forward_matches_embedding_bag_in_fp64():
    """On the valid IDs, SUM/MEAN pooling is torch.nn.functional.embedding_bag
    (library routine) over the same CSR offsets; empty bags give the default."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for seed in range(6):
        w = synth.random_small(seed, allow_padded=False, allow_trunc=False, allow_weights=False)
        tabs = _tables(w)
        out, _, rows = oracle.forward(w.columns, w.B, w.offsets, w.values, tabs, want_rows=True)
        col0 = 0
        for ci, c in enumerate(w.columns):
            r = rows[ci]
            off = w.offsets[ci].astype(np.int64)
            keep = r >= 0
            bag = np.repeat(np.arange(w.B), np.diff(off))[keep]
            new_off = np.searchsorted(bag, np.arange(w.B + 1), side="left")
            ref = F.embedding_bag(torch.from_numpy(r[keep]), torch.from_numpy(tabs[c.table]).double(),
                                  torch.from_numpy(new_off[:-1]), mode=c.pooling).numpy()
            nv = np.diff(new_off)
            dft = np.zeros(c.dim) if c.default is None else c.default.astype(np.float64)
            ref[nv == 0] = dft
            got = out[:, col0:col0 + c.dim]
            np.testing.assert_allclose(got, ref, rtol=1e-6, atol=1e-7)
            col0 += c.dim


def test_forward_invariants():
    rng = np.random.default_rng(3)
    E = rng.standard_normal((50, 8)).astype(np.float32)
    F_ = rng.standard_normal((50, 8)).astype(np.float32)
    B = 40
    lens = rng.integers(0, 9, B)
    off = synth.bag_offsets(lens)
    ids = rng.integers(-3, 53, int(lens.sum())).astype(np.int64)
    s = [ColumnSpec("identity", "sum", 50, 8, 0)]
    m = [ColumnSpec("identity", "mean", 50, 8, 0)]
    # single valid ID, mean pooling -> exactly its row
    one = np.array([7], np.int64)
    y, _ = oracle.forward(m, 1, [np.array([0, 1], np.int32)], [one], [E])
    assert np.array_equal(y[0], E[7])
    # all IDs dropped -> default vector (zeros when none)
    bad = np.array([-1, 50, 99], np.int64)
    y, _ = oracle.forward(s, 1, [np.array([0, 3], np.int32)], [bad], [E])
    assert np.array_equal(y[0], np.zeros(8, np.float32))
    # linearity: pool(aE + bF) = a pool(E) + b pool(F)
    a, b = 0.75, -2.5
    yE, _ = oracle.forward(s, B, [off], [ids], [E])
    yF, _ = oracle.forward(s, B, [off], [ids], [F_])
    yL, _ = oracle.forward(s, B, [off], [ids], [(a * E.astype(np.float64) + b * F_).astype(np.float32)])
    np.testing.assert_allclose(yL, a * yE.astype(np.float64) + b * yF, rtol=1e-5, atol=1e-5)
    # order of IDs inside a bag does not matter (up to rounding)
    perm = ids.copy()
    for i in range(B):
        rng.shuffle(perm[off[i]:off[i + 1]])
    yP, _ = oracle.forward(s, B, [off], [perm], [E])
    np.testing.assert_allclose(yP, yE, rtol=1e-6, atol=1e-6)


def test_forward_rejects_bad_offsets():
    E = _hand_table()
    col = [ColumnSpec("identity", "sum", 4, 2, 0)]
    with pytest.raises(ValueError):
        oracle.forward(col, 2, [np.array([1, 2, 3], np.int32)], [np.zeros(3, np.int64)], [E])
    with pytest.raises(ValueError):
        oracle.forward(col, 2, [np.array([0, 2, 1], np.int32)], [np.zeros(2, np.int64)], [E])


# ----------------------------------------------------------------- backward

def test_local_reduce_matches_recis_figure3():
    """Unique rows + counts of a batch reproduce Figure 3's local reduce-ID:
    same set of reduced IDs; counts rebuild the queries' multiplicity."""
    for line in _golden("recis_fig3_local_reduce.txt"):
        dev, q, red = [p.strip() for p in line.split("|")]
        q = np.array([int(x) for x in q.split()], np.int64)
        red = [int(x) for x in red.split()]
        col = [ColumnSpec("identity", "sum", 10000, 2, 0)]
        off = np.array([0, q.size], np.int32)
        W = [np.zeros((10000, 2), np.float32)]
        A = [np.zeros((10000, 2), np.float32)]
        G = np.ones((1, 2), np.float32)
        res = oracle.backward_adagrad(col, 1, [off], [q], G, None, W, A, 0.01, 1e-10)
        assert set(res["row"].tolist()) == set(red)
        assert res["row"].tolist() == sorted(red)
        inv = {r: n for r, n in zip(res["row"].tolist(), res["count"].tolist())}
        rebuilt = sorted(sum([[r] * n for r, n in inv.items()], []))
        assert rebuilt == sorted(q.tolist())


def test_backward_matches_embedding_bag_autograd():
    """The aggregated gradient of each unique row is the dense gradient that
    autograd of torch.nn.functional.embedding_bag (fp64) gives that row; rows
    the batch does not touch receive nothing."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for seed in range(5):
        w = synth.random_small(seed + 10, allow_padded=False, shared_tables=False, allow_trunc=False,
                               allow_weights=False)
        tabs = _tables(w)
        width = sum(c.dim for c in w.columns)
        G = synth.make_grad((w.B, width), seed).numpy()
        W = [t.copy() for t in tabs]
        A = [np.zeros_like(t) for t in tabs]
        res = oracle.backward_adagrad(w.columns, w.B, w.offsets, w.values, G, None, W, A, 0.05, 1e-10)
        col0 = 0
        for ci, c in enumerate(w.columns):
            r = oracle.column_rows(c, w.values[ci])
            off = w.offsets[ci].astype(np.int64)
            keep = r >= 0
            bag = np.repeat(np.arange(w.B), np.diff(off))[keep]
            new_off = np.searchsorted(bag, np.arange(w.B + 1), side="left")
            E = torch.from_numpy(tabs[c.table]).double().requires_grad_(True)
            y = F.embedding_bag(torch.from_numpy(r[keep]), E, torch.from_numpy(new_off[:-1]), mode=c.pooling)
            y.backward(torch.from_numpy(G[:, col0:col0 + c.dim]).double())
            dense = E.grad.numpy()
            sel = res["table"] == c.table
            touched = res["row"][sel]
            got = np.array([g for g, s in zip(res["grad"], sel) if s]).reshape(-1, c.dim)
            np.testing.assert_allclose(got, dense[touched], rtol=1e-6, atol=1e-6)
            untouched = np.setdiff1d(np.arange(c.num_rows), touched)
            assert np.all(dense[untouched] == 0)
            assert np.array_equal(np.sort(touched), np.unique(r[keep]))
            assert res["count"][sel].sum() == keep.sum()
            col0 += c.dim


def test_backward_gradient_sum_invariant():
    """Sum over unique rows of the aggregated gradient = sum over valid
    contributions of scale * G[bag] (per column and element, fp64)."""
    w = synth.random_small(77, C=4, B=50, allow_padded=False, shared_tables=False, allow_trunc=False,
                           allow_weights=False)
    tabs = _tables(w)
    width = sum(c.dim for c in w.columns)
    G = synth.make_grad((w.B, width), 5).numpy().astype(np.float64)
    W = [t.copy() for t in tabs]
    A = [np.zeros_like(t) for t in tabs]
    res = oracle.backward_adagrad(w.columns, w.B, w.offsets, w.values, G.astype(np.float32), None,
                                  W, A, 0.01, 1e-10)
    col0 = 0
    for ci, c in enumerate(w.columns):
        r = oracle.column_rows(c, w.values[ci])
        off = w.offsets[ci]
        want = np.zeros(c.dim)
        for b in range(w.B):
            rr = r[off[b]:off[b + 1]]
            nv = int((rr >= 0).sum())
            if nv:
                scale = 1.0 / nv if c.pooling == "mean" else 1.0
                want += nv * scale * G[b, col0:col0 + c.dim].astype(np.float32).astype(np.float64)
        sel = res["table"] == c.table
        got = np.sum([g.astype(np.float64) for g, s in zip(res["grad"], sel) if s], axis=0) if sel.any() else 0
        np.testing.assert_allclose(got, want, rtol=1e-5, atol=1e-4)
        col0 += c.dim


def test_adagrad_first_step_closed_form_and_torch():
    """From acc = 0 one step gives acc = g^2 and W - lr*g/(|g| + eps); the
    update is torch.optim.Adagrad's (library routine) with the aggregated
    gradient as the dense gradient."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    rows, dim, B = 30, 8, 25
    lens = rng.integers(0, 6, B)
    off = synth.bag_offsets(lens)
    ids = rng.integers(0, rows, int(lens.sum())).astype(np.int64)
    col = [ColumnSpec("identity", "sum", rows, dim, 0)]
    W0 = rng.standard_normal((rows, dim)).astype(np.float32)
    G = rng.standard_normal((B, dim)).astype(np.float32)
    lr, eps = 0.01, 1e-10
    W = [W0.copy()]
    A = [np.zeros_like(W0)]
    res = oracle.backward_adagrad(col, B, [off], [ids], G, None, W, A, lr, eps)
    g = np.zeros_like(W0)
    for r, gr in zip(res["row"], res["grad"]):
        g[r] = gr
    # closed form
    np.testing.assert_array_equal(A[0], g * g)
    touched = np.zeros(rows, bool)
    touched[res["row"]] = True
    cf = W0.astype(np.float64) - lr * g / (np.abs(g.astype(np.float64)) + eps)
    np.testing.assert_allclose(W[0][touched], cf[touched], rtol=1e-6, atol=1e-7)
    assert np.array_equal(W[0][~touched], W0[~touched])
    # torch.optim.Adagrad, two steps
    p = torch.nn.Parameter(torch.from_numpy(W0.copy()))
    opt = torch.optim.Adagrad([p], lr=lr, eps=eps, initial_accumulator_value=0.0)
    p.grad = torch.from_numpy(g.copy())
    opt.step()
    np.testing.assert_allclose(p.detach().numpy(), W[0], rtol=1e-6, atol=1e-7)
    res2 = oracle.backward_adagrad(col, B, [off], [ids], G, None, W, A, lr, eps)
    g2 = np.zeros_like(W0)
    for r, gr in zip(res2["row"], res2["grad"]):
        g2[r] = gr
    p.grad = torch.from_numpy(g2.copy())
    opt.step()
    np.testing.assert_allclose(p.detach().numpy(), W[0], rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(opt.state[p]["sum"].numpy(), A[0], rtol=1e-6, atol=1e-7)


def test_backward_mean_and_padded_hand_example():
    """Bag [1, 1, 3, 99] with MEAN (3 valid IDs): row 1 gets 2/3 G, row 3 gets
    1/3 G.  PADDED column, pad 2, bag [2, 0, 1]: position 2 is cut, row 2 gets
    Gseq[0,0], row 0 gets Gseq[0,1]."""
    E = np.zeros((4, 2), np.float32)
    off = np.array([0, 4], np.int32)
    ids = np.array([1, 1, 3, 99], np.int64)
    G = np.array([[3.0, -6.0]], np.float32)
    res = oracle.backward_adagrad([ColumnSpec("identity", "mean", 4, 2, 0)], 1, [off], [ids], G, None,
                                  [E.copy()], [E.copy()], 0.1, 1e-10)
    assert res["row"].tolist() == [1, 3] and res["count"].tolist() == [2, 1]
    np.testing.assert_allclose(res["grad"][0], [2.0, -4.0], rtol=1e-7)
    np.testing.assert_allclose(res["grad"][1], [1.0, -2.0], rtol=1e-7)
    off = np.array([0, 3], np.int32)
    ids = np.array([2, 0, 1], np.int64)
    Gs = np.array([[[1.0, 2.0], [3.0, 4.0]]], np.float32)
    res = oracle.backward_adagrad([ColumnSpec("identity", "padded", 4, 2, 0, pad_len=2)], 1, [off], [ids],
                                  None, [Gs], [E.copy()], [E.copy()], 0.1, 1e-10)
    assert res["row"].tolist() == [0, 2] and res["count"].tolist() == [1, 1]
    assert res["grad"][0].tolist() == [3.0, 4.0] and res["grad"][1].tolist() == [1.0, 2.0]


def test_backward_shared_table_merges_columns():
    """Two columns reading one physical table: a row touched by both is one
    unique row whose gradient sums both columns' contributions."""
    off = np.array([0, 1], np.int32)
    cols = [ColumnSpec("identity", "sum", 5, 2, 0), ColumnSpec("identity", "sum", 5, 2, 0)]
    G = np.array([[1.0, 2.0, 10.0, 20.0]], np.float32)
    E = np.zeros((5, 2), np.float32)
    res = oracle.backward_adagrad(cols, 1, [off, off], [np.array([4]), np.array([4])], G, None,
                                  [E.copy()], [E.copy()], 0.1, 1e-10)
    assert res["row"].tolist() == [4] and res["count"].tolist() == [2]
    assert res["grad"][0].tolist() == [11.0, 22.0]


# --------------------------------------------------------------- hash table

def test_hash_hand_traced_scenario():
    """Threshold 3, ttl 2, capacity 3 rows.  Traced by hand:
    step 0: A A B B B C -> B reaches 3 (row 0, same call); A, C count.
    step 1: A C D      -> A reaches 3 (row 1); C=2, D=1.
    step 4: evict(now=4, ttl=2): B (seen 0), A, C, D (seen 1) idle > 2 -> all go;
            rows 0, 1 return to the free list.
    step 5: E E E F F F -> E, F admitted in key order, lowest free rows 0, 1.
    step 6: G G G H H H -> G row 2 (bump), H finds no row: TABLE_FULL, -1.
    step 7: H          -> still no row (count 4).
    evict(now=8, ttl=2): E, F (seen 5) go, rows 1 and 0 are free again.
    step 8: H          -> H (count 5, still above the threshold) takes row 0."""
    h = oracle.Hash(3, 2, 3, 42, 0.5)
    A, B_, C, D, E, F_, G_, H = 100, 50, 7, 8, 30, 20, 9, 10
    rows, st = h.lookup_or_insert([0] * 6, [A, A, B_, B_, B_, C], 0)
    assert st == 0 and rows.tolist() == [-1, -1, 0, 0, 0, -1]
    assert h.last_admitted().tolist() == [0]
    rows, st = h.lookup_or_insert([0] * 3, [A, C, D], 1)
    assert rows.tolist() == [1, -1, -1]
    assert h.last_admitted().tolist() == [1]
    ex = h.export()
    assert dict(zip(ex["key"].tolist(), ex["count"].tolist())) == {A: 3, B_: 3, C: 2, D: 1}
    assert h.evict(3, 2) == 1            # only B (idle 3 > 2) at now = 3
    assert h.evict(4, 2) == 3
    assert h.size() == 0 and h.free_count() == 2
    rows, st = h.lookup_or_insert([0] * 6, [E, E, E, F_, F_, F_], 5)
    assert st == 0 and rows.tolist() == [1, 1, 1, 0, 0, 0]   # F < E: F takes row 0
    assert h.last_admitted().tolist() == [0, 1]               # admission order: F, then E
    rows, st = h.lookup_or_insert([0] * 6, [G_, G_, G_, H, H, H], 6)
    assert st == oracle.ERR_FULL and rows.tolist() == [2, 2, 2, -1, -1, -1]
    assert h.last_admitted().tolist() == [2]
    # H stays counting and is admitted as soon as a row is free again
    rows, st = h.lookup_or_insert([0], [H], 7)
    assert st == oracle.ERR_FULL and rows.tolist() == [-1]
    assert h.last_admitted().tolist() == []
    assert h.evict(8, 2) == 2
    rows, st = h.lookup_or_insert([0], [H], 8)
    assert st == 0 and rows.tolist() == [0]
    assert h.last_admitted().tolist() == [0]


def test_hash_init_values_are_exact_and_in_range():
    vals = np.array([oracle.hash_init_value(5, 3, 123456789, d, 1.0) for d in range(64)])
    assert np.all(vals >= -1.0) and np.all(vals < 1.0)
    assert np.all(vals * 2 ** 23 == np.round(vals * 2 ** 23))   # 24-bit grid
    v2 = np.array([oracle.hash_init_value(5, 3, 123456789, d, 0.01) for d in range(64)])
    np.testing.assert_array_equal(v2, (vals.astype(np.float32) * np.float32(0.01)).astype(np.float32))
    h = oracle.splitmix64(123456789 ^ (3 << 48) ^ 5 ^ 0)
    assert vals[0] == ((h >> 40) - 2 ** 23) / 2 ** 23


def _dict_model(stream, threshold, ttl, cap):
    """Independent brute-force model of the table rules, with Python dicts
    and a sorted list of free rows (used only on tiny streams)."""
    ent, free, bump, outs = {}, [], 0, []
    for step, tids, keys in stream:
        for k in zip(tids, keys):
            e = ent.setdefault(k, dict(count=0, row=-1, seen=step))
            e["seen"] = step
            if e["row"] < 0:
                e["count"] += 1
        new = sorted(k for k, e in ent.items() if e["row"] < 0 and e["count"] >= threshold)
        free.sort()
        for k in new:
            if free:
                ent[k]["row"] = free.pop(0)
            elif bump < cap:
                ent[k]["row"] = bump
                bump += 1
        outs.append([ent[k]["row"] for k in zip(tids, keys)])
        for k in [k for k, e in ent.items() if step - e["seen"] > ttl]:
            if ent[k]["row"] >= 0:
                free.append(ent[k]["row"])
            del ent[k]
    return outs, ent


def test_hash_matches_dict_model_and_invariants():
    rng = np.random.default_rng(9)
    thr, ttl, cap = 3, 4, 40
    stream = []
    for step in range(40):
        n = int(rng.integers(0, 30))
        keys = synth.zipf(rng, 60, 1.1, n)
        tids = rng.integers(0, 3, n)
        stream.append((step, tids.tolist(), keys.tolist()))
    want, ent = _dict_model(stream, thr, ttl, cap)
    h = oracle.Hash(cap, 4, thr, 1, 0.1)
    for (step, tids, keys), w in zip(stream, want):
        rows, _ = h.lookup_or_insert(tids, keys, step)
        assert rows.tolist() == w
        h.evict(step, ttl)
        ex = h.export()
        adm = ex["row"] >= 0
        # injective key -> row, rows in range
        assert len(set(ex["row"][adm].tolist())) == int(adm.sum())
        assert np.all(ex["row"][adm] < cap)
        # threshold rule: admitted entries reached it; counting ones did not
        # (unless the pool is exhausted)
        assert np.all(ex["count"][adm] >= thr)
        if h.bump() < cap or h.free_count() > 0:
            assert np.all(ex["count"][~adm] < thr)
        # after the sweep no entry is idle longer than ttl
        assert np.all(step - ex["last_seen"].astype(np.int64) <= ttl)
        # free rows and used rows partition the rows handed out so far
        assert int(adm.sum()) + h.free_count() == h.bump()
    ex = h.export()
    assert sorted(zip(ex["tid"].tolist(), ex["key"].tolist())) == sorted(ent.keys())


def _seq_grads(w, seed):
    """Upstream gradients of the padded columns ([B, pad_len, dim] each)."""
    r = np.random.default_rng(seed)
    return [r.standard_normal((w.B, c.pad_len, c.dim)).astype(np.float32) if c.pooling == "padded" else None
            for c in w.columns]


def test_backward_rows_equals_the_full_backward_on_its_rows():
    """backward_rows over every touched row (and over a subset) gives the
    counts, fp32 aggregated gradients and updated W/acc of backward_adagrad
    bit for bit: the same contributions summed in the same order."""
    for seed in range(8):
        w = synth.random_small(seed)
        tabs = _tables(w)
        width = sum(c.dim for c in w.columns if c.pooling != "padded")
        G = synth.make_grad((w.B, max(width, 1)), 9 + seed).numpy()[:, :width]
        Gs = _seq_grads(w, seed)
        W = [None if t is None else t.copy() for t in tabs]
        A = [None if t is None else np.full_like(t, 0.25) for t in tabs]
        Wl = [x if x is not None else np.zeros((1, 1), np.float32) for x in W]
        Al = [x if x is not None else np.zeros((1, 1), np.float32) for x in A]
        W0 = [x.copy() for x in Wl]
        A0 = [x.copy() for x in Al]
        ref = oracle.backward_adagrad(w.columns, w.B, w.offsets, w.values, G, Gs, Wl, Al, w.lr, w.eps,
                                      weights=w.weights)
        n = len(ref["row"])
        if n == 0:
            continue
        dims = {c.table: c.dim for c in w.columns}
        ld = max(dims.values())
        for pick in (np.arange(n), np.arange(n)[::3]):
            targets = [(int(ref["table"][i]), int(ref["row"][i])) for i in pick]
            Wr = np.zeros((len(targets), ld), np.float32)
            Ar = np.zeros((len(targets), ld), np.float32)
            for k, (t, r) in enumerate(targets):
                Wr[k, :dims[t]] = W0[t][r]
                Ar[k, :dims[t]] = A0[t][r]
            got = oracle.backward_rows(w.columns, w.B, w.offsets, w.values, G, Gs, targets, Wr, Ar, w.lr, w.eps,
                                       weights=w.weights)
            assert np.array_equal(got["count"], ref["count"][pick]), seed
            for k, (i, (t, r)) in enumerate(zip(pick, targets)):
                d = dims[t]
                assert np.array_equal(got["grad"][k, :d], ref["grad"][i]), (seed, t, r)
                assert np.array_equal(Wr[k, :d], Wl[t][r]), (seed, t, r)
                assert np.array_equal(Ar[k, :d], Al[t][r]), (seed, t, r)
                assert np.all(got["absgrad"][k, :d] >= np.abs(got["grad"][k, :d]) * (1 - 1e-6)), (seed, t, r)


def test_backward_rows_magnitudes_are_the_sum_of_abs_terms():
    """absgrad of a row = the aggregated gradient of |G| (checked on a hand
    example: MEAN bag [1, 1, 3], G = [3, -6] -> row 1 gets 2/3 |G|)."""
    off = np.array([0, 3], np.int32)
    ids = np.array([1, 1, 3], np.int64)
    G = np.array([[3.0, -6.0]], np.float32)
    Wr = np.zeros((2, 2), np.float32)
    Ar = np.zeros((2, 2), np.float32)
    got = oracle.backward_rows([ColumnSpec("identity", "mean", 4, 2, 0)], 1, [off], [ids], G, None,
                               [(0, 1), (0, 3)], Wr, Ar, 0.1, 1e-10)
    assert got["count"].tolist() == [2, 1]
    np.testing.assert_allclose(got["grad"], [[2.0, -4.0], [1.0, -2.0]], rtol=1e-7)
    np.testing.assert_allclose(got["absgrad"], [[2.0, 4.0], [1.0, 2.0]], rtol=1e-12)


def test_unique_counts_equals_the_backward_listing():
    """numpy.unique over the valid rows (library routine) lists the same
    (table, row, count) as the C oracle's sorted run listing."""
    for seed in range(10):
        w = synth.random_small(100 + seed)
        tabs = _tables(w)
        width = sum(c.dim for c in w.columns if c.pooling != "padded")
        G = np.zeros((w.B, max(width, 1)), np.float32)
        Gs = _seq_grads(w, seed)
        Wl = [x.copy() if x is not None else np.zeros((1, 1), np.float32) for x in tabs]
        Al = [np.zeros_like(x) for x in Wl]
        ref = oracle.backward_adagrad(w.columns, w.B, w.offsets, w.values, G, Gs, Wl, Al, w.lr, w.eps)
        got = oracle.unique_counts(w.columns, w.B, w.offsets, w.values)
        assert np.array_equal(got["table"], ref["table"].astype(np.int64)), seed
        assert np.array_equal(got["row"], ref["row"]), seed
        assert np.array_equal(got["count"], ref["count"]), seed


def test_truncation_hand_example():
    """SUM with max_len 2 on bag [1, 2, 3, 99] pools rows 1 and 2; MEAN with
    max_len 3 on [1, 99, 3, 2] averages rows 1 and 3 (99 is dropped inside the
    kept prefix, 2 lies past it); only the kept values receive gradient."""
    E = np.arange(40, dtype=np.float32).reshape(10, 4)
    off = np.array([0, 4], np.int32)
    cs = ColumnSpec("identity", "sum", 10, 4, 0, max_len=2)
    out, _ = oracle.forward([cs], 1, [off], [np.array([1, 2, 3, 99], np.int64)], [E])
    assert np.array_equal(out[0], E[1] + E[2])
    cm = ColumnSpec("identity", "mean", 10, 4, 0, max_len=3)
    out, _ = oracle.forward([cm], 1, [off], [np.array([1, 99, 3, 2], np.int64)], [E])
    assert np.array_equal(out[0], (E[1] + E[3]) / 2)
    G = np.ones((1, 4), np.float32)
    res = oracle.backward_adagrad([cm], 1, [off], [np.array([1, 99, 3, 2], np.int64)], G, None,
                                  [E.copy()], [np.zeros_like(E)], 0.1, 1e-10)
    assert res["row"].tolist() == [1, 3] and res["count"].tolist() == [1, 1]
    np.testing.assert_allclose(res["grad"][0], [0.5] * 4)


def test_truncation_equals_cut_inputs():
    """A truncated column gives the forward, backward and unique counts of the
    same column fed only each bag's first max_len values (the plain
    definition, by numpy slicing)."""
    from dataclasses import replace
    for seed in range(12):
        w = synth.random_small(300 + seed, allow_padded=False)
        if not any(c.max_len for c in w.columns):
            continue
        cut_cols, cut_offs, cut_vals, cut_wts = [], [], [], []
        wts = w.weights or [None] * len(w.columns)
        for c, o, v, wt in zip(w.columns, w.offsets, w.values, wts):
            if c.max_len:
                lens = np.minimum(np.diff(o), c.max_len)
                keep = np.concatenate([np.arange(o[b], o[b] + lens[b]) for b in range(w.B)] or
                                      [np.zeros(0, np.int64)]).astype(np.int64)
                cut_offs.append(synth.bag_offsets(lens))
                cut_vals.append(v[keep])
                cut_wts.append(None if wt is None else wt[keep])
                cut_cols.append(replace(c, max_len=0))
            else:
                cut_offs.append(o)
                cut_vals.append(v)
                cut_wts.append(wt)
                cut_cols.append(c)
        cw = None if w.weights is None else cut_wts
        tabs = _tables(w)
        a, _ = oracle.forward(w.columns, w.B, w.offsets, w.values, tabs, weights=w.weights)
        b, _ = oracle.forward(cut_cols, w.B, cut_offs, cut_vals, tabs, weights=cw)
        assert np.array_equal(a, b), seed
        ua = oracle.unique_counts(w.columns, w.B, w.offsets, w.values)
        ub = oracle.unique_counts(cut_cols, w.B, cut_offs, cut_vals)
        for k in ("table", "row", "count"):
            assert np.array_equal(ua[k], ub[k]), (seed, k)
        width = sum(c.dim for c in w.columns)
        G = synth.make_grad((w.B, max(width, 1)), seed).numpy()[:, :width]
        dummy = np.zeros((1, 1), np.float32)   # placeholders keep the list indexed by table
        Wa = [x.copy() if x is not None else dummy.copy() for x in tabs]
        Wb = [x.copy() if x is not None else dummy.copy() for x in tabs]
        Aa = [np.zeros_like(x) for x in Wa]
        Ab = [np.zeros_like(x) for x in Wb]
        oracle.backward_adagrad(w.columns, w.B, w.offsets, w.values, G, None, Wa, Aa, w.lr, w.eps,
                                weights=w.weights)
        oracle.backward_adagrad(cut_cols, w.B, cut_offs, cut_vals, G, None, Wb, Ab, w.lr, w.eps, weights=cw)
        for x, y in zip(Wa + Aa, Wb + Ab):
            assert np.array_equal(x, y), seed


def test_weighted_bag_hand_example():
    """SUM bag [1, 2, 1] with weights [0.5, 2, -1] pools -0.5 E1 + 2 E2; the
    backward passes -0.5 G to row 1 and 2 G to row 2; MEAN and PADDED columns
    ignore weights."""
    E = np.arange(40, dtype=np.float32).reshape(10, 4)
    off = np.array([0, 3], np.int32)
    ids = np.array([1, 2, 1], np.int64)
    wts = [np.array([0.5, 2.0, -1.0], np.float32)]
    cs = ColumnSpec("identity", "sum", 10, 4, 0)
    out, _ = oracle.forward([cs], 1, [off], [ids], [E], weights=wts)
    np.testing.assert_allclose(out[0], -0.5 * E[1] + 2 * E[2], rtol=1e-7)
    G = np.array([[1.0, -2.0, 3.0, 4.0]], np.float32)
    res = oracle.backward_adagrad([cs], 1, [off], [ids], G, None, [E.copy()], [np.zeros_like(E)], 0.1, 1e-10,
                                  weights=wts)
    assert res["row"].tolist() == [1, 2] and res["count"].tolist() == [2, 1]
    np.testing.assert_allclose(res["grad"][0], -0.5 * G[0], rtol=1e-7)
    np.testing.assert_allclose(res["grad"][1], 2.0 * G[0], rtol=1e-7)
    cm = ColumnSpec("identity", "mean", 10, 4, 0)
    out_w, _ = oracle.forward([cm], 1, [off], [ids], [E], weights=wts)
    out_u, _ = oracle.forward([cm], 1, [off], [ids], [E])
    assert np.array_equal(out_w, out_u)


def test_weighted_bags_match_embedding_bag_per_sample_weights():
    """Weighted SUM pooling and its backward are torch embedding_bag with
    per_sample_weights (library routine) in fp64, forward and autograd."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(3)
    for trial in range(4):
        rows, dim, B = int(rng.integers(5, 300)), int(rng.choice([4, 8, 16])), int(rng.integers(1, 40))
        lens = rng.integers(0, 12, B)
        off = synth.bag_offsets(lens)
        n = int(lens.sum())
        ids = rng.integers(-2, rows + 2, n).astype(np.int64)   # some dropped
        wts = rng.uniform(-1, 2, n).astype(np.float32)
        E = rng.standard_normal((rows, dim)).astype(np.float32)
        G = rng.standard_normal((B, dim)).astype(np.float32)
        cs = ColumnSpec("identity", "sum", rows, dim, 0)
        out, _ = oracle.forward([cs], B, [off], [ids], [E], weights=[wts])
        keep = (ids >= 0) & (ids < rows)
        bag = np.repeat(np.arange(B), lens)[keep]
        new_off = np.searchsorted(bag, np.arange(B), side="left")
        Et = torch.from_numpy(E).double().requires_grad_(True)
        ref = F.embedding_bag(torch.from_numpy(ids[keep]), Et, torch.from_numpy(new_off), mode="sum",
                              per_sample_weights=torch.from_numpy(wts[keep]).double())
        np.testing.assert_allclose(out, ref.detach().numpy(), rtol=1e-6, atol=1e-6)
        ref.backward(torch.from_numpy(G).double())
        res = oracle.backward_adagrad([cs], B, [off], [ids], G, None, [E.copy()], [np.zeros_like(E)], 0.1, 1e-10,
                                      weights=[wts])
        g = Et.grad.numpy()
        for r, gr in zip(res["row"], res["grad"]):
            np.testing.assert_allclose(gr, g[r], rtol=1e-5, atol=1e-6)
        touched = np.zeros(rows, bool)
        touched[res["row"]] = True
        assert np.all(g[~touched] == 0)


def _copy_column(dim, rows):
    """A padded column of pad_len 1 with one value per bag: the forward copies
    each bag's row (no pooling arithmetic)."""
    return [ColumnSpec("identity", "padded", rows, dim, 0, pad_len=1)], synth.bag_offsets(np.ones(rows, np.int64))


def test_bf16_rows_hand_values():
    """bfloat16 is the upper half of a binary32: 0x3F80 = 1, 0xC000 = -2,
    0x4049 = 3.140625, 0x0001 = 2^-133, 0x7F80 = inf, 0x8000 = -0."""
    cols, off = _copy_column(4, 2)
    E = np.array([[0x3F80, 0xC000, 0x4049, 0x0001], [0x7F80, 0x8000, 0x3F00, 0xBF80]], np.uint16)
    _, seq = oracle.forward(cols, 2, [off], [np.arange(2)], [E], table_dtypes=["bf16"])
    want = np.array([[1.0, -2.0, 3.140625, 2.0 ** -133], [np.inf, -0.0, 0.5, -1.0]], np.float32)
    assert np.array_equal(seq[0][:, 0, :], want)
    assert np.signbit(seq[0][1, 0, 1])


def test_bf16_rows_match_torch_conversion():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    bits = rng.integers(0, 1 << 16, (500, 8)).astype(np.uint16)
    cols, off = _copy_column(8, 500)
    _, seq = oracle.forward(cols, 500, [off], [np.arange(500)], [bits], table_dtypes=["bf16"])
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = seq[0][:, 0, :]
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_f16_rows_every_bit_pattern():
    """All 65536 binary16 patterns against numpy's float16 -> float32."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16).reshape(-1, 4)
    rows = bits.shape[0]
    cols, off = _copy_column(4, rows)
    _, seq = oracle.forward(cols, rows, [off], [np.arange(rows)], [bits], table_dtypes=["f16"])
    ref = bits.view(np.float16).astype(np.float32)
    got = seq[0][:, 0, :]
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_int8_rows_are_scale_times_q():
    """Every q in [-128, 127] with a power-of-two scale (exact), and a hand
    example pooled: rows (2, -3) x 0.5 and (100, 1) x 0.25 sum to (26, -1.25)."""
    q = np.arange(-128, 128, dtype=np.int16).astype(np.int8).reshape(-1, 4)
    rows = q.shape[0]
    cols, off = _copy_column(4, rows)
    scale = np.full(rows, 0.25, np.float32)
    _, seq = oracle.forward(cols, rows, [off], [np.arange(rows)], [q], table_dtypes=["i8"], row_scales=[scale])
    assert np.array_equal(seq[0][:, 0, :], q.astype(np.float32) / 4)
    E = np.array([[2, -3, 0, 0], [100, 1, 0, 0]], np.int8)
    cs = [ColumnSpec("identity", "sum", 2, 4, 0)]
    out, _ = oracle.forward(cs, 1, [np.array([0, 2], np.int32)], [np.array([0, 1])], [E], table_dtypes=["i8"],
                            row_scales=[np.array([0.5, 0.25], np.float32)])
    assert np.array_equal(out[0], np.array([26.0, -1.25, 0, 0], np.float32))


def test_low_precision_tables_pool_like_their_fp32_values():
    """A low-precision table pools exactly like an fp32 table holding its
    element values (where those are fp32-representable): every pooling, the
    padded copy, weights, shared tables."""
    torch = pytest.importorskip("torch")
    for seed in range(6):
        w = synth.random_small(400 + seed, train=False)
        dts, scales, tabs_lp, tabs_32 = [], [], [], []
        rng = np.random.default_rng(seed)
        for t, spec in enumerate(w.tables):
            if spec is None:
                dts.append("f32"), scales.append(None), tabs_lp.append(np.zeros((1, 4), np.float32))
                tabs_32.append(np.zeros((1, 4), np.float32))
                continue
            E = rng.standard_normal((spec.num_rows, spec.dim)).astype(np.float32)
            dt = ["bf16", "f16", "i8", "f32"][(seed + t) % 4]
            if dt == "bf16":
                b = torch.from_numpy(E).to(torch.bfloat16)
                lp, e32 = b.view(torch.int16).numpy().view(np.uint16), b.float().numpy()
                sc = None
            elif dt == "f16":
                h = E.astype(np.float16)
                lp, e32, sc = h.view(np.uint16), h.astype(np.float32), None
            elif dt == "i8":
                lp = rng.integers(-128, 128, E.shape).astype(np.int8)
                sc = (2.0 ** rng.integers(-8, 0, spec.num_rows)).astype(np.float32)   # exact products
                e32 = lp.astype(np.float32) * sc[:, None]
            else:
                lp, e32, sc = E, E, None
            dts.append(dt), scales.append(sc), tabs_lp.append(lp), tabs_32.append(e32)
        a = oracle.forward(w.columns, w.B, w.offsets, w.values, tabs_lp, weights=w.weights, table_dtypes=dts,
                           row_scales=scales)
        b = oracle.forward(w.columns, w.B, w.offsets, w.values, tabs_32, weights=w.weights)
        assert np.array_equal(a[0], b[0])
        for x, y in zip(a[1], b[1]):
            assert (x is None and y is None) or np.array_equal(x, y)
