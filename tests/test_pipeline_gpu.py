"""GPU parity of the pipelined dynamic-table step (the lookup of step t+1 and
the expiry of step t on a low-priority stream beside step t's backward)
against the oracle run step by step in order: every step's rows bit-exact,
pooled outputs within 1e-5 rel / 1e-6 abs, the final map identical and the
row pool's weights and accumulators within 1e-5 rel / 1e-6 abs (exclusions:
elements the fp32 sum left ill-conditioned at some step, counted)."""
import numpy as np
import pytest

import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import build as slbuild
from sparse_lookup_gb300 import synth
from sparse_lookup_gb300.pipeline import DynamicPipeline

from helpers import OraclePool, assert_close_skip, compare_hash_maps

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    slbuild.build()
    sl.lib()


def _steps(seed, C, B, steps, alpha, key_bits, max_len):
    import torch
    out = []
    for t in range(steps):
        offs, keys = synth.dynamic_keys(seed, t, C, B, alpha, key_bits, max_len)
        tids = np.concatenate([np.full(k.size, c, np.int32) for c, k in enumerate(keys)])
        allk = np.concatenate(keys)
        ids_off = np.concatenate([[0], np.cumsum(np.concatenate([np.diff(o) for o in offs]))]).astype(np.int32)
        out.append(dict(offs=offs, tids=tids, keys=allk, tids_d=torch.from_numpy(tids).cuda(),
                        keys_d=torch.from_numpy(allk).cuda(), off_d=torch.from_numpy(ids_off).cuda()))
    return out


@pytest.mark.parametrize("ttl,thr", [(4, 3), (0, 1), (1, 2)])
def test_pipelined_steps_match_the_oracle_in_order(ttl, thr):
    import torch
    C, B, steps, dim, seed, lr = 8, 512, 16, 32, 1007, 0.01
    cap, num_slots, max_len = 1 << 13, 1 << 16, 5
    data = _steps(seed, C, B, steps, 1.2, 20, max_len)
    max_keys = C * B * max_len
    ht = sl.HashTable(num_slots, cap, dim, thr, 128, seed, 0.01, max_keys)
    cols = [synth.ColumnSpec("rows_given", "sum", cap, dim, 0) for _ in range(C)]
    plan = sl.Plan(cols, [ht.weight], [ht.acc], max_batch=B, max_ids=max_keys, training=True)
    pipe = DynamicPipeline(ht, plan, ttl, B, max_keys)
    Gs = [synth.make_grad((B, plan.out_width), 500 + t, "cuda") for t in range(steps)]
    outs = [torch.empty((B, plan.out_width), device="cuda") for _ in range(steps)]
    rows = [torch.empty(d["keys"].size, dtype=torch.int64, device="cuda") for d in data]
    torch.cuda.synchronize()
    pipe.prefetch(0, data[0]["tids_d"], data[0]["keys_d"])
    for t in range(steps):
        pipe.forward(t, data[t]["off_d"], outs[t], rows_copy=rows[t])
        if t + 1 < steps:
            pipe.prefetch(t + 1, data[t + 1]["tids_d"], data[t + 1]["keys_d"])
        pipe.backward(Gs[t], lr, 1e-10)
    pipe.finish()
    torch.cuda.synchronize()
    assert ht.device_status() in (0, 5) and plan.device_status() == 0

    pool = OraclePool(cap, dim, thr, seed, cols, B, lr, 1e-10)
    for t in range(steps):
        d = data[t]
        o = pool.step(d["tids"], d["keys"], t, d["offs"], Gs[t].cpu().numpy(), ttl)
        assert np.array_equal(rows[t].cpu().numpy(), o["rows"]), "rows step %d" % t
        assert_close_skip(outs[t].cpu().numpy(), o["out"], o["out_skip"], what="pooled step %d" % t)
    compare_hash_maps(ht.export(), pool.oh.export(), "final map")
    pool.check_pool(ht.weight, ht.acc)


def test_forward_before_prefetch_is_rejected():
    import torch
    ht = sl.HashTable(1024, 64, 4, 1, 64, 1, 0.01, 64)
    cols = [synth.ColumnSpec("rows_given", "sum", 64, 4, 0)]
    plan = sl.Plan(cols, [ht.weight], [ht.acc], max_batch=2, max_ids=64, training=True)
    pipe = DynamicPipeline(ht, plan, 1, 2, 64)
    with pytest.raises(RuntimeError):
        pipe.forward(0, torch.zeros(3, dtype=torch.int32, device="cuda"), torch.empty((2, 4), device="cuda"))
