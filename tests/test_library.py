"""CPU checks of the C-ABI library: it builds for sm_103a, loads, exports
every entry point include/emb.h declares, rejects bad arguments before any
device work, and its host copy of the hash-mod arithmetic agrees with the
oracle.  No GPU compute."""
import os
import re

import numpy as np
import pytest

import oracle
import sparse_lookup_gb300 as sl
from sparse_lookup_gb300 import build as slbuild
from sparse_lookup_gb300.synth import ColumnSpec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    slbuild.build()
    return sl.lib()


def declared_functions():
    txt = open(os.path.join(ROOT, "include", "emb.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:emb_status|const char\*)\s+(\w+)\s*\(", txt, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("emb_plan_create", "emb_forward", "emb_backward_update", "hash_lookup_or_insert",
                 "hash_evict_expired"):
        assert must in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    assert set(declared_functions()) == set(sl.EXPORTED)


def test_library_is_built_for_sm103a(L):
    assert "sm_103a" in sl.emb_version()
    with open(sl.LIB_PATH, "rb") as f:
        blob = f.read()
    assert b"sm_103a" in blob or b"sm_103" in blob


def test_host_hash_mod_matches_oracle(L):
    rng = np.random.default_rng(5)
    ids = rng.integers(-2 ** 63, 2 ** 63 - 1, 4000, dtype=np.int64, endpoint=True)
    ids[:6] = [-2 ** 63, -1, 0, 1, 2 ** 63 - 1, 2 ** 62]
    sizes = [1, 2, 3, 7, 1000, 1024, 999_983, 10 ** 6, 2 ** 20 + 1, 2 ** 31 - 1]
    sizes += [int(x) for x in rng.integers(1, 2 ** 31 - 1, 20)]
    for rows in sizes:
        got = sl.emb_selftest_hash_mod(ids, rows)
        want = oracle.column_rows(ColumnSpec("hash_mod", "sum", rows, 4, 0), ids)
        assert np.array_equal(got, want), rows


def test_plan_create_rejects_bad_arguments_on_host(L):
    # all of these fail validation before any CUDA call
    d = sl.EmbColumnDesc()
    d.transform, d.pooling, d.num_rows, d.dim = 0, 0, 10, 6      # dim % 4 != 0
    d.weight = 16
    with pytest.raises(sl.EmbError) as e:
        sl.emb_plan_create([d], 4, 0, 0)
    assert e.value.status == 1
    d.dim = 8
    d.weight = 8                                                   # misaligned table
    with pytest.raises(sl.EmbError) as e:
        sl.emb_plan_create([d], 4, 0, 0)
    assert e.value.status == 1
    d.weight = 16
    d.transform = 2                                                # bucketize without boundaries
    with pytest.raises(sl.EmbError) as e:
        sl.emb_plan_create([d], 4, 0, 0)
    assert e.value.status == 1
    d.transform, d.dim = 0, 512                                    # dim above the limit
    with pytest.raises(sl.EmbError) as e:
        sl.emb_plan_create([d], 4, 0, 0)
    assert e.value.status == 2
    d.dim = 8
    with pytest.raises(sl.EmbError) as e:                          # training without accumulator
        sl.emb_plan_create([d], 4, 100, sl.PLAN_TRAINING)
    assert e.value.status == 1
    with pytest.raises(sl.EmbError) as e:                          # atomic backward without training
        sl.emb_plan_create([d], 4, 100, sl.PLAN_ATOMIC_BACKWARD)
    assert e.value.status == 1
    with pytest.raises(sl.EmbError) as e:                          # unknown flag bit
        sl.emb_plan_create([d], 4, 100, 4)
    assert e.value.status == 1
    with pytest.raises(sl.EmbError):
        sl.emb_plan_create([d], 0, 0, 0)                           # batch 0
