"""The native admission scheduler (libpkv, include/pkv_sched.h) against the
admission oracle, through the C ABI, on the CPU: every returned id, batch,
block table and counter identical over random continuous and static traces,
plus the budget arithmetic and argument errors."""

import random

import numpy as np
import pytest

import paged_kv_cache_210_gb300 as pkv
from oracle import admission as A
from paged_kv_cache_210_gb300 import build as lib_build

STATUS = {pkv.PKV_OK: A.OK, pkv.PKV_ERR_REJECTED: A.REJECTED, pkv.PKV_ERR_INVALID_ARG: A.INVALID}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    lib_build.build()
    pkv.load()


def _call(fn, *args):
    try:
        return A.OK, fn(*args)
    except pkv.PkvError as e:
        return STATUS[e.status], None


def test_budget_arithmetic_matches_oracle():
    rng = random.Random(3)
    cases = [(1, 16), (1, 17), (16, 1), (17, 1), (2000, 128), (1000, 5000), (2047, 64)]
    cases += [(rng.randint(1, 2047), rng.randint(1, 3000)) for _ in range(2000)]
    for p, n in cases:
        allowed, prefix, budget = pkv.pkv_sched_budget(p, n)
        assert allowed == A.allowed_new_tokens(p, n, 2048)
        assert prefix == A.processed_prefix(p, n, 2048)
        assert budget == A.budget_pages(p, n)
    for p, n in ((0, 1), (2048, 1), (10, 0)):
        with pytest.raises(pkv.PkvError) as e:
            pkv.pkv_sched_budget(p, n)
        assert e.value.status == pkv.PKV_ERR_INVALID_ARG


def _compare(native, orc, pool):
    snap = orc.snapshot()
    got = pkv.pkv_sched_get_stats(native)
    for key, value in snap.items():
        assert got[key] == value, key


@pytest.mark.parametrize("static", [False, True])
@pytest.mark.parametrize("seed", [1, 2, 3])
def test_random_trace_identical_to_oracle(static, seed):
    rng = random.Random(seed * 10 + static)
    pool = rng.choice([256, 1024, 4096])
    native = pkv.pkv_sched_create(pool, static_batching=static)
    orc = A.AdmissionScheduler(pool, static_batching=static)
    lengths = {}
    for step in range(300):
        for _ in range(rng.randint(0, 3)):
            p, n = rng.randint(0, 900), rng.randint(0, 900)
            st_n, rid_n = _call(pkv.pkv_sched_submit, native, p, n)
            st_o, rid_o = orc.submit(p, n)
            assert (st_n, rid_n) == (st_o, rid_o)
        adm_n = pkv.pkv_sched_admit(native)
        adm_o = orc.admit()
        assert adm_n == adm_o
        for rid in adm_o:
            lengths[rid] = orc.requests[rid].prompt_tokens
        batch = pkv.pkv_sched_decode_batch(native)
        assert batch == orc.decode_batch()
        for rid in batch:
            st_n, _ = _call(pkv.pkv_sched_extend, native, rid, lengths[rid])
            assert st_n == orc.extend(rid, lengths[rid]) == A.OK
        if batch:
            tab_n = pkv.pkv_sched_block_tables(native, batch, max_batch=len(batch) + 2)
            tab_o = np.full_like(tab_n, -1)
            tab_o[:, :len(batch)] = np.array(orc.block_tables(batch, 128), np.int32)
            assert np.array_equal(tab_n, tab_o)
        for rid in batch:
            prefix = orc.requests[rid].prefix
            if lengths[rid] >= prefix or rng.random() < 0.03:
                _call(pkv.pkv_sched_finish, native, rid)
                orc.finish(rid)
                del lengths[rid]
            else:
                lengths[rid] = min(prefix, lengths[rid] + rng.randint(1, 48))
        # an invalid growth is refused by both without side effects
        if batch and rng.random() < 0.2:
            rid = batch[0]
            if rid in lengths:
                bad = orc.requests[rid].prefix + 1
                assert _call(pkv.pkv_sched_extend, native, rid, bad)[0] == orc.extend(rid, bad)
        _compare(native, orc, pool)
    pkv.pkv_sched_destroy(native)


def test_argument_errors():
    with pytest.raises(pkv.PkvError):
        pkv.pkv_sched_create(0)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_sched_create(16, max_seq_len=2047)
    s = pkv.pkv_sched_create(64)
    with pytest.raises(pkv.PkvError) as e:
        pkv.pkv_sched_submit(s, 1000, 1000)     # 2048 pages > 64
    assert e.value.status == pkv.PKV_ERR_REJECTED
    rid = pkv.pkv_sched_submit(s, 10, 10)
    for fn, args in ((pkv.pkv_sched_extend, (rid, 5)), (pkv.pkv_sched_finish, (rid,)),
                     (pkv.pkv_sched_extend, (99, 5))):
        with pytest.raises(pkv.PkvError) as e:
            fn(s, *args)                          # not admitted yet / unknown
        assert e.value.status == pkv.PKV_ERR_INVALID_ARG
    assert pkv.pkv_sched_admit(s) == [rid]
    with pytest.raises(pkv.PkvError):
        pkv.pkv_sched_block_tables(s, [rid], max_batch=0)
    pkv.pkv_sched_extend(s, rid, 19)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_sched_block_tables(s, [rid], max_pages=1)
    tab = pkv.pkv_sched_block_tables(s, [rid], max_pages=2)
    assert tab.shape == (16, 1, 2) and np.all(tab >= 0)
    pkv.pkv_sched_finish(s, rid)
    assert pkv.pkv_sched_get_stats(s)["free_pages"] == 64


def test_extend_batch_and_reused_tables():
    a = pkv.pkv_sched_create(4096)
    b = A.AdmissionScheduler(4096)
    ids = [pkv.pkv_sched_submit(a, 40 + 7 * i, 300) for i in range(6)]
    assert [b.submit(40 + 7 * i, 300)[1] for i in range(6)] == ids
    assert pkv.pkv_sched_admit(a) == b.admit() == ids
    lengths = [41, 16, 17, 200, 1, 64]
    pkv.pkv_sched_extend_batch(a, ids, lengths)
    for rid, n in zip(ids, lengths):
        assert b.extend(rid, n) == A.OK
    full = pkv.pkv_sched_block_tables(a, ids, max_batch=8)
    ref = np.full_like(full, -1)
    ref[:, :6] = np.array(b.block_tables(ids, 128), np.int32)
    assert np.array_equal(full, ref)
    # without clearing, entries past each row's pages keep what was there
    buf = np.full((16, 8, 128), 7777, np.int32)
    pkv.pkv_sched_block_tables(a, ids, 8, 128, buf, clear_tail=False)
    for r, n in enumerate(lengths):
        pages = -(-n // 16)
        assert np.array_equal(buf[:, r, :pages], full[:, r, :pages])
        assert np.all(buf[:, r, pages:] == 7777)
    assert np.all(buf[:, 6:] == 7777)
    # a failing entry stops the batch and reports it
    with pytest.raises(pkv.PkvError):
        pkv.pkv_sched_extend_batch(a, [ids[0], 12345], [50, 10])
    with pytest.raises(ValueError):
        pkv.pkv_sched_extend_batch(a, ids, lengths[:-1])
