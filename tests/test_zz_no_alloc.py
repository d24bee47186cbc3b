"""The decode entry point that allocates nothing, against the oracle and the
pooled entry point.

Some callers of this library may not allocate device memory: they run under
another component's allocator that owns every device allocation, or in a
latency-critical loop that cannot take an allocation's synchronisation or
out-of-memory risk. pkv_decode_attention_noalloc serves them with scratch in
the library's own static device array. This file is collected last so that a
run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_210_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceState, assert_close, bits, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_210_gb300 import build
    build.build()
    return pkv.load()


def _noalloc(lib, st, wl, layer, out, num_splits, err, q=None):
    s = torch.cuda.current_stream().cuda_stream
    q = st.q[layer] if q is None else q
    return lib.pkv_decode_attention_noalloc(
        layer, q.data_ptr(), st.k_pool.data_ptr(), st.v_pool.data_ptr(),
        st.table.data_ptr(), st.lens.data_ptr(), out.data_ptr(), wl.num_layers, wl.num_pages,
        wl.batch, pkv.MAX_SEQ_LEN, wl.batch, num_splits, err.data_ptr(), s)


def _appended_state(wl):
    """Device state with every layer's new token appended, and the oracle's
    output for it (FP64, computed from the host copies of the pools)."""
    st = DeviceState(wl)
    pool = pkv.pkv_pool_create(wl.num_layers, wl.num_pages, wl.batch)
    for layer in range(wl.num_layers):
        pkv.pkv_append(pool, layer, st.k_new[layer], st.v_new[layer], st.k_pool, st.v_pool,
                       st.table, st.positions)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, _, _ = oracle_step(wl, st.host_k, st.host_v, bits(st.q.cpu()), bits(st.k_new.cpu()),
                            bits(st.v_new.cpu()))
    return st, pool, ref


def test_noalloc_matches_oracle_and_pooled_entry_point_on_two_calls(lib):
    wl = W.custom([1, 16, 17, 300, 2047, 2048, 40, 1000], num_layers=2, seed=400,
                  name="noalloc")
    st, pool, oracle_ref = _appended_state(wl)
    for splits in (4, 1, 16):
        ref = torch.full_like(st.out, float("nan"))
        for layer in range(wl.num_layers):
            pkv.pkv_decode_attention(pool, layer, st.q[layer], st.k_pool, st.v_pool, st.table,
                                     st.lens, ref[layer], num_splits=splits)
        assert pkv.pkv_get_error(pool) == pkv.PKV_OK
        # two calls in a row sharing the static scratch: layer 0, then layer 1
        got = torch.full_like(st.out, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for layer in range(wl.num_layers):
            assert _noalloc(lib, st, wl, layer, got[layer], splits, err) == pkv.PKV_OK
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for layer in range(wl.num_layers):
            # against the FP64 oracle, and against the pooled entry point
            assert_close(got[layer].cpu().numpy(), oracle_ref[layer],
                         f"oracle, layer {layer} S={splits}")
            assert_close(got[layer].cpu().numpy(), ref[layer].cpu().double().numpy(),
                         f"pooled, layer {layer} S={splits}")


@pytest.mark.parametrize("batch,splits", [(32, 8), (16, 16), (256, 1)])
def test_noalloc_at_the_scratch_limit_matches_oracle(lib, batch, splits):
    """batch x splits = 256 (sequence, split) rows, the whole static scratch,
    on two calls in a row (layer 0, then layer 1)."""
    rng = np.random.default_rng(402 + batch)
    lens = rng.integers(1, 2049 if batch <= 32 else 400, batch).astype(np.int32)
    lens[:4] = [1, 16, 17, 2048 if batch <= 32 else 399]
    wl = W.custom(lens, num_layers=2, seed=403 + batch, hole_every=3, name="noalloc-limit")
    st, _, oracle_ref = _appended_state(wl)
    got = torch.full_like(st.out, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for layer in range(wl.num_layers):
        assert _noalloc(lib, st, wl, layer, got[layer], splits, err) == pkv.PKV_OK
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_close(got.cpu().numpy(), oracle_ref, f"B={batch} S={splits}")


def test_noalloc_rejects_requests_beyond_its_scratch(lib):
    wl = W.custom([64] * 32, num_layers=1, seed=401, name="noalloc-limits")
    st = DeviceState(wl)
    out = torch.zeros_like(st.out[0])
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    # 32 sequences x 16 splits > 256 (sequence, split) rows
    assert _noalloc(lib, st, wl, 0, out, 16, err) == pkv.PKV_ERR_STATIC_LIMIT
    assert _noalloc(lib, st, wl, 0, out, 0, err) == pkv.PKV_ERR_STATIC_LIMIT
    assert _noalloc(lib, st, wl, 0, out, 17, err) == pkv.PKV_ERR_STATIC_LIMIT
    assert _noalloc(lib, st, wl, 1, out, 2, err, q=st.q[0]) == pkv.PKV_ERR_INVALID_ARG  # layer
    assert _noalloc(lib, st, wl, 0, out, 8, err) == pkv.PKV_OK                # 256 rows
    torch.cuda.synchronize()
    assert lib.pkv_status_string(pkv.PKV_ERR_STATIC_LIMIT).startswith(b"request exceeds")
