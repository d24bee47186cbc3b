"""The multi-layer fused step (pkv_append_attend_layers: several layers in one
persistent launch) against the CPU oracle and against the per-layer launches,
through the C ABI (needs a GPU).

Pools after the step: bit-exact. Outputs: the FP64 tolerance gate (max |d| <=
5e-4, row-normwise <= 1e-3), and bit-identical to the per-layer cluster
kernel with the same number of splits, which runs the same arithmetic.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_210_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceState, assert_close, bits, oracle_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_210_gb300 import build
    build.build()
    pkv.load()


def _pool(wl, flags=0):
    return pkv.pkv_pool_create(wl.num_layers, wl.num_pages, wl.batch, flags=flags)


def _host_inputs(st):
    return bits(st.q.cpu()), bits(st.k_new.cpu()), bits(st.v_new.cpu())


def _per_layer(wl, st, splits):
    """The same step as one fused launch per layer; returns (out, k_pool, v_pool)."""
    pool = _pool(wl)
    k0, v0 = st.k_pool.clone(), st.v_pool.clone()
    out = torch.full_like(st.out, float("nan"))
    for layer in range(wl.num_layers):
        pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer], k0, v0,
                              st.table, st.lens, out[layer], num_splits=splits)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    return out, k0, v0


WORKLOADS = {
    # 1 layer: no waits at all
    "tiny": lambda: W.tiny(False),
    # batch 2, 16 layers, full and partial last pages: S = 16 clusters
    "b2-16layers": lambda: W.custom([2048, 1000], num_layers=16, seed=701, name="b2-16"),
    # every page-boundary case, 3 layers, fragmented pool
    "edges": lambda: W.custom([1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 1000, 2047, 2048],
                              num_layers=3, seed=702, hole_every=3, name="edges"),
    # 16 sequences: S = 2, so 4 layers per launch and 20 layers take 5 launches
    "b16-20layers": lambda: W.custom(list(np.random.default_rng(703).integers(1, 300, 16)),
                                     num_layers=20, seed=703, name="b16-20"),
}


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_layers_match_oracle(name):
    wl = WORKLOADS[name]()
    st = DeviceState(wl)
    pool = _pool(wl)
    pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                 st.table, st.lens, st.out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    assert np.array_equal(bits(st.k_pool), ok) and np.array_equal(bits(st.v_pool), ov)
    assert_close(st.out.cpu().numpy(), ref, f"{name} layers")


@pytest.mark.parametrize("name", ["b2-16layers", "edges", "b16-20layers"])
def test_layers_bit_identical_to_per_layer_cluster_launches(name):
    """Same split count, same page order per warp, same merges: the same bits
    as one of the per-layer cluster plans (which one depends on the device's
    cluster residency)."""
    wl = WORKLOADS[name]()
    st = DeviceState(wl, host_pools=False)
    k0, v0 = st.k_pool.clone(), st.v_pool.clone()
    pool = _pool(wl)
    pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, k0, v0, st.table, st.lens,
                                 st.out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    got = st.out.cpu()
    matched = []
    for splits in (16, 8, 4, 2):
        out, kp, vp = _per_layer(wl, st, splits)
        assert torch.equal(kp.view(torch.int16), k0.view(torch.int16))
        assert torch.equal(vp.view(torch.int16), v0.view(torch.int16))
        if torch.equal(out.cpu().view(torch.int32), got.view(torch.int32)):
            matched.append(splits)
    assert matched, "no per-layer cluster plan gives the same bits"


def test_layer_range_leaves_other_layers_alone():
    wl = W.custom([300, 45, 2048], num_layers=5, seed=704, name="range")
    st = DeviceState(wl)
    pool = _pool(wl)
    out = torch.full((2, wl.batch, W.NUM_Q_HEADS, W.HEAD_DIM), float("nan"), device="cuda")
    pkv.pkv_append_attend_layers(pool, 2, st.q[2:4], st.k_new[2:4], st.v_new[2:4], st.k_pool,
                                 st.v_pool, st.table, st.lens, out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    q_b, kn_b, vn_b = _host_inputs(st)
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, q_b, kn_b, vn_b, layers=[2, 3])
    assert np.array_equal(bits(st.k_pool), ok) and np.array_equal(bits(st.v_pool), ov)
    assert_close(out.cpu().numpy(), ref, "layers 2..3")


def test_large_batch_runs_per_layer_launches():
    """A batch whose clusters cannot all be resident goes through the
    per-layer path: same results."""
    lens = np.random.default_rng(705).integers(1, 80, 160)
    wl = W.custom(list(lens), num_layers=2, seed=705, name="b160")
    st = DeviceState(wl)
    pool = _pool(wl)
    pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                 st.table, st.lens, st.out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    assert np.array_equal(bits(st.k_pool), ok) and np.array_equal(bits(st.v_pool), ov)
    assert_close(st.out.cpu().numpy(), ref, "b160 layers")


def test_graph_replay_repeats_the_step():
    """Captured in a CUDA graph (the counter reset is a node of it) and
    replayed: the append rewrites the same slots with the same bits, so every
    replay gives the first run's outputs."""
    wl = WORKLOADS["b2-16layers"]()
    st = DeviceState(wl, host_pools=False)
    pool = _pool(wl)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())   # the inputs were made on the current stream
    with torch.cuda.stream(s):
        pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                     st.table, st.lens, st.out, stream=s)
    s.synchronize()
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    first = st.out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                     st.table, st.lens, st.out, stream=torch.cuda.current_stream())
    for _ in range(3):
        st.out.fill_(float("nan"))
        with torch.cuda.stream(s):
            graph.replay()
        s.synchronize()
        assert torch.equal(st.out.view(torch.int32), first.view(torch.int32))
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK


def test_invalid_length_skips_only_that_sequence():
    wl = W.custom([700, 33, 2048], num_layers=4, seed=706, name="badlen")
    st = DeviceState(wl)
    bad = st.lens.clone()
    bad[1] = 5000
    pool = _pool(wl)
    pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                 st.table, bad, st.out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    got = st.out.cpu().numpy()
    assert np.all(np.isnan(got[:, 1]))            # untouched
    ref, _, _ = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    keep = [0, 2]
    assert_close(got[:, keep], ref[:, keep], "valid sequences")


def test_invalid_page_id_is_flagged():
    wl = W.custom([200, 64], num_layers=3, seed=707, name="badpage")
    st = DeviceState(wl)
    table = st.table.clone()
    table[1, 0, 3] = wl.num_pages + 7
    pool = _pool(wl)
    pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                 table, st.lens, st.out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    ref, _, _ = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    got = st.out.cpu().numpy()
    # layers 0 and 2 and the other sequence are unaffected
    assert_close(got[[0, 2]], ref[[0, 2]], "other layers")
    assert_close(got[1, 1:], ref[1, 1:], "other sequence")


def test_host_argument_checks():
    wl = W.tiny(False)
    st = DeviceState(wl, host_pools=False)
    pool = _pool(wl)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_append_attend_layers(pool, 1, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                     st.table, st.lens, st.out)   # layers 1..1 of a 1-layer pool
    with pytest.raises(pkv.PkvError):
        pkv.pkv_append_attend_layers(pool, -1, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                     st.table, st.lens, st.out)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                     st.table, st.lens, st.out, num_layers=2)
    # zero layers: a no-op
    pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                 st.table, st.lens, st.out, num_layers=0)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK


def test_layer_wait_timeout_is_flagged_and_the_context_stays_usable():
    """Failure detection without a GPU fault: the test hook makes every
    between-layer wait unreachable, so each block gives up after its bounded
    wait (about two seconds), flags the timeout and finishes; the host reads
    PKV_ERR_DEVICE_TIMEOUT, and the next normal step is correct."""
    wl = W.custom([300, 2048], num_layers=2, seed=708, name="timeout")
    st = DeviceState(wl)
    pool = _pool(wl)
    kp, vp = st.k_pool.clone(), st.v_pool.clone()
    out = torch.full_like(st.out, float("nan"))
    pkv.pkv_test_layers_wait_timeout(pool, 0, st.q, st.k_new, st.v_new, kp, vp, st.table,
                                     st.lens, out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_DEVICE_TIMEOUT
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK          # the flag was cleared
    pkv.pkv_append_attend_layers(pool, 0, st.q, st.k_new, st.v_new, st.k_pool, st.v_pool,
                                 st.table, st.lens, st.out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    assert np.array_equal(bits(st.k_pool), ok) and np.array_equal(bits(st.v_pool), ov)
    assert_close(st.out.cpu().numpy(), ref, "after a timeout")


def test_pool_device_figures_and_plan():
    """The handle's device figures (occupancy of the three decode shapes,
    cluster limit) feed the same planner the CPU tests check."""
    wl = W.tiny(False)
    pool = pkv.pkv_pool_create(1, wl.num_pages, 4, max_splits=32)
    f = pkv.pkv_pool_device_figures(pool)
    assert f.num_sms == torch.cuda.get_device_properties(0).multi_processor_count
    assert min(f.ticket_blocks_per_sm, f.narrow_blocks_per_sm, f.wide_blocks_per_sm) >= 1
    assert f.narrow_blocks_per_sm <= f.wide_blocks_per_sm
    assert f.max_cluster in (0, 2, 4, 8, 16)
    assert (f.max_splits, f.max_seq_len) == (32, 2048)
    p = pkv.pkv_plan_decode(f, 2)
    if f.max_cluster >= 2:
        assert p.cluster >= 2 and p.shape in (pkv.PKV_SHAPE_NARROW, pkv.PKV_SHAPE_WIDE)
    pool.close()
