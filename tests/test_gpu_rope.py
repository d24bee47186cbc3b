"""Rotary position embedding on the decode path against the oracle (needs a
GPU): the appended key rotated to its position and stored as BF16 (bit-exact
pools), the queries rotated to the same position (output within the FP32
tolerance), through the standalone append, the unfused attention and the
fused append-attend launch, on the cluster-merge and ticket-merge paths.

Angles: the Llama 3 base (500000) and, where the rotation must visibly move
the scores, the classic base 10000, as FP32 tables [2048][32].
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_210_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceState, assert_close, bits, oracle_step

pytestmark = pytest.mark.gpu

EDGE_LENGTHS = [1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 1000, 2047, 2048]


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_210_gb300 import build
    build.build()
    pkv.load()


WORKLOADS = {
    "tiny": lambda: W.tiny(False),
    "edges": lambda: W.custom(EDGE_LENGTHS, num_layers=2, seed=401, name="edges"),
    "edges-holes": lambda: W.custom(EDGE_LENGTHS[::-1], num_layers=2, seed=402, hole_every=3,
                                    name="edges-holes"),
}


def _tables(base):
    cos_t, sin_t = W.rope_tables(base=base)
    return (cos_t, sin_t), torch.from_numpy(cos_t).cuda(), torch.from_numpy(sin_t).cuda()


def _pool(wl, flags=0):
    return pkv.pkv_pool_create(wl.num_layers, wl.num_pages, wl.batch, flags=flags)


def _host_inputs(st):
    return bits(st.q.cpu()), bits(st.k_new.cpu()), bits(st.v_new.cpu())


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("base", [10000.0, 500000.0])
def test_rope_append_bit_exact(name, base):
    wl = WORKLOADS[name]()
    st = DeviceState(wl)
    host, cos_d, sin_d = _tables(base)
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        pkv.pkv_append_rope(pool, layer, st.k_new[layer], st.v_new[layer], st.k_pool, st.v_pool,
                            st.table, st.positions, cos_d, sin_d)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    _, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st), rope=host)
    assert np.array_equal(bits(st.k_pool), ok)
    assert np.array_equal(bits(st.v_pool), ov)


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_rope_append_then_decode_matches_oracle(name, splits):
    wl = WORKLOADS[name]()
    st = DeviceState(wl)
    host, cos_d, sin_d = _tables(10000.0)
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        pkv.pkv_append_rope(pool, layer, st.k_new[layer], st.v_new[layer], st.k_pool, st.v_pool,
                            st.table, st.positions, cos_d, sin_d)
        pkv.pkv_decode_attention_rope(pool, layer, st.q[layer], st.k_pool, st.v_pool, st.table,
                                      st.lens, cos_d, sin_d, st.out[layer], num_splits=splits)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, _, _ = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st), rope=host)
    assert_close(st.out.cpu().numpy(), ref, f"{name} rope S={splits}")


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_rope_fused_matches_oracle(name, splits):
    wl = WORKLOADS[name]()
    st = DeviceState(wl)
    host, cos_d, sin_d = _tables(10000.0)
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        pkv.pkv_append_attend_rope(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                                   st.k_pool, st.v_pool, st.table, st.lens, cos_d, sin_d,
                                   st.out[layer], num_splits=splits)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st), rope=host)
    assert np.array_equal(bits(st.k_pool), ok) and np.array_equal(bits(st.v_pool), ov)
    assert_close(st.out.cpu().numpy(), ref, f"{name} fused rope S={splits}")


def test_rope_changes_the_output():
    """The rotation is applied: with base 10000 the output moves well past
    the tolerance from the unrotated oracle."""
    wl = WORKLOADS["edges"]()
    st = DeviceState(wl)
    host, cos_d, sin_d = _tables(10000.0)
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        pkv.pkv_append_attend_rope(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                                   st.k_pool, st.v_pool, st.table, st.lens, cos_d, sin_d,
                                   st.out[layer])
    plain, _, _ = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    got = st.out.cpu().numpy()
    assert np.abs(got - plain).max() > 100 * 5e-4


@pytest.mark.parametrize("fused", [True, False])
def test_rope_identity_tables_reproduce_the_plain_path(fused):
    """cos = 1, sin = 0: the rotated path returns bit for bit what the plain path does."""
    wl = WORKLOADS["edges-holes"]()
    a = DeviceState(wl)
    b = DeviceState(wl)
    cos_d = torch.ones((W.MAX_SEQ_LEN, W.HEAD_DIM // 2), device="cuda")
    sin_d = torch.zeros_like(cos_d)
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        if fused:
            pkv.pkv_append_attend(pool, layer, a.q[layer], a.k_new[layer], a.v_new[layer],
                                  a.k_pool, a.v_pool, a.table, a.lens, a.out[layer])
            pkv.pkv_append_attend_rope(pool, layer, b.q[layer], b.k_new[layer], b.v_new[layer],
                                       b.k_pool, b.v_pool, b.table, b.lens, cos_d, sin_d,
                                       b.out[layer])
        else:
            pkv.pkv_append(pool, layer, a.k_new[layer], a.v_new[layer], a.k_pool, a.v_pool,
                           a.table, a.positions)
            pkv.pkv_decode_attention(pool, layer, a.q[layer], a.k_pool, a.v_pool, a.table,
                                     a.lens, a.out[layer])
            pkv.pkv_append_rope(pool, layer, b.k_new[layer], b.v_new[layer], b.k_pool, b.v_pool,
                                b.table, b.positions, cos_d, sin_d)
            pkv.pkv_decode_attention_rope(pool, layer, b.q[layer], b.k_pool, b.v_pool, b.table,
                                          b.lens, cos_d, sin_d, b.out[layer])
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    assert np.array_equal(bits(a.k_pool), bits(b.k_pool))
    assert torch.equal(a.out.view(torch.int32), b.out.view(torch.int32))


@pytest.mark.parametrize("pdl", [False, True])
def test_rope_many_sequences_chain_matches_oracle(pdl):
    """42 ragged sequences over a fragmented pool (the ticket-merge plan),
    3 layers of the fused rotated step, inside a CUDA graph with programmatic
    dependent launch when pdl is set."""
    wl = W.custom(EDGE_LENGTHS * 3, num_layers=3, seed=430, hole_every=3, name="many")
    st = DeviceState(wl)
    host, cos_d, sin_d = _tables(500000.0)
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st), rope=host)
    pool = _pool(wl, flags=pkv.PKV_FLAG_PDL if pdl else 0)

    def chain():
        for layer in range(wl.num_layers):
            pkv.pkv_append_attend_rope(pool, layer, st.q[layer], st.k_new[layer],
                                       st.v_new[layer], st.k_pool, st.v_pool, st.table, st.lens,
                                       cos_d, sin_d, st.out[layer])

    if pdl:
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            chain()
        g.replay()
        torch.cuda.synchronize()
    else:
        chain()
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    assert np.array_equal(bits(st.k_pool), ok) and np.array_equal(bits(st.v_pool), ov)
    assert_close(st.out.cpu().numpy(), ref, f"many rope pdl={pdl}")


def test_rope_full_size_llama_step():
    """The full 16-layer batch-2 step at 2048 tokens, fused and rotated, all
    outputs against the oracle, pools bit-exact."""
    wl = W.llama_default()
    st = DeviceState(wl)
    host, cos_d, sin_d = _tables(500000.0)
    pool = _pool(wl, flags=pkv.PKV_FLAG_PDL)
    for layer in range(wl.num_layers):
        pkv.pkv_append_attend_rope(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                                   st.k_pool, st.v_pool, st.table, st.lens, cos_d, sin_d,
                                   st.out[layer])
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st), rope=host)
    assert np.array_equal(bits(st.k_pool), ok) and np.array_equal(bits(st.v_pool), ov)
    assert_close(st.out.cpu().numpy(), ref, "llama rope")


def test_rope_tables_are_checked():
    wl = W.tiny()
    st = DeviceState(wl)
    _, cos_d, sin_d = _tables(10000.0)
    pool = _pool(wl)
    odd = torch.empty(W.MAX_SEQ_LEN * 32 + 1, device="cuda")[1:]   # 4-byte offset
    for cs, sn in ((None, sin_d), (cos_d, None), (odd, sin_d)):
        with pytest.raises(pkv.PkvError):
            pkv.pkv_append_attend_rope(pool, 0, st.q[0], st.k_new[0], st.v_new[0], st.k_pool,
                                       st.v_pool, st.table, st.lens, cs, sn, st.out[0])
        with pytest.raises(pkv.PkvError):
            pkv.pkv_append_rope(pool, 0, st.k_new[0], st.v_new[0], st.k_pool, st.v_pool,
                                st.table, st.positions, cs, sn)
        with pytest.raises(pkv.PkvError):
            pkv.pkv_decode_attention_rope(pool, 0, st.q[0], st.k_pool, st.v_pool, st.table,
                                          st.lens, cs, sn, st.out[0])
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
