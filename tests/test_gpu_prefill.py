"""Prefill over pages on the tensor cores against the oracle (needs a GPU):
the fill bit-exact, causal attention of every chunk token within the FP32
tolerance, for whole prompts, chunked prompts continuing a cached prefix,
several sequences per call, a full 2,048-token prompt, and device-side
index errors flagged without a fault."""

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_210_gb300 as pkv
import workloads as W
from gpu_helpers import assert_close, bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_210_gb300 import build
    build.build()
    pkv.load()


class State:
    def __init__(self, wl):
        self.wl = wl
        kp, vp = wl.pools("cpu", "nan")
        self.host_k, self.host_v = bits(kp), bits(vp)
        self.k_pool, self.v_pool = kp.cuda(), vp.cuda()
        self.q, self.k, self.v = wl.q(), wl.k(), wl.v()
        self.qd, self.kd, self.vd = self.q.cuda(), self.k.cuda(), self.v.cuda()
        self.table = torch.from_numpy(wl.block_tables).cuda()
        self.cu = torch.from_numpy(wl.cu_tokens).cuda()
        self.start = torch.from_numpy(wl.start_pos).cuda()
        self.out = torch.full((wl.num_layers, wl.total_tokens, 32, 64), float("nan"),
                              device="cuda")
        self.max_chunk = int(wl.chunk_lens.max())


def oracle_prefill(st, layers=None):
    wl = st.wl
    orc = oracle.load()
    g = oracle.geometry(wl.num_layers, wl.num_pages, wl.batch)
    kp, vp = st.host_k.copy(), st.host_v.copy()
    outs = []
    for layer in (range(wl.num_layers) if layers is None else layers):
        assert orc.prefill_fill(g, layer, bits(st.k[layer]), bits(st.v[layer]), kp, vp,
                                wl.block_tables, wl.cu_tokens, wl.start_pos) == oracle.OK
        s, out = orc.prefill_attention(g, layer, bits(st.q[layer]), kp, vp, wl.block_tables,
                                       wl.cu_tokens, wl.start_pos, threads=8)
        assert s == oracle.OK
        outs.append(out)
    return np.stack(outs), kp, vp


def run(st, pool, layers=None):
    for layer in (range(st.wl.num_layers) if layers is None else layers):
        pkv.pkv_prefill(pool, layer, st.qd[layer], st.kd[layer], st.vd[layer], st.k_pool,
                        st.v_pool, st.table, st.cu, st.start, st.out[layer], st.max_chunk)


CASES = {
    "one-token": lambda: W.prefill([1], seed=701, name="one-token"),
    "prompt-100": lambda: W.prefill([100], seed=702, name="prompt-100"),
    "ragged-3": lambda: W.prefill([33, 64, 5], seed=703, name="ragged-3", num_layers=2),
    "chunked": lambda: W.prefill([40, 77, 16, 1], [100, 3, 512, 63], seed=704, hole_every=3,
                                 name="chunked"),
}


@pytest.mark.parametrize("name", list(CASES))
def test_prefill_matches_oracle(name):
    st = State(CASES[name]())
    pool = pkv.pkv_pool_create(st.wl.num_layers, st.wl.num_pages, st.wl.batch)
    run(st, pool)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, ok, ov = oracle_prefill(st)
    assert np.array_equal(bits(st.k_pool.cpu()), ok)
    assert np.array_equal(bits(st.v_pool.cpu()), ov)
    assert_close(st.out.cpu().numpy(), ref, name)


def test_fill_alone_is_bit_exact():
    st = State(CASES["chunked"]())
    pool = pkv.pkv_pool_create(1, st.wl.num_pages, st.wl.batch)
    pkv.pkv_prefill_fill(pool, 0, st.kd[0], st.vd[0], st.k_pool, st.v_pool, st.table, st.cu,
                         st.start, st.max_chunk)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    _, ok, ov = oracle_prefill(st)
    assert np.array_equal(bits(st.k_pool.cpu()), ok) and np.array_equal(bits(st.v_pool.cpu()), ov)


def test_full_prompt_2048():
    """One 2,048-token prompt (64 query tiles, up to 2,048 keys), 2 layers."""
    st = State(W.prefill([2048], num_layers=2, seed=705, name="p2048"))
    pool = pkv.pkv_pool_create(2, st.wl.num_pages, 1)
    run(st, pool)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, _, _ = oracle_prefill(st)
    assert_close(st.out.cpu().numpy(), ref, "p2048")


def test_prefill_then_decode_step():
    """A prompt prefilled in two chunks, then one fused decode step appending
    the next token: the decode output equals the oracle on the final pool."""
    n = 300
    wl = W.prefill([n], num_layers=1, seed=706, name="then-decode")
    # the block table must also cover the decoded token at position n
    dec = W.custom([n + 1], num_layers=1, seed=706)
    st = State(W.PrefillWorkload("chunks", 1, dec.num_pages, np.array([0], np.int32),
                                 np.array([n], np.int32), dec.block_tables, wl.seed))
    st.host_k[:] = W.BF16_NAN_BITS
    st.host_v[:] = W.BF16_NAN_BITS
    st.k_pool.copy_(torch.from_numpy(st.host_k.view(np.int16)).view(torch.bfloat16))
    st.v_pool.copy_(torch.from_numpy(st.host_v.view(np.int16)).view(torch.bfloat16))
    pool = pkv.pkv_pool_create(1, dec.num_pages, 1)
    for s0, s1 in ((0, 128), (128, n)):
        cu = torch.tensor([0, s1 - s0], dtype=torch.int32, device="cuda")
        start = torch.tensor([s0], dtype=torch.int32, device="cuda")
        out = torch.empty((s1 - s0, 32, 64), device="cuda")
        pkv.pkv_prefill(pool, 0, st.qd[0, s0:s1], st.kd[0, s0:s1], st.vd[0, s0:s1], st.k_pool,
                        st.v_pool, st.table, cu, start, out, s1 - s0)
        st.out[0, s0:s1] = out
    q = dec.q("cpu")[0]
    kn, vn = dec.k_new("cpu")[0], dec.v_new("cpu")[0]
    lens = torch.tensor([n + 1], dtype=torch.int32, device="cuda")
    dout = torch.empty((1, 32, 64), device="cuda")
    pkv.pkv_append_attend(pool, 0, q.cuda(), kn.cuda(), vn.cuda(), st.k_pool, st.v_pool,
                          st.table, lens, dout)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, kp, vp = oracle_prefill(st)
    assert_close(st.out.cpu().numpy(), ref, "chunked prefill")
    orc = oracle.load()
    g = oracle.geometry(1, dec.num_pages, 1)
    assert orc.append(g, 0, bits(kn), bits(vn), kp, vp, dec.block_tables,
                      np.array([n], np.int32)) == oracle.OK
    s, dref, _, _ = orc.decode_attention(g, 0, bits(q), kp, vp, dec.block_tables,
                                         np.array([n + 1], np.int32))
    assert s == oracle.OK
    assert_close(dout.cpu().numpy(), dref, "decode after prefill")


def test_device_index_errors_are_flagged():
    st = State(W.prefill([40, 20], seed=707, name="errors"))
    pool = pkv.pkv_pool_create(1, st.wl.num_pages, 2)
    table = st.table.clone()
    table[0, 1, 0] = st.wl.num_pages + 5          # a page outside the pool
    pkv.pkv_prefill(pool, 0, st.qd[0], st.kd[0], st.vd[0], st.k_pool, st.v_pool, table, st.cu,
                    st.start, st.out[0], st.max_chunk)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    start = st.start.clone()
    start[0] = 2040                                # runs past the context
    pkv.pkv_prefill(pool, 0, st.qd[0], st.kd[0], st.vd[0], st.k_pool, st.v_pool, st.table,
                    st.cu, start, st.out[0], st.max_chunk)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    cu = st.cu.clone()
    cu[2] = st.wl.total_tokens + 7                 # rows past the buffers
    pkv.pkv_prefill(pool, 0, st.qd[0], st.kd[0], st.vd[0], st.k_pool, st.v_pool, st.table, cu,
                    st.start, st.out[0], st.max_chunk)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    # the pool still works afterwards
    run(st, pool)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK


def test_host_argument_errors():
    st = State(CASES["one-token"]())
    pool = pkv.pkv_pool_create(1, st.wl.num_pages, 1)
    for kwargs in ({"max_chunk_tokens": 0}, {"max_chunk_tokens": 4096}):
        with pytest.raises(pkv.PkvError):
            pkv.pkv_prefill(pool, 0, st.qd[0], st.kd[0], st.vd[0], st.k_pool, st.v_pool,
                            st.table, st.cu, st.start, st.out[0], **kwargs)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_prefill(pool, 1, st.qd[0], st.kd[0], st.vd[0], st.k_pool, st.v_pool, st.table,
                        st.cu, st.start, st.out[0], 1)
    odd = torch.empty(st.out[0].numel() + 1, device="cuda")[1:].view(st.out[0].shape)
    with pytest.raises(pkv.PkvError):
        pkv.pkv_prefill(pool, 0, st.qd[0], st.kd[0], st.vd[0], st.k_pool, st.v_pool, st.table,
                        st.cu, st.start, odd, 1)


def test_late_large_scores_rescale_o():
    """Key rows at positions 200..215 and 700..703 scaled by 16 (exact in
    BF16): every later query's row max jumps by far more than the kernel's
    2^8 lazy threshold several steps into the key range, so O is rescaled in
    tensor memory mid-sequence; the result must still match the oracle."""
    wl = W.prefill([900, 257], [0, 150], num_layers=1, seed=708, name="rescale")
    st = State(wl)
    k = st.k.clone()
    cu = wl.cu_tokens
    for b in range(wl.batch):
        for pos in list(range(200, 216)) + list(range(700, 704)):
            i = pos - int(wl.start_pos[b])
            if 0 <= i < int(wl.chunk_lens[b]):
                k[0, cu[b] + i] = k[0, cu[b] + i] * 16
    st.k, st.kd = k, k.cuda()
    pool = pkv.pkv_pool_create(1, wl.num_pages, wl.batch)
    run(st, pool)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, ok, ov = oracle_prefill(st)
    assert np.array_equal(bits(st.k_pool.cpu()), ok)
    assert_close(st.out.cpu().numpy(), ref, "late large scores")
