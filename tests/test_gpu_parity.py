"""CUDA path against the CPU oracle, through the C ABI (needs a GPU).

Append and pool state: bit-exact. Attention output (FP32 from BF16 inputs):
max |d| <= 5e-4 and row-normwise relative error <= 1e-3 against FP64.
Unused slots and pages hold BF16 NaN sentinels, so any stray read shows up.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_210_gb300 as pkv
import workloads as W
from gpu_helpers import DeviceState, assert_close, bits, compact_sample, oracle_step

pytestmark = pytest.mark.gpu

EDGE_LENGTHS = [1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 1000, 2047, 2048]


@pytest.fixture(scope="module", autouse=True)
def _library():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_210_gb300 import build
    build.build()
    pkv.load()


def _pool(wl, max_splits=0, flags=0):
    return pkv.pkv_pool_create(wl.num_layers, wl.num_pages, wl.batch, max_splits=max_splits,
                               flags=flags)


def _host_inputs(st):
    return bits(st.q.cpu()), bits(st.k_new.cpu()), bits(st.v_new.cpu())


WORKLOADS = {
    "tiny": lambda: W.tiny(False),
    "tiny-b": lambda: W.tiny(True),
    "edges": lambda: W.custom(EDGE_LENGTHS, num_layers=2, seed=301, name="edges"),
    "edges-holes": lambda: W.custom(EDGE_LENGTHS[::-1], num_layers=3, seed=302, hole_every=3,
                                    name="edges-holes"),
}


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_append_bit_exact(name):
    wl = WORKLOADS[name]()
    st = DeviceState(wl)
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        pkv.pkv_append(pool, layer, st.k_new[layer], st.v_new[layer], st.k_pool, st.v_pool,
                       st.table, st.positions)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    q_b, kn_b, vn_b = _host_inputs(st)
    _, ok, ov = oracle_step(wl, st.host_k, st.host_v, q_b, kn_b, vn_b)
    assert np.array_equal(bits(st.k_pool), ok)
    assert np.array_equal(bits(st.v_pool), ov)


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("splits", [1, 2, 3, 0])
def test_append_then_decode_matches_oracle(name, splits):
    wl = WORKLOADS[name]()
    st = DeviceState(wl)
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        pkv.pkv_append(pool, layer, st.k_new[layer], st.v_new[layer], st.k_pool, st.v_pool,
                       st.table, st.positions)
        pkv.pkv_decode_attention(pool, layer, st.q[layer], st.k_pool, st.v_pool, st.table,
                                 st.lens, st.out[layer], num_splits=splits)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, _, _ = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    assert_close(st.out.cpu().numpy(), ref, f"{name} S={splits}")


@pytest.mark.parametrize("name", list(WORKLOADS))
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_fused_append_attend_matches_oracle(name, splits):
    wl = WORKLOADS[name]()
    st = DeviceState(wl)
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                              st.k_pool, st.v_pool, st.table, st.lens, st.out[layer],
                              num_splits=splits)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    assert np.array_equal(bits(st.k_pool), ok) and np.array_equal(bits(st.v_pool), ov)
    assert_close(st.out.cpu().numpy(), ref, f"{name} fused S={splits}")


@pytest.mark.parametrize("batch", [1, 4])
def test_split_counts_against_unsplit_oracle(batch):
    wl = W.custom([2048] * batch, num_layers=2, seed=303 + batch, name="long")
    st = DeviceState(wl)
    q_b, kn_b, vn_b = _host_inputs(st)
    ref, _, _ = oracle_step(wl, st.host_k, st.host_v, q_b, kn_b, vn_b)
    results = {}
    for splits in (1, 2, 3, 4, 5, 8, 16, 32, 64, 128, 0):
        pool = _pool(wl, max_splits=128)
        k0, v0 = st.k_pool.clone(), st.v_pool.clone()
        out = torch.full_like(st.out, float("nan"))
        for layer in range(wl.num_layers):
            pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                                  k0, v0, st.table, st.lens, out[layer], num_splits=splits)
        assert pkv.pkv_get_error(pool) == pkv.PKV_OK
        results[splits] = out.cpu().numpy()
        assert_close(results[splits], ref, f"B={batch} S={splits}")
    # S = 1 and S = 32 agree to within rounding
    assert np.abs(results[1] - results[32]).max() <= 2 * 5e-4


@pytest.mark.parametrize("batch", [5, 8, 16, 32])
def test_library_cluster_plans_match_oracle(batch):
    """Batches whose library plan is the wide cluster shape (2 page stages, 4
    blocks per SM; S = 8 for 5..8 sequences, 4 for 16, 2 for 32), with
    mixed lengths, fused and unfused, against the unsplit oracle."""
    rng = np.random.default_rng(310 + batch)
    lens = rng.integers(1, 2049, batch)
    lens[0] = 2048
    wl = W.custom(list(lens), num_layers=2, seed=310 + batch, name=f"wide-b{batch}")
    st = DeviceState(wl)
    q_b, kn_b, vn_b = _host_inputs(st)
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, q_b, kn_b, vn_b)
    for fused in (True, False):
        pool = _pool(wl)
        k0, v0 = st.k_pool.clone(), st.v_pool.clone()
        out = torch.full_like(st.out, float("nan"))
        for layer in range(wl.num_layers):
            if fused:
                pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                                      k0, v0, st.table, st.lens, out[layer])
            else:
                pkv.pkv_append(pool, layer, st.k_new[layer], st.v_new[layer], k0, v0, st.table,
                               st.positions)
                pkv.pkv_decode_attention(pool, layer, st.q[layer], k0, v0, st.table, st.lens,
                                         out[layer])
        assert pkv.pkv_get_error(pool) == pkv.PKV_OK
        assert np.array_equal(bits(k0), ok) and np.array_equal(bits(v0), ov)
        assert_close(out.cpu().numpy(), ref, f"B={batch} fused={fused}")


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("graph", [False, True])
def test_programmatic_dependent_launch_chain_matches_oracle(fused, graph):
    """Layers launched back to back with programmatic dependent launch (each
    launch may start before the previous one ends): the unfused chain
    alternates append and decode, so decode must not prefetch the page the
    preceding append writes."""
    wl = W.custom([1, 16, 17, 300, 2047, 2048, 2048, 40], num_layers=4, seed=320,
                  name="pdl-chain")
    st = DeviceState(wl)
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    for splits in (0, 4, 32):
        pool = _pool(wl, flags=pkv.PKV_FLAG_PDL)
        kp, vp = st.k_pool.clone(), st.v_pool.clone()
        out = torch.full_like(st.out, float("nan"))

        def chain():
            for layer in range(wl.num_layers):
                if fused:
                    pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer],
                                          st.v_new[layer], kp, vp, st.table, st.lens, out[layer],
                                          num_splits=splits)
                else:
                    pkv.pkv_append(pool, layer, st.k_new[layer], st.v_new[layer], kp, vp,
                                   st.table, st.positions)
                    pkv.pkv_decode_attention(pool, layer, st.q[layer], kp, vp, st.table, st.lens,
                                             out[layer], num_splits=splits)

        if graph:
            s = torch.cuda.Stream()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                chain()
            g.replay()
            torch.cuda.synchronize()
        else:
            chain()
        assert pkv.pkv_get_error(pool) == pkv.PKV_OK
        assert np.array_equal(bits(kp), ok) and np.array_equal(bits(vp), ov)
        assert_close(out.cpu().numpy(), ref, f"pdl fused={fused} graph={graph} S={splits}")


@pytest.mark.parametrize("layers,first_lens", [
    (2, [1, 15, 16, 31, 200, 2040]),                      # a cluster-merge plan
    (3, [1, 15, 16, 17, 33, 100, 300, 511, 1000, 2040] * 4),   # 40 sequences: ticket merge
])
def test_consecutive_decode_steps_under_pdl_match_oracle(layers, first_lens):
    """Several decode steps of a 2- or 3-layer model, every layer's fused
    launch chained to the one before by programmatic dependent launch inside
    one CUDA graph. Step s appends each sequence's token at position
    first_len + s - 1 and attends first_len + s tokens, so the launch of a
    layer at step s + 1 reads, before its wait, the row that the same layer's
    launch of step s wrote a few launches earlier; a launch must not run
    ahead of those writes. Rows that no step has written yet hold NaN."""
    steps = 5
    first = np.asarray(first_lens, np.int32)
    final = first + steps - 1
    wl = W.custom(final, num_layers=layers, seed=460 + layers, name="pdl-steps")
    kp_h, vp_h = (bits(p) for p in wl.pools("cpu", "nan"))
    nan = np.uint16(W.BF16_NAN_BITS)
    for layer in range(layers):
        for b in range(wl.batch):
            for p in range(int(first[b]) - 1, int(final[b])):
                page = wl.block_tables[layer, b, p // 16]
                kp_h[page, :, p % 16, :] = nan
                vp_h[page, :, p % 16, :] = nan
    gen = torch.Generator().manual_seed(470 + layers)

    def draws(shape):
        return torch.randn(shape, generator=gen).to(torch.bfloat16)

    q = [draws((layers, wl.batch, 32, 64)) for _ in range(steps)]
    kn = [draws((layers, wl.batch, 8, 64)) for _ in range(steps)]
    vn = [draws((layers, wl.batch, 8, 64)) for _ in range(steps)]
    lens = [torch.from_numpy(first + s) for s in range(steps)]

    # oracle: the steps in order on host copies of the pools
    refs = []
    ok, ov = kp_h.copy(), vp_h.copy()
    for s in range(steps):
        ref, ok, ov = oracle_step(wl, ok, ov, bits(q[s]), bits(kn[s]), bits(vn[s]),
                                  lens=(first + s).astype(np.int32))
        refs.append(ref)

    dev = "cuda"
    table = torch.from_numpy(wl.block_tables).to(dev)
    q_d = [x.to(dev) for x in q]
    kn_d = [x.to(dev) for x in kn]
    vn_d = [x.to(dev) for x in vn]
    lens_d = [x.to(dev) for x in lens]
    for splits in (0, 32):
        pool = _pool(wl, flags=pkv.PKV_FLAG_PDL)
        kp = torch.from_numpy(kp_h.view(np.int16)).view(torch.bfloat16).to(dev)
        vp = torch.from_numpy(vp_h.view(np.int16)).view(torch.bfloat16).to(dev)
        out = [torch.full((layers, wl.batch, 32, 64), float("nan"), device=dev)
               for _ in range(steps)]
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for step in range(steps):
                for layer in range(layers):
                    pkv.pkv_append_attend(pool, layer, q_d[step][layer], kn_d[step][layer],
                                          vn_d[step][layer], kp, vp, table, lens_d[step],
                                          out[step][layer], num_splits=splits,
                                          stream=torch.cuda.current_stream())
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert pkv.pkv_get_error(pool) == pkv.PKV_OK
        assert np.array_equal(bits(kp), ok) and np.array_equal(bits(vp), ov)
        for step in range(steps):
            assert_close(out[step].cpu().numpy(), refs[step], f"step {step} S={splits}")


@pytest.mark.parametrize("fused", [True, False])
@pytest.mark.parametrize("pdl", [False, True])
def test_many_sequences_chain_matches_oracle(fused, pdl):
    """A batch too large for a cluster split (the library then picks page
    ranges merged by ticket): 42 ragged sequences (every edge length three
    times) over a fragmented pool, 3 layers, launched back to back (inside a
    CUDA graph with programmatic dependent launch)."""
    wl = W.custom(EDGE_LENGTHS * 3, num_layers=3, seed=330, hole_every=3, name="many")
    st = DeviceState(wl)
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    pool = _pool(wl, flags=pkv.PKV_FLAG_PDL if pdl else 0)
    out = torch.full_like(st.out, float("nan"))

    def chain():
        for layer in range(wl.num_layers):
            if fused:
                pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                                      st.k_pool, st.v_pool, st.table, st.lens, out[layer])
            else:
                pkv.pkv_append(pool, layer, st.k_new[layer], st.v_new[layer], st.k_pool,
                               st.v_pool, st.table, st.positions)
                pkv.pkv_decode_attention(pool, layer, st.q[layer], st.k_pool, st.v_pool,
                                         st.table, st.lens, out[layer])

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
    got = out.cpu().numpy()
    assert_close(got, ref, f"many fused={fused} pdl={pdl}")
    if pdl:   # a second replay: the tickets were reset by the first
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert pkv.pkv_get_error(pool) == pkv.PKV_OK
        assert_close(out.cpu().numpy(), ref, "second replay")


def test_output_independent_of_physical_pages():
    """The same logical cache under two page permutations gives bit-identical
    output for a fixed split plan."""
    lens = [1, 17, 40, 300, 2048]
    a = W.custom(lens, num_layers=1, seed=310, name="perm-a")
    b = W.custom(lens, num_layers=1, seed=311, num_pages=a.num_pages + 40, name="perm-b")
    sa = DeviceState(a, fill="nan")
    # rebuild b's pools holding a's logical contents at b's physical pages
    kb = torch.full((b.num_pages, 8, 16, 64), float("nan"), dtype=torch.bfloat16)
    vb = kb.clone()
    ka, va = sa.k_pool.cpu(), sa.v_pool.cpu()
    for seq, n in enumerate(lens):
        for lp in range(-(-n // 16)):
            kb[b.block_tables[0, seq, lp]] = ka[a.block_tables[0, seq, lp]]
            vb[b.block_tables[0, seq, lp]] = va[a.block_tables[0, seq, lp]]
    kb, vb = kb.cuda(), vb.cuda()
    tb = torch.from_numpy(b.block_tables).cuda()
    for splits in (1, 4, 0):
        pool_a, pool_b = _pool(a), _pool(b)
        oa = torch.empty((a.batch, 32, 64), device="cuda")
        ob = torch.empty_like(oa)
        pkv.pkv_append_attend(pool_a, 0, sa.q[0], sa.k_new[0], sa.v_new[0], sa.k_pool.clone(),
                              sa.v_pool.clone(), sa.table, sa.lens, oa, num_splits=splits)
        pkv.pkv_append_attend(pool_b, 0, sa.q[0], sa.k_new[0], sa.v_new[0], kb.clone(),
                              vb.clone(), tb, sa.lens, ob, num_splits=splits)
        assert pkv.pkv_get_error(pool_a) == pkv.PKV_OK and pkv.pkv_get_error(pool_b) == pkv.PKV_OK
        assert torch.equal(oa, ob), f"S={splits}"


def test_single_token_returns_v_row_exactly():
    wl = W.custom([1] * 7, num_layers=1, seed=312)
    st = DeviceState(wl)
    pool = _pool(wl)
    out = st.out[0]
    pkv.pkv_append_attend(pool, 0, st.q[0], st.k_new[0], st.v_new[0], st.k_pool, st.v_pool,
                          st.table, st.lens, out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    v = st.v_new[0].float()                       # [B][8][64]
    expect = v.repeat_interleave(4, dim=1)        # query head h reads kv head h // 4
    assert torch.equal(out, expect)


def test_zero_query_gives_mean_of_values():
    lens = [5, 16, 33, 700]
    wl = W.custom(lens, num_layers=1, seed=313)
    st = DeviceState(wl)
    pool = _pool(wl)
    q0 = torch.zeros_like(st.q[0])
    pkv.pkv_append_attend(pool, 0, q0, st.k_new[0], st.v_new[0], st.k_pool, st.v_pool,
                          st.table, st.lens, st.out[0], num_splits=3)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    vp = st.v_pool.cpu().float().numpy()
    for b, n in enumerate(lens):
        t = np.arange(n)
        rows = vp[wl.block_tables[0, b, t // 16], :, t % 16, :]   # [n][8][64]
        mean = rows.astype(np.float64).mean(axis=0).repeat(4, axis=0)
        assert_close(st.out[0, b].cpu().numpy(), mean, f"seq {b}")


def test_device_index_errors_are_flagged_not_faulted():
    wl = W.custom([20, 40], num_layers=1, seed=314)
    st = DeviceState(wl)
    pool = _pool(wl)
    # page id past the pool in sequence 1
    bad = st.table.clone()
    bad[0, 1, 1] = wl.num_pages + 5
    pkv.pkv_decode_attention(pool, 0, st.q[0], st.k_pool, st.v_pool, bad, st.lens, st.out[0])
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    bad[0, 1, 1] = -3
    pkv.pkv_append_attend(pool, 0, st.q[0], st.k_new[0], st.v_new[0], st.k_pool, st.v_pool,
                          bad, st.lens, st.out[0])
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    # positions out of range: nothing is written
    before = st.k_pool.clone()
    for pos in ([2048, 3], [-1, 3], [5, 4096]):
        pkv.pkv_append(pool, 0, st.k_new[0], st.v_new[0], st.k_pool, st.v_pool, st.table,
                       torch.tensor(pos, dtype=torch.int32, device="cuda"))
        assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    # only valid positions were written: compare against a clean append of those
    # seq_len out of range
    for lens in ([0, 40], [20, 2049], [-7, 40]):
        pkv.pkv_decode_attention(pool, 0, st.q[0], st.k_pool, st.v_pool, st.table,
                                 torch.tensor(lens, dtype=torch.int32, device="cuda"), st.out[0])
        assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    # the flag is cleared by reading it, and the context still works
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    pkv.pkv_decode_attention(pool, 0, st.q[0], st.k_pool, st.v_pool, st.table, st.lens,
                             st.out[0])
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    del before


def test_host_argument_errors():
    wl = W.custom([20, 40], num_layers=2, seed=315)
    st = DeviceState(wl)
    pool = _pool(wl, max_splits=8)
    L = pool._lib
    h = pool.handle
    s = torch.cuda.current_stream().cuda_stream
    q, kp, vp, t, n, o = (x.data_ptr() for x in (st.q[0], st.k_pool, st.v_pool, st.table,
                                                st.lens, st.out[0]))
    assert L.pkv_decode_attention(h, 0, None, kp, vp, t, n, o, 2, 0, s) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_decode_attention(h, 0, q + 2, kp, vp, t, n, o, 2, 0, s) == \
        pkv.PKV_ERR_INVALID_ARG                                   # misaligned
    assert L.pkv_decode_attention(h, 2, q, kp, vp, t, n, o, 2, 0, s) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_decode_attention(h, -1, q, kp, vp, t, n, o, 2, 0, s) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_decode_attention(h, 0, q, kp, vp, t, n, o, 3, 0, s) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_decode_attention(h, 0, q, kp, vp, t, n, o, 2, 9, s) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_decode_attention(h, 0, q, kp, vp, t, n, o, 0, 0, s) == pkv.PKV_OK
    assert L.pkv_append(h, 0, None, None, kp, vp, t, n, 2, s) == pkv.PKV_ERR_INVALID_ARG
    assert L.pkv_append_attend(h, 0, q, None, None, kp, vp, t, n, o, 2, 0, s) == \
        pkv.PKV_ERR_INVALID_ARG
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK


# ------------------------------------------------------------ full-size configurations
FULL = {
    "llama-b2-2048": (W.llama_default, None),
    "mix-b64": (W.continuous_mix, [0, 1, 2, 7, 20, 33, 50, 63]),
    "ragged-b256": (W.large_ragged, [0, 1, 2, 3, 4, 5, 100, 200, 255]),
    "long-b1": (lambda: W.long_context(1), None),
    "long-b4": (lambda: W.long_context(4), None),
    "long-b8": (lambda: W.long_context(8), None),              # wide cluster shape, S = 8
    "long-b16": (lambda: W.long_context(16), [0, 3, 7, 8, 12, 15]),   # wide, S = 4
}


@pytest.mark.parametrize("name", list(FULL))
def test_full_size_fused_step_matches_oracle(name):
    """Every layer of the workload through the fused step with the library's
    own split choice (the benchmark's launch configuration); sampled sequences
    (or all, for small batches) compared with the oracle, and the whole pool
    checked against the closed-form append."""
    make, sample = FULL[name]
    wl = make()
    st = DeviceState(wl, host_pools=False)
    sample = list(range(wl.batch)) if sample is None else sample
    table_s, hk, hv = compact_sample(wl, sample, st.k_pool, st.v_pool)
    k_before = st.k_pool.clone()
    v_before = st.v_pool.clone()
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                              st.k_pool, st.v_pool, st.table, st.lens, st.out[layer])
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    # whole pool: exactly the appended rows changed, at the closed-form address
    pos = st.positions.long()
    for layer in range(wl.num_layers):
        pages = st.table[layer].long().gather(1, (pos // 16).unsqueeze(1)).squeeze(1)
        k_before[pages, :, pos % 16, :] = st.k_new[layer]
        v_before[pages, :, pos % 16, :] = st.v_new[layer]
    assert torch.equal(k_before.view(torch.int16), st.k_pool.view(torch.int16))
    assert torch.equal(v_before.view(torch.int16), st.v_pool.view(torch.int16))
    del k_before, v_before
    # sampled sequences against the oracle
    q_b, kn_b, vn_b = (bits(x[:, sample].cpu()) for x in (st.q, st.k_new, st.v_new))
    lens = wl.seq_lens[sample].copy()
    ref, _, _ = oracle_step(wl, hk, hv, q_b, kn_b, vn_b, table=table_s, lens=lens, threads=16)
    got = st.out[:, sample].cpu().numpy()
    assert_close(got, ref, name)


@pytest.mark.parametrize("batch", [1, 4])
@pytest.mark.parametrize("splits", [1, 4, 16, 32])
def test_long_context_split_counts_full_size(batch, splits):
    wl = W.long_context(batch)
    st = DeviceState(wl, host_pools=False)
    sample = list(range(batch))
    table_s, hk, hv = compact_sample(wl, sample, st.k_pool, st.v_pool)
    pool = _pool(wl)
    for layer in range(wl.num_layers):
        pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                              st.k_pool, st.v_pool, st.table, st.lens, st.out[layer],
                              num_splits=splits)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    q_b, kn_b, vn_b = (bits(x.cpu()) for x in (st.q, st.k_new, st.v_new))
    ref, _, _ = oracle_step(wl, hk, hv, q_b, kn_b, vn_b, table=table_s, lens=wl.seq_lens.copy(),
                            threads=16)
    assert_close(st.out.cpu().numpy(), ref, f"B={batch} S={splits}")


def test_longest_first_order_large_batch():
    """A batch of 400 ragged sequences (more than one wave of blocks, so the
    decode launch hands out sequences longest first): every output against
    the oracle; then one invalid length is flagged while the other
    sequences still match."""
    rng = np.random.default_rng(440)
    lens = rng.integers(1, 300, size=400).astype(np.int32)
    lens[:5] = [1, 16, 17, 299, 2]
    wl = W.custom(lens, num_layers=1, seed=441, name="longest-first")
    st = DeviceState(wl)
    pool = _pool(wl)
    pkv.pkv_append_attend(pool, 0, st.q[0], st.k_new[0], st.v_new[0], st.k_pool, st.v_pool,
                          st.table, st.lens, st.out[0])
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    assert np.array_equal(bits(st.k_pool), ok) and np.array_equal(bits(st.v_pool), ov)
    assert_close(st.out.cpu().numpy(), ref, "longest first")
    # an invalid length: flagged, its rows untouched, the others unchanged
    bad = st.lens.clone()
    bad[7] = 0
    out = torch.full_like(st.out[0], float("nan"))
    pkv.pkv_decode_attention(pool, 0, st.q[0], st.k_pool, st.v_pool, st.table, bad, out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    got = out.cpu().numpy()
    assert np.all(np.isnan(got[7]))
    keep = np.ones(wl.batch, bool)
    keep[7] = False
    assert_close(got[keep], ref[0][keep], "others with one invalid length")


@pytest.mark.parametrize("pdl", [False, True])
def test_large_batch_fused_chain_matches_oracle(pdl):
    """The fused step at a large batch (the library's ticket-merge plan,
    sequences handed out longest first): lengths over the whole range,
    page-boundary cases, a fragmented pool, three layers chained (with
    programmatic dependent launch, also replayed from a CUDA graph), against
    the oracle; then one invalid length is flagged and skipped."""
    rng = np.random.default_rng(450)
    lens = rng.integers(1, 2049, size=120).astype(np.int32)
    lens[:8] = [1, 16, 17, 128, 129, 2047, 2048, 8 * 16 + 1]
    wl = W.custom(lens, num_layers=3, seed=451, hole_every=3, name="large-fused")
    st = DeviceState(wl)
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st))
    pool = _pool(wl, flags=pkv.PKV_FLAG_PDL if pdl else 0)
    kp, vp = st.k_pool.clone(), st.v_pool.clone()
    out = torch.full_like(st.out, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())   # the copies above run on the current stream

    def chain(stream):
        for layer in range(wl.num_layers):
            pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer], kp,
                                  vp, st.table, st.lens, out[layer], stream=stream)

    with torch.cuda.stream(s):
        chain(s)
    s.synchronize()
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    assert np.array_equal(bits(kp), ok) and np.array_equal(bits(vp), ov)
    assert_close(out.cpu().numpy(), ref, f"large batch pdl={pdl}")
    if pdl:
        first = out.clone()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            chain(torch.cuda.current_stream())
        for _ in range(2):
            out.fill_(float("nan"))
            with torch.cuda.stream(s):
                graph.replay()
            s.synchronize()
            assert torch.equal(out.view(torch.int32), first.view(torch.int32))
        assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    bad = st.lens.clone()
    bad[9] = 0
    out2 = torch.full_like(st.out[0], float("nan"))
    kp2, vp2 = kp.clone(), vp.clone()
    pkv.pkv_append_attend(pool, 0, st.q[0], st.k_new[0], st.v_new[0], kp2, vp2, st.table, bad,
                          out2)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    got = out2.cpu().numpy()
    assert np.all(np.isnan(got[9]))
    keep = np.ones(wl.batch, bool)
    keep[9] = False
    assert_close(got[keep], ref[0][keep], "large batch, one invalid length")


# ------------------------------------------------------------ large-batch plans
@pytest.mark.parametrize("case", ["mix", "equal-lengths", "2048-short", "units-near-bound",
                                  "one-long", "ranges-just-past"])
@pytest.mark.parametrize("fused", [True, False])
def test_large_batch_plans_match_oracle(case, fused):
    """Batches the library splits into page ranges merged by ticket and hands
    out longest sequence first, ranges sized to the batch's pages: a
    log-uniform length mix with page-boundary lengths, many sequences of
    equal length (ranks among equals), 2048 short sequences, 43 sequences of
    17 pages beside one of one page (16-page ranges: 87 units, three short
    of the grid's batch + range_div on a 152-SM device), one 2048-token
    sequence beside 63 one-token ones (eight 16-page ranges), and 44
    sequences of 25 pages (1100 pages: 24-page ranges on a 152-SM device,
    so every sequence ends in a one-page range); two layers chained with programmatic dependent
    launch in a CUDA graph, replayed twice (the tickets must come back to
    zero), against the oracle."""
    rng = np.random.default_rng(480)
    if case == "mix":
        lens = np.clip(np.round(np.exp(rng.uniform(np.log(16), np.log(2048), 72))), 1, 2048)
        lens[:8] = [1, 16, 17, 512, 513, 2047, 2048, 33]
    elif case == "equal-lengths":
        lens = np.array([300] * 50 + [16] * 30 + [2048] * 5 + [1] * 10)
    elif case == "units-near-bound":
        lens = np.array([16 * 17] * 43 + [16])
    elif case == "one-long":
        lens = np.array([2048] + [1] * 63)
    elif case == "ranges-just-past":
        lens = np.array([16 * 24 + 1] * 44)
    else:
        lens = rng.integers(1, 40, 2048)
    wl = W.custom(lens.astype(np.int32), num_layers=2, seed=481, hole_every=3, name=case)
    st = DeviceState(wl)
    ref, ok, ov = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st), threads=16)
    pool = _pool(wl, flags=pkv.PKV_FLAG_PDL)
    plan = pkv.pkv_plan_decode(pkv.pkv_pool_device_figures(pool), wl.batch, 0)
    assert plan.cluster == 0 and plan.longest_first == 1
    kp, vp = st.k_pool.clone(), st.v_pool.clone()
    out = torch.full_like(st.out, float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for layer in range(wl.num_layers):
            cs = torch.cuda.current_stream()
            if fused:
                pkv.pkv_append_attend(pool, layer, st.q[layer], st.k_new[layer], st.v_new[layer],
                                      kp, vp, st.table, st.lens, out[layer], stream=cs)
            else:
                pkv.pkv_append(pool, layer, st.k_new[layer], st.v_new[layer], kp, vp, st.table,
                               st.positions, stream=cs)
                pkv.pkv_decode_attention(pool, layer, st.q[layer], kp, vp, st.table, st.lens,
                                         out[layer], stream=cs)
    for replay in range(2):
        out.fill_(float("nan"))
        kp.copy_(st.k_pool)
        vp.copy_(st.v_pool)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert pkv.pkv_get_error(pool) == pkv.PKV_OK
        assert np.array_equal(bits(kp), ok) and np.array_equal(bits(vp), ov)
        assert_close(out.cpu().numpy(), ref, f"{case} fused={fused} replay {replay}")


def test_large_batch_launch_flags_bad_data_and_recovers():
    """Invalid lengths are flagged and their rows left untouched; a page id
    out of range is flagged and skipped; the next launch on the same handle
    is correct (the tickets were reset)."""
    rng = np.random.default_rng(490)
    lens = rng.integers(1, 2049, 100).astype(np.int32)
    wl = W.custom(lens, num_layers=1, seed=491, name="large-batch-errors")
    st = DeviceState(wl)
    ref, _, _ = oracle_step(wl, st.host_k, st.host_v, *_host_inputs(st), threads=16)
    pool = _pool(wl)
    kp, vp = st.k_pool.clone(), st.v_pool.clone()
    bad_lens = st.lens.clone()
    bad_lens[3] = 0
    bad_lens[50] = 4096
    out = torch.full_like(st.out[0], float("nan"))
    pkv.pkv_append_attend(pool, 0, st.q[0], st.k_new[0], st.v_new[0], kp, vp, st.table,
                          bad_lens, out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    got = out.cpu().numpy()
    assert np.all(np.isnan(got[3])) and np.all(np.isnan(got[50]))
    keep = np.ones(wl.batch, bool)
    keep[[3, 50]] = False
    assert_close(got[keep], ref[0][keep], "others beside invalid lengths")
    bad_table = st.table.clone()
    bad_table[0, 7, 0] = wl.num_pages + 3
    pkv.pkv_decode_attention(pool, 0, st.q[0], kp, vp, bad_table, st.lens, out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_ERR_OUT_OF_RANGE
    # a clean launch afterwards
    kp, vp = st.k_pool.clone(), st.v_pool.clone()
    out.fill_(float("nan"))
    pkv.pkv_append_attend(pool, 0, st.q[0], st.k_new[0], st.v_new[0], kp, vp, st.table, st.lens,
                          out)
    assert pkv.pkv_get_error(pool) == pkv.PKV_OK
    assert_close(out.cpu().numpy(), ref[0], "after the flagged launches")
