"""Checks that tie the CPU oracle to facts outside itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with a fact fixed by the samir-vllm pages or by
mathematics: hand-derived closed forms (tests/golden), the single-token and
zero-query special cases, normalisation of the softmax weights, a dominant
key, invariance of the paged result under page permutations (against a
contiguous-cache statement), a library routine (torch's scaled dot-product
attention in float64 on the CPU), the split/merge algebra, and the closed-form
address of the decode-time append. The same functions run against builds of
the oracle with planted mistakes, each of which must fail at least one pin.
"""

import json
import math
import os

import numpy as np
import torch

import oracle as oracle_pkg
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HQ, HKV, D, P = W.NUM_Q_HEADS, W.NUM_KV_HEADS, W.HEAD_DIM, W.PAGE_SIZE


# ---------------------------------------------------------------- helpers
def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> uint16 bit patterns (numpy)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bits(x: np.ndarray) -> np.ndarray:
    """Exact for values representable in BF16 (used for hand-built cases only)."""
    f = np.asarray(x, np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not exact in BF16"
    return (b >> 16).astype(np.uint16)


def normal_bits(rng, shape, scale=1.0):
    x = (rng.standard_normal(shape) * scale).astype(np.float32)
    return bits(torch.from_numpy(x).to(torch.bfloat16))


def scatter_tokens(k_tokens, v_tokens, pages, num_pages, fill=W.BF16_NAN_BITS):
    """Pools [num_pages][Hkv][P][D] holding token t of a contiguous cache
    [len][Hkv][D] at page pages[t // P], slot t % P (the test's own statement
    of the layout); every other slot holds `fill`."""
    k_pool = np.full((num_pages, HKV, P, D), fill, np.uint16)
    v_pool = np.full_like(k_pool, fill)
    n = k_tokens.shape[0]
    t = np.arange(n)
    k_pool[np.asarray(pages)[t // P], :, t % P, :] = k_tokens
    v_pool[np.asarray(pages)[t // P], :, t % P, :] = v_tokens
    return k_pool, v_pool


def one_sequence(orc, q, k_pool, v_pool, pages, seq_len, num_pages):
    g = oracle_pkg.geometry(1, num_pages, 1)
    table = np.full((1, 1, W.MAX_PAGES_PER_SEQ), -1, np.int32)
    table[0, 0, :len(pages)] = pages
    st, out, lse, wsum = orc.decode_attention(g, 0, q.reshape(1, HQ, D).copy(), k_pool, v_pool,
                                              table, np.array([seq_len], np.int32))
    assert st == oracle_pkg.OK, f"status {st}"
    return out[0], lse[0], wsum[0]


def tiny_state(alt=False):
    """Tiny workload with the new tokens already appended (by the test's own
    numpy scatter), as uint16 arrays."""
    wl = W.tiny(alt)
    kp, vp = (bits(p) for p in wl.pools("cpu", "nan"))
    q, kn, vn = bits(wl.q()), bits(wl.k_new()), bits(wl.v_new())
    pos = wl.positions
    for b in range(wl.batch):
        page = wl.block_tables[0, b, pos[b] // P]
        kp[page, :, pos[b] % P, :] = kn[0, b]
        vp[page, :, pos[b] % P, :] = vn[0, b]
    return wl, q, kp, vp


def gather(table_row, seq_len, pool):
    """[len][Hkv][D] rows of one sequence, walked through its block table."""
    t = np.arange(seq_len)
    return pool[table_row[t // P], :, t % P, :]


def sdpa_reference(q_bits, k_rows_bits, v_rows_bits):
    """torch float64 scaled_dot_product_attention, GQA expanded by
    repeat_interleave (query head h reads KV head h // 4)."""
    group = HQ // HKV
    qf = torch.from_numpy(bits_to_f64(q_bits)).reshape(1, HQ, 1, D)
    k = torch.from_numpy(bits_to_f64(k_rows_bits)).permute(1, 0, 2)  # [Hkv][L][D]
    v = torch.from_numpy(bits_to_f64(v_rows_bits)).permute(1, 0, 2)
    k = k.repeat_interleave(group, dim=0).unsqueeze(0)
    v = v.repeat_interleave(group, dim=0).unsqueeze(0)
    out = torch.nn.functional.scaled_dot_product_attention(qf, k, v)
    return out.reshape(HQ, D).numpy()


# ---------------------------------------------------------------- pins
def pin_golden_closed_form(orc):
    with open(os.path.join(GOLDEN, "two_token_closed_form.json")) as f:
        spec = json.load(f)
    env = {"e": math.e}
    for case in spec["cases"]:
        k = np.zeros((case["num_pages"], HKV, P, D), np.float64)
        v = np.zeros_like(k)
        kv = case["kv_head"]
        for t, row in case["k_rows"].items():
            for d, x in row.items():
                t_ = int(t)
                k[case["block_table"][t_ // P], kv, t_ % P, int(d)] = x
        for t, row in case["v_rows"].items():
            for d, x in row.items():
                t_ = int(t)
                v[case["block_table"][t_ // P], kv, t_ % P, int(d)] = x
        q = np.zeros((HQ, D), np.float64)
        for h, row in case["q_heads"].items():
            for d, x in row.items():
                q[int(h), int(d)] = x
        out, lse, _ = one_sequence(orc, f64_to_bits(q), f64_to_bits(k), f64_to_bits(v),
                                   case["block_table"], case["seq_len"], case["num_pages"])
        for e in case["expected"]:
            closed = eval(e["formula"], {"__builtins__": {}}, env)  # formula text -> number
            assert abs(closed - e["value"]) < 1e-15, f"fixture value disagrees with {e}"
            got = out[e["head"], e["dim"]]
            assert abs(got - e["value"]) < 1e-14, f"{case['name']}: {e} got {got}"
        if case["seq_len"] == 2:  # lse of head 5 is log(1 + e), of head 4 is log 2
            assert abs(lse[5] - math.log(1 + math.e)) < 1e-14
            assert abs(lse[4] - math.log(2)) < 1e-14


def pin_pool_geometry_facts(orc):
    with open(os.path.join(GOLDEN, "pool_geometry.json")) as f:
        spec = json.load(f)
    facts, derived = spec["facts"], spec["derived"]
    assert facts["page_size_tokens"]["value"] == P
    assert facts["context_tokens"]["value"] // P == derived["max_pages_per_sequence"]["value"]
    assert W.PAGE_BYTES_KV == derived["bytes_per_page_kv"]["value"]
    assert W.pages_for_pool_mib(facts["default_pool_mib"]["value"]) == \
        derived["pages_in_default_pool"]["value"]
    assert HQ * D == facts["hidden_width"]["value"]
    # two sequences at full context in every layer fill the default pool exactly
    wl = W.llama_default()
    assert wl.num_pages == derived["pages_for_two_full_sequences_all_layers"]["value"]
    assert np.all(wl.block_tables >= 0)
    assert np.unique(wl.block_tables).size == wl.num_pages


def pin_single_token_returns_v_row(orc):
    rng = np.random.default_rng(11)
    q = normal_bits(rng, (HQ, D))
    kt, vt = normal_bits(rng, (1, HKV, D)), normal_bits(rng, (1, HKV, D))
    kp, vp = scatter_tokens(kt, vt, [3], 5)
    out, lse, wsum = one_sequence(orc, q, kp, vp, [3], 1, 5)
    for h in range(HQ):
        assert np.array_equal(out[h], bits_to_f64(vt[0, h // (HQ // HKV)])), f"head {h}"
    assert np.all(wsum == 1.0)


def pin_zero_query_gives_mean_of_v(orc):
    rng = np.random.default_rng(12)
    n = 37
    q = np.zeros((HQ, D), np.uint16)
    kt, vt = normal_bits(rng, (n, HKV, D)), normal_bits(rng, (n, HKV, D))
    pages = [4, 0, 2]
    kp, vp = scatter_tokens(kt, vt, pages, 6)
    out, lse, _ = one_sequence(orc, q, kp, vp, pages, n, 6)
    mean = bits_to_f64(vt).mean(axis=0)  # [Hkv][D]
    for h in range(HQ):
        np.testing.assert_allclose(out[h], mean[h // (HQ // HKV)], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, math.log(n), rtol=0, atol=1e-13)


def pin_weights_sum_to_one(orc):
    wl, q, kp, vp = tiny_state()
    g = oracle_pkg.geometry(1, wl.num_pages, wl.batch)
    st, out, lse, wsum = orc.decode_attention(g, 0, q[0].copy(), kp, vp, wl.block_tables,
                                              wl.seq_lens)
    assert st == oracle_pkg.OK
    assert np.all(np.isfinite(out))
    np.testing.assert_allclose(wsum, 1.0, rtol=0, atol=1e-12)


def pin_dominant_key(orc):
    rng = np.random.default_rng(13)
    n = 29
    q = normal_bits(rng, (HQ, D))
    kt, vt = normal_bits(rng, (n, HKV, D)), normal_bits(rng, (n, HKV, D))
    star = 17
    # key `star` of every KV head points along sign(q) of head 4*kv with
    # magnitude 256: its score exceeds every other by > 1000, so the softmax
    # puts all weight (to double precision) on it for those heads
    qf = bits_to_f64(q)
    for kv in range(HKV):
        kt[star, kv] = f64_to_bits(256.0 * np.sign(qf[kv * (HQ // HKV)]))
    pages = [1, 5]
    kp, vp = scatter_tokens(kt, vt, pages, 7)
    out, _, _ = one_sequence(orc, q, kp, vp, pages, n, 7)
    for kv in range(HKV):
        assert np.array_equal(out[kv * (HQ // HKV)], bits_to_f64(vt[star, kv]))


def pin_paged_equals_contiguous(orc):
    rng = np.random.default_rng(14)
    for n in (1, 15, 16, 17, 40, 128, 300):
        q = normal_bits(rng, (HQ, D))
        kt, vt = normal_bits(rng, (n, HKV, D)), normal_bits(rng, (n, HKV, D))
        st, ref = orc.contiguous_attention(q, kt, vt)
        assert st == oracle_pkg.OK
        need = -(-n // P)
        results = []
        for trial in range(2):
            num_pages = need + 5
            pages = rng.permutation(num_pages)[:need].astype(np.int32)
            kp, vp = scatter_tokens(kt, vt, pages, num_pages)
            out, _, _ = one_sequence(orc, q, kp, vp, pages, n, num_pages)
            results.append(out)
        assert np.array_equal(results[0], ref), f"len {n}"
        assert np.array_equal(results[1], ref), f"len {n}"


def pin_contiguous_matches_sdpa(orc):
    rng = np.random.default_rng(15)
    for n in (1, 33):
        q = normal_bits(rng, (HQ, D))
        kt, vt = normal_bits(rng, (n, HKV, D)), normal_bits(rng, (n, HKV, D))
        st, out = orc.contiguous_attention(q, kt, vt)
        assert st == oracle_pkg.OK
        np.testing.assert_allclose(out, sdpa_reference(q, kt, vt), rtol=0, atol=1e-12)


def pin_paged_matches_sdpa(orc):
    for alt in (False, True):
        wl, q, kp, vp = tiny_state(alt)
        g = oracle_pkg.geometry(1, wl.num_pages, wl.batch)
        st, out, _, _ = orc.decode_attention(g, 0, q[0].copy(), kp, vp, wl.block_tables,
                                             wl.seq_lens)
        assert st == oracle_pkg.OK
        for b in range(wl.batch):
            n = int(wl.seq_lens[b])
            ref = sdpa_reference(q[0, b], gather(wl.block_tables[0, b], n, kp),
                                 gather(wl.block_tables[0, b], n, vp))
            np.testing.assert_allclose(out[b], ref, rtol=0, atol=1e-12)


def pin_split_equals_unsplit(orc):
    lens = [1, 16, 17, 40, 200, 2048]
    wl = W.custom(lens, num_layers=2, seed=217)
    kp, vp = (bits(p) for p in wl.pools("cpu", "zero"))
    q = bits(wl.q())
    g = oracle_pkg.geometry(2, wl.num_pages, wl.batch)
    for layer in (0, 1):
        st, ref, _, _ = orc.decode_attention(g, layer, q[layer].copy(), kp, vp,
                                             wl.block_tables, wl.seq_lens)
        assert st == oracle_pkg.OK
        for S in (1, 2, 4, 16, 32):
            st, out, po, pm, pl = orc.decode_attention_split(g, layer, q[layer].copy(), kp, vp,
                                                            wl.block_tables, wl.seq_lens, S)
            assert st == oracle_pkg.OK
            np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
            # S = 1: the single partial normalised is the answer
            if S == 1:
                np.testing.assert_allclose(po[:, :, 0] / pl[:, :, 0:1], ref, rtol=1e-12,
                                           atol=1e-13)
            # empty splits carry m = -inf, l = 0
            for b, n in enumerate(lens):
                n_pages = -(-n // P)
                chunk = -(-n_pages // S)
                for s in range(S):
                    if s * chunk >= n_pages:
                        assert np.all(pl[b, :, s] == 0) and np.all(np.isneginf(pm[b, :, s]))
                    else:
                        assert np.all(pl[b, :, s] >= 1.0)  # the max term contributes exp(0)


def pin_mt_matches_single_thread(orc):
    wl = W.custom([5, 16, 33, 64, 100, 250, 1], num_layers=1, seed=218)
    kp, vp = (bits(p) for p in wl.pools("cpu", "zero"))
    q = bits(wl.q())
    g = oracle_pkg.geometry(1, wl.num_pages, wl.batch)
    st, ref, _, _ = orc.decode_attention(g, 0, q[0].copy(), kp, vp, wl.block_tables,
                                         wl.seq_lens)
    for nthreads in (1, 3):
        st2, out = orc.decode_attention_mt(g, 0, q[0].copy(), kp, vp, wl.block_tables,
                                           wl.seq_lens, nthreads)
        assert st == st2 == oracle_pkg.OK
        assert np.array_equal(out, ref)


def pin_append_closed_form(orc):
    wl = W.custom([1, 16, 17, 32, 2048, 100], num_layers=3, seed=219)
    kp, vp = (bits(p) for p in wl.pools("cpu", "nan"))
    kn, vn = bits(wl.k_new()), bits(wl.v_new())
    g = oracle_pkg.geometry(3, wl.num_pages, wl.batch)
    pos = wl.positions
    for layer in range(3):
        exp_k, exp_v = kp.copy(), vp.copy()
        for b in range(wl.batch):
            page = wl.block_tables[layer, b, pos[b] // P]
            exp_k[page, :, pos[b] % P, :] = kn[layer, b]
            exp_v[page, :, pos[b] % P, :] = vn[layer, b]
        st = orc.append(g, layer, kn[layer].copy(), vn[layer].copy(), kp, vp, wl.block_tables,
                        pos)
        assert st == oracle_pkg.OK
        assert np.array_equal(kp, exp_k) and np.array_equal(vp, exp_v), f"layer {layer}"


def pin_append_rejects_out_of_range(orc):
    wl = W.custom([20, 20], num_layers=1, seed=220)
    kp, vp = (bits(p) for p in wl.pools("cpu", "zero"))
    before_k, before_v = kp.copy(), vp.copy()
    kn, vn = bits(wl.k_new()), bits(wl.v_new())
    g = oracle_pkg.geometry(1, wl.num_pages, wl.batch)
    table = wl.block_tables.copy()
    table[0, 1, 1] = wl.num_pages  # page id past the pool
    for pos in ([2048, 19], [-1, 19], [19, 19]):
        st = orc.append(g, 0, kn[0].copy(), vn[0].copy(), kp, vp, table,
                        np.array(pos, np.int32))
        assert st == oracle_pkg.OUT_OF_RANGE
        # sequence 1 (bad page) is never written; sequence 0 only when its position is valid
        assert np.array_equal(kp[table[0, 1, 0]], before_k[table[0, 1, 0]])
        if pos[0] < 0 or pos[0] >= 2048:
            assert np.array_equal(kp, before_k) and np.array_equal(vp, before_v)


def _rope_case(seed, n_pos=40):
    rng = np.random.default_rng(seed)
    wl = W.custom([n_pos, 7, 33], num_layers=1, seed=seed)
    kp, vp = (bits(p) for p in wl.pools("cpu", "zero"))
    kn, vn = bits(wl.k_new()), bits(wl.v_new())
    g = oracle_pkg.geometry(1, wl.num_pages, wl.batch)
    return rng, wl, kp, vp, kn, vn, g


def pin_rope_zero_angle_is_identity(orc):
    rng, wl, kp, vp, kn, vn, g = _rope_case(501)
    cos_t = np.ones((W.MAX_SEQ_LEN, D // 2), np.float32)
    sin_t = np.zeros_like(cos_t)
    a_k, a_v = kp.copy(), vp.copy()
    assert orc.append(g, 0, kn[0].copy(), vn[0].copy(), a_k, a_v, wl.block_tables,
                      wl.positions) == oracle_pkg.OK
    assert orc.append_rope(g, 0, kn[0].copy(), vn[0].copy(), kp, vp, wl.block_tables,
                           wl.positions, cos_t, sin_t) == oracle_pkg.OK
    assert np.array_equal(kp, a_k) and np.array_equal(vp, a_v)
    q = normal_bits(rng, (3, HQ, D))
    st, q64 = orc.rope_queries(q, wl.positions, cos_t, sin_t)
    assert st == oracle_pkg.OK and np.array_equal(q64, bits_to_f64(q))


def pin_rope_quarter_turn_swaps_halves(orc):
    """cos = 0, sin = 1: x'[i] = -x[i + D/2] and x'[i + D/2] = x[i], exactly."""
    rng, wl, kp, vp, kn, vn, g = _rope_case(502)
    cos_t = np.zeros((W.MAX_SEQ_LEN, D // 2), np.float32)
    sin_t = np.ones_like(cos_t)
    assert orc.append_rope(g, 0, kn[0].copy(), vn[0].copy(), kp, vp, wl.block_tables,
                           wl.positions, cos_t, sin_t) == oracle_pkg.OK
    half = D // 2
    for b in range(wl.batch):
        pos = int(wl.positions[b])
        got = bits_to_f64(kp[wl.block_tables[0, b, pos // P], :, pos % P, :])
        x = bits_to_f64(kn[0, b])
        np.testing.assert_array_equal(got[:, :half], -x[:, half:])
        np.testing.assert_array_equal(got[:, half:], x[:, :half])
    q = normal_bits(rng, (3, HQ, D))
    st, q64 = orc.rope_queries(q, wl.positions, cos_t, sin_t)
    qf = bits_to_f64(q)
    np.testing.assert_array_equal(q64[..., :half], -qf[..., half:])
    np.testing.assert_array_equal(q64[..., half:], qf[..., :half])


def pin_rope_key_uses_its_own_position(orc):
    """Decode appends each token at its absolute rotary position (samir-vllm:
    Build LLM Inference From Scratch in C++ and CUDA, "Architecture
    walkthrough", KV cache paragraph), so the key takes the angle row of its
    own position and of no other. Tables here hold a quarter turn at each
    sequence's position, a half turn (plain negation) at the rows next to it
    and no rotation anywhere else: the stored key must be the quarter turn,
    exactly, and V must be stored unrotated."""
    _, wl, kp, vp, kn, vn, g = _rope_case(504)
    half = D // 2
    cos_t = np.ones((W.MAX_SEQ_LEN, half), np.float32)
    sin_t = np.zeros_like(cos_t)
    pos = [int(p) for p in wl.positions]
    for p in pos:
        for r in (p - 1, p + 1):
            cos_t[r] = -1.0
    for p in pos:
        cos_t[p], sin_t[p] = 0.0, 1.0
    assert len(set(pos)) == len(pos) and min(pos) >= 1
    assert orc.append_rope(g, 0, kn[0].copy(), vn[0].copy(), kp, vp, wl.block_tables,
                           wl.positions, cos_t, sin_t) == oracle_pkg.OK
    for b, p in enumerate(pos):
        page, slot = wl.block_tables[0, b, p // P], p % P
        got = bits_to_f64(kp[page, :, slot, :])
        x = bits_to_f64(kn[0, b])
        np.testing.assert_array_equal(got[:, :half], -x[:, half:])
        np.testing.assert_array_equal(got[:, half:], x[:, :half])
        np.testing.assert_array_equal(vp[page, :, slot, :], vn[0, b])


def pin_rope_key_within_rounding_of_exact_rotation(orc):
    """At general angles (base 10000, positions spread over the context) the
    stored key is the exact rotation of the BF16 input by the table's FP32
    angles, rounded to BF16: each stored value lies within half a BF16 unit
    in the last place of the exact value, widened only by the FP32 rounding of
    the two products and their sum, 2^-23 (|x c| + |y s|)."""
    _, wl, kp, vp, kn, vn, g = _rope_case(505)
    half = D // 2
    cos_t, sin_t = W.rope_tables(base=10000.0)
    positions = np.array([1999, 517, 3], np.int32)
    table = wl.block_tables.copy()
    for b, p in enumerate(positions.tolist()):        # the pages those positions need
        table[0, b, p // P] = table[0, b, 0]
    assert orc.append_rope(g, 0, kn[0].copy(), vn[0].copy(), kp, vp, table, positions,
                           cos_t, sin_t) == oracle_pkg.OK
    for b, p in enumerate(positions.tolist()):
        got = bits_to_f64(kp[table[0, b, p // P], :, p % P, :])
        x = bits_to_f64(kn[0, b])[:, :half]
        y = bits_to_f64(kn[0, b])[:, half:]
        c = cos_t[p].astype(np.float64)
        s = sin_t[p].astype(np.float64)
        exact = np.concatenate([x * c - y * s, y * c + x * s], axis=1)
        f32_err = 2.0 ** -23 * np.concatenate([np.abs(x * c) + np.abs(y * s),
                                               np.abs(y * c) + np.abs(x * s)], axis=1)
        mag = np.abs(exact) + f32_err
        half_ulp = np.where(mag > 0, 2.0 ** (np.floor(np.log2(np.maximum(mag, 1e-300))) - 8),
                            0.0)
        assert np.all(np.abs(got - exact) <= half_ulp + f32_err), (b, p)
        # and the rotation is not the identity at these angles
        assert np.any(got != bits_to_f64(kn[0, b]))


def pin_rope_keeps_pair_norms_and_relative_scores(orc):
    """A rotation keeps |(x_i, x_{i+D/2})|, and q_p . k_t depends on p - t only."""
    rng = np.random.default_rng(503)
    cos_t, sin_t = W.rope_tables(base=10000.0)
    half = D // 2
    q = normal_bits(rng, (1, HQ, D))
    k = normal_bits(rng, (1, HQ, D))
    def rot(x, p):
        st, r = orc.rope_queries(x, np.array([p], np.int32), cos_t, sin_t)
        assert st == oracle_pkg.OK
        return r[0]
    qf = bits_to_f64(q)[0]
    r = rot(q, 777)
    np.testing.assert_allclose(r[:, :half] ** 2 + r[:, half:] ** 2,
                               qf[:, :half] ** 2 + qf[:, half:] ** 2, rtol=1e-6, atol=1e-9)
    d1 = np.sum(rot(q, 100) * rot(k, 40), axis=-1)
    d2 = np.sum(rot(q, 1100) * rot(k, 1040), axis=-1)
    d0 = np.sum(rot(q, 60) * bits_to_f64(k)[0], axis=-1)
    np.testing.assert_allclose(d1, d2, rtol=0, atol=2e-4)
    np.testing.assert_allclose(d1, d0, rtol=0, atol=2e-4)


# ---------------------------------------------------------------- prefill
def _prefill_state(chunk_lens, start_pos, seed):
    wl = W.prefill(chunk_lens, start_pos, num_layers=1, seed=seed)
    kp, vp = (bits(t) for t in wl.pools("cpu", "nan"))
    return wl, kp, vp, bits(wl.q()[0]), bits(wl.k()[0]), bits(wl.v()[0])


def _prefill_run(orc, wl, kp, vp, q, k, v):
    g = oracle_pkg.geometry(1, wl.num_pages, wl.batch)
    assert orc.prefill_fill(g, 0, k, v, kp, vp, wl.block_tables, wl.cu_tokens,
                            wl.start_pos) == oracle_pkg.OK
    st, out = orc.prefill_attention(g, 0, q, kp, vp, wl.block_tables, wl.cu_tokens,
                                    wl.start_pos, threads=3)
    assert st == oracle_pkg.OK
    return out


def pin_prefill_matches_causal_sdpa(orc):
    """Against torch float64 scaled_dot_product_attention with a causal mask
    offset by the chunk's start, on K/V gathered by the test's own reading of
    the layout (GQA expanded); chunks starting at 0 and mid-prompt."""
    chunk, start = [20, 37, 9], [0, 5, 30]
    wl, kp, vp, q, k, v = _prefill_state(chunk, start, 601)
    before_k = kp.copy()
    out = _prefill_run(orc, wl, kp, vp, q, k, v)
    cu = wl.cu_tokens
    for b in range(wl.batch):
        n, s0 = int(chunk[b]), int(start[b])
        L = s0 + n
        rows = wl.block_tables[0, b]
        t = np.arange(L)
        kk = bits_to_f64(kp[rows[t // P], :, t % P, :])      # [L][Hkv][D]
        vv = bits_to_f64(vp[rows[t // P], :, t % P, :])
        # the chunk's rows come from k/v, the earlier ones were already cached
        np.testing.assert_array_equal(kp[rows[t[s0:] // P], :, t[s0:] % P, :],
                                      k[cu[b]:cu[b + 1]])
        np.testing.assert_array_equal(kp[rows[t[:s0] // P], :, t[:s0] % P, :],
                                      before_k[rows[t[:s0] // P], :, t[:s0] % P, :])
        qq = torch.from_numpy(bits_to_f64(q[cu[b]:cu[b + 1]])).permute(1, 0, 2)   # [Hq][n][D]
        kt = torch.from_numpy(kk).permute(1, 0, 2).repeat_interleave(HQ // HKV, dim=0)
        vt = torch.from_numpy(vv).permute(1, 0, 2).repeat_interleave(HQ // HKV, dim=0)
        mask = torch.arange(L)[None, :] <= (s0 + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qq, kt, vt, attn_mask=mask)
        np.testing.assert_allclose(out[cu[b]:cu[b + 1]], ref.permute(1, 0, 2).numpy(),
                                   rtol=0, atol=1e-12)


def pin_prefill_first_token_returns_its_v_row(orc):
    wl, kp, vp, q, k, v = _prefill_state([16, 1], [0, 0], 602)
    out = _prefill_run(orc, wl, kp, vp, q, k, v)
    for b, row in ((0, 0), (1, 16)):
        for h in range(HQ):
            np.testing.assert_array_equal(out[row, h], bits_to_f64(v[row, h // (HQ // HKV)]))


def pin_prefill_chunks_compose(orc):
    """Prefilling [0, a) then [a, n) gives the rows of a single [0, n) call,
    bit for bit, and the last token equals decode attention at length n."""
    n, a = 45, 17
    whole, kp, vp, q, k, v = _prefill_state([n], [0], 603)
    out_whole = _prefill_run(orc, whole, kp.copy(), vp.copy(), q, k, v)
    parts = []
    kp2, vp2 = kp.copy(), vp.copy()
    for s0, s1 in ((0, a), (a, n)):
        wl = W.PrefillWorkload("part", 1, whole.num_pages, np.array([s0], np.int32),
                               np.array([s1 - s0], np.int32), whole.block_tables, whole.seed)
        parts.append(_prefill_run(orc, wl, kp2, vp2, q[s0:s1].copy(), k[s0:s1].copy(),
                                  v[s0:s1].copy()))
    np.testing.assert_array_equal(np.concatenate(parts), out_whole)
    g = oracle_pkg.geometry(1, whole.num_pages, 1)
    st, dec, _, _ = orc.decode_attention(g, 0, q[n - 1:n].copy(), kp2, vp2, whole.block_tables,
                                         np.array([n], np.int32))
    assert st == oracle_pkg.OK
    np.testing.assert_array_equal(dec[0], out_whole[n - 1])


def pin_prefill_fill_closed_form(orc):
    """Every chunk row lands at page table[(s + i) // 16], slot (s + i) % 16,
    and nothing else changes; a position past the table is reported."""
    wl, kp, vp, q, k, v = _prefill_state([33, 4], [3, 60], 604)
    kp0, vp0 = kp.copy(), vp.copy()
    g = oracle_pkg.geometry(1, wl.num_pages, wl.batch)
    assert orc.prefill_fill(g, 0, k, v, kp, vp, wl.block_tables, wl.cu_tokens,
                            wl.start_pos) == oracle_pkg.OK
    ek, ev = kp0.copy(), vp0.copy()
    for b in range(wl.batch):
        for i in range(int(wl.chunk_lens[b])):
            pos = int(wl.start_pos[b]) + i
            row = int(wl.cu_tokens[b]) + i
            page = wl.block_tables[0, b, pos // P]
            ek[page, :, pos % P] = k[row]
            ev[page, :, pos % P] = v[row]
    assert np.array_equal(kp, ek) and np.array_equal(vp, ev)
    bad = wl.start_pos.copy()
    bad[1] = 2048 - 2                      # runs past the 128-page table
    assert orc.prefill_fill(g, 0, k, v, kp, vp, wl.block_tables, wl.cu_tokens,
                            bad) == oracle_pkg.OUT_OF_RANGE


ALL_PINS = [pin_golden_closed_form, pin_pool_geometry_facts, pin_single_token_returns_v_row,
            pin_zero_query_gives_mean_of_v, pin_weights_sum_to_one, pin_dominant_key,
            pin_paged_equals_contiguous, pin_contiguous_matches_sdpa, pin_paged_matches_sdpa,
            pin_split_equals_unsplit, pin_mt_matches_single_thread, pin_append_closed_form,
            pin_append_rejects_out_of_range, pin_rope_zero_angle_is_identity,
            pin_rope_quarter_turn_swaps_halves, pin_rope_key_uses_its_own_position,
            pin_rope_key_within_rounding_of_exact_rotation,
            pin_rope_keeps_pair_norms_and_relative_scores,
            pin_prefill_matches_causal_sdpa, pin_prefill_first_token_returns_its_v_row,
            pin_prefill_chunks_compose, pin_prefill_fill_closed_form]
