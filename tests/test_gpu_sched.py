"""Continuous batching driven by the native admission scheduler (needs a
GPU): requests are admitted against their page budgets, their prompts'
K/V are written into the pages the scheduler assigns, and every decode step
runs the fused append-attend launch on the scheduler's block tables. Each
step's output and pool are checked against the oracle on the same tables."""

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


def _bf16_normal(gen, shape):
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(torch.bfloat16)


@pytest.mark.parametrize("static", [False, True])
def test_scheduler_driven_decode_matches_oracle(static):
    layers, num_pages, max_batch = 2, 40, 12
    gen = torch.Generator().manual_seed(4210 + static)
    rng = np.random.default_rng(4210 + static)
    sched = pkv.pkv_sched_create(num_pages, num_layers=layers, static_batching=static)
    orc = oracle.load()
    g = oracle.geometry(layers, num_pages, max_batch)
    k_host = np.full((num_pages, 8, 16, 64), W.BF16_NAN_BITS, np.uint16)
    v_host = k_host.copy()
    k_pool = torch.from_numpy(k_host.view(np.int16)).view(torch.bfloat16).cuda()
    v_pool = torch.from_numpy(v_host.view(np.int16)).view(torch.bfloat16).cuda()
    pool = pkv.pkv_pool_create(layers, num_pages, max_batch)

    # requests: (prompt tokens, max new tokens); budgets of 2..14 pages in a
    # 40-page pool, so admission has to wait and finishing frees room
    specs = [(int(rng.integers(1, 60)), int(rng.integers(2, 40))) for _ in range(12)]
    ids = [pkv.pkv_sched_submit(sched, p, n) for p, n in specs]
    remaining = {rid: n for rid, (p, n) in zip(ids, specs)}
    length = {}
    steps = 0
    while remaining:
        for rid in pkv.pkv_sched_admit(sched):
            p = specs[ids.index(rid)][0]
            # prefill stand-in: the prompt's K/V (positions < p - 1) written
            # into the assigned pages; the decode step appends position p - 1
            pkv.pkv_sched_extend(sched, rid, p)
            tab = pkv.pkv_sched_block_tables(sched, [rid], max_batch=1)
            kv = bits(_bf16_normal(gen, (2, layers, p, 8, 64)))
            for layer in range(layers):
                for t in range(p - 1):
                    page = tab[layer, 0, t // 16]
                    k_host[page, :, t % 16] = kv[0, layer, t]
                    v_host[page, :, t % 16] = kv[1, layer, t]
            length[rid] = p
        k_pool.copy_(torch.from_numpy(k_host.view(np.int16)).view(torch.bfloat16))
        v_pool.copy_(torch.from_numpy(v_host.view(np.int16)).view(torch.bfloat16))
        batch = pkv.pkv_sched_decode_batch(sched)
        assert 0 < len(batch) <= max_batch
        for rid in batch:
            pkv.pkv_sched_extend(sched, rid, length[rid])
        table = pkv.pkv_sched_block_tables(sched, batch, max_batch=max_batch)
        lens = np.array([length[r] for r in batch], np.int32)
        B = len(batch)
        q = _bf16_normal(gen, (layers, B, 32, 64))
        kn = _bf16_normal(gen, (layers, B, 8, 64))
        vn = _bf16_normal(gen, (layers, B, 8, 64))
        out = torch.full((layers, B, 32, 64), float("nan"), device="cuda")
        table_d, lens_d = torch.from_numpy(table).cuda(), torch.from_numpy(lens).cuda()
        qd, knd, vnd = q.cuda(), kn.cuda(), vn.cuda()
        for layer in range(layers):
            pkv.pkv_append_attend(pool, layer, qd[layer], knd[layer], vnd[layer], k_pool, v_pool,
                                  table_d, lens_d, out[layer])
        assert pkv.pkv_get_error(pool) == pkv.PKV_OK
        ref = []
        for layer in range(layers):
            assert orc.append(g, layer, bits(kn[layer]), bits(vn[layer]), k_host, v_host, table,
                              lens - 1) == oracle.OK
            st, o = orc.decode_attention_mt(g, layer, bits(q[layer]), k_host, v_host, table,
                                            lens, 4)
            assert st == oracle.OK
            ref.append(o)
        assert np.array_equal(bits(k_pool.cpu()), k_host)
        assert np.array_equal(bits(v_pool.cpu()), v_host)
        assert_close(out.cpu().numpy(), np.stack(ref), f"step {steps}")
        # one token generated per request; a request ends at its reserved
        # prefix (its last token is returned, not appended) or early
        for rid in batch:
            prefix = pkv.pkv_sched_budget(*specs[ids.index(rid)], num_layers=layers)[1]
            if length[rid] >= prefix or rng.random() < 0.05:
                pkv.pkv_sched_finish(sched, rid)
                del remaining[rid]
            else:
                length[rid] += 1
        steps += 1
        assert steps < 200
    stats = pkv.pkv_sched_get_stats(sched)
    assert stats["finished"] == len(ids) and stats["free_pages"] == num_pages
    assert stats["admission_waits"] > 0 and stats["peak_assigned_pages"] <= num_pages
