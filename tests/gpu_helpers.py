"""Shared plumbing for the GPU parity tests: device copies of a workload,
oracle runs on host copies, and the tolerance gate.

Tolerance (float outputs, FP32 from BF16 inputs, against the FP64 oracle):
max |d| <= 5e-4 over all elements and, per (sequence, query head) row,
max_d |d| / max_d |ref| <= 1e-3. Pools after an append: bit-exact.
"""

import numpy as np
import torch

import oracle
import workloads as W

ATOL = 5e-4
ROW_RTOL = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16).copy()


def assert_close(got, ref, what=""):
    got = np.asarray(got, np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    row = err.max(axis=-1) / np.maximum(np.abs(ref).max(axis=-1), 1e-30)
    assert err.max() <= ATOL, f"{what}: max|d| {err.max():.3e}"
    assert row.max() <= ROW_RTOL, f"{what}: row-normwise rel {row.max():.3e}"
    return float(err.max()), float(row.max())


class DeviceState:
    """A workload's inputs resident on the GPU (and the host state the oracle needs)."""

    def __init__(self, wl: W.Workload, device="cuda", fill="nan", host_pools=True):
        self.wl = wl
        self.device = device
        gen_dev = "cpu" if host_pools else device
        kp, vp = wl.pools(gen_dev, fill)
        self.k_pool = kp.to(device)
        self.v_pool = vp.to(device)
        self.host_k = bits(kp) if host_pools else None
        self.host_v = bits(vp) if host_pools else None
        self.q = wl.q(gen_dev).to(device)
        self.k_new = wl.k_new(gen_dev).to(device)
        self.v_new = wl.v_new(gen_dev).to(device)
        self.table = torch.from_numpy(wl.block_tables).to(device)
        self.lens = torch.from_numpy(wl.seq_lens).to(device)
        self.positions = torch.from_numpy(wl.positions).to(device)
        self.out = torch.full((wl.num_layers, wl.batch, W.NUM_Q_HEADS, W.HEAD_DIM),
                              float("nan"), device=device)


def oracle_step(wl, host_k, host_v, q_bits, kn_bits, vn_bits, layers=None, threads=8,
                table=None, lens=None, rope=None):
    """Oracle append then attention for each layer, on (copies of) host pools.
    rope = (cos, sin) FP32 tables: the key and the queries are rotated to
    their position first. Returns (out [len(layers)][B][32][64], pool_k,
    pool_v after the appends)."""
    orc = oracle.load()
    table = wl.block_tables if table is None else table
    lens = wl.seq_lens if lens is None else lens
    layers = range(wl.num_layers) if layers is None else layers
    num_pages = host_k.shape[0]
    g = oracle.geometry(wl.num_layers, num_pages, lens.shape[0])
    kp, vp = host_k.copy(), host_v.copy()
    outs = []
    positions = (lens - 1).astype(np.int32)
    for layer in layers:
        if rope is None:
            st = orc.append(g, layer, kn_bits[layer].copy(), vn_bits[layer].copy(), kp, vp,
                            table, positions)
            assert st == oracle.OK, st
            st, out = orc.decode_attention_mt(g, layer, q_bits[layer].copy(), kp, vp, table,
                                              lens, threads)
        else:
            st = orc.append_rope(g, layer, kn_bits[layer].copy(), vn_bits[layer].copy(), kp, vp,
                                 table, positions, rope[0], rope[1])
            assert st == oracle.OK, st
            st, q64 = orc.rope_queries(q_bits[layer].copy(), positions, rope[0], rope[1])
            assert st == oracle.OK, st
            st, out = orc.decode_attention_q64(g, layer, q64, kp, vp, table, lens)
        assert st == oracle.OK, st
        outs.append(out)
    return np.stack(outs), kp, vp


def compact_sample(wl, sample, k_pool_dev, v_pool_dev):
    """Host copy of just the pages the sampled sequences use (all layers), with
    their block tables renumbered into the compact pool. Copies the state as it
    is now, so call it before any kernel writes the pool."""
    sample = np.asarray(sample)
    tab = wl.block_tables[:, sample, :]
    used = np.unique(tab[tab >= 0])
    remap = np.full(wl.num_pages, -1, np.int64)
    remap[used] = np.arange(used.size)
    new_tab = np.where(tab >= 0, remap[np.maximum(tab, 0)], -1).astype(np.int32)
    idx = torch.from_numpy(used.astype(np.int64)).to(k_pool_dev.device)
    hk = bits(k_pool_dev.index_select(0, idx))
    hv = bits(v_pool_dev.index_select(0, idx))
    return np.ascontiguousarray(new_tab), hk, hv
