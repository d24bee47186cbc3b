"""Seeded synthetic inputs for paged decode attention.

This module only draws inputs: sequence lengths, page assignments (block
tables), and BF16 values for q, the new token's k/v and the cached pool. It
holds none of the attention arithmetic, and both the CUDA path's tests and
the CPU oracle take their inputs from it.

Geometry is that of a Llama-3.2-1B decode step: 16 layers, 32 query heads over
8 KV heads, head_dim 64, 16-token pages, at most 2,048 tokens of context
(128 pages per sequence and layer). Values are BF16, rounded to nearest-even
from FP32 N(0, 1) draws. Pools are laid out [page][kv_head][token][dim], K
and V in separate pools, page ids global over one pool shared by all layers.
Block tables are int32 [layer][batch][128]; entries past a sequence's last
page hold -1.

Cache state before the step: every position < seq_len - 1 holds a value; the
slot at position seq_len - 1 (where the step appends) and every slot or page
that no sequence owns hold the fill value: a BF16 NaN sentinel for parity
runs, so a stray read shows up, or zero for timed runs.

Workloads (seed 210 + index, one sub-stream per quantity):
  1 tiny      1 layer, batch 2, seq_lens {17, 40}, 8-page pool, seeded permutation
  1b          the same with seq_lens {18, 41} (the other reading of the lengths)
  2 llama     16 layers, batch 2 at 2,048, 4,096-page (128 MiB) pool, shuffled
  3 mix       16 layers, batch 64, lengths log-uniform in [16, 2048], 4 GiB pool,
              fragmented free list (every 3rd page of the shuffle held back)
  4 ragged    16 layers, batch 256, lengths uniform in [1, 2048] with
              {1, 16, 32, 2048, 17, 1024} forced first, pool sized to fit, K x 4
  5 long      16 layers, batch 1 or 4 at 2,048, 1 GiB pool, scattered pages

Prefill chunks (PrefillWorkload): for each sequence, a chunk of n_b prompt
tokens at positions start_b .. start_b + n_b - 1, packed token-major into
q [L][T][32][64] and k/v [L][T][8][64] (T = sum n_b, rows cu_tokens[b] ..
cu_tokens[b+1] - 1); positions < start_b are already cached (earlier chunks);
the chunk's own slots hold the fill value until the prefill writes them.
"""

from dataclasses import dataclass, field

import numpy as np
import torch

PAGE_SIZE = 16
NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 64
MAX_SEQ_LEN = 2048
MAX_PAGES_PER_SEQ = MAX_SEQ_LEN // PAGE_SIZE
BASE_SEED = 210
BF16_NAN_BITS = 0x7FC0
# bytes of one page of one layer: 16 tokens x 8 heads x 64 dims x BF16, K and V
PAGE_BYTES_KV = PAGE_SIZE * NUM_KV_HEADS * HEAD_DIM * 2 * 2
MIB = 1 << 20

_STREAMS = {"q": 0, "k_new": 1, "v_new": 2, "k_pool": 3, "v_pool": 4, "lengths": 5,
            "pages": 6}


def pages_for_pool_mib(mib: int) -> int:
    """Number of pages a pool of `mib` MiB holds (K and V together)."""
    return (mib * MIB) // PAGE_BYTES_KV


def rope_tables(max_seq_len=MAX_SEQ_LEN, head_dim=HEAD_DIM, base=500000.0):
    """Rotary angles as FP32 tables (cos, sin) of shape [max_seq_len][head_dim / 2]:
    angle(p, i) = p * base^(-2 i / head_dim), taken in float64 then rounded.
    The base is an input (the pages give neither it nor Llama 3.2's frequency
    scaling); 500000 is the Llama 3 base."""
    half = head_dim // 2
    inv = base ** (-2.0 * np.arange(half, dtype=np.float64) / head_dim)
    ang = np.arange(max_seq_len, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def _rng(seed: int, stream: str) -> np.random.Generator:
    return np.random.default_rng([seed, _STREAMS[stream]])


def assign_pages(seq_lens, num_layers, num_pages, rng, hole_every=0):
    """Block tables from a seeded shuffle of all page ids.

    Pages are handed out one at a time, round-robin over (layer, sequence),
    logical page by logical page, the way a decode loop grows sequences. With
    hole_every = n, every n-th id of the shuffle is held back first, so the
    free list is fragmented.
    """
    seq_lens = np.asarray(seq_lens, np.int64)
    batch = seq_lens.shape[0]
    free = rng.permutation(num_pages).astype(np.int32)
    if hole_every:
        keep = (np.arange(num_pages) % hole_every) != hole_every - 1
        free = free[keep]
    n_pages = (seq_lens + PAGE_SIZE - 1) // PAGE_SIZE
    table = np.full((num_layers, batch, MAX_PAGES_PER_SEQ), -1, np.int32)
    nxt = 0
    for i in range(int(n_pages.max()) if batch else 0):
        growing = np.nonzero(n_pages > i)[0]
        for layer in range(num_layers):
            take = growing.shape[0]
            if nxt + take > free.shape[0]:
                raise ValueError("pool too small for the requested sequences")
            table[layer, growing, i] = free[nxt:nxt + take]
            nxt += take
    return table


def _bf16(x: torch.Tensor) -> torch.Tensor:
    """FP32 -> BF16, round to nearest even (torch's conversion)."""
    return x.to(torch.bfloat16)


@dataclass
class Workload:
    name: str
    num_layers: int
    num_pages: int
    seq_lens: np.ndarray          # int32 [B]: attended length after the append
    block_tables: np.ndarray      # int32 [L][B][128]
    seed: int
    k_scale: float = 1.0
    note: str = ""
    _live: np.ndarray = field(default=None, repr=False)

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def positions(self) -> np.ndarray:
        """Absolute position of the token this step appends."""
        return (self.seq_lens - 1).astype(np.int32)

    def _normal(self, shape, stream, device, scale=1.0):
        gen = torch.Generator(device=device)
        gen.manual_seed(self.seed * 1000 + _STREAMS[stream])
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)  # a power of two: exact, commutes with rounding
        return _bf16(x)

    def q(self, device="cpu") -> torch.Tensor:
        """bf16 [L][B][32][64]."""
        return self._normal((self.num_layers, self.batch, NUM_Q_HEADS, HEAD_DIM), "q", device)

    def k_new(self, device="cpu") -> torch.Tensor:
        """bf16 [L][B][8][64]: the appended token's keys."""
        return self._normal((self.num_layers, self.batch, NUM_KV_HEADS, HEAD_DIM), "k_new",
                            device, self.k_scale)

    def v_new(self, device="cpu") -> torch.Tensor:
        """bf16 [L][B][8][64]: the appended token's values."""
        return self._normal((self.num_layers, self.batch, NUM_KV_HEADS, HEAD_DIM), "v_new",
                            device)

    def live_slots(self) -> np.ndarray:
        """bool [num_pages][16]: slots that hold a cached token before the step."""
        if self._live is None:
            live = np.zeros((self.num_pages, PAGE_SIZE), bool)
            for b in range(self.batch):
                cached = int(self.seq_lens[b]) - 1
                if cached <= 0:
                    continue
                t = np.arange(cached)
                for layer in range(self.num_layers):
                    pages = self.block_tables[layer, b, t // PAGE_SIZE]
                    live[pages, t % PAGE_SIZE] = True
            self._live = live
        return self._live

    def pools(self, device="cpu", fill="nan", chunk_pages=8192):
        """(k_pool, v_pool): bf16 [num_pages][8][16][64] holding the cache state
        before the step; slots no cached token owns hold `fill` ('nan' or 'zero')."""
        shape = (self.num_pages, NUM_KV_HEADS, PAGE_SIZE, HEAD_DIM)
        out = []
        live = torch.from_numpy(self.live_slots()).to(device)
        for stream, scale in (("k_pool", self.k_scale), ("v_pool", 1.0)):
            pool = torch.empty(shape, dtype=torch.bfloat16, device=device)
            gen = torch.Generator(device=device)
            gen.manual_seed(self.seed * 1000 + _STREAMS[stream])
            for p0 in range(0, self.num_pages, chunk_pages):
                p1 = min(self.num_pages, p0 + chunk_pages)
                x = torch.randn((p1 - p0,) + shape[1:], generator=gen, device=device,
                                dtype=torch.float32)
                if scale != 1.0:
                    x.mul_(scale)
                pool[p0:p1] = _bf16(x)
            dead = ~live  # [P][16]
            fill_bits = BF16_NAN_BITS if fill == "nan" else 0
            view = pool.view(torch.int16).permute(0, 2, 1, 3)  # [P][16][8][64]
            view[dead] = np.int16(fill_bits)
            out.append(pool)
        return out[0], out[1]


def tiny(alt_lengths=False) -> Workload:
    seed = BASE_SEED + 1
    lens = np.array([18, 41] if alt_lengths else [17, 40], np.int32)
    table = assign_pages(lens, 1, 8, _rng(seed, "pages"))
    return Workload("tiny" + ("-b" if alt_lengths else ""), 1, 8, lens, table, seed,
                    note="1 layer, batch 2, 8-page pool")


def llama_default(num_layers=16) -> Workload:
    seed = BASE_SEED + 2
    lens = np.full(2, MAX_SEQ_LEN, np.int32)
    num_pages = pages_for_pool_mib(128)
    table = assign_pages(lens, num_layers, num_pages, _rng(seed, "pages"))
    return Workload("llama-b2-2048", num_layers, num_pages, lens, table, seed,
                    note="16 layers, batch 2 at 2048, 128 MiB pool")


def continuous_mix(batch=64, num_layers=16) -> Workload:
    seed = BASE_SEED + 3
    r = _rng(seed, "lengths")
    u = r.uniform(np.log(16), np.log(MAX_SEQ_LEN), size=batch)
    lens = np.clip(np.round(np.exp(u)), 16, MAX_SEQ_LEN).astype(np.int32)
    num_pages = pages_for_pool_mib(4096) * num_layers // 16
    table = assign_pages(lens, num_layers, num_pages, _rng(seed, "pages"), hole_every=3)
    return Workload("mix-b64", num_layers, num_pages, lens, table, seed,
                    note="16 layers, batch 64 log-uniform lengths, 4 GiB pool, fragmented")


def large_ragged(batch=256, num_layers=16) -> Workload:
    seed = BASE_SEED + 4
    r = _rng(seed, "lengths")
    lens = r.integers(1, MAX_SEQ_LEN + 1, size=batch).astype(np.int32)
    forced = [1, 16, 32, 2048, 17, 1024]
    lens[:len(forced)] = forced[:batch]
    n_pages = int(((lens.astype(np.int64) + PAGE_SIZE - 1) // PAGE_SIZE).sum()) * num_layers
    table = assign_pages(lens, num_layers, n_pages, _rng(seed, "pages"))
    return Workload("ragged-b256", num_layers, n_pages, lens, table, seed, k_scale=4.0,
                    note="16 layers, batch 256 uniform lengths, K x 4")


def long_context(batch=1, num_layers=16) -> Workload:
    seed = BASE_SEED + 5
    lens = np.full(batch, MAX_SEQ_LEN, np.int32)
    num_pages = pages_for_pool_mib(1024) * num_layers // 16
    table = assign_pages(lens, num_layers, num_pages, _rng(seed, "pages"))
    return Workload(f"long-b{batch}", num_layers, num_pages, lens, table, seed,
                    note=f"16 layers, batch {batch} at 2048, 1 GiB pool")


def custom(seq_lens, num_layers=1, num_pages=None, seed=BASE_SEED + 9, k_scale=1.0,
           hole_every=0, name="custom") -> Workload:
    """Any lengths; the pool defaults to exactly what the sequences need."""
    lens = np.asarray(seq_lens, np.int32)
    need = int(((lens.astype(np.int64) + PAGE_SIZE - 1) // PAGE_SIZE).sum()) * num_layers
    if num_pages is None:
        # with holes, one id in hole_every is held back
        num_pages = need if not hole_every else -(-need * hole_every // (hole_every - 1)) + 1
        num_pages = max(1, num_pages)
    table = assign_pages(lens, num_layers, num_pages, _rng(seed, "pages"), hole_every)
    return Workload(name, num_layers, num_pages, lens, table, seed, k_scale=k_scale)


@dataclass
class PrefillWorkload:
    name: str
    num_layers: int
    num_pages: int
    start_pos: np.ndarray         # int32 [B]: position of each chunk's first token
    chunk_lens: np.ndarray        # int32 [B]: tokens in each chunk
    block_tables: np.ndarray      # int32 [L][B][128], covering start + n tokens
    seed: int
    note: str = ""

    @property
    def batch(self) -> int:
        return int(self.chunk_lens.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.chunk_lens.sum())

    @property
    def cu_tokens(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.chunk_lens)]).astype(np.int32)

    @property
    def seq_lens(self) -> np.ndarray:
        """Length of each sequence once the chunk is in the cache."""
        return (self.start_pos + self.chunk_lens).astype(np.int32)

    def _normal(self, shape, stream, device):
        gen = torch.Generator(device=device)
        gen.manual_seed(self.seed * 1000 + _STREAMS[stream])
        return _bf16(torch.randn(shape, generator=gen, device=device, dtype=torch.float32))

    def q(self, device="cpu") -> torch.Tensor:
        """bf16 [L][T][32][64]."""
        return self._normal((self.num_layers, self.total_tokens, NUM_Q_HEADS, HEAD_DIM), "q",
                            device)

    def k(self, device="cpu") -> torch.Tensor:
        """bf16 [L][T][8][64]: the chunk tokens' keys."""
        return self._normal((self.num_layers, self.total_tokens, NUM_KV_HEADS, HEAD_DIM),
                            "k_new", device)

    def v(self, device="cpu") -> torch.Tensor:
        return self._normal((self.num_layers, self.total_tokens, NUM_KV_HEADS, HEAD_DIM),
                            "v_new", device)

    def pools(self, device="cpu", fill="nan"):
        """Pools holding positions < start_pos (the earlier chunks); every
        other slot holds `fill`."""
        lens = self.start_pos.astype(np.int32) + 1   # a Workload caches seq_len - 1 tokens
        base = Workload(self.name, self.num_layers, self.num_pages, lens, self.block_tables,
                        self.seed)
        return base.pools(device, fill)


def prefill(chunk_lens, start_pos=None, num_layers=1, num_pages=None, seed=BASE_SEED + 30,
            hole_every=0, name="prefill") -> PrefillWorkload:
    """Chunks of the given lengths; the pool defaults to exactly the pages the
    sequences need once their chunks are in."""
    n = np.asarray(chunk_lens, np.int32)
    start = np.zeros_like(n) if start_pos is None else np.asarray(start_pos, np.int32)
    total = (start + n).astype(np.int64)
    need = int(((total + PAGE_SIZE - 1) // PAGE_SIZE).sum()) * num_layers
    if num_pages is None:
        num_pages = need if not hole_every else -(-need * hole_every // (hole_every - 1)) + 1
        num_pages = max(1, num_pages)
    table = assign_pages(total, num_layers, num_pages, _rng(seed, "pages"), hole_every)
    return PrefillWorkload(name, num_layers, num_pages, start, n, table, seed)


def prefill_prompt(prompt_len=2048, num_layers=16) -> PrefillWorkload:
    """One prompt prefilled at once, the pages' engine's way (one prompt at a
    time between decode iterations): 16 layers, 2,048 tokens, 128 MiB pool."""
    return prefill([prompt_len], num_layers=num_layers, num_pages=pages_for_pool_mib(128),
                   seed=BASE_SEED + 6, name=f"prefill-{prompt_len}")
