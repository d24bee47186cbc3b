"""CPU oracle for paged decode attention (TEST INFRASTRUCTURE ONLY).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never does, and this
package never imports the CUDA library.

Thin ctypes wrappers over ``pkv_oracle.cpp`` (plain FP64 C++). Arrays are
numpy: BF16 values are ``uint16`` bit patterns, indices ``int32``, results
``float64``. See the C source for the definitions and the passages of the
samir-vllm pages each one follows.
"""

import ctypes

import numpy as np

from . import build as _build

OK, BAD_ARG, OUT_OF_RANGE = 0, 1, 2


class Geometry(ctypes.Structure):
    _fields_ = [(name, ctypes.c_int) for name in (
        "num_layers", "num_pages", "page_size", "num_q_heads", "num_kv_heads",
        "head_dim", "max_batch", "max_pages_per_seq")]


def geometry(num_layers, num_pages, max_batch, page_size=16, num_q_heads=32,
             num_kv_heads=8, head_dim=64, max_pages_per_seq=128):
    return Geometry(num_layers, num_pages, page_size, num_q_heads, num_kv_heads,
                    head_dim, max_batch, max_pages_per_seq)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(a, dtype):
    if not (isinstance(a, np.ndarray) and a.dtype == dtype and a.flags.c_contiguous):
        raise TypeError(f"expected a C-contiguous {np.dtype(dtype)} array")
    return a


class Oracle:
    """The oracle functions bound to one compiled copy of ``pkv_oracle.cpp``."""

    def __init__(self, path):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        G = ctypes.POINTER(Geometry)
        i = ctypes.c_int
        lib.pkv_oracle_append.argtypes = [G, i, P, P, P, P, P, P, i]
        lib.pkv_oracle_decode_attention.argtypes = [G, i, P, P, P, P, P, i, P, P, P]
        lib.pkv_oracle_decode_attention_mt.argtypes = [G, i, P, P, P, P, P, i, P, i]
        lib.pkv_oracle_decode_attention_split.argtypes = [G, i, P, P, P, P, P, i, i,
                                                          P, P, P, P]
        lib.pkv_oracle_contiguous_attention.argtypes = [P, P, P, i, i, i, i, P]
        lib.pkv_oracle_append_rope.argtypes = [G, i, P, P, P, P, P, P, i, P, P, i]
        lib.pkv_oracle_rope_queries.argtypes = [P, i, i, i, P, P, P, i, P]
        lib.pkv_oracle_decode_attention_q64.argtypes = [G, i, P, P, P, P, P, i, P]
        lib.pkv_oracle_prefill_fill.argtypes = [G, i, P, P, P, P, P, P, P, i]
        lib.pkv_oracle_prefill_attention.argtypes = [G, i, P, P, P, P, P, P, i, P, i]
        for name in ("pkv_oracle_append", "pkv_oracle_decode_attention",
                     "pkv_oracle_decode_attention_mt", "pkv_oracle_decode_attention_split",
                     "pkv_oracle_contiguous_attention", "pkv_oracle_append_rope",
                     "pkv_oracle_rope_queries", "pkv_oracle_decode_attention_q64",
                     "pkv_oracle_prefill_fill", "pkv_oracle_prefill_attention"):
            getattr(lib, name).restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def append(self, g, layer, k_new, v_new, k_pool, v_pool, block_tables, positions):
        """Scatter one new token per sequence into the pools, in place. Returns status."""
        for a in (k_new, v_new, k_pool, v_pool):
            _check(a, np.uint16)
        _check(block_tables, np.int32)
        _check(positions, np.int32)
        return self.lib.pkv_oracle_append(ctypes.byref(g), layer, _ptr(k_new), _ptr(v_new),
                                          _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                          _ptr(positions), int(positions.shape[0]))

    def decode_attention(self, g, layer, q, k_pool, v_pool, block_tables, seq_lens):
        """Returns (status, out[B][Hq][D], lse[B][Hq], weight_sum[B][Hq]) in float64."""
        for a in (q, k_pool, v_pool):
            _check(a, np.uint16)
        _check(block_tables, np.int32)
        _check(seq_lens, np.int32)
        B = int(seq_lens.shape[0])
        out = np.zeros((B, g.num_q_heads, g.head_dim), np.float64)
        lse = np.zeros((B, g.num_q_heads), np.float64)
        wsum = np.zeros((B, g.num_q_heads), np.float64)
        st = self.lib.pkv_oracle_decode_attention(ctypes.byref(g), layer, _ptr(q),
                                                  _ptr(k_pool), _ptr(v_pool),
                                                  _ptr(block_tables), _ptr(seq_lens), B,
                                                  _ptr(out), _ptr(lse), _ptr(wsum))
        return st, out, lse, wsum

    def decode_attention_mt(self, g, layer, q, k_pool, v_pool, block_tables, seq_lens,
                            nthreads, out=None):
        """Same as decode_attention (output only), sequences spread over nthreads threads."""
        for a in (q, k_pool, v_pool):
            _check(a, np.uint16)
        _check(block_tables, np.int32)
        _check(seq_lens, np.int32)
        B = int(seq_lens.shape[0])
        if out is None:
            out = np.zeros((B, g.num_q_heads, g.head_dim), np.float64)
        st = self.lib.pkv_oracle_decode_attention_mt(ctypes.byref(g), layer, _ptr(q),
                                                     _ptr(k_pool), _ptr(v_pool),
                                                     _ptr(block_tables), _ptr(seq_lens), B,
                                                     _ptr(out), int(nthreads))
        return st, out

    def decode_attention_split(self, g, layer, q, k_pool, v_pool, block_tables, seq_lens,
                               num_splits):
        """Returns (status, out, part_o[B][Hq][S][D], part_m[B][Hq][S], part_l[B][Hq][S])."""
        for a in (q, k_pool, v_pool):
            _check(a, np.uint16)
        _check(block_tables, np.int32)
        _check(seq_lens, np.int32)
        B = int(seq_lens.shape[0])
        S = int(num_splits)
        out = np.zeros((B, g.num_q_heads, g.head_dim), np.float64)
        po = np.zeros((B, g.num_q_heads, S, g.head_dim), np.float64)
        pm = np.zeros((B, g.num_q_heads, S), np.float64)
        pl = np.zeros((B, g.num_q_heads, S), np.float64)
        st = self.lib.pkv_oracle_decode_attention_split(ctypes.byref(g), layer, _ptr(q),
                                                        _ptr(k_pool), _ptr(v_pool),
                                                        _ptr(block_tables), _ptr(seq_lens),
                                                        B, S, _ptr(out), _ptr(po), _ptr(pm),
                                                        _ptr(pl))
        return st, out, po, pm, pl

    def append_rope(self, g, layer, k_new, v_new, k_pool, v_pool, block_tables, positions,
                    cos_t, sin_t):
        """append() with each new key rotated to its position (FP32, then BF16)."""
        for a in (k_new, v_new, k_pool, v_pool):
            _check(a, np.uint16)
        _check(block_tables, np.int32)
        _check(positions, np.int32)
        _check(cos_t, np.float32)
        _check(sin_t, np.float32)
        return self.lib.pkv_oracle_append_rope(ctypes.byref(g), layer, _ptr(k_new), _ptr(v_new),
                                               _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                               _ptr(positions), int(positions.shape[0]),
                                               _ptr(cos_t), _ptr(sin_t), int(cos_t.shape[0]))

    def rope_queries(self, q, positions, cos_t, sin_t):
        """q [B][Hq][D] BF16 patterns -> (status, q rotated to its position, float64)."""
        _check(q, np.uint16)
        _check(positions, np.int32)
        _check(cos_t, np.float32)
        _check(sin_t, np.float32)
        B, Hq, D = q.shape
        out = np.zeros((B, Hq, D), np.float64)
        st = self.lib.pkv_oracle_rope_queries(_ptr(q), B, Hq, D, _ptr(positions), _ptr(cos_t),
                                              _ptr(sin_t), int(cos_t.shape[0]), _ptr(out))
        return st, out

    def decode_attention_q64(self, g, layer, q64, k_pool, v_pool, block_tables, seq_lens):
        """decode_attention() with float64 queries [B][Hq][D] -> (status, out)."""
        _check(q64, np.float64)
        for a in (k_pool, v_pool):
            _check(a, np.uint16)
        _check(block_tables, np.int32)
        _check(seq_lens, np.int32)
        B = int(seq_lens.shape[0])
        out = np.zeros((B, g.num_q_heads, g.head_dim), np.float64)
        st = self.lib.pkv_oracle_decode_attention_q64(ctypes.byref(g), layer, _ptr(q64),
                                                      _ptr(k_pool), _ptr(v_pool),
                                                      _ptr(block_tables), _ptr(seq_lens), B,
                                                      _ptr(out))
        return st, out

    def prefill_fill(self, g, layer, k, v, k_pool, v_pool, block_tables, cu_tokens, start_pos):
        """Writes chunk tokens' K/V (k, v: [total][Hkv][D] BF16 patterns) into the pools."""
        for a in (k, v, k_pool, v_pool):
            _check(a, np.uint16)
        for a in (block_tables, cu_tokens, start_pos):
            _check(a, np.int32)
        return self.lib.pkv_oracle_prefill_fill(ctypes.byref(g), layer, _ptr(k), _ptr(v),
                                                _ptr(k_pool), _ptr(v_pool), _ptr(block_tables),
                                                _ptr(cu_tokens), _ptr(start_pos),
                                                int(start_pos.shape[0]))

    def prefill_attention(self, g, layer, q, k_pool, v_pool, block_tables, cu_tokens, start_pos,
                          threads=8):
        """Causal attention over the pages for every chunk token -> (status, out
        [total][Hq][D] float64)."""
        _check(q, np.uint16)
        for a in (k_pool, v_pool):
            _check(a, np.uint16)
        for a in (block_tables, cu_tokens, start_pos):
            _check(a, np.int32)
        out = np.zeros((q.shape[0], g.num_q_heads, g.head_dim), np.float64)
        st = self.lib.pkv_oracle_prefill_attention(ctypes.byref(g), layer, _ptr(q), _ptr(k_pool),
                                                   _ptr(v_pool), _ptr(block_tables),
                                                   _ptr(cu_tokens), _ptr(start_pos),
                                                   int(start_pos.shape[0]), _ptr(out),
                                                   int(threads))
        return st, out

    def contiguous_attention(self, q, k, v):
        """q [Hq][D], k and v [len][Hkv][D] (uint16 BF16 patterns) -> (status, out [Hq][D])."""
        for a in (q, k, v):
            _check(a, np.uint16)
        Hq, D = q.shape
        L, Hkv, _ = k.shape
        out = np.zeros((Hq, D), np.float64)
        st = self.lib.pkv_oracle_contiguous_attention(_ptr(q), _ptr(k), _ptr(v), L, Hq, Hkv,
                                                      D, _ptr(out))
        return st, out


_default = None


def load() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(_build.build())
    return _default
