"""Paged KV cache decode path for one GB300 GPU: Python binding.

Argument marshalling only. Every step runs in the CUDA library
``_build/libpkv.so`` (built from ``csrc/`` by ``build.build()``) behind the C
ABI of ``include/pkv.h``; the functions here have the same names, take torch
tensors (or raw device addresses as ints), pass their device pointers and
the stream, and raise ``PkvError`` on a non-OK status. There is no fallback:
if the library is missing, every call raises.
"""

import ctypes
import os

from . import build as _build

PAGE_SIZE = 16
NUM_Q_HEADS = 32
NUM_KV_HEADS = 8
HEAD_DIM = 64
MAX_SEQ_LEN = 2048

STATUS = {0: "PKV_OK", 1: "PKV_ERR_INVALID_ARG", 2: "PKV_ERR_OUT_OF_RANGE", 3: "PKV_ERR_CUDA",
          4: "PKV_ERR_UNSUPPORTED", 5: "PKV_ERR_DEVICE_TIMEOUT", 6: "PKV_ERR_STATIC_LIMIT"}
PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_OUT_OF_RANGE, PKV_ERR_CUDA, PKV_ERR_UNSUPPORTED, \
    PKV_ERR_DEVICE_TIMEOUT, PKV_ERR_STATIC_LIMIT = range(7)

EXPORTED = ("pkv_pool_create", "pkv_pool_destroy", "pkv_append", "pkv_decode_attention",
            "pkv_append_attend", "pkv_append_rope", "pkv_decode_attention_rope",
            "pkv_append_attend_rope", "pkv_get_error", "pkv_decode_attention_noalloc",
            "pkv_status_string")


class PkvError(RuntimeError):
    def __init__(self, status, call):
        self.status = status
        super().__init__(f"{call}: {STATUS.get(status, status)}")


class PoolConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_layers", "num_pages", "page_size", "num_q_heads", "num_kv_heads", "head_dim",
        "max_seq_len", "max_batch", "max_splits", "flags")]


PKV_FLAG_PDL = 1


_lib = None


def library_path() -> str:
    return _build.LIBRARY


def load(path: str = None):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or _build.LIBRARY
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} (run paged_kv_cache_210_gb300.build)")
    lib = ctypes.CDLL(path)
    P, i = ctypes.c_void_p, ctypes.c_int
    lib.pkv_pool_create.argtypes = [ctypes.POINTER(PoolConfig), ctypes.POINTER(ctypes.c_void_p)]
    lib.pkv_pool_destroy.argtypes = [P]
    lib.pkv_append.argtypes = [P, i, P, P, P, P, P, P, i, P]
    lib.pkv_decode_attention.argtypes = [P, i, P, P, P, P, P, P, i, i, P]
    lib.pkv_append_attend.argtypes = [P, i, P, P, P, P, P, P, P, P, i, i, P]
    lib.pkv_append_rope.argtypes = [P, i, P, P, P, P, P, P, P, P, i, P]
    lib.pkv_decode_attention_rope.argtypes = [P, i, P, P, P, P, P, P, P, P, i, i, P]
    lib.pkv_append_attend_rope.argtypes = [P, i, P, P, P, P, P, P, P, P, P, P, i, i, P]
    lib.pkv_get_error.argtypes = [P, P]
    lib.pkv_decode_attention_noalloc.argtypes = [i, P, P, P, P, P, P, i, i, i, i, i, i, P, P]
    lib.pkv_status_string.argtypes = [i]
    lib.pkv_status_string.restype = ctypes.c_char_p
    for name in EXPORTED[:-1]:
        getattr(lib, name).restype = ctypes.c_int
    if path == _build.LIBRARY:
        _lib = lib
    return lib


def _addr(x):
    """Device address of a tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status, call):
    if status != PKV_OK:
        raise PkvError(status, call)


class Pool:
    """Owns a pkv_pool_t handle (the split workspace and the error flag)."""

    def __init__(self, handle, config, lib):
        self.handle = handle
        self.config = config
        self._lib = lib

    def close(self):
        if self.handle:
            _check(self._lib.pkv_pool_destroy(self.handle), "pkv_pool_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def pkv_pool_create(num_layers, num_pages, max_batch, max_seq_len=MAX_SEQ_LEN, max_splits=0,
                    flags=0, lib=None) -> Pool:
    lib = lib or load()
    cfg = PoolConfig(num_layers, num_pages, PAGE_SIZE, NUM_Q_HEADS, NUM_KV_HEADS, HEAD_DIM,
                     max_seq_len, max_batch, max_splits, flags)
    handle = ctypes.c_void_p()
    _check(lib.pkv_pool_create(ctypes.byref(cfg), ctypes.byref(handle)), "pkv_pool_create")
    return Pool(handle.value, cfg, lib)


def pkv_pool_destroy(pool: Pool):
    pool.close()


def _batch(x, batch):
    return int(x.shape[0]) if batch is None else int(batch)


def pkv_append(pool: Pool, layer, k, v, k_pool, v_pool, block_tables, positions, batch=None,
               stream=None):
    """k, v: bf16 [B][8][64]; pools bf16 [P][8][16][64]; tables int32 [L][max_batch][pages]."""
    st = pool._lib.pkv_append(pool.handle, int(layer), _addr(k), _addr(v), _addr(k_pool),
                              _addr(v_pool), _addr(block_tables), _addr(positions),
                              _batch(positions, batch), _stream(stream))
    _check(st, "pkv_append")


def pkv_decode_attention(pool: Pool, layer, q, k_pool, v_pool, block_tables, seq_lens, out,
                         batch=None, num_splits=0, stream=None):
    """q: bf16 [B][32][64]; out: fp32 [B][32][64]; seq_lens: int32 [B] (after the append)."""
    st = pool._lib.pkv_decode_attention(pool.handle, int(layer), _addr(q), _addr(k_pool),
                                        _addr(v_pool), _addr(block_tables), _addr(seq_lens),
                                        _addr(out), _batch(seq_lens, batch), int(num_splits),
                                        _stream(stream))
    _check(st, "pkv_decode_attention")


def pkv_append_attend(pool: Pool, layer, q, k, v, k_pool, v_pool, block_tables, seq_lens, out,
                      batch=None, num_splits=0, stream=None):
    """Fused append (at seq_lens - 1) and decode attention for one layer."""
    st = pool._lib.pkv_append_attend(pool.handle, int(layer), _addr(q), _addr(k), _addr(v),
                                     _addr(k_pool), _addr(v_pool), _addr(block_tables),
                                     _addr(seq_lens), _addr(out), _batch(seq_lens, batch),
                                     int(num_splits), _stream(stream))
    _check(st, "pkv_append_attend")


def pkv_append_rope(pool: Pool, layer, k, v, k_pool, v_pool, block_tables, positions,
                    rope_cos, rope_sin, batch=None, stream=None):
    """pkv_append with each key rotated to its position; rope_cos/rope_sin:
    fp32 [max_seq_len][32] on the device."""
    st = pool._lib.pkv_append_rope(pool.handle, int(layer), _addr(k), _addr(v), _addr(k_pool),
                                   _addr(v_pool), _addr(block_tables), _addr(positions),
                                   _addr(rope_cos), _addr(rope_sin), _batch(positions, batch),
                                   _stream(stream))
    _check(st, "pkv_append_rope")


def pkv_decode_attention_rope(pool: Pool, layer, q, k_pool, v_pool, block_tables, seq_lens,
                              rope_cos, rope_sin, out, batch=None, num_splits=0, stream=None):
    """pkv_decode_attention with each query rotated to position seq_lens - 1."""
    st = pool._lib.pkv_decode_attention_rope(pool.handle, int(layer), _addr(q), _addr(k_pool),
                                             _addr(v_pool), _addr(block_tables),
                                             _addr(seq_lens), _addr(rope_cos), _addr(rope_sin),
                                             _addr(out), _batch(seq_lens, batch),
                                             int(num_splits), _stream(stream))
    _check(st, "pkv_decode_attention_rope")


def pkv_append_attend_rope(pool: Pool, layer, q, k, v, k_pool, v_pool, block_tables, seq_lens,
                           rope_cos, rope_sin, out, batch=None, num_splits=0, stream=None):
    """pkv_append_attend with the key and the queries rotated to seq_lens - 1."""
    st = pool._lib.pkv_append_attend_rope(pool.handle, int(layer), _addr(q), _addr(k), _addr(v),
                                          _addr(k_pool), _addr(v_pool), _addr(block_tables),
                                          _addr(seq_lens), _addr(rope_cos), _addr(rope_sin),
                                          _addr(out), _batch(seq_lens, batch),
                                          int(num_splits), _stream(stream))
    _check(st, "pkv_append_attend_rope")


def pkv_get_error(pool: Pool, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the sticky device status."""
    return pool._lib.pkv_get_error(pool.handle, _stream(stream))


def pkv_decode_attention_noalloc(layer, q, k_pool, v_pool, block_tables, seq_lens, out,
                                 num_layers, num_pages, max_batch, max_seq_len=MAX_SEQ_LEN,
                                 batch=None, num_splits=1, error_bits=None, stream=None,
                                 lib=None):
    """Decode attention for callers that may not allocate device memory: no
    pool handle, scratch in the library's own static device array (limits and
    the one-time set-up on first use are described in include/pkv.h)."""
    lib = lib or load()
    st = lib.pkv_decode_attention_noalloc(int(layer), _addr(q), _addr(k_pool), _addr(v_pool),
                                          _addr(block_tables), _addr(seq_lens), _addr(out),
                                          int(num_layers), int(num_pages), int(max_batch),
                                          int(max_seq_len), _batch(seq_lens, batch),
                                          int(num_splits), _addr(error_bits), _stream(stream))
    _check(st, "pkv_decode_attention_noalloc")
