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
          4: "PKV_ERR_UNSUPPORTED", 5: "PKV_ERR_DEVICE_TIMEOUT", 6: "PKV_ERR_STATIC_LIMIT",
          7: "PKV_ERR_REJECTED"}
PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_OUT_OF_RANGE, PKV_ERR_CUDA, PKV_ERR_UNSUPPORTED, \
    PKV_ERR_DEVICE_TIMEOUT, PKV_ERR_STATIC_LIMIT, PKV_ERR_REJECTED = range(8)

EXPORTED = ("pkv_pool_create", "pkv_pool_destroy", "pkv_append", "pkv_decode_attention",
            "pkv_append_attend", "pkv_append_rope", "pkv_decode_attention_rope",
            "pkv_append_attend_rope", "pkv_append_attend_layers", "pkv_test_layers_wait_timeout",
            "pkv_get_error", "pkv_decode_attention_noalloc",
            "pkv_sched_budget", "pkv_sched_create", "pkv_sched_destroy", "pkv_sched_submit",
            "pkv_sched_admit", "pkv_sched_extend", "pkv_sched_extend_batch", "pkv_sched_finish",
            "pkv_sched_decode_batch",
            "pkv_sched_block_tables", "pkv_sched_get_stats", "pkv_prefill_fill",
            "pkv_prefill_attention", "pkv_prefill", "pkv_plan_decode",
            "pkv_pool_device_figures", "pkv_status_string")


class PkvError(RuntimeError):
    def __init__(self, status, call):
        self.status = status
        super().__init__(f"{call}: {STATUS.get(status, status)}")


class SchedConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_layers", "num_pages", "page_size", "max_seq_len", "static_batching")]


class SchedStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "pool_pages", "submitted", "rejected", "admitted", "finished", "peak_active",
        "largest_decode_batch", "peak_assigned_pages", "admission_waits", "free_pages",
        "free_credits", "active", "waiting")]


class PoolConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_layers", "num_pages", "page_size", "num_q_heads", "num_kv_heads", "head_dim",
        "max_seq_len", "max_batch", "max_splits", "flags")]


PKV_FLAG_PDL = 1


class DeviceFigures(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "num_sms", "ticket_blocks_per_sm", "narrow_blocks_per_sm", "wide_blocks_per_sm",
        "max_cluster", "max_splits", "max_seq_len")]


class Plan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "shape", "cluster", "num_splits", "chunk_pages", "range_div", "grid_splits",
        "grid_units", "longest_first")]


PKV_SHAPE_TICKET, PKV_SHAPE_NARROW, PKV_SHAPE_WIDE = 0, 1, 2


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
    lib.pkv_append_attend_layers.argtypes = [P, i, i, P, P, P, P, P, P, P, P, i, P]
    lib.pkv_test_layers_wait_timeout.argtypes = [P, i, i, P, P, P, P, P, P, P, P, i, P]
    lib.pkv_get_error.argtypes = [P, P]
    lib.pkv_decode_attention_noalloc.argtypes = [i, P, P, P, P, P, P, i, i, i, i, i, i, P, P]
    SC, SP = ctypes.POINTER(SchedConfig), ctypes.POINTER(ctypes.c_int)
    lib.pkv_sched_budget.argtypes = [SC, i, i, SP, SP, ctypes.POINTER(ctypes.c_int64)]
    lib.pkv_sched_create.argtypes = [SC, ctypes.POINTER(ctypes.c_void_p)]
    lib.pkv_sched_destroy.argtypes = [P]
    lib.pkv_sched_submit.argtypes = [P, i, i, SP]
    lib.pkv_sched_admit.argtypes = [P, P, i, SP]
    lib.pkv_sched_extend.argtypes = [P, i, i]
    lib.pkv_sched_finish.argtypes = [P, i]
    lib.pkv_sched_decode_batch.argtypes = [P, P, i, SP]
    lib.pkv_sched_extend_batch.argtypes = [P, P, P, i]
    lib.pkv_sched_block_tables.argtypes = [P, P, i, P, i, i, i]
    lib.pkv_sched_get_stats.argtypes = [P, ctypes.POINTER(SchedStats)]
    lib.pkv_prefill_fill.argtypes = [P, i, P, P, P, P, P, P, P, i, i, i, P]
    lib.pkv_prefill_attention.argtypes = [P, i, P, P, P, P, P, P, P, i, i, i, P]
    lib.pkv_prefill.argtypes = [P, i, P, P, P, P, P, P, P, P, P, i, i, i, P]
    lib.pkv_plan_decode.argtypes = [ctypes.POINTER(DeviceFigures), i, i, ctypes.POINTER(Plan)]
    lib.pkv_pool_device_figures.argtypes = [P, ctypes.POINTER(DeviceFigures)]
    lib.pkv_status_string.argtypes = [i]
    lib.pkv_status_string.restype = ctypes.c_char_p
    for name in EXPORTED[:-1]:
        getattr(lib, name).restype = ctypes.c_int
    if path == _build.LIBRARY:
        _lib = lib
    return lib


def _addr(x, dtype=None, what="tensor"):
    """Address of a tensor (or an int address, or None). A tensor must be
    contiguous and, when `dtype` is given ("bfloat16", "float32", "int32"),
    of that dtype: the library reads raw memory in the layouts include/*.h
    documents."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError(f"{what}: the library takes contiguous tensors")
    if dtype is not None and str(x.dtype) != "torch." + dtype:
        raise ValueError(f"{what}: expected {dtype}, got {x.dtype}")
    return x.data_ptr()


def _i32(x, what):
    return _addr(x, "int32", what)


# the dtype of each tensor argument of the CUDA entry points, by parameter name
_DTYPES = {"q": "bfloat16", "k": "bfloat16", "v": "bfloat16", "k_pool": "bfloat16",
           "v_pool": "bfloat16", "block_tables": "int32", "positions": "int32",
           "seq_lens": "int32", "cu_tokens": "int32", "start_pos": "int32", "out": "float32",
           "rope_cos": "float32", "rope_sin": "float32"}


def _ptrs(**tensors):
    """Checked addresses of the named tensor arguments, in the order given."""
    return [_addr(t, _DTYPES[name], name) for name, t in tensors.items()]


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
    st = pool._lib.pkv_append(
        pool.handle, int(layer),
        *_ptrs(k=k, v=v, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables,
               positions=positions),
        _batch(positions, batch), _stream(stream))
    _check(st, "pkv_append")


def pkv_decode_attention(pool: Pool, layer, q, k_pool, v_pool, block_tables, seq_lens, out,
                         batch=None, num_splits=0, stream=None):
    """q: bf16 [B][32][64]; out: fp32 [B][32][64]; seq_lens: int32 [B] (after the append)."""
    st = pool._lib.pkv_decode_attention(
        pool.handle, int(layer),
        *_ptrs(q=q, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables, seq_lens=seq_lens,
               out=out),
        _batch(seq_lens, batch), int(num_splits), _stream(stream))
    _check(st, "pkv_decode_attention")


def pkv_append_attend(pool: Pool, layer, q, k, v, k_pool, v_pool, block_tables, seq_lens, out,
                      batch=None, num_splits=0, stream=None):
    """Fused append (at seq_lens - 1) and decode attention for one layer."""
    st = pool._lib.pkv_append_attend(
        pool.handle, int(layer),
        *_ptrs(q=q, k=k, v=v, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables,
               seq_lens=seq_lens, out=out),
        _batch(seq_lens, batch), int(num_splits), _stream(stream))
    _check(st, "pkv_append_attend")


def pkv_append_rope(pool: Pool, layer, k, v, k_pool, v_pool, block_tables, positions,
                    rope_cos, rope_sin, batch=None, stream=None):
    """pkv_append with each key rotated to its position; rope_cos/rope_sin:
    fp32 [max_seq_len][32] on the device."""
    st = pool._lib.pkv_append_rope(
        pool.handle, int(layer),
        *_ptrs(k=k, v=v, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables,
               positions=positions, rope_cos=rope_cos, rope_sin=rope_sin),
        _batch(positions, batch), _stream(stream))
    _check(st, "pkv_append_rope")


def pkv_decode_attention_rope(pool: Pool, layer, q, k_pool, v_pool, block_tables, seq_lens,
                              rope_cos, rope_sin, out, batch=None, num_splits=0, stream=None):
    """pkv_decode_attention with each query rotated to position seq_lens - 1."""
    st = pool._lib.pkv_decode_attention_rope(
        pool.handle, int(layer),
        *_ptrs(q=q, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables, seq_lens=seq_lens,
               rope_cos=rope_cos, rope_sin=rope_sin, out=out),
        _batch(seq_lens, batch), int(num_splits), _stream(stream))
    _check(st, "pkv_decode_attention_rope")


def pkv_append_attend_rope(pool: Pool, layer, q, k, v, k_pool, v_pool, block_tables, seq_lens,
                           rope_cos, rope_sin, out, batch=None, num_splits=0, stream=None):
    """pkv_append_attend with the key and the queries rotated to seq_lens - 1."""
    st = pool._lib.pkv_append_attend_rope(
        pool.handle, int(layer),
        *_ptrs(q=q, k=k, v=v, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables,
               seq_lens=seq_lens, rope_cos=rope_cos, rope_sin=rope_sin, out=out),
        _batch(seq_lens, batch), int(num_splits), _stream(stream))
    _check(st, "pkv_append_attend_rope")


def pkv_append_attend_layers(pool: Pool, layer_begin, q, k, v, k_pool, v_pool, block_tables,
                             seq_lens, out, num_layers=None, batch=None, stream=None):
    """Fused append + attend of layers layer_begin .. layer_begin + num_layers - 1
    in one persistent launch (several for long calls). q: bf16 [J][B][32][64];
    k, v: bf16 [J][B][8][64]; out: fp32 [J][B][32][64]; J = num_layers
    (default: q's first dimension)."""
    J = int(q.shape[0]) if num_layers is None else int(num_layers)
    st = pool._lib.pkv_append_attend_layers(
        pool.handle, int(layer_begin), J,
        *_ptrs(q=q, k=k, v=v, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables,
               seq_lens=seq_lens, out=out),
        _batch(seq_lens, batch), _stream(stream))
    _check(st, "pkv_append_attend_layers")


def pkv_test_layers_wait_timeout(pool: Pool, layer_begin, q, k, v, k_pool, v_pool,
                                 block_tables, seq_lens, out, num_layers=None, batch=None,
                                 stream=None):
    """Failure-detection test hook: pkv_append_attend_layers with every
    between-layer wait unreachable; the device flags a timeout."""
    J = int(q.shape[0]) if num_layers is None else int(num_layers)
    st = pool._lib.pkv_test_layers_wait_timeout(
        pool.handle, int(layer_begin), J,
        *_ptrs(q=q, k=k, v=v, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables,
               seq_lens=seq_lens, out=out),
        _batch(seq_lens, batch), _stream(stream))
    _check(st, "pkv_test_layers_wait_timeout")


def pkv_plan_decode(figures: DeviceFigures, batch, num_splits=0, lib=None) -> Plan:
    """The decode launch plan for a batch on a device (host arithmetic, no GPU)."""
    lib = lib or load()
    plan = Plan()
    _check(lib.pkv_plan_decode(ctypes.byref(figures), int(batch), int(num_splits),
                               ctypes.byref(plan)), "pkv_plan_decode")
    return plan


def pkv_pool_device_figures(pool: Pool) -> DeviceFigures:
    figures = DeviceFigures()
    _check(pool._lib.pkv_pool_device_figures(pool.handle, ctypes.byref(figures)),
           "pkv_pool_device_figures")
    return figures


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
    st = lib.pkv_decode_attention_noalloc(
        int(layer),
        *_ptrs(q=q, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables, seq_lens=seq_lens,
               out=out),
        int(num_layers), int(num_pages), int(max_batch), int(max_seq_len),
        _batch(seq_lens, batch), int(num_splits), _i32(error_bits, "error_bits"),
        _stream(stream))
    _check(st, "pkv_decode_attention_noalloc")


# ---------------------------------------------------------------- prefill
def pkv_prefill_fill(pool: Pool, layer, k, v, k_pool, v_pool, block_tables, cu_tokens, start_pos,
                     max_chunk_tokens, batch=None, total_tokens=None, stream=None):
    """Writes chunk tokens' K/V (bf16 [T][8][64]) into their pages."""
    batch = int(start_pos.shape[0]) if batch is None else int(batch)
    total = int(k.shape[0]) if total_tokens is None else int(total_tokens)
    st = pool._lib.pkv_prefill_fill(
        pool.handle, int(layer),
        *_ptrs(k=k, v=v, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables,
               cu_tokens=cu_tokens, start_pos=start_pos),
        batch, total, int(max_chunk_tokens), _stream(stream))
    _check(st, "pkv_prefill_fill")


def pkv_prefill_attention(pool: Pool, layer, q, k_pool, v_pool, block_tables, cu_tokens, start_pos,
                          out, max_chunk_tokens, batch=None, total_tokens=None, stream=None):
    """Causal attention of chunk tokens (q bf16 [T][32][64]) over the pages; out fp32."""
    batch = int(start_pos.shape[0]) if batch is None else int(batch)
    total = int(q.shape[0]) if total_tokens is None else int(total_tokens)
    st = pool._lib.pkv_prefill_attention(
        pool.handle, int(layer),
        *_ptrs(q=q, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables,
               cu_tokens=cu_tokens, start_pos=start_pos, out=out),
        batch, total, int(max_chunk_tokens), _stream(stream))
    _check(st, "pkv_prefill_attention")


def pkv_prefill(pool: Pool, layer, q, k, v, k_pool, v_pool, block_tables, cu_tokens, start_pos,
                out, max_chunk_tokens, batch=None, total_tokens=None, stream=None):
    """pkv_prefill_fill then pkv_prefill_attention."""
    batch = int(start_pos.shape[0]) if batch is None else int(batch)
    total = int(q.shape[0]) if total_tokens is None else int(total_tokens)
    st = pool._lib.pkv_prefill(
        pool.handle, int(layer),
        *_ptrs(q=q, k=k, v=v, k_pool=k_pool, v_pool=v_pool, block_tables=block_tables,
               cu_tokens=cu_tokens, start_pos=start_pos, out=out),
        batch, total, int(max_chunk_tokens), _stream(stream))
    _check(st, "pkv_prefill")


# ---------------------------------------------------------------- admission scheduler (host)
class Scheduler:
    """Owns a pkv_sched_t: admission credits and lazy page assignment for the
    shared pool (host only; see include/pkv_sched.h)."""

    def __init__(self, handle, config, lib):
        self.handle = handle
        self.config = config
        self._lib = lib

    def close(self):
        if self.handle:
            _check(self._lib.pkv_sched_destroy(self.handle), "pkv_sched_destroy")
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _sched_config(num_pages, num_layers, page_size, max_seq_len, static_batching):
    return SchedConfig(int(num_layers), int(num_pages), int(page_size), int(max_seq_len),
                       1 if static_batching else 0)


def pkv_sched_budget(prompt_tokens, max_new_tokens, num_layers=16, page_size=PAGE_SIZE,
                     max_seq_len=MAX_SEQ_LEN, lib=None):
    """(allowed new tokens, largest processed prefix, budget in pages)."""
    lib = lib or load()
    cfg = _sched_config(1, num_layers, page_size, max_seq_len, False)
    allowed, prefix, budget = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
    _check(lib.pkv_sched_budget(ctypes.byref(cfg), int(prompt_tokens), int(max_new_tokens),
                                ctypes.byref(allowed), ctypes.byref(prefix),
                                ctypes.byref(budget)), "pkv_sched_budget")
    return allowed.value, prefix.value, budget.value


def pkv_sched_create(num_pages, num_layers=16, page_size=PAGE_SIZE, max_seq_len=MAX_SEQ_LEN,
                     static_batching=False, lib=None) -> Scheduler:
    lib = lib or load()
    cfg = _sched_config(num_pages, num_layers, page_size, max_seq_len, static_batching)
    handle = ctypes.c_void_p()
    _check(lib.pkv_sched_create(ctypes.byref(cfg), ctypes.byref(handle)), "pkv_sched_create")
    return Scheduler(handle.value, cfg, lib)


def pkv_sched_destroy(sched: Scheduler):
    sched.close()


def pkv_sched_submit(sched: Scheduler, prompt_tokens, max_new_tokens) -> int:
    """Queues a request and returns its id; PkvError(PKV_ERR_REJECTED) when
    its budget exceeds the pool."""
    rid = ctypes.c_int(-1)
    _check(sched._lib.pkv_sched_submit(sched.handle, int(prompt_tokens), int(max_new_tokens),
                                       ctypes.byref(rid)), "pkv_sched_submit")
    return rid.value


def pkv_sched_get_stats(sched: Scheduler) -> dict:
    st = SchedStats()
    _check(sched._lib.pkv_sched_get_stats(sched.handle, ctypes.byref(st)), "pkv_sched_get_stats")
    return {name: getattr(st, name) for name, _ in SchedStats._fields_}


def _id_buffer(n):
    return (ctypes.c_int * max(1, n))()


def pkv_sched_admit(sched: Scheduler) -> list:
    """One admission pass; the admitted ids in order."""
    cap = pkv_sched_get_stats(sched)["waiting"]
    buf, count = _id_buffer(cap), ctypes.c_int()
    _check(sched._lib.pkv_sched_admit(sched.handle, buf, int(cap), ctypes.byref(count)),
           "pkv_sched_admit")
    return list(buf[:count.value])


def pkv_sched_extend(sched: Scheduler, request_id, length):
    _check(sched._lib.pkv_sched_extend(sched.handle, int(request_id), int(length)),
           "pkv_sched_extend")


def pkv_sched_extend_batch(sched: Scheduler, ids, lengths):
    """pkv_sched_extend for every (id, length) pair, in one call."""
    import numpy as np
    id_buf = np.ascontiguousarray(ids, dtype=np.intc)
    len_buf = np.ascontiguousarray(lengths, dtype=np.intc)
    if id_buf.shape != len_buf.shape or id_buf.ndim != 1:
        raise ValueError("ids and lengths must be 1-D and of one length")
    _check(sched._lib.pkv_sched_extend_batch(sched.handle, id_buf.ctypes.data, len_buf.ctypes.data,
                                             int(id_buf.shape[0])), "pkv_sched_extend_batch")


def pkv_sched_finish(sched: Scheduler, request_id):
    _check(sched._lib.pkv_sched_finish(sched.handle, int(request_id)), "pkv_sched_finish")


def pkv_sched_decode_batch(sched: Scheduler) -> list:
    """The active requests in admission order (one decode step's batch)."""
    cap = pkv_sched_get_stats(sched)["active"]
    buf, count = _id_buffer(cap), ctypes.c_int()
    _check(sched._lib.pkv_sched_decode_batch(sched.handle, buf, int(cap), ctypes.byref(count)),
           "pkv_sched_decode_batch")
    return list(buf[:count.value])


def pkv_sched_block_tables(sched: Scheduler, ids, max_batch=None, max_pages=None, out=None,
                           clear_tail=True):
    """Host block tables int32 [num_layers][max_batch][max_pages] for the batch
    `ids` (numpy array; `out` may supply a C-contiguous one to fill; with
    clear_tail False, entries past each row's pages are left as they were)."""
    import numpy as np
    ids = np.ascontiguousarray(ids, dtype=np.intc).reshape(-1)
    max_batch = len(ids) if max_batch is None else int(max_batch)
    max_pages = sched.config.max_seq_len // sched.config.page_size if max_pages is None \
        else int(max_pages)
    shape = (sched.config.num_layers, max_batch, max_pages)
    if out is None:
        out = np.empty(shape, np.int32)
    elif out.shape != shape or out.dtype != np.int32 or not out.flags.c_contiguous:
        raise ValueError(f"out must be a C-contiguous int32 array of shape {shape}")
    _check(sched._lib.pkv_sched_block_tables(sched.handle, ids.ctypes.data, len(ids),
                                             out.ctypes.data_as(ctypes.c_void_p), max_batch,
                                             max_pages, 1 if clear_tail else 0),
           "pkv_sched_block_tables")
    return out
