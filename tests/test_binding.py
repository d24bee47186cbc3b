"""The Python binding's argument marshalling, on the CPU: tensors must be
contiguous and of the dtype the C ABI reads (bf16 activations and pools,
int32 tables and lengths, fp32 outputs and rotary tables); a wrong one raises
before any library call."""

import pytest
import torch

import paged_kv_cache_210_gb300 as pkv


class _NoLibrary:
    """Stands in for the CUDA library: any call would be a failure."""

    def __getattr__(self, name):
        def call(*args):
            raise AssertionError(f"{name} reached the library")
        return call


POOL = pkv.Pool(handle=1, config=None, lib=_NoLibrary())


def _good(B=2, L=1, P=8):
    return dict(
        q=torch.zeros(B, 32, 64, dtype=torch.bfloat16),
        k=torch.zeros(B, 8, 64, dtype=torch.bfloat16),
        v=torch.zeros(B, 8, 64, dtype=torch.bfloat16),
        k_pool=torch.zeros(P, 8, 16, 64, dtype=torch.bfloat16),
        v_pool=torch.zeros(P, 8, 16, 64, dtype=torch.bfloat16),
        block_tables=torch.zeros(L, B, 128, dtype=torch.int32),
        seq_lens=torch.ones(B, dtype=torch.int32),
        out=torch.zeros(B, 32, 64, dtype=torch.float32),
    )


@pytest.mark.parametrize("name,bad", [
    ("q", torch.zeros(2, 32, 64, dtype=torch.float32)),
    ("k", torch.zeros(2, 8, 64, dtype=torch.float16)),
    ("k_pool", torch.zeros(8, 8, 16, 64, dtype=torch.int16)),
    ("block_tables", torch.zeros(1, 2, 128, dtype=torch.int64)),
    ("seq_lens", torch.ones(2, dtype=torch.int64)),
    ("out", torch.zeros(2, 32, 64, dtype=torch.bfloat16)),
    ("out", torch.zeros(2, 64, 32, dtype=torch.float32).transpose(1, 2)),   # not contiguous
])
def test_wrong_tensor_raises_before_the_library(name, bad):
    a = _good()
    a[name] = bad
    with pytest.raises(ValueError, match=name):
        pkv.pkv_append_attend(POOL, 0, a["q"], a["k"], a["v"], a["k_pool"], a["v_pool"],
                              a["block_tables"], a["seq_lens"], a["out"])


def test_rope_tables_must_be_fp32():
    a = _good()
    cos = torch.zeros(2048, 32, dtype=torch.float64)
    with pytest.raises(ValueError, match="rope_cos"):
        pkv.pkv_decode_attention_rope(POOL, 0, a["q"], a["k_pool"], a["v_pool"],
                                      a["block_tables"], a["seq_lens"], cos, cos, a["out"])


def test_int_addresses_and_none_pass_through():
    assert pkv._addr(None) is None
    assert pkv._addr(12345, "bfloat16") == 12345
    t = torch.zeros(4, dtype=torch.int32)
    assert pkv._i32(t, "t") == t.data_ptr()
    assert pkv._ptrs(q=None, out=7) == [None, 7]
