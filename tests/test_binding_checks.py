"""The Python binding validates tensor arguments before handing raw pointers
to the C ABI (no GPU needed: every case fails before any CUDA call)."""
import pytest
import torch

from mqa_decode_attention_paged_gb300 import _binding as mqa


def _mla_args(**kw):
    a = dict(q=torch.zeros(2, 16, 576, dtype=torch.bfloat16), kv=torch.zeros(4, 16, 576, dtype=torch.bfloat16),
             bt=torch.zeros(2, 2, dtype=torch.int32), sl=torch.zeros(2, dtype=torch.int32))
    a.update(kw)
    return a


def _call_mla(a, **kw):
    return mqa.mla_decode(a["q"], a["kv"], a["bt"], a["sl"], 0.07, **kw)


@pytest.mark.parametrize("kw,exc,msg", [
    (dict(q=torch.zeros(2, 16, 576, dtype=torch.float16)), TypeError, "q must have dtype"),
    (dict(bt=torch.zeros(2, 2, dtype=torch.int64)), TypeError, "block_table must have dtype"),
    (dict(sl=torch.zeros(2, dtype=torch.int64)), TypeError, "seq_lens must have dtype"),
    (dict(kv=torch.zeros(4, 16, 576, dtype=torch.float32)), TypeError, "kv_cache must be bf16"),
    (dict(q=torch.zeros(2, 576, 16, dtype=torch.bfloat16).transpose(1, 2)), ValueError, "q must be contiguous"),
    (dict(sl=torch.zeros(3, dtype=torch.int32)), ValueError, "seq_lens must have shape"),
    (dict(bt=torch.zeros(3, 2, dtype=torch.int32)), ValueError, r"block_table must be int32 \[batch"),
    (dict(), ValueError, "must be a CUDA tensor"),
])
def test_mla_decode_argument_checks(kw, exc, msg):
    with pytest.raises(exc, match=msg):
        _call_mla(_mla_args(**kw))


def test_output_and_status_checks():
    a = _mla_args()
    with pytest.raises(TypeError, match="out must have dtype"):
        _call_mla(a, out=torch.zeros(2, 16, 512, dtype=torch.float32))
    with pytest.raises(ValueError, match="out must have shape"):
        _call_mla(a, out=torch.zeros(2, 16, 448, dtype=torch.bfloat16))
    with pytest.raises(TypeError, match="lse must have dtype"):
        _call_mla(a, out=torch.zeros(2, 16, 512, dtype=torch.bfloat16), lse=torch.zeros(2, 16, dtype=torch.float64))
    with pytest.raises(TypeError, match="device_status must have dtype"):
        _call_mla(a, out=torch.zeros(2, 16, 512, dtype=torch.bfloat16), device_status=torch.zeros(1))


def test_gqa_sparse_merge_checks():
    q = torch.zeros(2, 8, 128, dtype=torch.bfloat16)
    bt = torch.zeros(2, 2, dtype=torch.int32)
    sl = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(TypeError, match="kv_cache must have 1-byte elements"):
        mqa.gqa_paged_decode(q, torch.zeros(4, 2, 16, 2, 132, dtype=torch.bfloat16), bt, sl, 0.1,
                             kv_dtype="int8_pth")
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        mqa.gqa_paged_decode(q, torch.zeros(4, 2, 16, 2, 132, dtype=torch.uint8), bt, sl, 0.1, kv_dtype="int8_pth")
    a = _mla_args()
    with pytest.raises(ValueError, match="indices must be int32"):
        mqa.mla_decode_sparse(a["q"], a["kv"], a["bt"], a["sl"], torch.zeros(2, 64, dtype=torch.int64), 0.07)
    with pytest.raises(TypeError, match="shard_out must have dtype"):
        mqa.lse_merge(torch.zeros(3, 4, 64), torch.zeros(3, 4))
    with pytest.raises(TypeError, match="shard_lse must have dtype"):
        mqa.lse_merge(torch.zeros(3, 4, 64, dtype=torch.bfloat16), torch.zeros(3, 4, dtype=torch.float64))
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        mqa.lse_merge(torch.zeros(3, 4, 64, dtype=torch.bfloat16), torch.zeros(3, 4))
