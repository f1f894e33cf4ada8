"""The allocation-free MLA entry point, for callers that cannot allocate device
memory (a plugin inside a host program whose pool owns all device memory, or a
hot loop that cannot pay for cudaMalloc/cudaFree synchronisation).

mla_decode_noalloc keeps its split partials in the library's own fixed device
array instead of a caller workspace.  Here it is called through the C ABI
twice in a row and each result is checked against mla_decode (caller
workspace) within the parity tolerances; the second call also shows that the
array's leftover contents from the first call do not leak into the result.
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from mqa_decode_attention_paged_gb300 import _binding as mqa
import synth

from helpers import OUT_ABS, OUT_REL_BF16, OUT_REL_FP8, LSE_ABS, to_device

pytestmark = pytest.mark.gpu


def _call_noalloc(case, dev, splits, out, lse):
    q, kv, bt, sl = dev
    B, H, D = q.shape
    code = mqa.KV_BF16 if case.kv_dtype == "bf16" else mqa.KV_FP8_E4M3
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    rc = mqa.lib.mla_decode_noalloc(P(q), P(kv), P(bt), P(sl), case.scale, case.k_scale, P(out), P(lse),
                                    B, H, D, case.kv_lora_rank, case.num_blocks, case.page,
                                    case.max_blocks, code, splits, None, stream)
    return rc


def _check(a_out, a_lse, b_out, b_lse, fp8):
    rel = OUT_REL_FP8 if fp8 else OUT_REL_BF16
    a_out, b_out = a_out.double().cpu().numpy(), b_out.double().cpu().numpy()
    a_lse, b_lse = a_lse.double().cpu().numpy(), b_lse.double().cpu().numpy()
    assert np.isfinite(a_out).all()
    assert (np.abs(a_out - b_out) <= OUT_ABS + rel * np.abs(b_out)).all()
    assert np.abs(a_lse - b_lse).max() <= LSE_ABS


@pytest.mark.parametrize("name,overrides,splits", [
    ("mla_v2lite", dict(B=16), 16),
    ("tiny_mla", dict(), 3),
    ("mla_v3_fp8", dict(B=4, seq_lens=("uniform", 500, 3000)), 8),
])
def test_noalloc_matches_workspace_entry_point_twice(name, overrides, splits):
    case = synth.workload(name, **overrides)
    dev = to_device(case)
    B, H, _ = dev[0].shape
    R = case.kv_lora_rank
    ref_out, ref_lse = mqa.mla_decode(*dev, case.scale, case.k_scale, num_kv_splits=splits,
                                      kv_lora_rank=R)
    for _ in range(2):
        out = torch.full((B, H, R), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_noalloc(case, dev, splits, out, lse) == mqa.OK
        torch.cuda.synchronize()
        _check(out, lse, ref_out, ref_lse, case.kv_dtype != "bf16")


def test_noalloc_rejects_work_beyond_its_array():
    case = synth.workload("tiny_mla")
    dev = to_device(case)
    B, H, _ = dev[0].shape
    out = torch.empty((B, H, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    # B * H * S * 513 * 4 bytes above 64 MiB
    too_many = mqa.NOALLOC_SCRATCH_BYTES // (B * H * 513 * 4) + 1
    assert _call_noalloc(case, dev, too_many, out, lse) == mqa.ERR_WORKSPACE_TOO_SMALL
