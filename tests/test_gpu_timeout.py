"""Failure detection on the GPU without a fault or a hang: the library's test
hooks (include/mqa_decode_testing.h) make the producer of one work unit
withhold all its tiles, so the consumers' bounded waits (2 s) run out.  This
is done for the bf16 GQA kernel and for both MLA kernels (the 2-CTA
tensor-core kernel of more than 32 heads, the warp-MMA kernel of 16 heads),
with bf16 and e4m3 caches.  The call must report MQA_ERR_DEVICE_TIMEOUT in
the status word, every block must return, the other request must still be
exact, and the context must stay usable for a normal call."""
import ctypes

import numpy as np
import pytest
import torch

from mqa_decode_attention_paged_gb300 import _binding as mqa
import synth

from helpers import assert_close, run_gpu, run_oracle, subset, to_device

pytestmark = pytest.mark.gpu


def test_withheld_tile_times_out_and_reports(monkeypatch):
    monkeypatch.setenv("MQA_ENABLE_TEST_HOOKS", "1")
    lib = mqa.lib
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fn = lib.mqa_test_gqa_withheld_arrive
    fn.restype = I
    fn.argtypes = [P, P, P, P, F, P, P, I, I, I, I, I, I, I, I, P, SZ, P, P, I]
    case = synth.make_gqa_case([100, 40], Hq=8, Hkv=2, D=128, page=16, seed=41)
    q, kv, bt, sl = to_device(case)
    B, Hq, D = q.shape
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(ptr(q), ptr(kv), ptr(bt), ptr(sl), case.scale, ptr(out), ptr(lse), B, Hq, case.num_kv_heads, D,
            case.num_blocks, case.page, case.max_blocks, 1, None, 0, ptr(status), stream, 0)
    assert rc == mqa.OK
    torch.cuda.synchronize()  # returns: every wait has a time limit
    assert int(status.item()) == mqa.ERR_DEVICE_TIMEOUT
    # request 1 (its own unit with num_kv_splits = 1) was not affected
    ref_out, ref_lse = run_oracle(subset(case, [1]))
    assert_close(out.double().cpu().numpy()[[1]], lse.double().cpu().numpy()[[1]], ref_out, ref_lse,
                 what="other request")
    # the context is usable: a normal call is exact
    o2, l2 = run_gpu(case, 2)
    ref_out, ref_lse = run_oracle(case)
    assert_close(o2, l2, ref_out, ref_lse, what="after the timeout")


def _mla_hook():
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fn = mqa.lib.mqa_test_mla_withheld_arrive
    fn.restype = I
    fn.argtypes = [P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, I, I, P, SZ, P, P, I]
    return fn


@pytest.mark.parametrize("H,kv_dtype", [(128, "bf16"), (128, "fp8_e4m3"), (16, "bf16"), (16, "fp8_e4m3")])
def test_mla_withheld_tile_times_out_and_reports(monkeypatch, H, kv_dtype):
    # More than 32 heads: the 2-CTA tensor-core cluster of unit 0 (both CTAs)
    # waits in vain for its first pair; 16 heads: the warp-MMA block of unit 0
    # waits in vain for its first tile.  Unit 1 (request 1) is untouched.
    monkeypatch.setenv("MQA_ENABLE_TEST_HOOKS", "1")
    fn = _mla_hook()
    case = synth.make_mla_case([300, 200], H=H, page=64, kv_dtype=kv_dtype, k_scale=0.05, seed=42)
    q, kv, bt, sl = to_device(case)
    B, Hh, D = q.shape
    R = case.kv_lora_rank
    out = torch.full((B, Hh, R), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hh), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    kvd = mqa.KV_BF16 if kv_dtype == "bf16" else mqa.KV_FP8_E4M3
    rc = fn(ptr(q), ptr(kv), ptr(bt), ptr(sl), case.scale, case.k_scale, ptr(out), ptr(lse), B, Hh, D, R,
            case.num_blocks, case.page, case.max_blocks, kvd, 1, None, 0, ptr(status), stream, 0)
    assert rc == mqa.OK
    torch.cuda.synchronize()  # returns: every wait has a time limit
    assert int(status.item()) == mqa.ERR_DEVICE_TIMEOUT
    ref_out, ref_lse = run_oracle(subset(case, [1]))
    assert_close(out.double().cpu().numpy()[[1]], lse.double().cpu().numpy()[[1]], ref_out, ref_lse,
                 fp8=kv_dtype != "bf16", what="other request")
    o2, l2 = run_gpu(case, 3)
    ref_out, ref_lse = run_oracle(case)
    assert_close(o2, l2, ref_out, ref_lse, fp8=kv_dtype != "bf16", what="after the timeout")


@pytest.mark.parametrize("warp", [2, 3, 7])
def test_mla_one_softmax_warp_gives_up(monkeypatch, warp):
    # e4m3 cache, 128 heads: one softmax warp of unit 0 stops before its first
    # pair while the other warps of its group go on.  Nothing in the kernel
    # may wait for that warp except a bounded mbarrier wait: the waits that
    # miss its arrivals run out, and the call returns with a timeout.
    monkeypatch.setenv("MQA_ENABLE_TEST_HOOKS", "1")
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fn = mqa.lib.mqa_test_mla_warp_gives_up
    fn.restype = I
    fn.argtypes = [P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, I, P, SZ, P, P, I, I]
    case = synth.make_mla_case([700, 300], H=128, page=64, kv_dtype="fp8_e4m3", k_scale=0.05, seed=43)
    q, kv, bt, sl = to_device(case)
    B, H, D = q.shape
    R = case.kv_lora_rank
    out = torch.full((B, H, R), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = fn(ptr(q), ptr(kv), ptr(bt), ptr(sl), case.scale, case.k_scale, ptr(out), ptr(lse), B, H, D, R,
            case.num_blocks, case.page, case.max_blocks, 1, None, 0, ptr(status), stream, 0, warp)
    assert rc == mqa.OK
    torch.cuda.synchronize()  # returns: no barrier is left waiting for the warp that gave up
    assert int(status.item()) == mqa.ERR_DEVICE_TIMEOUT
    ref_out, ref_lse = run_oracle(subset(case, [1]))
    assert_close(out.double().cpu().numpy()[[1]], lse.double().cpu().numpy()[[1]], ref_out, ref_lse, fp8=True,
                 what="other request")
    o2, l2 = run_gpu(case, 3)
    ref_out, ref_lse = run_oracle(case)
    assert_close(o2, l2, ref_out, ref_lse, fp8=True, what="after the timeout")
