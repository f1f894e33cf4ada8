"""Failure detection on the GPU without a fault or a hang: the library's test
hook (include/mqa_decode_testing.h) makes the producer of one work unit of
the bf16 GQA kernel withhold all its tiles, so the consumers' bounded wait (2 s) runs out.  The call must
report MQA_ERR_DEVICE_TIMEOUT in the status word, every block must return,
the other request must still be exact, and the context must stay usable."""
import ctypes

import numpy as np
import pytest
import torch

from mqa_decode_attention_paged_gb300 import _binding as mqa
from mqa_decode_attention_paged_gb300 import synth

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
