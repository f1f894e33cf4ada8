"""GPU parity of ``mla_decode_fixed_splits`` (one work unit per request and
split, every request cut into num_kv_splits equal page ranges, as the Triton
MLA backend splits: "Triton と MLA" page, 主要ファイル / データフロー) against
the fp64 oracle, on the warp-MMA path (16 heads) and the tensor-core path
(128 and 64 heads), bf16 and e4m3 caches, ragged and empty requests and a
poisoned cache; and its stated property: at ANY split count the result is
bitwise reproducible and independent of the rest of the batch."""
import numpy as np
import pytest
import torch

from mqa_decode_attention_paged_gb300 import _binding as mqa
import synth

from helpers import assert_close, run_gpu, run_oracle, subset, to_device

pytestmark = pytest.mark.gpu

RAGGED = [0, 1, 63, 64, 65, 300, 1000, 17, 129, 2000]


def run_fixed(case, splits, dev=None):
    q, kv, bt, sl = dev if dev is not None else to_device(case)
    B, H, D = q.shape
    R = case.kv_lora_rank
    need = mqa.mla_decode_workspace_bytes(B, H, R, splits)
    # NaN-filled workspace and outputs: an unwritten partial or output shows
    ws = torch.full((max(need, 16),), 0xFF, dtype=torch.uint8, device=q.device)
    out = torch.full((B, H, R), float("nan"), dtype=torch.bfloat16, device=q.device)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=q.device)
    mqa.mla_decode_fixed_splits(q, kv, bt, sl, case.scale, case.k_scale, out=out, lse=lse, num_kv_splits=splits,
                                kv_lora_rank=R, workspace=ws)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("H,kv_dtype,page", [(16, "bf16", 16), (16, "fp8_e4m3", 64), (128, "bf16", 64),
                                             (128, "fp8_e4m3", 64), (64, "bf16", 32), (128, "bf16", 16)])
def test_parity_ragged_poisoned(H, kv_dtype, page):
    fp8 = kv_dtype != "bf16"
    case = synth.poison(synth.make_mla_case(RAGGED, H=H, page=page, kv_dtype=kv_dtype, k_scale=0.05 if fp8 else 1.0,
                                            pool_factor=1.2, seed=140 + H + page, extra_cols=1))
    ref_out, ref_lse = run_oracle(case)
    dev = to_device(case)
    for splits in (1, 2, 3, 4, 16):
        out, lse = run_fixed(case, splits, dev)
        assert np.isfinite(out).all()
        assert_close(out, lse, ref_out, ref_lse, fp8=fp8, what=f"fixed H={H} {kv_dtype} P={page} S={splits}")


@pytest.mark.parametrize("H,kv_dtype", [(16, "bf16"), (128, "bf16"), (128, "fp8_e4m3")])
def test_batch_invariant_and_reproducible_at_any_split_count(H, kv_dtype):
    case = synth.make_mla_case(("uniform", 1, 3000), B=12, H=H, page=64, kv_dtype=kv_dtype, k_scale=0.05,
                               seed=150 + H)
    dev = to_device(case)
    rows = [9, 2, 5]
    sub = subset(case, rows)
    for splits in (2, 5, 16):
        a = run_fixed(case, splits, dev)
        b = run_fixed(case, splits, dev)
        assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
        c = run_fixed(sub, splits)
        assert np.array_equal(c[0], a[0][rows]) and np.array_equal(c[1], a[1][rows]), f"S={splits}"


def test_one_split_is_the_per_request_mode():
    case = synth.make_mla_case(RAGGED, H=128, page=64, seed=160)
    a = run_fixed(case, 1)
    b = run_gpu(case, 1)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_more_splits_than_pages_and_empty_batch_members():
    # most ranges are empty: requests of 0, 1 and 2 pages over 64 splits
    case = synth.make_mla_case([0, 16, 17, 32, 0, 5], H=16, page=16, seed=161)
    out, lse = run_fixed(case, 64)
    ref_out, ref_lse = run_oracle(case)
    assert (out[[0, 4]] == 0).all() and np.isneginf(lse[[0, 4]]).all()
    assert_close(out, lse, ref_out, ref_lse, what="S=64 over short requests")
    case = synth.make_mla_case([0, 64, 65, 128, 0, 5], H=128, page=64, seed=162)
    out, lse = run_fixed(case, 64)
    ref_out, ref_lse = run_oracle(case)
    assert (out[[0, 4]] == 0).all() and np.isneginf(lse[[0, 4]]).all()
    assert_close(out, lse, ref_out, ref_lse, what="S=64 over short requests, 128 heads")
