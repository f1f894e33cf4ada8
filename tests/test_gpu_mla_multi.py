"""GPU parity of multi-token MLA decode (q_len query tokens per request, each seeing the
keys up to its own position: tutorial page lshu.cn/news/265860, §10) against the fp64
oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth

from helpers import assert_close, run_gpu, to_device

pytestmark = pytest.mark.gpu

# lengths below q_len leave the first queries with nothing to see
RAGGED = [1, 3, 8, 15, 16, 17, 63, 64, 65, 200, 0, 129, 1000]


def run_multi(case, q_len, splits, dev=None):
    from mqa_decode_attention_paged_gb300 import _binding as mqa
    q, kv, bt, sl = dev if dev is not None else to_device(case)
    B, rows, D = q.shape
    H = rows // q_len
    R = case.kv_lora_rank
    out = torch.full((B, q_len, H, R), float("nan"), dtype=torch.bfloat16, device=q.device)
    lse = torch.full((B, q_len, H), float("nan"), dtype=torch.float32, device=q.device)
    need = mqa.mla_decode_workspace_bytes(B, rows, R, splits)
    ws = torch.full((max(need, 16),), 0xFF, dtype=torch.uint8, device=q.device)
    out, lse = mqa.mla_decode_multi(q.view(B, q_len, H, D), kv, bt, sl, case.scale, case.k_scale, out=out,
                                    lse=lse, num_kv_splits=splits, kv_lora_rank=R, workspace=ws)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def oracle_multi(case, q_len):
    B, rows, D = case.q.shape
    return oracle.mla_decode_multi(case.q.reshape(B, q_len, rows // q_len, D), case.kv, case.kv_dtype,
                                   case.block_table, case.seq_lens, case.scale, case.k_scale,
                                   kv_lora_rank=case.kv_lora_rank)


def check(case, q_len, splits, what):
    out, lse = run_multi(case, q_len, splits)
    ref_out, ref_lse = oracle_multi(case, q_len)
    assert_close(out.reshape(out.shape[0], -1, out.shape[-1]), lse.reshape(lse.shape[0], -1),
                 ref_out.reshape(out.shape[0], -1, out.shape[-1]), ref_lse.reshape(lse.shape[0], -1),
                 fp8=case.kv_dtype != "bf16", what=what)


@pytest.mark.parametrize("q_len,H", [(2, 8), (4, 8), (2, 16), (3, 5)])
@pytest.mark.parametrize("page", [16, 64])
@pytest.mark.parametrize("splits", [1, 3])
def test_multi_warp_mma_path(q_len, H, page, splits):
    # q_len x H <= 32 rows: the warp-MMA kernel, 16 rows per block
    case = synth.poison(synth.make_mla_case(RAGGED, H=q_len * H, page=page, pool_factor=1.2, seed=41,
                                            extra_cols=1))
    check(case, q_len, splits, f"mma q_len={q_len} H={H} P={page} S={splits}")


@pytest.mark.parametrize("q_len,H", [(8, 16), (4, 32), (6, 12), (4, 16), (3, 11)])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("page,splits", [(64, 1), (64, 4), (16, 3)])
def test_multi_tensor_core_path(q_len, H, kv_dtype, page, splits):
    # 33..128 rows: the 2-CTA tcgen05 clusters
    case = synth.poison(synth.make_mla_case(RAGGED, H=q_len * H, page=page, kv_dtype=kv_dtype, k_scale=0.05,
                                            pool_factor=1.2, seed=42, extra_cols=1))
    check(case, q_len, splits, f"tc q_len={q_len} H={H} {kv_dtype} P={page} S={splits}")


@pytest.mark.parametrize("H", [16, 128])
def test_one_query_is_plain_decode(H):
    case = synth.make_mla_case([77, 300, 1, 0], H=H, page=64, seed=43)
    dev = to_device(case)
    for splits in (1, 3):
        out_m, lse_m = run_multi(case, 1, splits, dev)
        out, lse = run_gpu(case, splits, dev)
        assert np.array_equal(out_m[:, 0], out) and np.array_equal(lse_m[:, 0], lse)


def test_full_size_mtp_sampled():
    # the bench's multi-token workload (64 requests of 1024..8192 tokens, 8 new
    # positions, 16 heads -> 128 rows) in its timed launch configuration,
    # checked on sampled requests
    from helpers import subset
    case = synth.workload("mla_mtp")
    q_len = case.meta["q_len"]
    out, lse = run_multi(case, q_len, 16)
    rows = [0, 33]
    ref_out, ref_lse = oracle_multi(subset(case, rows), q_len)
    B = len(rows)
    assert_close(out[rows].reshape(B, -1, out.shape[-1]), lse[rows].reshape(B, -1),
                 ref_out.reshape(B, -1, ref_out.shape[-1]), ref_lse.reshape(B, -1), what="mla_mtp")
    assert np.isfinite(out).all() and np.isfinite(lse).all()
