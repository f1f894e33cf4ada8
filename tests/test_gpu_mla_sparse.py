"""GPU parity of sparse (top-k) MLA decode (each query attends only the positions its
request's index list selects, found through the block table: tutorial page
lshu.cn/news/265860, §13) against the fp64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth

from helpers import assert_close, subset, to_device

pytestmark = pytest.mark.gpu

RAGGED = [1, 3, 40, 0, 63, 64, 65, 200, 129, 1000, 2500]


def run_sparse(case, idx, splits, dev=None, status=None):
    from mqa_decode_attention_paged_gb300 import _binding as mqa
    q, kv, bt, sl = dev if dev is not None else to_device(case)
    B, H, D = q.shape
    R = case.kv_lora_rank
    # NaN-filled outputs and workspace: anything left unwritten shows up
    out = torch.full((B, H, R), float("nan"), dtype=torch.bfloat16, device=q.device)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=q.device)
    need = mqa.mla_decode_workspace_bytes(B, H, R, splits)
    ws = torch.full((max(need, 16),), 0xFF, dtype=torch.uint8, device=q.device)
    ii = torch.from_numpy(np.ascontiguousarray(idx, dtype=np.int32)).to(q.device)
    out, lse = mqa.mla_decode_sparse(q, kv, bt, sl, ii, case.scale, case.k_scale, out=out, lse=lse,
                                     num_kv_splits=splits, kv_lora_rank=R, workspace=ws, device_status=status)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def oracle_sparse(case, idx):
    return oracle.mla_decode_sparse(case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens,
                                    np.ascontiguousarray(idx, dtype=np.int32), case.scale, case.k_scale,
                                    kv_lora_rank=case.kv_lora_rank)


def check(case, idx, splits, what):
    out, lse = run_sparse(case, idx, splits)
    ref_out, ref_lse = oracle_sparse(case, idx)
    assert_close(out, lse, ref_out, ref_lse, fp8=case.kv_dtype != "bf16", what=what)


@pytest.mark.parametrize("H", [1, 16, 40, 128])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("page,splits", [(64, 1), (16, 3), (8, 2)])
@pytest.mark.parametrize("topk", [40, 300])
def test_sparse_parity(H, kv_dtype, page, splits, topk):
    # ragged lengths (0, shorter than topk: -1 padding), 20 % extra padding,
    # NaN in every cache slot no token owns: none of it may reach a result
    case = synth.poison(synth.make_mla_case(RAGGED, H=H, page=page, kv_dtype=kv_dtype, k_scale=0.05,
                                            pool_factor=1.2, seed=61))
    idx = synth.draw_topk_indices(np.random.default_rng(62), case.seq_lens, topk, pad=0.2)
    check(case, idx, splits, f"sparse H={H} {kv_dtype} P={page} S={splits} topk={topk}")


@pytest.mark.parametrize("H", [16, 128])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_sparse_parity_head_320(H, kv_dtype):
    # head 320 (kv_lora_rank 256): a row is 640 (bf16) or 320 (e4m3) bytes,
    # so the four-row gathers take boxes of 84 or 40 eight-byte elements
    case = synth.poison(synth.make_mla_case(RAGGED, H=H, D=320, page=16, kv_dtype=kv_dtype, k_scale=0.05,
                                            pool_factor=1.2, seed=63))
    idx = synth.draw_topk_indices(np.random.default_rng(64), case.seq_lens, 300, pad=0.2)
    for splits in (1, 3):
        check(case, idx, splits, f"sparse D=320 H={H} {kv_dtype} S={splits}")


def test_out_of_range_and_duplicate_entries():
    case = synth.poison(synth.make_mla_case([90, 200, 5], H=16, page=16, seed=63))
    idx = synth.draw_topk_indices(np.random.default_rng(64), case.seq_lens, 64)
    # negative, at the end, far past the end (and past what the table maps)
    # entries select nothing; a repeated position counts twice
    extra = np.array([[-1, 90, 1 << 20, 3, 3], [-7, 200, 5000, 0, 199], [5, 6, -2, 4, 4]], np.int32)
    idx = np.concatenate([idx, extra], axis=1)
    for splits in (1, 2):
        check(case, idx, splits, f"out-of-range S={splits}")


def test_selecting_every_position_matches_dense_oracle():
    case = synth.make_mla_case([37, 100, 1, 64, 513], H=16, page=64, seed=65)
    topk = int(case.seq_lens.max())
    idx = np.full((case.batch, topk), -1, np.int32)
    for b, n in enumerate(case.seq_lens):
        idx[b, :n] = np.arange(n)
    out, lse = run_sparse(case, idx, 2)
    ref_out, ref_lse = oracle.mla_decode(case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens,
                                         case.scale, kv_lora_rank=case.kv_lora_rank)
    assert_close(out, lse, ref_out, ref_lse, what="sparse(all) vs dense")


def test_single_split_is_deterministic():
    case = synth.make_mla_case([500, 3000, 77], H=16, page=64, seed=66)
    idx = synth.draw_topk_indices(np.random.default_rng(67), case.seq_lens, 512)
    dev = to_device(case)
    a = run_sparse(case, idx, 1, dev)
    b = run_sparse(case, idx, 1, dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_bad_block_id_is_reported_and_skipped():
    case = synth.make_mla_case([300, 200], H=16, page=16, seed=68)
    idx = synth.draw_topk_indices(np.random.default_rng(69), case.seq_lens, 128)
    bt = case.block_table.copy()
    bt[0, 3] = -1                      # page 3 of request 0 (tokens 48..63)
    bt[1, 2] = case.num_blocks + 5     # page 2 of request 1 (tokens 32..47)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_sparse(synth.replace(case, block_table=bt), idx, 2, status=status)
    assert int(status.item()) == 5
    # the rows of those pages are skipped: the result is the oracle's over
    # the remaining entries
    drop = idx.copy()
    drop[0][(drop[0] >= 48) & (drop[0] < 64)] = -1
    drop[1][(drop[1] >= 32) & (drop[1] < 48)] = -1
    ref_out, ref_lse = oracle_sparse(case, drop)
    assert_close(out, lse, ref_out, ref_lse, what="bad block ids")


def test_full_size_sparse_sampled():
    # the bench's sparse workload (64 requests of 16k..40k tokens, 2048
    # selected positions each, 16 heads) in its timed launch configuration
    # (splits as mqa_num_kv_splits gives for max_seq_len = topk), checked on
    # sampled requests
    from mqa_decode_attention_paged_gb300 import _binding as mqa
    case = synth.workload("mla_sparse")
    idx = case.meta["indices"]
    splits = mqa.num_kv_splits(idx.shape[1], mqa.device_sm_count(), False)
    out, lse = run_sparse(case, idx, splits)
    rows = [0, 41]
    ref_out, ref_lse = oracle_sparse(subset(case, rows), idx[rows])
    assert_close(out[rows], lse[rows], ref_out, ref_lse, what="mla_sparse")
    assert np.isfinite(out).all() and np.isfinite(lse).all()
