"""GPU parity of MLA decode (C ABI -> sm_103a kernels) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import synth

from helpers import assert_close, run_gpu, run_oracle, subset, to_device

pytestmark = pytest.mark.gpu

RAGGED = [1, 15, 16, 17, 63, 64, 65, 200, 0, 129]


@pytest.mark.parametrize("splits", [1, 2, 3])
def test_tiny_config(splits):
    case = synth.workload("tiny_mla")
    out, lse = run_gpu(case, splits)
    ref_out, ref_lse = run_oracle(case)
    assert_close(out, lse, ref_out, ref_lse, what=f"tiny S={splits}")


@pytest.mark.parametrize("splits", [1, 2, 3])
def test_tiny_config_poisoned(splits):
    case = synth.poison(synth.workload("tiny_mla", pool_factor=1.5, extra_cols=3), table_fill=2**31 - 1)
    out, lse = run_gpu(case, splits)
    ref_out, ref_lse = run_oracle(synth.workload("tiny_mla", pool_factor=1.5, extra_cols=3))
    assert np.isfinite(out).all()
    assert_close(out, lse, ref_out, ref_lse, what=f"poisoned S={splits}")


@pytest.mark.parametrize("D", [576, 320])
@pytest.mark.parametrize("page", [16, 64])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
@pytest.mark.parametrize("splits", [1, 4])
def test_ragged_shapes(D, page, kv_dtype, splits):
    case = synth.poison(synth.make_mla_case(RAGGED, H=16, D=D, page=page, kv_dtype=kv_dtype,
                                            k_scale=0.05, pool_factor=1.2, seed=7, extra_cols=1))
    out, lse = run_gpu(case, splits)
    ref_out, ref_lse = run_oracle(case)
    assert_close(out, lse, ref_out, ref_lse, fp8=kv_dtype != "bf16",
                 what=f"D={D} P={page} {kv_dtype} S={splits}")


@pytest.mark.parametrize("D", [576, 320])
@pytest.mark.parametrize("page", [16, 64])
@pytest.mark.parametrize("splits", [1, 4])
def test_tensor_core_path_ragged(D, page, splits):
    # 33..128 heads over a bf16 cache run on the 2-CTA tcgen05 clusters.
    case = synth.poison(synth.make_mla_case(RAGGED, H=128, D=D, page=page, pool_factor=1.2, seed=8,
                                            extra_cols=1))
    out, lse = run_gpu(case, splits)
    ref_out, ref_lse = run_oracle(case)
    assert_close(out, lse, ref_out, ref_lse, what=f"tc D={D} P={page} S={splits}")


@pytest.mark.parametrize("page", [32, 48, 128])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_tensor_core_path_other_page_sizes(page, kv_dtype):
    # Pages of 32 tokens (one box each), 48 (boxes straddle no page, pairs do)
    # and 128 (two pairs per page) on the tensor-core clusters.
    case = synth.poison(synth.make_mla_case(RAGGED + [300, 1000], H=128, D=576, page=page, kv_dtype=kv_dtype,
                                            k_scale=0.05, pool_factor=1.2, seed=19, extra_cols=1))
    for splits in (1, 3):
        out, lse = run_gpu(case, splits)
        ref_out, ref_lse = run_oracle(case)
        assert_close(out, lse, ref_out, ref_lse, fp8=kv_dtype != "bf16", what=f"tc P={page} {kv_dtype} S={splits}")


@pytest.mark.parametrize("D", [576, 320])
@pytest.mark.parametrize("page", [16, 64])
@pytest.mark.parametrize("splits", [1, 4])
def test_tensor_core_path_fp8_ragged(D, page, splits):
    # The e4m3 cache on the tensor-core clusters: the tile is widened to f16 in
    # shared memory and k_scale scales the logits and the output.
    case = synth.poison(synth.make_mla_case(RAGGED, H=128, D=D, page=page, kv_dtype="fp8_e4m3", k_scale=0.05,
                                            pool_factor=1.2, seed=18, extra_cols=1))
    out, lse = run_gpu(case, splits)
    ref_out, ref_lse = run_oracle(case)
    assert_close(out, lse, ref_out, ref_lse, fp8=True, what=f"tc fp8 D={D} P={page} S={splits}")


def test_tensor_core_path_multi_tile_and_rescale():
    # Long pieces (many tiles), and a late key with a much larger logit so the
    # running max jumps by more than 2^8 mid-sequence (forces the O rescale).
    case = synth.make_mla_case([1500, 700, 64, 2200], H=128, page=64, seed=9)
    kv = case.kv.copy()
    blk = case.block_table[0, 1500 // 64]
    qf = torch.from_numpy(case.q[0].view(np.int16)).view(torch.bfloat16).float().numpy()
    kv[blk, 1500 % 64 - 10] = synth.to_bf16_bits(np.clip(qf.mean(axis=0) * 40.0, -200, 200))
    case = synth.replace(case, kv=kv)
    ref_out, ref_lse = run_oracle(case)
    for splits in (1, 5):
        out, lse = run_gpu(case, splits)
        assert_close(out, lse, ref_out, ref_lse, what=f"tc rescale S={splits}")


@pytest.mark.parametrize("H", [1, 5, 16, 32, 33, 40, 64, 80, 100, 128])
def test_head_counts(H):
    case = synth.make_mla_case([77, 300, 1], H=H, page=64, seed=11)
    for splits in (1, 3):
        out, lse = run_gpu(case, splits)
        ref_out, ref_lse = run_oracle(case)
        assert_close(out, lse, ref_out, ref_lse, what=f"H={H} S={splits}")


@pytest.mark.parametrize("H", [33, 64])
def test_mid_head_counts_fp8(H):
    # 33..64 heads of an e4m3 cache on the tcgen05 clusters (M = 128 padded)
    case = synth.poison(synth.make_mla_case(RAGGED, H=H, page=64, kv_dtype="fp8_e4m3", k_scale=0.05,
                                            pool_factor=1.2, seed=44, extra_cols=1))
    for splits in (1, 3):
        out, lse = run_gpu(case, splits)
        ref_out, ref_lse = run_oracle(case)
        assert_close(out, lse, ref_out, ref_lse, fp8=True, what=f"fp8 H={H} S={splits}")


def test_many_units_and_tiles():
    # Spans many work units, several tiles per piece and ragged tails.
    case = synth.make_mla_case(("uniform", 1, 3000), B=24, H=16, page=64, pool_factor=1.5, seed=12)
    ref_out, ref_lse = run_oracle(case)
    for splits in (1, 2, 7, 16, 64):
        out, lse = run_gpu(case, splits)
        assert_close(out, lse, ref_out, ref_lse, what=f"S={splits}")


def test_empty_requests():
    case = synth.make_mla_case([0, 50, 0, 0, 130, 0], H=16, page=16, seed=13)
    for splits in (1, 2, 5):
        out, lse = run_gpu(case, splits)
        assert (out[[0, 2, 3, 5]] == 0).all() and np.isneginf(lse[[0, 2, 3, 5]]).all()
        ref_out, ref_lse = run_oracle(case)
        assert_close(out, lse, ref_out, ref_lse, what=f"empty S={splits}")


def test_single_split_is_bitwise_deterministic_and_batch_invariant():
    case = synth.make_mla_case(("uniform", 100, 4000), B=12, H=16, page=64, seed=14)
    dev = to_device(case)
    out1, lse1 = run_gpu(case, 1, dev)
    out2, lse2 = run_gpu(case, 1, dev)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)
    rows = [3, 7, 0]
    out3, lse3 = run_gpu(subset(case, rows), 1)
    assert np.array_equal(out3, out1[rows]) and np.array_equal(lse3, lse1[rows])


def test_split_run_is_reproducible():
    case = synth.make_mla_case(("uniform", 100, 4000), B=12, H=16, page=64, seed=15)
    dev = to_device(case)
    a = run_gpu(case, 8, dev)
    b = run_gpu(case, 8, dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_request_isolation():
    case = synth.make_mla_case([300, 500], H=16, page=16, seed=16)
    out, lse = run_gpu(case, 1)
    kv = case.kv.copy()
    n1 = (500 + 15) // 16
    kv[case.block_table[1, :n1]] = synth.to_bf16_bits(np.full(kv.shape[1:], 2.0, np.float32))
    out2, lse2 = run_gpu(synth.replace(case, kv=kv), 1)
    assert np.array_equal(out[0], out2[0]) and np.array_equal(lse[0], lse2[0])


def test_device_checks_report_bad_block_ids_and_lengths():
    case = synth.make_mla_case([40, 70], H=16, page=16, seed=17)
    bt = case.block_table.copy()
    bt[1, 2] = case.num_blocks + 5  # out of range
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_gpu(synth.replace(case, block_table=bt), 2, status=status)
    assert int(status.item()) == 5
    sl = case.seq_lens.copy()
    sl[0] = case.max_blocks * 16 + 1  # longer than the block table allows
    status.zero_()
    out, _ = run_gpu(synth.replace(case, seq_lens=sl), 1, status=status)
    assert int(status.item()) == 5 and np.isfinite(out).all()


@pytest.mark.parametrize("name,rows,heads,splits", [
    ("mla_v2lite", [0, 17, 63], None, 16),
    ("mla_v3_fp8", [5, 77], list(range(0, 128, 37)), 64),
    ("mla_longctx", [2], [0, 64, 127], 256),
    ("mla_longctx", [1], [3], 1),
])
def test_full_size_configs_sampled(name, rows, heads, splits):
    case = synth.workload(name)
    out, lse = run_gpu(case, splits)
    sub = subset(case, rows, heads)
    ref_out, ref_lse = run_oracle(sub)
    got_o = out[rows] if heads is None else out[np.ix_(rows, heads)]
    got_l = lse[rows] if heads is None else lse[np.ix_(rows, heads)]
    assert_close(got_o, got_l, ref_out, ref_lse, fp8=case.kv_dtype != "bf16", what=name)
    # Properties of every output row: finite, and (a convex combination of V
    # rows) no entry larger than the largest |V| entry of the cache.
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    R = case.kv_lora_rank
    if case.kv_dtype == "bf16":
        vmax = torch.from_numpy(case.kv[..., :R].view(np.int16)).view(torch.bfloat16).abs().max().item()
    else:
        vmax = torch.from_numpy(case.kv[..., :R]).view(torch.float8_e4m3fn).float().abs().max().item()
        vmax *= case.k_scale
    assert np.abs(out).max() <= vmax * (1 + 1e-2)
