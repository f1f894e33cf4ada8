"""GPU parity of decode context parallelism through the C ABI.

- ``mqa_dcp_scale_shard`` against the oracle's share e^{lse_g - lse} O_g on
  seeded shard results (rows where some or every shard is empty included),
  in the head-chunk order a reduce-scatter wants, with fp32 and bf16 output.
- The whole path with the ranks taken one after another on one GPU: the
  library plans each rank's pages (``mqa_dcp_shard``, both layouts), decodes
  them (``mla_decode`` / ``gqa_paged_decode``), and the shards are merged both
  ways: stacked as an all-gather leaves them and merged by ``mqa_lse_merge``,
  or scaled by ``mqa_dcp_scale_shard`` and summed over the ranks as a sum
  reduce-scatter does.  Both must give the oracle's decode of the whole
  sequences.  (The collectives themselves are covered on CPU ranks in
  test_dcp_host.py.)
"""
import numpy as np
import pytest
import torch

import oracle
from mqa_decode_attention_paged_gb300 import _binding as mqa
import synth

from helpers import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu


def _shard_inputs(G, B, H, D, seed):
    rng = np.random.default_rng(seed)
    outs = synth.to_bf16_bits(rng.standard_normal((G, B, H, D), dtype=np.float32))
    lses = (rng.standard_normal((G, B, H)) * 6.0).astype(np.float32)
    lses[rng.random((G, B, H)) < 0.15] = -np.inf   # empty shards
    lses[:, 1, : H // 2] = -np.inf                 # rows no shard holds a token of
    if G > 1:
        lses[0, 2] = lses[1, 2] + 30.0             # one shard far ahead
    return outs, lses


def _bf16_to_f64(bits):
    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("G,H,D", [(1, 16, 512), (2, 16, 512), (3, 6, 256), (4, 128, 512), (8, 32, 128),
                                   (2, 2, 8)])
@pytest.mark.parametrize("fp32", [True, False])
def test_scale_shard_matches_oracle_share(G, H, D, fp32):
    B = 5
    outs, lses = _shard_inputs(G, B, H, D, seed=90 + G + D)
    gl = torch.from_numpy(lses).cuda()
    hc = H // G
    for rank in range(G):
        so = torch.from_numpy(outs[rank].view(np.int16)).view(torch.bfloat16).cuda()
        scaled = torch.full((G, B, hc, D), float("nan"), dtype=torch.float32 if fp32 else torch.bfloat16,
                            device="cuda")
        lse = torch.full((B, H), float("nan"), dtype=torch.float32, device="cuda")
        mqa.dcp_scale_shard(so, gl, rank, scaled=scaled, lse=lse, scaled_fp32=fp32)
        torch.cuda.synchronize()
        share, ref_lse = oracle.lse_share(_bf16_to_f64(outs[rank]), lses.astype(np.float64), rank)
        ref = share.reshape(B, G, hc, D).transpose(1, 0, 2, 3)
        got = scaled.double().cpu().numpy()
        # fp32: the weight e^{lse_g - m} / sum is good to ~1e-6 relative;
        # bf16 adds one rounding of the product
        rel = 1e-5 if fp32 else 2.0 ** -8
        assert np.all(np.abs(got - ref) <= 1e-30 + rel * np.abs(ref)), f"rank {rank}"
        lg = lse.double().cpu().numpy()
        fin = np.isfinite(ref_lse)
        assert np.array_equal(np.isfinite(lg), fin) and np.isneginf(lg[~fin]).all()
        assert np.all(np.abs(lg[fin] - ref_lse[fin]) <= 1e-5 * np.maximum(1.0, np.abs(ref_lse[fin])))


def test_scale_shard_argument_checks():
    so = torch.zeros((2, 4, 64), dtype=torch.bfloat16, device="cuda")
    gl = torch.zeros((3, 2, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):          # 4 heads over 3 ranks
        mqa.dcp_scale_shard(so, gl, 0)
    gl = torch.zeros((2, 2, 4), dtype=torch.float32, device="cuda")
    with pytest.raises(mqa.MqaError):        # rank outside [0, G)
        mqa.dcp_scale_shard(so, gl, 2)
    with pytest.raises(TypeError):
        mqa.dcp_scale_shard(so, gl.double(), 0)


def _rank_results(case, G, layout, splits):
    outs, lses = [], []
    for g in range(G):
        table, lens = mqa.dcp_shard(case.block_table, case.seq_lens, case.page, G, g, layout)
        sh = synth.replace(case, block_table=table, seq_lens=lens)
        o, l = run_gpu(sh, splits)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


CASES = {
    "mla_h16": (lambda: synth.make_mla_case([37, 100, 16, 1, 0, 700, 17], H=16, D=576, page=16, seed=64), False),
    "mla_h128_fp8": (lambda: synth.make_mla_case([300, 64, 129, 1000], H=128, D=576, page=64, kv_dtype="fp8_e4m3",
                                                 k_scale=0.05, seed=65), True),
    "mla_h128_bf16": (lambda: synth.make_mla_case([513, 64, 1, 2000], H=128, D=576, page=64, seed=66), False),
    "gqa": (lambda: synth.make_gqa_case([19, 4, 70, 333], Hq=32, Hkv=8, D=128, page=16, seed=67), False),
}


@pytest.mark.parametrize("layout", ["round_robin", "contiguous"])
@pytest.mark.parametrize("G", [2, 4])
@pytest.mark.parametrize("name", list(CASES))
def test_ranks_on_one_gpu_equal_whole_sequence(name, G, layout):
    make, fp8 = CASES[name]
    case = make()
    ref_out, ref_lse = run_oracle(case)
    outs, lses = _rank_results(case, G, layout, splits=2)
    B, H, D = outs.shape[1:]
    # the all-gather exchange: stacked shards, merged by mqa_lse_merge
    so = torch.from_numpy(outs).to(torch.bfloat16).cuda()   # exact: bf16 decode outputs
    sl = torch.from_numpy(lses).to(torch.float32).cuda()
    out, lse = mqa.lse_merge(so, sl)
    torch.cuda.synchronize()
    assert_close(out.double().cpu().numpy(), lse.double().cpu().numpy(), ref_out, ref_lse, fp8=fp8,
                 what=f"all-gather merge {name} G={G} {layout}")
    # the reduce-scatter exchange: each rank's scaled shard, summed over ranks
    total = np.zeros((G, B, H // G, D))
    for g in range(G):
        scaled, mlse = mqa.dcp_scale_shard(so[g].contiguous(), sl, g)
        torch.cuda.synchronize()
        total += scaled.double().cpu().numpy()
    merged = total.transpose(1, 0, 2, 3).reshape(B, H, D)
    assert_close(merged, mlse.double().cpu().numpy(), ref_out, ref_lse, fp8=fp8,
                 what=f"reduce-scatter merge {name} G={G} {layout}")
