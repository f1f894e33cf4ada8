"""GPU parity of the merge of sequence-shard results (decode context
parallelism: each shard of a request's KV pages decoded on its own, then the
shards' (output, lse) merged by LogSumExp; tutorial page lshu.cn/news/265860,
§12) through the C ABI, against the fp64 oracle.

The shards are decoded by the library itself (one decode call per shard, as
each rank would), merged by `mqa_lse_merge`, and compared with the oracle's
decode of the whole sequences (the bf16 tolerance of the helpers) and with
the oracle's merge of the same shard results (one bf16 rounding apart).
"""
import numpy as np
import pytest
import torch

import oracle
import synth

from helpers import assert_close, run_gpu, run_oracle, subset

pytestmark = pytest.mark.gpu


def _shard_results(case, G, splits, poison_empty=True):
    outs, lses = [], []
    for sh in synth.shard_case(case, G):
        o, l = run_gpu(sh, splits)
        if poison_empty:
            o[np.isneginf(l)] = np.nan  # an empty shard's output must not be read
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)


def _merge_gpu(outs, lses):
    from mqa_decode_attention_paged_gb300 import _binding as mqa
    so = torch.from_numpy(outs).to(torch.bfloat16).cuda()
    sl = torch.from_numpy(lses).to(torch.float32).cuda()
    out, lse = mqa.lse_merge(so, sl)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def _check_against_oracle_merge(out, lse, outs, lses):
    # the kernel merges the same bf16 shard outputs in fp32 and rounds once to
    # bf16: elementwise, half a bf16 ulp of the result (2^-9 relative, taken
    # as 2^-8) plus the fp32 error of the weighted sum, bounded by 1e-5 times
    # the same merge of the outputs' magnitudes
    # (the kernel reads the shard outputs as bf16: round them the same way)
    as_bf16 = torch.from_numpy(np.ascontiguousarray(outs, dtype=np.float32)).to(torch.bfloat16).double().numpy()
    clean = np.nan_to_num(as_bf16)
    ref_o, ref_l = oracle.lse_merge(clean, lses)
    mag, _ = oracle.lse_merge(np.abs(clean), lses)
    assert np.all(np.abs(out - ref_o) <= 2.0 ** -8 * np.abs(ref_o) + 1e-5 * mag + 1e-30)
    fin = np.isfinite(ref_l)
    assert np.array_equal(fin, np.isfinite(lse))
    assert np.abs(lse[fin] - ref_l[fin]).max() <= 1e-4


@pytest.mark.parametrize("G", [1, 2, 3, 5])
@pytest.mark.parametrize("make,fp8", [
    (lambda: synth.make_mla_case([37, 100, 16, 1, 0, 700], H=16, D=576, page=16, seed=61), False),
    (lambda: synth.make_mla_case([300, 64, 129], H=128, D=576, page=64, kv_dtype="fp8_e4m3", k_scale=0.05,
                                 seed=62), True),
    (lambda: synth.make_gqa_case([19, 4, 70, 333], Hq=32, Hkv=8, D=128, page=16, seed=63), False),
], ids=["mla_h16", "mla_h128_fp8", "gqa"])
def test_merged_shards_match_whole_sequence(G, make, fp8):
    case = make()
    ref_out, ref_lse = run_oracle(case)
    outs, lses = _shard_results(case, G, splits=2)
    out, lse = _merge_gpu(outs, lses)
    assert_close(out, lse, ref_out, ref_lse, fp8=fp8, what=f"G={G}")
    _check_against_oracle_merge(out, lse, outs, lses)


def test_all_shards_empty_and_determinism():
    rng = np.random.default_rng(3)
    outs = rng.standard_normal((4, 3, 8, 64)).astype(np.float32)
    lses = rng.standard_normal((4, 3, 8)).astype(np.float32)
    lses[:, 1] = -np.inf           # row group 1: nothing anywhere
    outs[:, 1] = np.nan
    lses[2, 0] = -np.inf           # one empty shard elsewhere
    outs[2, 0] = np.nan
    a = _merge_gpu(outs, lses)
    b = _merge_gpu(outs, lses)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert (a[0][1] == 0).all() and np.isneginf(a[1][1]).all()
    assert np.isfinite(a[0]).all()
    _check_against_oracle_merge(a[0], a[1], outs, lses)


def test_many_shards_and_widths():
    rng = np.random.default_rng(4)
    for G, D in ((37, 8), (64, 136), (3, 4096)):
        outs = rng.standard_normal((G, 5, 2, D)).astype(np.float32)
        lses = (3 * rng.standard_normal((G, 5, 2))).astype(np.float32)
        out, lse = _merge_gpu(outs, lses)
        _check_against_oracle_merge(out, lse, outs.astype(np.float32), lses)


def test_full_size_long_context_over_8_shards():
    # the long-context batch (B=4, H=128, 65k-131k tokens) over 8 shards,
    # checked on sampled (request, head) rows
    case = synth.workload("mla_longctx")
    outs, lses = _shard_results(case, 8, splits=32, poison_empty=False)
    out, lse = _merge_gpu(outs, lses)
    rows, heads = [2], [0, 64, 127]
    ref_out, ref_lse = run_oracle(subset(case, rows, heads))
    assert_close(out[np.ix_(rows, heads)], lse[np.ix_(rows, heads)], ref_out, ref_lse, what="longctx dcp8")
    assert np.isfinite(out).all() and np.isfinite(lse).all()
