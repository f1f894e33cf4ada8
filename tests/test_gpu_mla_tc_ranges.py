"""Value ranges on the H = 128 tensor-core MLA path.

- Every finite e4m3 code (254 of the 256; 0x7F / 0xFF are NaN) in valid
  tokens, K and V columns alike, against the fp64 oracle on the same decoded
  values: the e4m3 -> f16 widening in shared memory must be exact, the
  subnormal codes (exponent field 0) included.
- Query magnitudes.  With a bf16 cache the query stays bf16, so a power of
  two on q (compensated by the softmax scale) changes nothing, even at 2^17 or
  2^-20.  With an e4m3 cache this path takes the query in f16 (the header
  states the range): powers of two that keep it inside f16's normal range
  (2^12, 2^-8 here) still change nothing, and a row with an entry beyond
  +-65504 affects no other row.
"""
import numpy as np
import pytest
import torch

import synth

from helpers import assert_close, run_gpu, run_oracle

pytestmark = pytest.mark.gpu

LENS = [70, 1, 300, 129, 64, 1000]


def _all_codes_case(seed, H=128, D=576, page=64):
    case = synth.make_mla_case(LENS, H=H, D=D, page=page, kv_dtype="fp8_e4m3", k_scale=0.05, pool_factor=1.2,
                               seed=seed)
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    kv = case.kv.copy()
    rng = np.random.default_rng(seed)
    for b, n in enumerate(case.seq_lens):
        for t in range(int(n)):
            blk, slot = case.block_table[b, t // page], t % page
            kv[blk, slot] = finite[(rng.integers(0, 254) + np.arange(D)) % 254]
    return synth.replace(case, kv=kv)


@pytest.mark.parametrize("D", [576, 320])
def test_every_finite_e4m3_code(D):
    case = _all_codes_case(61 + D, D=D)
    ref_out, ref_lse = run_oracle(case)
    for splits in (1, 3):
        out, lse = run_gpu(case, splits)
        assert np.isfinite(out).all()
        assert_close(out, lse, ref_out, ref_lse, fp8=True, what=f"all e4m3 codes D={D} S={splits}")


def _scaled_query_case(kv_dtype, log2_factor):
    base = synth.make_mla_case(LENS, H=128, page=64, kv_dtype=kv_dtype, k_scale=0.05, pool_factor=1.2, seed=62)
    qf = torch.from_numpy(base.q.view(np.int16)).view(torch.bfloat16).double()
    q = (qf * 2.0 ** log2_factor).to(torch.bfloat16)  # exact: a power of two on bf16 values
    assert torch.isfinite(q.double()).all() and (q.double() != 0).any()
    return synth.replace(base, q=np.ascontiguousarray(q.view(torch.int16).numpy().view(np.uint16)),
                         scale=base.scale * 2.0 ** -log2_factor)


@pytest.mark.parametrize("kv_dtype,log2_factor", [("bf16", 17), ("bf16", -20), ("fp8_e4m3", 12),
                                                  ("fp8_e4m3", -8)])
def test_query_magnitudes(kv_dtype, log2_factor):
    case = _scaled_query_case(kv_dtype, log2_factor)
    ref_out, ref_lse = run_oracle(case)
    for splits in (1, 4):
        out, lse = run_gpu(case, splits)
        assert np.isfinite(out).all() and np.isfinite(lse).all()
        assert_close(out, lse, ref_out, ref_lse, fp8=kv_dtype != "bf16",
                     what=f"|q| x 2^{log2_factor} {kv_dtype} S={splits}")


def test_query_beyond_f16_affects_only_its_row():
    # One row of one request gets an entry of 2^17 (no f16 value): on the e4m3
    # tensor-core path that row's result is undefined (the header says so),
    # every other row stays exact; with 32 heads (the warp-MMA path, bf16
    # query) the same entry is exact as well.
    base = synth.make_mla_case(LENS, H=128, page=64, kv_dtype="fp8_e4m3", k_scale=0.05, pool_factor=1.2, seed=63)
    q = base.q.copy()
    q[2, 40, 7] = synth.to_bf16_bits(np.array([131072.0], np.float32))[0]
    case = synth.replace(base, q=q)
    ref_out, ref_lse = run_oracle(case)
    for splits in (1, 3):
        out, lse = run_gpu(case, splits)
        keep = np.ones(out.shape[:2], bool)
        keep[2, 40] = False
        assert_close(out[keep], lse[keep], ref_out[keep], ref_lse[keep], fp8=True, what=f"other rows S={splits}")
    small = synth.replace(case, q=np.ascontiguousarray(case.q[:, :32]))
    small = synth.replace(small, q=small.q.copy())
    small.q[2, 8, 7] = synth.to_bf16_bits(np.array([131072.0], np.float32))[0]
    out, lse = run_gpu(small, 2)
    ref_out, ref_lse = run_oracle(small)
    assert np.isfinite(out).all()
    keep = np.ones(out.shape[:2], bool)
    keep[2, 8] = False
    assert_close(out[keep], lse[keep], ref_out[keep], ref_lse[keep], fp8=True, what="2^17 entry, 32 heads")
    # that row's logits reach ~1e4: its lse is good to fp32's relative
    # precision there, its output to the usual tolerance
    assert abs(lse[2, 8] - ref_lse[2, 8]) <= 1e-6 * abs(ref_lse[2, 8])
    assert np.all(np.abs(out[2, 8] - ref_out[2, 8]) <= 1e-2 + 3e-2 * np.abs(ref_out[2, 8]))
