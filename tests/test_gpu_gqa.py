"""GPU parity of GQA paged decode (C ABI -> sm_103a kernels) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import synth

from helpers import assert_close, run_gpu, run_oracle, subset, to_device

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 8, 128), (16, 1, 64), (12, 4, 64), (6, 3, 128)])
@pytest.mark.parametrize("splits", [1, 3])
def test_ragged_shapes(Hq, Hkv, D, splits):
    case = synth.poison(synth.make_gqa_case([1, 15, 16, 17, 40, 0, 100], Hq=Hq, Hkv=Hkv, D=D,
                                            page=16, pool_factor=1.3, seed=21, extra_cols=2))
    out, lse = run_gpu(case, splits)
    ref_out, ref_lse = run_oracle(case)
    assert_close(out, lse, ref_out, ref_lse, what=f"Hq={Hq} Hkv={Hkv} D={D} S={splits}")


@pytest.mark.parametrize("page", [16, 32])
def test_multi_unit(page):
    case = synth.make_gqa_case(("lognormal", 300, 1.0, 2000), B=20, page=page, seed=22)
    ref_out, ref_lse = run_oracle(case)
    for splits in (1, 2, 8, 32):
        out, lse = run_gpu(case, splits)
        assert_close(out, lse, ref_out, ref_lse, what=f"P={page} S={splits}")


def test_single_split_deterministic():
    case = synth.make_gqa_case(("uniform", 10, 900), B=9, seed=23)
    dev = to_device(case)
    a = run_gpu(case, 1, dev)
    b = run_gpu(case, 1, dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    rows = [4, 1]
    c = run_gpu(subset(case, rows), 1)
    assert np.array_equal(c[0], a[0][rows])


def test_full_size_config_sampled():
    case = synth.workload("gqa")
    splits = 32
    out, lse = run_gpu(case, splits)
    rows = [0, 101, 255]
    ref_out, ref_lse = run_oracle(subset(case, rows))
    assert_close(out[rows], lse[rows], ref_out, ref_lse, what="gqa full")
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    vmax = torch.from_numpy(case.kv[:, 1].view(np.int16)).view(torch.bfloat16).abs().max().item()
    assert np.abs(out).max() <= vmax * (1 + 1e-2)
