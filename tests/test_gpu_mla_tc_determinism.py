"""Bitwise determinism and batch invariance of the H = 128 tensor-core MLA path
(the 2-CTA tcgen05 clusters), on batches of the long-context shape: 128 heads,
head 576, pages of 64 tokens, lengths 131072 / 98304 / 65536 / 120000.

With num_kv_splits = 1 every request runs on one cluster in a fixed order
("Triton と MLA" page, データフロー: the batch-invariant branch forces a single
split for a deterministic reduction), so a second run must reproduce the
first bit for bit, and a sub-batch must reproduce the same requests' rows of
the full batch bit for bit.  Split runs (the heuristic's 256 splits) use a
fixed page-to-unit mapping and a fixed merge order, so they are reproducible
run to run as well."""
import numpy as np
import pytest

import synth

from helpers import assert_close, run_gpu, run_oracle, subset, to_device

pytestmark = pytest.mark.gpu

LONG = [131072, 98304, 65536, 120000]


def _long_case(kv_dtype):
    if kv_dtype == "bf16":
        return synth.workload("mla_longctx")
    return synth.make_mla_case(LONG, H=128, D=576, page=64, kv_dtype="fp8_e4m3", k_scale=0.05, seed=1012)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_single_split_bitwise_deterministic_and_batch_invariant(kv_dtype):
    case = _long_case(kv_dtype)
    dev = to_device(case)
    out1, lse1 = run_gpu(case, 1, dev)
    out2, lse2 = run_gpu(case, 1, dev)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2), "S=1 run to run"
    # a sub-batch (other requests, other order, other grid) gives the same rows
    rows = [2, 0]
    out3, lse3 = run_gpu(subset(case, rows), 1)
    assert np.array_equal(out3, out1[rows]) and np.array_equal(lse3, lse1[rows]), "S=1 sub-batch"
    # and the rows are right: a sample of heads of the shortest request
    heads = [0, 63, 64, 127]
    ref_out, ref_lse = run_oracle(subset(case, [2], heads))
    assert_close(out1[np.ix_([2], heads)], lse1[np.ix_([2], heads)], ref_out, ref_lse,
                 fp8=kv_dtype != "bf16", what=f"long {kv_dtype} S=1")


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_split_run_reproducible(kv_dtype):
    case = _long_case(kv_dtype)
    dev = to_device(case)
    a = run_gpu(case, 256, dev)
    b = run_gpu(case, 256, dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_single_split_batch_invariant_mixed_lengths():
    # A ragged batch of short and long requests, fp8 and bf16 alike: each
    # request's rows do not depend on which other requests share the call.
    for kv_dtype in ("bf16", "fp8_e4m3"):
        case = synth.make_mla_case([5000, 1, 0, 64, 777, 12345, 65], H=128, D=576, page=64,
                                   kv_dtype=kv_dtype, k_scale=0.05, seed=1013)
        out, lse = run_gpu(case, 1)
        for rows in ([5], [1, 3], [6, 0, 4]):
            o, l = run_gpu(subset(case, rows), 1)
            assert np.array_equal(o, out[rows]) and np.array_equal(l, lse[rows]), (kv_dtype, rows)
