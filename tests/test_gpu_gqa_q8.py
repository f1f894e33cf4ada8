"""GPU parity of GQA paged decode over 8-bit caches (C ABI -> sm_103a kernel)
against the fp64 oracle: e4m3 with one k_scale / v_scale, and the
per-token-head e4m3 / int8 formats whose rows carry their own scale.

Tolerance: the fp8 bound of the helpers (|out - ref| <= 1e-2 + 3e-2 |ref|,
|lse - ref| <= 1e-3), the oracle running on the same codes and scales.
"""
import numpy as np
import pytest
import torch

import synth

from helpers import assert_close, run_gpu, run_oracle, subset, to_device

pytestmark = pytest.mark.gpu

FORMATS = [dict(kv_dtype="fp8_e4m3", k_scale=0.05, v_scale=0.03),
           dict(kv_dtype="fp8_e4m3_pth"),
           dict(kv_dtype="int8_pth"),
           dict(kv_dtype="int4_pth")]
IDS = ["e4m3", "e4m3_pth", "int8_pth", "int4_pth"]


@pytest.mark.parametrize("fmt", FORMATS, ids=IDS)
@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (8, 8, 128), (16, 1, 64), (12, 4, 64), (6, 3, 128),
                                      (7, 7, 64), (5, 5, 128)])
@pytest.mark.parametrize("splits", [1, 3])
def test_ragged_shapes(fmt, Hq, Hkv, D, splits):
    # lengths around the 16-token tile (tails of 1, 15, 16, 17 tokens), an
    # empty request, NaN-poisoned padding and block-table tails
    case = synth.poison(synth.make_gqa_case([1, 15, 16, 17, 40, 0, 100], Hq=Hq, Hkv=Hkv, D=D, page=16,
                                            pool_factor=1.3, seed=31, extra_cols=2, **fmt))
    out, lse = run_gpu(case, splits)
    ref_out, ref_lse = run_oracle(case)
    assert_close(out, lse, ref_out, ref_lse, fp8=True, what=f"{fmt['kv_dtype']} Hq={Hq} Hkv={Hkv} D={D} S={splits}")


@pytest.mark.parametrize("fmt", FORMATS, ids=IDS)
@pytest.mark.parametrize("page", [16, 32, 64])
def test_multi_unit(fmt, page):
    case = synth.make_gqa_case(("lognormal", 300, 1.0, 2000), B=20, page=page, seed=32, **fmt)
    ref_out, ref_lse = run_oracle(case)
    for splits in (1, 2, 8, 32):
        out, lse = run_gpu(case, splits)
        assert_close(out, lse, ref_out, ref_lse, fp8=True, what=f"{fmt['kv_dtype']} P={page} S={splits}")


@pytest.mark.parametrize("fmt", FORMATS, ids=IDS)
def test_single_split_deterministic(fmt):
    case = synth.make_gqa_case(("uniform", 10, 900), B=9, seed=33, **fmt)
    dev = to_device(case)
    a = run_gpu(case, 1, dev)
    b = run_gpu(case, 1, dev)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    rows = [4, 1]
    c = run_gpu(subset(case, rows), 1)
    assert np.array_equal(c[0], a[0][rows])


def test_per_token_scales_are_applied_per_row():
    # Scale one token's K row and V row of one KV head by large factors (the
    # codes unchanged): only the query heads of that KV head change, as the
    # oracle says.
    case = synth.make_gqa_case([48, 20], Hq=8, Hkv=2, D=128, page=16, kv_dtype="int8_pth", seed=34)
    kv = case.kv.copy()
    blk, slot = case.block_table[0, 1], 5  # token 21 of request 0, KV head 1
    for plane, f in ((0, 4.0), (1, 8.0)):
        sc = np.ascontiguousarray(kv[blk, plane, slot, 1, -4:]).view("<f4") * np.float32(f)
        kv[blk, plane, slot, 1, -4:] = sc.view(np.uint8)
    mod = synth.replace(case, kv=kv)
    out, lse = run_gpu(mod, 2)
    ref_out, ref_lse = run_oracle(mod)
    assert_close(out, lse, ref_out, ref_lse, fp8=True, what="scaled row")
    base_out, _ = run_gpu(case, 2)
    assert np.array_equal(out[:, :4], base_out[:, :4])  # KV head 0's query heads untouched
    assert not np.array_equal(out[0, 4:], base_out[0, 4:])


@pytest.mark.parametrize("kv_dtype", ["fp8_e4m3_pth", "int8_pth", "int4_pth"])
def test_extreme_scale_magnitudes(kv_dtype):
    # Rows whose scales span many orders of magnitude (tiny whole requests,
    # single huge V scales late in a sequence): the P.V power-of-two factor
    # keeps every product a normal f16 number.
    case = synth.make_gqa_case([300, 90, 40], Hq=8, Hkv=2, D=128, page=16, kv_dtype=kv_dtype, seed=36)
    kv = case.kv.copy()
    rng = np.random.default_rng(7)

    def scale_rows(blocks, plane, f):
        sc = np.ascontiguousarray(kv[blocks, plane, ..., -4:]).view("<f4") * np.float32(f)
        kv[blocks, plane, ..., -4:] = sc.view(np.uint8)

    n0 = (300 + 15) // 16
    scale_rows(case.block_table[1, :6], 1, 1e-7)                      # request 1: tiny V scales
    scale_rows(case.block_table[1, :6], 0, 1e-3)                      # and small K scales
    scale_rows(case.block_table[0, n0 - 3:n0], 1, 3e4)                # request 0: V scales jump late
    for t in rng.choice(40, size=5, replace=False):                    # request 2: scattered spikes
        blk, slot = case.block_table[2, t // 16], t % 16
        sc = np.ascontiguousarray(kv[blk, 1, slot, :, -4:]).view("<f4") * np.float32(1e5)
        kv[blk, 1, slot, :, -4:] = sc.view(np.uint8)
    mod = synth.replace(case, kv=kv)
    ref_out, ref_lse = run_oracle(mod)
    for splits in (1, 4):
        out, lse = run_gpu(mod, splits)
        # relative to each row's magnitude: the tiny-scale request has outputs ~1e-7
        for b in range(3):
            mag = max(np.abs(ref_out[b]).max(), 1e-30)
            assert np.abs(out[b] - ref_out[b]).max() <= 3e-2 * mag, (kv_dtype, splits, b)
        assert np.abs(lse - ref_lse).max() <= 1e-3


def test_device_check_reports_bad_block_id():
    case = synth.make_gqa_case([40, 70], Hq=8, Hkv=2, D=128, page=16, kv_dtype="fp8_e4m3_pth", seed=35)
    bt = case.block_table.copy()
    bt[1, 2] = case.num_blocks + 5  # out of range
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = run_gpu(synth.replace(case, block_table=bt), 2, status=status)
    assert int(status.item()) == 5
    assert np.isfinite(out).all()
    # request 0 does not touch the bad entry and is still exact
    ref_out, ref_lse = run_oracle(subset(case, [0]))
    assert_close(out[[0]], lse[[0]], ref_out, ref_lse, fp8=True, what="bad block, other request")


@pytest.mark.parametrize("name", ["gqa_fp8_pth", "gqa_int8_pth", "gqa_int4_pth"])
def test_full_size_config_sampled(name):
    case = synth.workload(name)
    splits = 32
    out, lse = run_gpu(case, splits)
    rows = [0, 101, 255]
    ref_out, ref_lse = run_oracle(subset(case, rows))
    assert_close(out[rows], lse[rows], ref_out, ref_lse, fp8=True, what=name)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    # a convex combination of V rows: no entry above the largest |V| of the cache
    v = case.kv[:, 1]
    sc = np.ascontiguousarray(v[..., -4:]).view("<f4")[..., 0].astype(np.float64)
    top = {"gqa_fp8_pth": 448.0, "gqa_int8_pth": 128.0, "gqa_int4_pth": 8.0}[name]
    assert np.abs(out).max() <= (sc.max() * top) * (1 + 1e-2)
