"""Pins for the oracle's per-token-head quantised GQA decode (no GPU).

The cache format ("Triton と MLA" page, 役割 / 設計動機 / 主要ファイル:
fp8_per_token_head and int8_per_token_head caches keep one scale per
(token, KV head) inline, with head_dim padded to hold it) is read here as
rows of D codes followed by the row's little-endian fp32 scale.  The oracle
is checked against a numpy reference that decodes the rows by an independent
route (torch's e4m3 cast, numpy's int8 view, numpy's float32 view of the
scale bytes), against the per-tensor e4m3 oracle when every scale is 1,
against closed forms, and against poisoned padding.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

PTH = ["fp8_e4m3_pth", "int8_pth", "int4_pth"]


def _unpack_int4(codes):
    """uint8 [..., n] -> int [..., 2n]: element 2i from the low nibble of byte
    i, as a signed 4-bit number (shift the nibble into the top of an int8)."""
    lo = (codes << 4).view(np.int8) >> 4
    hi = codes.view(np.int8) >> 4
    out = np.empty(codes.shape[:-1] + (2 * codes.shape[-1],), dtype=np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def _decode_rows(rows, kv_dtype):
    """rows uint8 [..., C + 4] -> float64 [..., D] by an independent route."""
    codes = np.ascontiguousarray(rows[..., :-4])
    if kv_dtype == "fp8_e4m3_pth":
        vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    elif kv_dtype == "int4_pth":
        vals = _unpack_int4(codes).astype(np.float64)
    else:
        vals = codes.view(np.int8).astype(np.float64)
    sc = np.ascontiguousarray(rows[..., -4:]).view("<f4").astype(np.float64)
    return vals * sc


def _dense_pth(case):
    qd = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).double().numpy()
    B, Hq, D = case.q.shape
    grp = Hq // case.num_kv_heads
    out = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    for b in range(B):
        n = int(case.seq_lens[b])
        for h in range(Hq):
            if n == 0:
                lse[b, h] = -np.inf
                continue
            g = h // grp
            rows = lambda plane: np.stack([case.kv[case.block_table[b, t // case.page], plane, t % case.page, g]
                                           for t in range(n)])
            K = _decode_rows(rows(0), case.kv_dtype)
            V = _decode_rows(rows(1), case.kv_dtype)
            s = case.scale * (K @ qd[b, h])
            m = s.max()
            w = np.exp(s - m)
            lse[b, h] = m + np.log(w.sum())
            out[b, h] = (w / w.sum()) @ V
    return out, lse


def _run(case):
    return oracle.gqa_paged_decode(case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens,
                                   case.scale)


def test_int4_decoder_exhaustive():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    got = oracle.int4_values(codes[None, :])[0]
    assert np.array_equal(got, _unpack_int4(codes[None, :])[0].astype(np.float64))
    assert got[2 * 0x80] == 0 and got[2 * 0x80 + 1] == -8 and got[2 * 0x7F] == -1 and got[2 * 0x7F + 1] == 7
    assert set(got.tolist()) == set(range(-8, 8))


def test_int8_decoder_exhaustive():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    assert np.array_equal(oracle.int8_values(codes), codes.view(np.int8).astype(np.float64))
    assert oracle.int8_values(np.array([0x80, 0x7F, 0xFF], dtype=np.uint8)).tolist() == [-128.0, 127.0, -1.0]


@pytest.mark.parametrize("kv_dtype", PTH)
def test_encoder_round_trip_is_within_half_a_code(kv_dtype):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 7, 128), dtype=np.float32)
    rows = synth.encode_pth_rows(x, kv_dtype)
    assert rows.shape == (5, 7, (64 if kv_dtype == "int4_pth" else 128) + 4) and rows.dtype == np.uint8
    sc = np.ascontiguousarray(rows[..., -4:]).view("<f4")[..., 0]
    top = {"fp8_e4m3_pth": 448.0, "int8_pth": 127.0, "int4_pth": 7.0}[kv_dtype]
    assert np.allclose(sc, np.abs(x).max(axis=-1) / top, rtol=1e-6)
    y = _decode_rows(rows, kv_dtype)
    # e4m3: 3 mantissa bits -> relative error <= 2^-4; int8: half a code step
    err = np.abs(y - x)
    if kv_dtype in ("int8_pth", "int4_pth"):
        assert (err <= 0.5 * sc[..., None] * (1 + 1e-6)).all()
    else:
        assert (err <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * sc[..., None]) * (1 + 1e-6)).all()


@pytest.mark.parametrize("kv_dtype", PTH)
@pytest.mark.parametrize("spec", [
    dict(seq_lens=[1, 17, 40], Hq=4, Hkv=2, D=64, page=16, seed=1),
    dict(seq_lens=[33, 5], Hq=8, Hkv=8, D=128, page=16, seed=2),
    dict(seq_lens=[70], Hq=6, Hkv=1, D=128, page=32, seed=3, pool_factor=2.0),
])
def test_brute_force_tiny(kv_dtype, spec):
    case = synth.make_gqa_case(kv_dtype=kv_dtype, **spec)
    out, lse = _run(case)
    ref_out, ref_lse = _dense_pth(case)
    assert np.abs(out - ref_out).max() <= 1e-12 * max(1.0, np.abs(ref_out).max())
    assert np.abs(lse - ref_lse).max() <= 1e-12


def test_unit_scales_reduce_to_per_tensor_e4m3():
    # With every inline scale 1.0 the format is the plain e4m3 cache with
    # k_scale = v_scale = 1, which the per-tensor oracle computes.
    g = synth.make_gqa_case(seq_lens=[37, 100], Hq=8, Hkv=2, D=64, page=16, kv_dtype="fp8_e4m3",
                            k_scale=1.0, v_scale=1.0, seed=4)
    one = np.frombuffer(np.float32(1.0).astype("<f4").tobytes(), dtype=np.uint8)
    kv = np.concatenate([g.kv, np.broadcast_to(one, g.kv.shape[:-1] + (4,))], axis=-1)
    pth = synth.replace(g, kv=np.ascontiguousarray(kv), kv_dtype="fp8_e4m3_pth")
    o1, l1 = oracle.gqa_paged_decode(g.q, g.kv, "fp8_e4m3", g.block_table, g.seq_lens, g.scale, 1.0, 1.0)
    o2, l2 = _run(pth)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def _set_scale(kv, blk, plane, slot, head, value):
    kv[blk, plane, slot, head, -4:] = np.frombuffer(np.float32(value).astype("<f4").tobytes(), dtype=np.uint8)


@pytest.mark.parametrize("kv_dtype", PTH)
def test_one_token_closed_form(kv_dtype):
    # One token: out = vs * V codes, lse = scale * ks * <q, K codes>.
    case = synth.make_gqa_case(seq_lens=[1], Hq=2, Hkv=1, D=64, page=16, kv_dtype=kv_dtype, seed=5)
    kv = case.kv.copy()
    blk = case.block_table[0, 0]
    _set_scale(kv, blk, 0, 0, 0, 0.25)
    _set_scale(kv, blk, 1, 0, 0, 3.0)
    out, lse = _run(synth.replace(case, kv=kv))
    dec = {"fp8_e4m3_pth": oracle.e4m3_values, "int8_pth": oracle.int8_values,
           "int4_pth": lambda c: oracle.int4_values(c[None, :])[0]}[kv_dtype]
    kc = dec(kv[blk, 0, 0, 0, :-4])
    vc = dec(kv[blk, 1, 0, 0, :-4])
    qd = oracle.bf16_values(case.q[0])
    for h in range(2):
        assert np.allclose(out[0, h], 3.0 * vc, rtol=0, atol=1e-12)
        assert math.isclose(lse[0, h], case.scale * 0.25 * float(qd[h] @ kc), rel_tol=1e-12, abs_tol=1e-12)


@pytest.mark.parametrize("kv_dtype", PTH)
def test_key_scale_zero_gives_uniform_weights(kv_dtype):
    # Every K scale 0: all logits 0, so out = mean of the dequantised V rows
    # (each with its own scale) and lse = ln n.
    case = synth.make_gqa_case(seq_lens=[21], Hq=3, Hkv=1, D=64, page=16, kv_dtype=kv_dtype, seed=6)
    kv = case.kv.copy()
    for t in range(21):
        _set_scale(kv, case.block_table[0, t // 16], 0, t % 16, 0, 0.0)
    out, lse = _run(synth.replace(case, kv=kv))
    V = np.stack([_decode_rows(kv[case.block_table[0, t // 16], 1, t % 16, 0], kv_dtype) for t in range(21)])
    assert np.abs(out[0] - V.mean(axis=0)).max() <= 1e-12
    assert np.abs(lse[0] - math.log(21)).max() <= 1e-12


@pytest.mark.parametrize("kv_dtype", PTH)
def test_value_scale_is_per_token(kv_dtype):
    # Doubling one token's V scale changes the output by exactly that token's
    # weighted value: out' - out = w_t * V_t, with w_t = exp(s_t - lse).
    case = synth.make_gqa_case(seq_lens=[30], Hq=2, Hkv=1, D=64, page=16, kv_dtype=kv_dtype, seed=7)
    out, lse = _run(case)
    kv = case.kv.copy()
    t = 19
    blk, slot = case.block_table[0, t // 16], t % 16
    row = kv[blk, 1, slot, 0].copy()
    sc = float(np.ascontiguousarray(row[-4:]).view("<f4")[0])
    _set_scale(kv, blk, 1, slot, 0, 2.0 * sc)
    out2, lse2 = _run(synth.replace(case, kv=kv))
    assert np.array_equal(lse, lse2)
    K = _decode_rows(kv[blk, 0, slot, 0], kv_dtype)
    qd = oracle.bf16_values(case.q[0])
    for h in range(2):
        w = math.exp(case.scale * float(qd[h] @ K) - lse[0, h])
        assert np.abs((out2[0, h] - out[0, h]) - w * _decode_rows(row, kv_dtype)).max() <= 1e-12


@pytest.mark.parametrize("kv_dtype", PTH)
def test_poisoned_padding_is_never_read(kv_dtype):
    case = synth.make_gqa_case(seq_lens=[19, 4, 32], Hq=4, Hkv=2, D=64, page=16, kv_dtype=kv_dtype,
                               seed=8, pool_factor=1.5, extra_cols=1)
    o1, l1 = _run(case)
    o2, l2 = _run(synth.poison(case))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.isfinite(o1).all()


def test_empty_sequence_and_bad_block():
    case = synth.make_gqa_case(seq_lens=[0, 5], Hq=2, Hkv=1, D=64, page=16, kv_dtype="int8_pth", seed=9)
    out, lse = _run(case)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()
    bt = case.block_table.copy()
    bt[1, 0] = case.num_blocks
    with pytest.raises(ValueError):
        oracle.gqa_paged_decode(case.q, case.kv, "int8_pth", bt, case.seq_lens, case.scale)
