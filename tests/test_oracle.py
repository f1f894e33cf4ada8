"""Pins for the CPU fp64 oracle (no GPU).

The oracle is checked against things other than itself: values the pages
print (paging example, split-count rule), closed forms, invariants, brute
force on tiny inputs written independently with numpy, and exhaustive decoder
comparisons against torch's host casts.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- decoders --

def test_bf16_decoder_exhaustive_against_torch():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.bf16_values(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def test_bf16_decoder_closed_forms():
    v = oracle.bf16_values(np.array([0x3F80, 0xC000, 0x0001, 0x7F80, 0x8000, 0x3FC0], dtype=np.uint16))
    assert v[0] == 1.0 and v[1] == -2.0
    assert v[2] == 2.0 ** -133  # smallest subnormal
    assert v[3] == math.inf
    assert v[4] == 0.0 and math.copysign(1.0, v[4]) == -1.0
    assert v[5] == 1.5


def test_e4m3_decoder_exhaustive_against_torch():
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    mine = oracle.e4m3_values(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert nan.sum() == 2  # 0x7F and 0xFF only: e4m3fn has no infinities
    assert np.array_equal(mine[~nan], ref[~nan])


def test_e4m3_decoder_closed_forms():
    # OCP FP8 E4M3: bias 7, subnormal m * 2^-9, max 448, S.1111.111 = NaN.
    table = {0x38: 1.0, 0x3C: 1.5, 0x7E: 448.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9,
             0x08: 2.0 ** -6, 0xB8: -1.0, 0x40: 2.0, 0x30: 0.5}
    for code, want in table.items():
        assert oracle.e4m3_values(np.array([code], dtype=np.uint8))[0] == want, hex(code)
    assert np.isnan(oracle.e4m3_values(np.array([0x7F, 0xFF], dtype=np.uint8))).all()


# ------------------------------------------------------- page-printed values --

def test_num_kv_splits_rule():
    with open(os.path.join(GOLDEN, "num_kv_splits.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        assert oracle.num_kv_splits(c["max_seq_len"], c["sm_count"], c["batch_invariant"]) == c["splits"], c


def test_paging_example():
    with open(os.path.join(GOLDEN, "paging_example.json")) as f:
        g = json.load(f)
    pos = g["position"]
    for c in g["cases"]:
        P = c["block_size"]
        assert pos // P == c["logical_block"]
        table = np.full((2, c["logical_block"] + 1), -1, dtype=np.int32)
        table[0, c["logical_block"]] = g["requests"]["A"]
        table[1, c["logical_block"]] = g["requests"]["B"]
        assert oracle.physical_slot(table, 0, pos, P) == c["slot_A"]
        assert oracle.physical_slot(table, 1, pos, P) == c["slot_B"]


# ------------------------------------------------------------- brute force --

def _dense_mla(case):
    """Independent numpy float64 reference: gather every token row by an
    explicit loop, then softmax(scale q K^T) V with V = K[:, :R]."""
    dec = (lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()) \
        if case.kv_dtype == "bf16" else \
        (lambda x: torch.from_numpy(x).view(torch.float8_e4m3fn).double().numpy() * case.k_scale)
    qd = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).double().numpy()
    R = case.kv_lora_rank
    B, H, D = case.q.shape
    out = np.zeros((B, H, R))
    lse = np.zeros((B, H))
    for b in range(B):
        n = int(case.seq_lens[b])
        rows = [case.kv[case.block_table[b, t // case.page], t % case.page] for t in range(n)]
        if n == 0:
            lse[b] = -np.inf
            continue
        K = dec(np.stack(rows))
        s = case.scale * (qd[b] @ K.T)  # [H, n]
        m = s.max(axis=1, keepdims=True)
        w = np.exp(s - m)
        lse[b] = (m[:, 0] + np.log(w.sum(axis=1)))
        out[b] = (w / w.sum(axis=1, keepdims=True)) @ K[:, :R]
    return out, lse


def _dense_gqa(case):
    dec = (lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()) \
        if case.kv_dtype == "bf16" else \
        (lambda x: torch.from_numpy(x).view(torch.float8_e4m3fn).double().numpy())
    ks = case.k_scale if case.kv_dtype != "bf16" else 1.0
    vs = case.v_scale if case.kv_dtype != "bf16" else 1.0
    qd = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).double().numpy()
    B, Hq, D = case.q.shape
    Hkv = case.num_kv_heads
    grp = Hq // Hkv
    out = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    for b in range(B):
        n = int(case.seq_lens[b])
        for h in range(Hq):
            g = h // grp
            K = ks * dec(np.stack([case.kv[case.block_table[b, t // case.page], 0, t % case.page, g]
                                   for t in range(n)]))
            V = vs * dec(np.stack([case.kv[case.block_table[b, t // case.page], 1, t % case.page, g]
                                   for t in range(n)]))
            s = case.scale * (K @ qd[b, h])
            m = s.max()
            w = np.exp(s - m)
            lse[b, h] = m + np.log(w.sum())
            out[b, h] = (w / w.sum()) @ V
    return out, lse


def _run(case, form="direct", **kw):
    args = (case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens, case.scale)
    if case.kind == "gqa":
        return oracle.gqa_paged_decode(*args, k_scale=case.k_scale, v_scale=case.v_scale)
    if form == "streaming":
        return oracle.mla_decode_streaming(*args, k_scale=case.k_scale, kv_lora_rank=case.kv_lora_rank, **kw)
    if form == "split":
        return oracle.mla_decode_split(*args, k_scale=case.k_scale, kv_lora_rank=case.kv_lora_rank, **kw)
    return oracle.mla_decode(*args, k_scale=case.k_scale, kv_lora_rank=case.kv_lora_rank)


TINY = [
    dict(seq_lens=[37, 40], H=4, D=576, page=16, kv_dtype="bf16", seed=1),
    dict(seq_lens=[1, 33], H=3, D=320, page=16, kv_dtype="bf16", seed=2),
    dict(seq_lens=[17, 29], H=2, D=576, page=32, kv_dtype="fp8_e4m3", k_scale=0.05, seed=3),
    dict(seq_lens=[40], H=4, D=320, page=16, kv_dtype="fp8_e4m3", k_scale=0.5, seed=4),
]


@pytest.mark.parametrize("spec", TINY)
def test_mla_brute_force_tiny(spec):
    case = synth.make_mla_case(**spec)
    out, lse = _run(case)
    ref_out, ref_lse = _dense_mla(case)
    assert np.abs(out - ref_out).max() <= 1e-12 * max(1.0, np.abs(ref_out).max())
    assert np.abs(lse - ref_lse).max() <= 1e-12 * max(1.0, np.abs(ref_lse).max())


@pytest.mark.parametrize("spec", [
    dict(seq_lens=[21, 3], Hq=4, Hkv=2, D=128, page=16, kv_dtype="bf16", seed=5),
    dict(seq_lens=[35], Hq=8, Hkv=1, D=64, page=16, kv_dtype="bf16", seed=6),
    dict(seq_lens=[18, 7], Hq=6, Hkv=3, D=128, page=16, kv_dtype="fp8_e4m3", k_scale=0.1,
         v_scale=0.2, seed=7),
])
def test_gqa_brute_force_tiny(spec):
    case = synth.make_gqa_case(**spec)
    out, lse = _run(case)
    ref_out, ref_lse = _dense_gqa(case)
    assert np.abs(out - ref_out).max() <= 1e-12 * max(1.0, np.abs(ref_out).max())
    assert np.abs(lse - ref_lse).max() <= 1e-12


def test_lse_equals_log_sum_exp_fsum():
    case = synth.make_mla_case(seq_lens=[23], H=2, D=576, page=16, seed=11)
    _, lse = _run(case)
    qd = synth_bf16(case.q)
    for h in range(2):
        s = []
        for t in range(23):
            row = synth_bf16(case.kv[case.block_table[0, t // 16], t % 16])
            s.append(case.scale * math.fsum(float(a) * float(b) for a, b in zip(qd[0, h], row)))
        assert abs(lse[0, h] - math.log(math.fsum(math.exp(x) for x in s))) < 1e-12


def synth_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


# ------------------------------------------------------ closed forms --------

def test_one_token_returns_v0():
    case = synth.make_mla_case(seq_lens=[1, 1], H=5, D=576, page=16, seed=21)
    out, lse = _run(case)
    for b in range(2):
        row = synth_bf16(case.kv[case.block_table[b, 0], 0])
        assert np.array_equal(out[b], np.broadcast_to(row[:512], (5, 512)))
        for h in range(5):
            s0 = case.scale * math.fsum(float(a) * float(c) for a, c in
                                        zip(synth_bf16(case.q[b, h]), row))
            assert abs(lse[b, h] - s0) < 1e-12


def test_equal_logits_give_mean_of_values():
    # q is zero on the latent dims and every token shares one rope part, so all
    # logits are equal: out = mean_t V_t, lse = s + ln n.
    case = synth.make_mla_case(seq_lens=[45, 9], H=3, D=576, page=16, seed=22)
    q = case.q.copy()
    q[:, :, :512] = 0
    kv = case.kv.copy()
    kv[:, :, 512:] = case.kv[0, 0, 512:]
    case = synth.replace(case, q=q, kv=kv)
    out, lse = _run(case)
    for b, n in enumerate(case.seq_lens):
        V = np.stack([synth_bf16(kv[case.block_table[b, t // 16], t % 16])[:512] for t in range(n)])
        for h in range(3):
            s = case.scale * math.fsum(float(a) * float(c) for a, c in
                                       zip(synth_bf16(q[b, h, 512:]), synth_bf16(kv[0, 0, 512:])))
            assert np.abs(out[b, h] - V.mean(axis=0)).max() < 1e-12
            assert abs(lse[b, h] - (s + math.log(n))) < 1e-12


def test_zero_query_fp8_gives_scaled_mean_and_log_n():
    case = synth.make_mla_case(seq_lens=[30], H=2, D=576, page=16, kv_dtype="fp8_e4m3",
                               k_scale=0.05, seed=23)
    case = synth.replace(case, q=np.zeros_like(case.q))
    out, lse = _run(case)
    codes = np.stack([case.kv[case.block_table[0, t // 16], t % 16, :512] for t in range(30)])
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    assert np.abs(out[0] - 0.05 * vals.mean(axis=0)).max() < 1e-12
    assert np.abs(lse - math.log(30)).max() < 1e-12


def test_dominant_key_selects_its_value():
    # A large scale turns the softmax into an argmax over distinct logits.
    case = synth.make_mla_case(seq_lens=[50], H=2, D=576, page=16, seed=24, scale=1e3)
    out, lse = _run(case)
    qd = synth_bf16(case.q)
    rows = np.stack([synth_bf16(case.kv[case.block_table[0, t // 16], t % 16]) for t in range(50)])
    for h in range(2):
        s = rows @ qd[0, h]
        j = int(np.argmax(s))
        gap = np.sort(s)[-1] - np.sort(s)[-2]
        assert gap * 1e3 > 50  # the runner-up weight is below e^-50
        assert np.abs(out[0, h] - rows[j, :512]).max() < 1e-12


def test_empty_sequence():
    case = synth.make_mla_case(seq_lens=[0, 5], H=2, D=576, page=16, seed=25)
    out, lse = _run(case)
    assert np.all(out[0] == 0) and np.all(lse[0] == -np.inf)
    assert np.all(np.isfinite(out[1]))


# --------------------------------------------------------------- invariants --

def test_block_permutation_invariance():
    case = synth.make_mla_case(seq_lens=[37, 100], H=4, D=576, page=16, pool_factor=1.5, seed=31)
    out, lse = _run(case)
    rng = np.random.default_rng(5)
    perm = rng.permutation(case.num_blocks)
    kv2 = np.empty_like(case.kv)
    kv2[perm] = case.kv
    table2 = np.where(case.block_table >= 0, perm[np.maximum(case.block_table, 0)], -1).astype(np.int32)
    out2, lse2 = _run(synth.replace(case, kv=kv2, block_table=table2))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


@pytest.mark.parametrize("fill", [-1, 2**31 - 1])
def test_poisoned_padding_is_never_read(fill):
    case = synth.make_mla_case(seq_lens=[37, 100, 16], H=3, D=576, page=16, pool_factor=1.3,
                               seed=32, extra_cols=2)
    out, lse = _run(case)
    out2, lse2 = _run(synth.poison(case, table_fill=fill))
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)
    g = synth.make_gqa_case(seq_lens=[19, 4], Hq=4, Hkv=2, D=64, page=16, seed=33, extra_cols=1)
    o1, l1 = _run(g)
    o2, l2 = _run(synth.poison(g, table_fill=fill))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 5, 7, 12])
def test_split_merge_equals_direct(splits):
    # Includes more splits than pages (empty segments with weight 0).
    case = synth.make_mla_case(seq_lens=[37, 100, 5], H=3, D=576, page=16, seed=41)
    out, lse = _run(case)
    out_s, lse_s = _run(case, "split", num_splits=splits)
    assert np.abs(out - out_s).max() < 1e-12
    assert np.abs(lse - lse_s).max() < 1e-12


@pytest.mark.parametrize("tile", [1, 3, 16, 64])
def test_streaming_equals_direct(tile):
    case = synth.make_mla_case(seq_lens=[37, 100], H=3, D=320, page=16, kv_dtype="fp8_e4m3",
                               k_scale=0.05, seed=42)
    out, lse = _run(case)
    out_s, lse_s = _run(case, "streaming", tile=tile)
    assert np.abs(out - out_s).max() < 1e-12
    assert np.abs(lse - lse_s).max() < 1e-12


def test_request_isolation():
    case = synth.make_mla_case(seq_lens=[37, 100], H=2, D=576, page=16, seed=43)
    out, lse = _run(case)
    kv = case.kv.copy()
    for blk in case.block_table[1, :7]:
        kv[blk] = synth.to_bf16_bits(np.full(kv.shape[1:], 3.0, dtype=np.float32))
    out2, lse2 = _run(synth.replace(case, kv=kv))
    assert np.array_equal(out[0], out2[0]) and np.array_equal(lse[0], lse2[0])
    assert not np.array_equal(out[1], out2[1])


def test_gqa_kv_head_swap_permutes_groups():
    case = synth.make_gqa_case(seq_lens=[20, 13], Hq=4, Hkv=2, D=64, page=16, seed=44)
    out, lse = _run(case)
    kv = case.kv[:, :, :, ::-1, :].copy()  # swap the two KV heads
    q = np.concatenate([case.q[:, 2:], case.q[:, :2]], axis=1)  # swap query groups too
    out2, lse2 = _run(synth.replace(case, kv=kv, q=q))
    assert np.array_equal(out2[:, :2], out[:, 2:]) and np.array_equal(out2[:, 2:], out[:, :2])
    assert np.array_equal(lse2[:, :2], lse[:, 2:])


def test_bad_block_id_is_rejected():
    case = synth.make_mla_case(seq_lens=[20], H=2, D=576, page=16, seed=45)
    bt = case.block_table.copy()
    bt[0, 1] = case.num_blocks
    with pytest.raises(ValueError):
        _run(synth.replace(case, block_table=bt))
