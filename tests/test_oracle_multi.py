"""Pins of the fp64 oracle for multi-token decode (tutorial page lshu.cn/news/265860,
§10: query i of q_len sits at context_length + i and sees the keys at positions <= its
own), checked against things other than the oracle's own code: a dense numpy reference
with an explicit causal mask, reductions to single-query decode, and causality."""
import numpy as np
import pytest
import torch

import oracle
import synth


def _dense_multi(case, q_len):
    """Independent reference: gather every cached row of a request by an explicit
    loop, mask key t for query i unless t <= kv_length - q_len + i, softmax, times V."""
    dec = (lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()) \
        if case.kv_dtype == "bf16" else \
        (lambda x: torch.from_numpy(x).view(torch.float8_e4m3fn).double().numpy() * case.k_scale)
    B, rows, D = case.q.shape
    H = rows // q_len
    qd = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).double().numpy().reshape(B, q_len, H, D)
    R = case.kv_lora_rank
    out = np.zeros((B, q_len, H, R))
    lse = np.full((B, q_len, H), -np.inf)
    for b in range(B):
        n = int(case.seq_lens[b])
        if n == 0:
            continue
        K = dec(np.stack([case.kv[case.block_table[b, t // case.page], t % case.page] for t in range(n)]))
        for i in range(q_len):
            visible = np.arange(n) <= n - q_len + i
            if not visible.any():
                continue
            s = case.scale * (qd[b, i] @ K.T)  # [H, n]
            s = np.where(visible[None, :], s, -np.inf)
            m = s.max(axis=1, keepdims=True)
            w = np.exp(s - m)
            lse[b, i] = m[:, 0] + np.log(w.sum(axis=1))
            out[b, i] = (w / w.sum(axis=1, keepdims=True)) @ K[:, :R]
    return out, lse


def _multi(case, q_len):
    B, rows, D = case.q.shape
    return oracle.mla_decode_multi(case.q.reshape(B, q_len, rows // q_len, D), case.kv, case.kv_dtype,
                                   case.block_table, case.seq_lens, case.scale, case.k_scale,
                                   kv_lora_rank=case.kv_lora_rank)


@pytest.mark.parametrize("q_len,H", [(1, 4), (2, 3), (3, 2), (6, 2)])
@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_multi_brute_force_tiny(q_len, H, kv_dtype):
    # lengths below q_len leave the first queries with no visible key
    case = synth.make_mla_case([5, 40, 3, 1, 0, 17], H=q_len * H, page=16, kv_dtype=kv_dtype, k_scale=0.05,
                               seed=31)
    out, lse = _multi(case, q_len)
    ref_out, ref_lse = _dense_multi(case, q_len)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    assert np.allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)
    assert np.allclose(out, ref_out, rtol=0, atol=1e-12)
    assert (out[~fin] == 0).all()


def test_one_query_is_single_decode():
    case = synth.make_mla_case([37, 100, 1], H=8, page=16, seed=32)
    out1, lse1 = _multi(case, 1)
    out, lse = oracle.mla_decode(case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens, case.scale)
    assert np.array_equal(out1[:, 0], out) and np.array_equal(lse1[:, 0], lse)


@pytest.mark.parametrize("q_len", [2, 5])
def test_query_i_is_single_decode_of_its_prefix(q_len):
    # query i sees exactly the first kv_length - q_len + i + 1 tokens
    H = 3
    case = synth.make_mla_case([9, 64, 130], H=q_len * H, page=16, seed=33)
    out, lse = _multi(case, q_len)
    B, rows, D = case.q.shape
    q4 = case.q.reshape(B, q_len, H, D)
    for i in range(q_len):
        sub = synth.replace(case, q=np.ascontiguousarray(q4[:, i]),
                            seq_lens=(case.seq_lens - q_len + i + 1).astype(np.int32))
        o1, l1 = oracle.mla_decode(sub.q, sub.kv, sub.kv_dtype, sub.block_table, sub.seq_lens, sub.scale)
        assert np.array_equal(out[:, i], o1) and np.array_equal(lse[:, i], l1)


def test_causality_new_key_reaches_only_later_queries():
    # changing the key at position kv_length - q_len + j (new token j) leaves
    # queries 0 .. j-1 unchanged and changes queries j .. q_len-1
    q_len, H = 4, 2
    case = synth.make_mla_case([50], H=q_len * H, page=16, seed=34)
    out, lse = _multi(case, q_len)
    n = int(case.seq_lens[0])
    for j in range(q_len):
        t = n - q_len + j
        kv = case.kv.copy()
        kv[case.block_table[0, t // case.page], t % case.page] = synth.to_bf16_bits(
            np.full(kv.shape[-1], 3.0, np.float32))
        out2, lse2 = _multi(synth.replace(case, kv=kv), q_len)
        assert np.array_equal(out2[0, :j], out[0, :j]) and np.array_equal(lse2[0, :j], lse[0, :j])
        assert not np.array_equal(lse2[0, j:], lse[0, j:])
