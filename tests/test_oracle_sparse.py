"""Pins of the fp64 oracle for sparse (top-k) MLA decode (tutorial page lshu.cn/news/265860,
§13: each query attends only its request's selected key positions, translated to physical
slots through the block table), checked against a dense numpy reference over the gathered
rows, reductions to dense decode, and invariants of the index list."""
import numpy as np
import pytest
import torch

import oracle
import synth


def _dec(case):
    if case.kv_dtype == "bf16":
        return lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double().numpy()
    return lambda x: torch.from_numpy(x).view(torch.float8_e4m3fn).double().numpy() * case.k_scale


def _dense_sparse(case, idx):
    """Gather the selected rows by an explicit loop, then softmax(scale q K^T) V."""
    dec = _dec(case)
    qd = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).double().numpy()
    B, H, D = case.q.shape
    R = case.kv_lora_rank
    out = np.zeros((B, H, R))
    lse = np.full((B, H), -np.inf)
    for b in range(B):
        sel = [int(t) for t in idx[b] if 0 <= t < case.seq_lens[b]]
        if not sel:
            continue
        K = dec(np.stack([case.kv[case.block_table[b, t // case.page], t % case.page] for t in sel]))
        s = case.scale * (qd[b] @ K.T)
        m = s.max(axis=1, keepdims=True)
        w = np.exp(s - m)
        lse[b] = m[:, 0] + np.log(w.sum(axis=1))
        out[b] = (w / w.sum(axis=1, keepdims=True)) @ K[:, :R]
    return out, lse


def _sparse(case, idx):
    return oracle.mla_decode_sparse(case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens, idx,
                                    case.scale, case.k_scale, kv_lora_rank=case.kv_lora_rank)


def _random_indices(case, topk, seed, pad=0.2):
    """Distinct positions per request, a share of them replaced by -1 padding."""
    rng = np.random.default_rng(seed)
    idx = np.full((case.batch, topk), -1, np.int32)
    for b, n in enumerate(case.seq_lens):
        k = min(topk, int(n))
        idx[b, :k] = rng.choice(int(n), size=k, replace=False)
        idx[b, rng.random(topk) < pad] = -1
    return idx


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_sparse_brute_force_tiny(kv_dtype):
    case = synth.make_mla_case([5, 40, 300, 1, 0, 129], H=4, page=16, kv_dtype=kv_dtype, k_scale=0.05, seed=51)
    idx = _random_indices(case, 24, 52)
    out, lse = _sparse(case, idx)
    ref_out, ref_lse = _dense_sparse(case, idx)
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    assert np.allclose(lse[fin], ref_lse[fin], rtol=0, atol=1e-12)
    assert np.allclose(out, ref_out, rtol=0, atol=1e-12)


def test_selecting_every_position_is_dense_decode():
    case = synth.make_mla_case([37, 100, 1, 64], H=8, page=16, seed=53)
    topk = int(case.seq_lens.max())
    idx = np.full((case.batch, topk), -1, np.int32)
    for b, n in enumerate(case.seq_lens):
        idx[b, :n] = np.arange(n)
    out, lse = _sparse(case, idx)
    ref_out, ref_lse = oracle.mla_decode(case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens,
                                         case.scale)
    assert np.allclose(out, ref_out, rtol=0, atol=1e-12) and np.allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_order_padding_and_out_of_range_entries():
    case = synth.make_mla_case([90, 200], H=4, page=16, seed=54)
    idx = _random_indices(case, 32, 55, pad=0.0)
    out, lse = _sparse(case, idx)
    perm = np.random.default_rng(56).permutation(idx.shape[1])
    out_p, lse_p = _sparse(case, np.ascontiguousarray(idx[:, perm]))
    assert np.allclose(out_p, out, rtol=0, atol=1e-12) and np.allclose(lse_p, lse, rtol=0, atol=1e-12)
    # -1 padding and positions at or past the sequence end select nothing
    extra = np.array([[-1, 90, 1 << 20], [-7, 200, 5000]], np.int32)
    out_x, lse_x = _sparse(case, np.concatenate([idx, extra], axis=1))
    assert np.array_equal(out_x, out) and np.array_equal(lse_x, lse)


def test_one_selected_token_returns_its_value():
    case = synth.make_mla_case([50], H=3, page=16, seed=57)
    t = 17
    out, lse = _sparse(case, np.array([[-1, t, -1]], np.int32))
    row = case.kv[case.block_table[0, t // case.page], t % case.page]
    K = _dec(case)(row[None])[0]
    qd = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).double().numpy()[0]
    assert np.allclose(out[0], np.broadcast_to(K[:case.kv_lora_rank], out[0].shape), rtol=0, atol=1e-12)
    assert np.allclose(lse[0], case.scale * (qd @ K), rtol=0, atol=1e-12)
