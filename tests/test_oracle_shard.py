"""Pins for the oracle's merge of sequence-shard results (no GPU).

Decode context parallelism places a request's KV pages on several ranks; each
computes its shard's (output, lse) and the results are merged by LogSumExp
(tutorial page lshu.cn/news/265860, §12; the "Triton と MLA" page, 設計動機:
lse is returned so that shards can be merged).  The merge is pinned by the
identity it must satisfy: merging the shard results of the oracle's own
decode gives the decode of the whole sequence; plus closed forms.
"""
import math

import numpy as np
import pytest

import oracle
import synth


def _decode(case):
    args = (case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens, case.scale)
    if case.kind == "mla":
        return oracle.mla_decode(*args, k_scale=case.k_scale, kv_lora_rank=case.kv_lora_rank)
    return oracle.gqa_paged_decode(*args, k_scale=case.k_scale, v_scale=case.v_scale)


@pytest.mark.parametrize("G", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("make", [
    lambda: synth.make_mla_case([37, 100, 16, 1, 0, 250], H=3, D=576, page=16, seed=51),
    lambda: synth.make_mla_case([90, 64], H=2, D=320, page=32, kv_dtype="fp8_e4m3", k_scale=0.05, seed=52),
    lambda: synth.make_gqa_case([19, 4, 70], Hq=4, Hkv=2, D=64, page=16, seed=53),
], ids=["mla576", "mla320_fp8", "gqa"])
def test_merged_shards_equal_whole_sequence(G, make):
    case = make()
    out, lse = _decode(case)
    parts = [_decode(sh) for sh in synth.shard_case(case, G)]
    m_out, m_lse = oracle.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    assert np.abs(m_out - out).max() <= 1e-12 * max(1.0, np.abs(out).max())
    fin = np.isfinite(lse)
    assert np.array_equal(fin, np.isfinite(m_lse))
    assert np.abs(m_lse[fin] - lse[fin]).max() <= 1e-12
    assert (m_out[~fin] == 0).all()


def test_shards_cover_each_sequence_once():
    case = synth.make_mla_case([37, 100, 0, 16], H=1, D=576, page=16, seed=54)
    for G in (1, 2, 3, 7):
        sh = synth.shard_case(case, G)
        assert (sum(s.seq_lens.astype(np.int64) for s in sh) == case.seq_lens).all()
        for b in range(case.batch):
            blocks = [int(x) for s in sh for x in s.block_table[b] if x >= 0]
            npg = (int(case.seq_lens[b]) + 15) // 16
            assert blocks == [int(x) for x in case.block_table[b, :npg]]


def test_closed_forms():
    rng = np.random.default_rng(5)
    o = rng.standard_normal((3, 2, 4, 8))
    # one shard: identity
    l1 = rng.standard_normal((1, 2, 4))
    out, lse = oracle.lse_merge(o[:1], l1)
    assert np.array_equal(out, o[0]) and np.array_equal(lse, l1[0])
    # equal lse: the mean of the shard outputs, lse + ln G
    leq = np.full((3, 2, 4), 0.7)
    out, lse = oracle.lse_merge(o, leq)
    assert np.abs(out - o.mean(axis=0)).max() < 1e-15
    assert np.abs(lse - (0.7 + math.log(3))).max() < 1e-15
    # an empty shard (lse -inf) has no weight, whatever its output holds
    l2 = rng.standard_normal((3, 2, 4))
    l2[1] = -np.inf
    o2 = o.copy()
    o2[1] = np.nan
    out, lse = oracle.lse_merge(o2, l2)
    ref, rl = oracle.lse_merge(o[[0, 2]], l2[[0, 2]])
    assert np.array_equal(out, ref) and np.array_equal(lse, rl)
    # two shards, one dominant by far: its output
    l3 = np.stack([np.full((2, 4), 50.0), np.full((2, 4), -50.0)])
    out, lse = oracle.lse_merge(o[:2], l3)
    assert np.abs(out - o[0]).max() < 1e-40 + 1e-30 * np.abs(o[1]).max() + 1e-15
    # nothing anywhere: zeros and -inf
    out, lse = oracle.lse_merge(o, np.full((3, 2, 4), -np.inf))
    assert (out == 0).all() and np.isneginf(lse).all()


@pytest.mark.parametrize("G", [2, 3, 5])
def test_shares_of_shards_sum_to_whole_sequence(G):
    # lse all-gather / output reduce-scatter: each shard's share
    # e^{lse_g - lse} O_g, summed over the shards, is the decode of the whole
    # sequence (an independent pin: the whole decode never merges anything)
    case = synth.make_mla_case([37, 100, 16, 1, 0, 250], H=4, D=576, page=16, seed=55)
    out, lse = _decode(case)
    parts = [_decode(sh) for sh in synth.shard_case(case, G)]
    lses = np.stack([p[1] for p in parts])
    total = np.zeros_like(out)
    for g, p in enumerate(parts):
        share, l = oracle.lse_share(p[0], lses, g)
        total += share
        fin = np.isfinite(lse)
        assert np.array_equal(np.isfinite(l), fin)
        assert np.abs(l[fin] - lse[fin]).max() <= 1e-12
    assert np.abs(total - out).max() <= 1e-12 * max(1.0, np.abs(out).max())


def test_share_closed_forms():
    rng = np.random.default_rng(6)
    o = rng.standard_normal((3, 2, 4, 8))
    lses = rng.standard_normal((3, 2, 4))
    # the shares add up to the merge, shard by shard in any order
    merged, mlse = oracle.lse_merge(o, lses)
    shares = [oracle.lse_share(o[g], lses, g) for g in range(3)]
    assert np.abs(sum(s[0] for s in shares) - merged).max() < 1e-14
    assert all(np.abs(s[1] - mlse).max() < 1e-15 for s in shares)
    # one shard: its own output, its own lse
    s, l = oracle.lse_share(o[0], lses[:1], 0)
    assert np.abs(s - o[0]).max() < 1e-15 and np.abs(l - lses[0]).max() < 1e-15
    # two shards of equal lse: half each, lse + ln 2
    eq = np.full((2, 2, 4), -1.5)
    s, l = oracle.lse_share(o[1], eq, 1)
    assert np.abs(s - 0.5 * o[1]).max() < 1e-15 and np.abs(l - (-1.5 + math.log(2))).max() < 1e-15
    # weights e^{lse_g - lse}: shard 0 of lse 0 against shard 1 of lse ln 3 -> 1/4
    l2 = np.stack([np.zeros((2, 4)), np.full((2, 4), math.log(3.0))])
    s, _ = oracle.lse_share(o[0], l2, 0)
    assert np.abs(s - 0.25 * o[0]).max() < 1e-15
    # an empty shard: share 0 whatever its output holds; the others keep theirs
    l3 = lses.copy()
    l3[2] = -np.inf
    s, _ = oracle.lse_share(np.full((2, 4, 8), np.nan), l3, 2)
    assert (s == 0).all()
    # nothing anywhere: zeros and -inf
    s, l = oracle.lse_share(o[0], np.full((3, 2, 4), -np.inf), 0)
    assert (s == 0).all() and np.isneginf(l).all()
