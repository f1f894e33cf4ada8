"""The library's decode-context-parallel page placement (host code of the C
ABI, no GPU): ``mqa_dcp_shard`` and ``mqa_dcp_locate``.

- The contiguous layout equals the test generator's own page-aligned shards
  (``synth.shard_case``, written independently).
- Under both layouts the ranks' shards cover every token of every sequence
  exactly once, in sequence order within a rank, every page but a
  sequence's last one full, and the last page last on its rank.
- ``mqa_dcp_locate`` agrees with the tables: token pos sits in the slot of
  its rank's shard that holds the same physical block and offset.
- A round-robin page never moves as its sequence grows.
- Bad arguments are refused before anything is written.
"""
import ctypes

import numpy as np
import pytest

from mqa_decode_attention_paged_gb300 import _binding as mqa
import synth

LAYOUTS = ["round_robin", "contiguous"]


def _case(seed=81, page=16):
    return synth.make_mla_case([37, 100, 0, 16, 1, 250, 64], H=1, D=576, page=page, pool_factor=1.3, seed=seed)


def test_shard_max_blocks():
    assert mqa.dcp_shard_max_blocks(16, 1) == 16
    assert mqa.dcp_shard_max_blocks(16, 3) == 6
    assert mqa.dcp_shard_max_blocks(1, 8) == 1
    for bad in ((0, 2), (4, 0), (-1, 1)):
        assert mqa.lib.mqa_dcp_shard_max_blocks(*bad) == -1


@pytest.mark.parametrize("G", [1, 2, 3, 4, 7])
def test_contiguous_matches_the_generator(G):
    case = _case()
    ref = synth.shard_case(case, G)
    for g in range(G):
        table, lens = mqa.dcp_shard(case.block_table, case.seq_lens, case.page, G, g, "contiguous")
        assert np.array_equal(lens, ref[g].seq_lens)
        w = ref[g].block_table.shape[1]
        assert table.shape[1] >= w
        assert np.array_equal(table[:, :w], ref[g].block_table)
        assert (table[:, w:] == -1).all()


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("G", [1, 2, 3, 5])
@pytest.mark.parametrize("page", [16, 64])
def test_shards_cover_each_token_once(layout, G, page):
    case = _case(seed=82, page=page)
    P = case.page
    shards = [mqa.dcp_shard(case.block_table, case.seq_lens, P, G, g, layout) for g in range(G)]
    assert (sum(s[1].astype(np.int64) for s in shards) == case.seq_lens).all()
    for b, n in enumerate(case.seq_lens):
        n = int(n)
        npg = (n + P - 1) // P
        seen = []
        for g, (table, lens) in enumerate(shards):
            k = (int(lens[b]) + P - 1) // P
            pages = [int(x) for x in table[b, :k]]
            assert (table[b, k:] == -1).all()
            seen += pages
            # every page of the shard but its last is full; a partial last
            # page is the sequence's last page
            if k and int(lens[b]) % P:
                assert pages[-1] == int(case.block_table[b, npg - 1])
            # the rank's pages in sequence order
            where = [list(case.block_table[b, :npg]).index(x) for x in pages]
            assert where == sorted(where)
            if layout == "round_robin":
                assert where == list(range(g, npg, G))
        assert sorted(seen) == sorted(int(x) for x in case.block_table[b, :npg])


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("G", [2, 3])
def test_locate_agrees_with_the_tables(layout, G):
    case = _case(seed=83)
    P = case.page
    shards = [mqa.dcp_shard(case.block_table, case.seq_lens, P, G, g, layout) for g in range(G)]
    for b, n in enumerate(case.seq_lens):
        for pos in range(int(n)):
            r, sp = mqa.dcp_locate(pos, int(n), P, G, layout)
            table, lens = shards[r]
            assert 0 <= sp < lens[b]
            assert table[b, sp // P] == case.block_table[b, pos // P] and sp % P == pos % P


def test_round_robin_pages_stay_put_as_a_sequence_grows():
    P, G = 16, 3
    for pos in range(0, 500, 7):
        homes = {mqa.dcp_locate(pos, n, P, G, "round_robin") for n in range(pos + 1, 600, 37)}
        assert len(homes) == 1
    # the contiguous layout moves pages when the sequence grows (why serving
    # keeps the round-robin one)
    assert mqa.dcp_locate(40, 64, P, 2, "contiguous") != mqa.dcp_locate(40, 400, P, 2, "contiguous")


def test_invalid_arguments_write_nothing():
    case = _case()
    bt = np.ascontiguousarray(case.block_table, dtype=np.int32)
    sl = np.ascontiguousarray(case.seq_lens, dtype=np.int32)
    B, mb = bt.shape
    w = mqa.dcp_shard_max_blocks(mb, 2)
    table = np.full((B, w), 777, dtype=np.int32)
    lens = np.full(B, 777, dtype=np.int32)
    f = mqa.lib.mqa_dcp_shard

    def call(bt_=bt, sl_=sl, B_=B, mb_=mb, P=case.page, G=2, g=0, layout=0, width=w):
        return f(bt_.ctypes.data, sl_.ctypes.data, B_, mb_, P, G, g, layout, table.ctypes.data, width,
                 lens.ctypes.data)

    assert call(g=2) == mqa.ERR_INVALID_ARG
    assert call(g=-1) == mqa.ERR_INVALID_ARG
    assert call(G=0) == mqa.ERR_INVALID_ARG
    assert call(layout=2) == mqa.ERR_INVALID_ARG
    assert call(width=w - 1) == mqa.ERR_INVALID_ARG
    assert call(B_=0) == mqa.ERR_INVALID_ARG
    assert call(P=0) == mqa.ERR_INVALID_ARG
    long_ = sl.copy()
    long_[3] = mb * case.page + 1
    assert call(sl_=long_) == mqa.ERR_INVALID_ARG
    neg = sl.copy()
    neg[5] = -1
    assert call(sl_=neg) == mqa.ERR_INVALID_ARG
    assert f(None, sl.ctypes.data, B, mb, case.page, 2, 0, 0, table.ctypes.data, w, lens.ctypes.data) == \
        mqa.ERR_INVALID_ARG
    assert (table == 777).all() and (lens == 777).all()
    assert call() == mqa.OK
    r, p = ctypes.c_int(), ctypes.c_int()
    loc = mqa.lib.mqa_dcp_locate
    assert loc(10, 10, 16, 2, 0, ctypes.byref(r), ctypes.byref(p)) == mqa.ERR_INVALID_ARG
    assert loc(-1, 10, 16, 2, 0, ctypes.byref(r), ctypes.byref(p)) == mqa.ERR_INVALID_ARG
    assert loc(3, 10, 16, 2, 5, ctypes.byref(r), ctypes.byref(p)) == mqa.ERR_INVALID_ARG
    assert loc(3, 10, 0, 2, 0, ctypes.byref(r), ctypes.byref(p)) == mqa.ERR_INVALID_ARG
    assert loc(3, 10, 16, 2, 0, None, ctypes.byref(p)) == mqa.ERR_INVALID_ARG
    with pytest.raises(ValueError):
        mqa.dcp_shard(bt, sl, case.page, 2, 0, "striped")
    with pytest.raises(mqa.MqaError):
        mqa.dcp_shard(bt, sl, case.page, 2, 3)
