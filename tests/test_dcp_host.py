"""Decode context parallelism on the CPU with gloo ranks, through this
library's host code: every rank asks the library (``dcp_shard``, the C ABI's
page planner) which pages of each request it holds, decodes them (here with
the fp64 oracle, which stands in for the GPU decode on a machine without
one), and the ranks exchange their results with the package's DCP helpers:

- ``all_gather_shards`` stacks every shard's (output, lse) in rank order, the
  layout ``mqa_lse_merge`` takes; the oracle's merge of it must be the decode
  of the whole sequences on every rank;
- ``reduce_scatter_heads`` sums the ranks' shares (each rank's output times
  its weight in the merge, computed here by the oracle and put in the
  head-chunk order ``mqa_dcp_scale_shard`` writes, whose GPU parity is in
  test_gpu_dcp.py): rank c must end with the whole decode of its heads.

Both placements (round-robin and contiguous pages) and world sizes 2 and 3
are covered."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    import synth
    return synth.make_mla_case([37, 100, 0, 300, 16], H=6, D=576, page=16, seed=71)


def _rank_main(rank, world, port, out_dir, layout):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from mqa_decode_attention_paged_gb300 import _binding as mqa
        from mqa_decode_attention_paged_gb300 import dcp
        import synth
        case = _case()
        table, lens = mqa.dcp_shard(case.block_table, case.seq_lens, case.page, world, rank, layout)
        shard = synth.replace(case, block_table=table, seq_lens=lens)
        out, lse = oracle.mla_decode(shard.q, shard.kv, shard.kv_dtype, shard.block_table, shard.seq_lens,
                                     shard.scale, kv_lora_rank=shard.kv_lora_rank)
        # exchange 1: all-gather of outputs and lse, merged on every rank
        so, sl = dcp.all_gather_shards(torch.from_numpy(out), torch.from_numpy(lse))
        assert tuple(so.shape) == (world,) + out.shape and tuple(sl.shape) == (world,) + lse.shape
        m_out, m_lse = oracle.lse_merge(so.numpy(), sl.numpy())
        np.save(os.path.join(out_dir, f"ag_out{rank}.npy"), m_out)
        np.save(os.path.join(out_dir, f"ag_lse{rank}.npy"), m_lse)
        # exchange 2: lse all-gather, own share in head chunks, reduce-scatter
        lses = [torch.empty(lse.shape, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(lses, torch.from_numpy(lse))
        share, _ = oracle.lse_share(out, np.stack([t.numpy() for t in lses]), rank)
        B, H, R = share.shape
        chunks = np.ascontiguousarray(share.reshape(B, world, H // world, R).transpose(1, 0, 2, 3))
        mine = dcp.reduce_scatter_heads(torch.from_numpy(chunks))
        np.save(os.path.join(out_dir, f"rs_out{rank}.npy"), mine.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("layout", ["round_robin", "contiguous"])
@pytest.mark.parametrize("world", [2, 3])
def test_context_parallel_decode_equals_whole(tmp_path, layout, world):
    import oracle
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path), layout), nprocs=world,
                       start_method="spawn", join=True)
    case = _case()
    ref_out, ref_lse = oracle.mla_decode(case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens,
                                         case.scale, kv_lora_rank=case.kv_lora_rank)
    fin = np.isfinite(ref_lse)
    hc = case.num_heads // world
    for r in range(world):
        out = np.load(tmp_path / f"ag_out{r}.npy")
        lse = np.load(tmp_path / f"ag_lse{r}.npy")
        assert np.abs(out - ref_out).max() <= 1e-12
        assert np.array_equal(fin, np.isfinite(lse))
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-12
        mine = np.load(tmp_path / f"rs_out{r}.npy")
        assert np.abs(mine - ref_out[:, r * hc:(r + 1) * hc]).max() <= 1e-12
