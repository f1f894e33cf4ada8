"""Decode context parallelism on the CPU with gloo: two ranks each hold the
page-aligned shards of every request that fall to them, compute their shards'
(output, lse) (here with the fp64 oracle, test infrastructure), all-gather
them over a gloo process group, and merge them with the oracle's LogSumExp
merge; every rank must end with the decode of the whole sequences.  This
covers the exchange that the single-GPU `mqa_lse_merge` follows (its GPU
parity is in test_gpu_shard_merge.py)."""
import os
import socket
import sys

import numpy as np
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
    from mqa_decode_attention_paged_gb300 import synth
    return synth.make_mla_case([37, 100, 0, 300, 16], H=4, D=576, page=16, seed=71)


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from mqa_decode_attention_paged_gb300 import synth
        case = _case()
        shard = synth.shard_case(case, world)[rank]
        out, lse = oracle.mla_decode(shard.q, shard.kv, shard.kv_dtype, shard.block_table, shard.seq_lens,
                                     shard.scale, kv_lora_rank=shard.kv_lora_rank)
        # the exchange: every rank gathers every shard's output and lse
        outs = [torch.empty(out.shape, dtype=torch.float64) for _ in range(world)]
        lses = [torch.empty(lse.shape, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(outs, torch.from_numpy(out))
        dist.all_gather(lses, torch.from_numpy(lse))
        m_out, m_lse = oracle.lse_merge(np.stack([t.numpy() for t in outs]), np.stack([t.numpy() for t in lses]))
        np.save(os.path.join(out_dir, f"out{rank}.npy"), m_out)
        np.save(os.path.join(out_dir, f"lse{rank}.npy"), m_lse)
    finally:
        dist.destroy_process_group()


def test_two_rank_context_parallel_decode_equals_whole(tmp_path):
    import oracle
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    case = _case()
    ref_out, ref_lse = oracle.mla_decode(case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens,
                                         case.scale, kv_lora_rank=case.kv_lora_rank)
    for r in range(world):
        out = np.load(tmp_path / f"out{r}.npy")
        lse = np.load(tmp_path / f"lse{r}.npy")
        assert np.abs(out - ref_out).max() <= 1e-12
        fin = np.isfinite(ref_lse)
        assert np.array_equal(fin, np.isfinite(lse))
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= 1e-12
