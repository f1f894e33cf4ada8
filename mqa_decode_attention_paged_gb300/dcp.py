"""Decode context parallelism (DCP) across ranks: the exchange around the
library's DCP calls.

Each rank holds some pages of every request (``dcp_shard`` plans which, and
``dcp_locate`` tells a cache writer where a token goes), decodes them with
``mla_decode`` / ``gqa_paged_decode`` and gets its shard's normalised output
and natural-log lse.  The shards are merged by LogSumExp ("Triton と MLA"
page, 設計動機: lse is returned so that DCP shards can be merged, by
cp_lse_ag_out_rs; tutorial page lshu.cn/news/265860, §12).  Two exchanges:

- :func:`merge_reduce_scatter` (lse all-gather, output reduce-scatter): every
  rank gathers the [B, H] lse of all shards, scales its own output by its
  weight in the merge (``mqa_dcp_scale_shard``, laid out by head chunks) and a
  sum reduce-scatter leaves rank c with the merged output of heads
  [c H / G, (c + 1) H / G).  Per rank it moves G x [B, H] lse and about
  [B, H, D] of output.
- :func:`merge_all_gather`: every rank gathers all shard outputs and merges
  them with ``mqa_lse_merge``; every rank ends with all heads, at G times the
  output bytes.

The collectives are ``torch.distributed``'s (NCCL on GPUs, gloo on CPU
tensors) and, like the library calls here, run in order on the current CUDA
stream; every arithmetic step runs in the library.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import _binding as _b


def all_gather_shards(out, lse, group=None):
    """Every rank's shard output and lse stacked in rank order: (shard_out
    [G, *out.shape], shard_lse [G, *lse.shape]), the layout ``lse_merge``
    takes."""
    return _gather(out, group), _gather(lse, group)


def _gather(t, group):
    # flat buffers: the concatenated form every backend accepts
    G = dist.get_world_size(group)
    res = torch.empty(G * t.numel(), dtype=t.dtype, device=t.device)
    dist.all_gather_into_tensor(res, t.contiguous().view(-1), group=group)
    return res.view((G,) + tuple(t.shape))


def reduce_scatter_heads(scaled, group=None):
    """Sum over the ranks of the [G, B, H / G, D] buffers ``dcp_scale_shard``
    writes; rank c receives chunk c, [B, H / G, D]."""
    G = dist.get_world_size(group)
    if scaled.shape[0] != G:
        raise ValueError(f"scaled must have {G} head chunks, got {scaled.shape[0]}")
    res = torch.empty(scaled[0].numel(), dtype=scaled.dtype, device=scaled.device)
    dist.reduce_scatter_tensor(res, scaled.contiguous().view(-1), op=dist.ReduceOp.SUM, group=group)
    return res.view(tuple(scaled.shape[1:]))


def merge_all_gather(out, lse, group=None):
    """Merged (output [B, H, D] bf16, lse [B, H]) of all ranks' shards, on
    every rank."""
    shard_out, shard_lse = all_gather_shards(out, lse, group)
    return _b.lse_merge(shard_out, shard_lse)


def merge_reduce_scatter(out, lse, group=None, scaled_fp32=True):
    """The lse-all-gather / output-reduce-scatter merge: returns (merged
    output of this rank's heads [B, H / G, D], fp32 if scaled_fp32 else bf16;
    merged lse of all heads [B, H] fp32)."""
    rank = dist.get_rank(group)
    gathered = _gather(lse, group)
    scaled, merged_lse = _b.dcp_scale_shard(out, gathered, rank, scaled_fp32=scaled_fp32)
    return reduce_scatter_heads(scaled, group), merged_lse
