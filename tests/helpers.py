"""Shared helpers for the GPU parity tests: device upload, C-ABI calls through
the binding, oracle on request subsets, and the tolerance checks.

Tolerances (elementwise, against the fp64 oracle on the same inputs):
  bf16 cache: |out - ref| <= 1e-2 + 2e-2 |ref|;  fp8 cache: <= 1e-2 + 3e-2 |ref|
  lse: |lse - ref| <= 1e-3 (and -inf exactly where the oracle has -inf).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth

OUT_ABS = 1e-2
OUT_REL_BF16 = 2e-2
OUT_REL_FP8 = 3e-2
LSE_ABS = 1e-3


def to_device(case: synth.PagedCase, device="cuda"):
    q = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).to(device)
    if case.kv_dtype == "bf16":
        kv = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(device)
    elif case.kv_dtype in synth.PTH_DTYPES:
        kv = torch.from_numpy(case.kv).to(device)  # uint8 rows: codes + inline scale
    else:
        kv = torch.from_numpy(case.kv).view(torch.float8_e4m3fn).to(device)
    bt = torch.from_numpy(case.block_table).to(device)
    sl = torch.from_numpy(case.seq_lens).to(device)
    return q, kv, bt, sl


def run_gpu(case, num_kv_splits=1, dev=None, status=None):
    """Run the library on `case`; returns float64 numpy (out, lse)."""
    from mqa_decode_attention_paged_gb300 import _binding as mqa
    q, kv, bt, sl = dev if dev is not None else to_device(case)
    B, H, D = q.shape
    if case.kind == "mla":
        need = mqa.mla_decode_workspace_bytes(B, H, case.kv_lora_rank, num_kv_splits)
    else:
        need = mqa.gqa_paged_decode_workspace_bytes(B, H, D, num_kv_splits)
    # NaN-filled workspace and outputs: reading a partial slot that was never
    # written, or leaving an output element unwritten, shows up as NaN.
    ws = torch.full((max(need, 16),), 0xFF, dtype=torch.uint8, device=q.device)
    R = case.kv_lora_rank if case.kind == "mla" else D
    out = torch.full((B, H, R), float("nan"), dtype=torch.bfloat16, device=q.device)
    lse = torch.full((B, H), float("nan"), dtype=torch.float32, device=q.device)
    if case.kind == "mla":
        out, lse = mqa.mla_decode(q, kv, bt, sl, case.scale, case.k_scale, out=out, lse=lse,
                                  num_kv_splits=num_kv_splits, kv_lora_rank=case.kv_lora_rank,
                                  workspace=ws, device_status=status)
    else:
        out, lse = mqa.gqa_paged_decode(q, kv, bt, sl, case.scale, case.k_scale, case.v_scale,
                                        out=out, lse=lse, num_kv_splits=num_kv_splits,
                                        workspace=ws, device_status=status,
                                        kv_dtype=case.kv_dtype if case.kv_dtype in synth.PTH_DTYPES else None)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def subset(case, rows, heads=None):
    """The same cache with only requests `rows` (and optionally query heads `heads`)."""
    rows = np.asarray(rows)
    q = case.q[rows]
    if heads is not None:
        q = q[:, heads]
    return synth.replace(case, q=np.ascontiguousarray(q),
                         block_table=np.ascontiguousarray(case.block_table[rows]),
                         seq_lens=np.ascontiguousarray(case.seq_lens[rows]))


def run_oracle(case):
    args = (case.q, case.kv, case.kv_dtype, case.block_table, case.seq_lens, case.scale)
    if case.kind == "mla":
        return oracle.mla_decode(*args, k_scale=case.k_scale, kv_lora_rank=case.kv_lora_rank)
    return oracle.gqa_paged_decode(*args, k_scale=case.k_scale, v_scale=case.v_scale)


def assert_close(out, lse, ref_out, ref_lse, fp8=False, what=""):
    rel = OUT_REL_FP8 if fp8 else OUT_REL_BF16
    err = np.abs(out - ref_out)
    bound = OUT_ABS + rel * np.abs(ref_out)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: out mismatch at {tuple(idx)}: got {out[tuple(idx)]}, "
                             f"ref {ref_out[tuple(idx)]} ({bad.sum()} of {bad.size} outside tolerance)")
    inf_ref = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(lse), inf_ref), f"{what}: lse -inf pattern differs"
    d = np.abs(lse[~inf_ref] - ref_lse[~inf_ref])
    assert d.size == 0 or d.max() <= LSE_ABS, f"{what}: lse max err {d.max()}"
