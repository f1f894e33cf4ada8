"""ctypes binding of ``libmqa_decode.so`` (the C ABI declared in include/mqa_decode.h).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  torch supplies device memory and the current stream.  When the
shared library is missing this module raises at import time instead of falling
back to anything else.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_WORKSPACE_TOO_SMALL = 3
ERR_CUDA = 4
ERR_DEVICE_CHECK = 5
ERR_DEVICE_TIMEOUT = 6

KV_BF16 = 0
KV_FP8_E4M3 = 1
KV_FP8_E4M3_PER_TOKEN_HEAD = 2
KV_INT8_PER_TOKEN_HEAD = 3
KV_INT4_PER_TOKEN_HEAD = 4
_KV_NAMES = {"bf16": KV_BF16, "fp8_e4m3": KV_FP8_E4M3, "fp8_e4m3_pth": KV_FP8_E4M3_PER_TOKEN_HEAD,
             "int8_pth": KV_INT8_PER_TOKEN_HEAD, "int4_pth": KV_INT4_PER_TOKEN_HEAD}

LIB_PATH = _build.LIB_PATH


class MqaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        msg = f"{where}: {status_string(code)} (status {code})"
        if self.code == ERR_CUDA:
            msg += f": {lib.mqa_last_cuda_error_string().decode()}"
        super().__init__(msg)


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first with `python -m mqa_decode_attention_paged_gb300.build` "
            "(requires nvcc); there is no fallback implementation")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.mqa_abi_version.restype = I
    lib.mqa_abi_version.argtypes = []
    lib.mqa_status_string.restype = ctypes.c_char_p
    lib.mqa_status_string.argtypes = [I]
    lib.mqa_device_sm_count.restype = I
    lib.mqa_device_sm_count.argtypes = []
    lib.mqa_last_cuda_error.restype = I
    lib.mqa_last_cuda_error.argtypes = []
    lib.mqa_last_cuda_error_string.restype = ctypes.c_char_p
    lib.mqa_last_cuda_error_string.argtypes = []
    lib.mqa_num_kv_splits.restype = I
    lib.mqa_num_kv_splits.argtypes = [I, I, I]
    lib.mla_decode_workspace_bytes.restype = SZ
    lib.mla_decode_workspace_bytes.argtypes = [I, I, I, I]
    lib.gqa_paged_decode_workspace_bytes.restype = SZ
    lib.gqa_paged_decode_workspace_bytes.argtypes = [I, I, I, I]
    lib.mla_decode.restype = I
    lib.mla_decode.argtypes = [P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, I, I, P, SZ, P, P]
    lib.mla_decode_fixed_splits.restype = I
    lib.mla_decode_fixed_splits.argtypes = [P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, I, I, P, SZ, P, P]
    lib.mla_decode_multi.restype = I
    lib.mla_decode_multi.argtypes = [P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, I, I, I, P, SZ, P, P]
    lib.mla_decode_sparse.restype = I
    lib.mla_decode_sparse.argtypes = [P, P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, I, I, I, P, SZ, P, P]
    lib.mla_decode_noalloc.restype = I
    lib.mla_decode_noalloc.argtypes = [P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, I, I, P, P]
    lib.gqa_paged_decode.restype = I
    lib.gqa_paged_decode.argtypes = [P, P, P, P, F, F, F, P, P, I, I, I, I, I, I, I, I, I, P, SZ, P, P]
    lib.mqa_lse_merge.restype = I
    lib.mqa_lse_merge.argtypes = [P, P, P, P, I, ctypes.c_longlong, I, P]
    lib.mqa_dcp_shard_max_blocks.restype = I
    lib.mqa_dcp_shard_max_blocks.argtypes = [I, I]
    lib.mqa_dcp_shard.restype = I
    lib.mqa_dcp_shard.argtypes = [P, P, I, I, I, I, I, I, P, I, P]
    lib.mqa_dcp_locate.restype = I
    lib.mqa_dcp_locate.argtypes = [I, I, I, I, I, ctypes.POINTER(I), ctypes.POINTER(I)]
    lib.mqa_dcp_scale_shard.restype = I
    lib.mqa_dcp_scale_shard.argtypes = [P, P, P, P, I, I, I, I, I, I, P]
    return lib


lib = _load()


def abi_version() -> int:
    return int(lib.mqa_abi_version())


def status_string(code: int) -> str:
    return lib.mqa_status_string(int(code)).decode()


def device_sm_count() -> int:
    return int(lib.mqa_device_sm_count())


def num_kv_splits(max_seq_len: int, sm_count: int, batch_invariant: bool = False) -> int:
    return int(lib.mqa_num_kv_splits(int(max_seq_len), int(sm_count), int(bool(batch_invariant))))


def mla_decode_workspace_bytes(batch: int, num_heads: int, kv_lora_rank: int, num_kv_splits: int) -> int:
    return int(lib.mla_decode_workspace_bytes(batch, num_heads, kv_lora_rank, num_kv_splits))


def gqa_paged_decode_workspace_bytes(batch: int, num_q_heads: int, head_size: int, num_kv_splits: int) -> int:
    return int(lib.gqa_paged_decode_workspace_bytes(batch, num_q_heads, head_size, num_kv_splits))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(t, name, dtypes=None, shape=None, optional=False, elt=None):
    """Validate the layout of a tensor argument before its pointer is handed to
    the C ABI: dtype (or element size), shape and contiguity.  The library
    reads raw pointers, so a wrong layout would otherwise be read as garbage."""
    if t is None:
        if optional:
            return
        raise ValueError(f"{name} is required")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype {' or '.join(str(d) for d in dtypes)}, got {t.dtype}")
    if elt is not None and t.element_size() != elt:
        raise TypeError(f"{name} must have {elt}-byte elements, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on_device(named):
    """Every given tensor must live on the CUDA device of the first."""
    dev = None
    for name, t in named:
        if t is None:
            continue
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor, got one on {t.device}")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"{name} is on {t.device}, the call runs on {dev}")


def _check_common(q, kv_cache, code, block_table, seq_lens, out, out_shape, lse, lse_shape, workspace,
                  device_status, extra=()):
    import torch
    _check(q, "q", (torch.bfloat16,))
    _check(kv_cache, "kv_cache", elt=2 if code == KV_BF16 else 1)
    _check(block_table, "block_table", (torch.int32,))
    if block_table.dim() != 2 or block_table.shape[0] != out_shape[0]:
        raise ValueError("block_table must be int32 [batch, max_blocks]")
    _check(seq_lens, "seq_lens", (torch.int32,), shape=(out_shape[0],))
    _check(out, "out", (torch.bfloat16,), shape=out_shape)
    _check(lse, "lse", (torch.float32,), shape=lse_shape, optional=True)
    _check(workspace, "workspace", optional=True)
    _check(device_status, "device_status", (torch.int32,), optional=True)
    _on_device([("q", q), ("kv_cache", kv_cache), ("block_table", block_table), ("seq_lens", seq_lens),
                ("out", out), ("lse", lse), ("workspace", workspace), ("device_status", device_status),
                *extra])


def _kv_code(kv_cache, kv_dtype):
    import torch
    if kv_dtype is not None:
        return _KV_NAMES[kv_dtype] if isinstance(kv_dtype, str) else int(kv_dtype)
    if kv_cache.dtype == torch.bfloat16:
        return KV_BF16
    if kv_cache.dtype == torch.float8_e4m3fn:
        return KV_FP8_E4M3
    raise TypeError("kv_cache must be bf16 or float8_e4m3fn (or pass kv_dtype with uint8 storage)")


def mla_decode(q, kv_cache, block_table, seq_lens, scale, k_scale=1.0, *, out=None, lse=None,
               num_kv_splits=1, workspace=None, kv_lora_rank=None, kv_dtype=None,
               device_status=None, stream=None, return_lse=True):
    """MLA decode through the C ABI.  q [B,H,D] bf16, kv_cache [num_blocks, page, D],
    block_table [B, max_blocks] int32, seq_lens [B] int32 (all on one CUDA device).
    Allocates out / lse / workspace with torch when they are not given."""
    return _mla_decode(lib.mla_decode, "mla_decode", q, kv_cache, block_table, seq_lens, scale, k_scale, out,
                       lse, num_kv_splits, workspace, kv_lora_rank, kv_dtype, device_status, stream, return_lse)


def mla_decode_fixed_splits(q, kv_cache, block_table, seq_lens, scale, k_scale=1.0, *, out=None, lse=None,
                            num_kv_splits=1, workspace=None, kv_lora_rank=None, kv_dtype=None,
                            device_status=None, stream=None, return_lse=True):
    """``mla_decode`` with one work unit per (request, split): every request
    cut into num_kv_splits equal page ranges (batch-invariant at any split
    count).  Same arguments and results as :func:`mla_decode`."""
    return _mla_decode(lib.mla_decode_fixed_splits, "mla_decode_fixed_splits", q, kv_cache, block_table,
                       seq_lens, scale, k_scale, out, lse, num_kv_splits, workspace, kv_lora_rank, kv_dtype,
                       device_status, stream, return_lse)


def _mla_decode(fn, name, q, kv_cache, block_table, seq_lens, scale, k_scale, out, lse, num_kv_splits, workspace,
                kv_lora_rank, kv_dtype, device_status, stream, return_lse):
    import torch
    B, H, D = q.shape
    nb, page, D2 = kv_cache.shape
    if D2 != D:
        raise ValueError("q and kv_cache head sizes differ")
    R = (D - 64) if kv_lora_rank is None else int(kv_lora_rank)
    code = _kv_code(kv_cache, kv_dtype)
    if out is None:
        out = torch.empty((B, H, R), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    need = mla_decode_workspace_bytes(B, H, R, num_kv_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check_common(q, kv_cache, code, block_table, seq_lens, out, (B, H, R), lse, (B, H), workspace,
                  device_status)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = fn(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), float(scale), float(k_scale), _ptr(out),
            _ptr(lse), B, H, D, R, nb, page, block_table.shape[1], code, int(num_kv_splits), _ptr(workspace),
            ws_bytes, _ptr(device_status), _stream(stream))
    if rc != OK:
        raise MqaError(rc, name)
    return out, lse


def mla_decode_multi(q, kv_cache, block_table, seq_lens, scale, k_scale=1.0, *, out=None, lse=None,
                     num_kv_splits=1, workspace=None, kv_lora_rank=None, kv_dtype=None,
                     device_status=None, stream=None, return_lse=True):
    """Multi-token MLA decode through the C ABI.  q [B, q_len, H, D] bf16 (query i of
    request b sits at position seq_lens[b] - q_len + i and sees the keys up to it);
    returns out [B, q_len, H, R] bf16 and lse [B, q_len, H] fp32."""
    import torch
    B, Lq, H, D = q.shape
    nb, page, D2 = kv_cache.shape
    if D2 != D:
        raise ValueError("q and kv_cache head sizes differ")
    R = (D - 64) if kv_lora_rank is None else int(kv_lora_rank)
    code = _kv_code(kv_cache, kv_dtype)
    if out is None:
        out = torch.empty((B, Lq, H, R), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Lq, H), dtype=torch.float32, device=q.device)
    need = mla_decode_workspace_bytes(B, Lq * H, R, num_kv_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check_common(q, kv_cache, code, block_table, seq_lens, out, (B, Lq, H, R), lse, (B, Lq, H), workspace,
                  device_status)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.mla_decode_multi(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), float(scale),
                              float(k_scale), _ptr(out), _ptr(lse), B, Lq, H, D, R, nb, page,
                              block_table.shape[1], code, int(num_kv_splits), _ptr(workspace), ws_bytes,
                              _ptr(device_status), _stream(stream))
    if rc != OK:
        raise MqaError(rc, "mla_decode_multi")
    return out, lse


def mla_decode_sparse(q, kv_cache, block_table, seq_lens, indices, scale, k_scale=1.0, *, out=None,
                      lse=None, num_kv_splits=1, workspace=None, kv_lora_rank=None, kv_dtype=None,
                      device_status=None, stream=None, return_lse=True):
    """Sparse (top-k) MLA decode through the C ABI.  q [B, H, D] bf16, indices [B, topk]
    int32 logical positions (entries outside [0, seq_lens[b]) select nothing); returns
    out [B, H, R] bf16 and lse [B, H] fp32."""
    import torch
    B, H, D = q.shape
    nb, page, D2 = kv_cache.shape
    if D2 != D:
        raise ValueError("q and kv_cache head sizes differ")
    if indices.dim() != 2 or indices.shape[0] != B or indices.dtype != torch.int32:
        raise ValueError("indices must be int32 [batch, topk]")
    topk = indices.shape[1]
    R = (D - 64) if kv_lora_rank is None else int(kv_lora_rank)
    code = _kv_code(kv_cache, kv_dtype)
    if out is None:
        out = torch.empty((B, H, R), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=q.device)
    need = mla_decode_workspace_bytes(B, H, R, num_kv_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(indices, "indices", (torch.int32,))
    _check_common(q, kv_cache, code, block_table, seq_lens, out, (B, H, R), lse, (B, H), workspace,
                  device_status, extra=[("indices", indices)])
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.mla_decode_sparse(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens), _ptr(indices),
                               float(scale), float(k_scale), _ptr(out), _ptr(lse), B, H, D, R, nb, page,
                               block_table.shape[1], topk, code, int(num_kv_splits), _ptr(workspace),
                               ws_bytes, _ptr(device_status), _stream(stream))
    if rc != OK:
        raise MqaError(rc, "mla_decode_sparse")
    return out, lse


def gqa_paged_decode(q, kv_cache, block_table, seq_lens, scale, k_scale=1.0, v_scale=1.0, *,
                     out=None, lse=None, num_kv_splits=1, workspace=None, kv_dtype=None,
                     device_status=None, stream=None, return_lse=True):
    """GQA paged decode through the C ABI.  q [B,Hq,D] bf16; kv_cache
    [num_blocks, 2, page, Hkv, D] bf16 or e4m3 (k_scale / v_scale), or, with
    kv_dtype "fp8_e4m3_pth" / "int8_pth", uint8 [num_blocks, 2, page, Hkv,
    D + 4] rows of D codes followed by their fp32 scale, or "int4_pth", uint8
    [..., D / 2 + 4] rows of packed 4-bit codes followed by the scale."""
    import torch
    B, Hq, D = q.shape
    nb, two, page, Hkv, D2 = kv_cache.shape
    code = _kv_code(kv_cache, kv_dtype)
    row = {KV_FP8_E4M3_PER_TOKEN_HEAD: D + 4, KV_INT8_PER_TOKEN_HEAD: D + 4,
           KV_INT4_PER_TOKEN_HEAD: D // 2 + 4}.get(code, D)
    if two != 2 or D2 != row:
        raise ValueError(f"kv_cache must be [num_blocks, 2, page, num_kv_heads, {row}]")
    if out is None:
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    need = gqa_paged_decode_workspace_bytes(B, Hq, D, num_kv_splits)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check_common(q, kv_cache, code, block_table, seq_lens, out, (B, Hq, D), lse, (B, Hq), workspace,
                  device_status)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.gqa_paged_decode(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
                              float(scale), float(k_scale), float(v_scale), _ptr(out), _ptr(lse),
                              B, Hq, Hkv, D, nb, page, block_table.shape[1], code,
                              int(num_kv_splits), _ptr(workspace), ws_bytes, _ptr(device_status),
                              _stream(stream))
    if rc != OK:
        raise MqaError(rc, "gqa_paged_decode")
    return out, lse


def lse_merge(shard_out, shard_lse, *, out=None, lse=None, stream=None, return_lse=True):
    """Merge sequence-shard results through the C ABI (decode context
    parallelism, after the caller has gathered the shards): shard_out bf16
    [G, ..., head_dim], shard_lse fp32 [G, ...]; returns (out [..., head_dim]
    bf16, lse [...] fp32)."""
    import torch
    G = shard_out.shape[0]
    D = shard_out.shape[-1]
    lead = tuple(shard_out.shape[1:-1])
    if tuple(shard_lse.shape) != (G,) + lead:
        raise ValueError("shard_lse must be [num_shards, *shard_out.shape[1:-1]]")
    rows = 1
    for x in lead:
        rows *= int(x)
    if out is None:
        out = torch.empty(lead + (D,), dtype=torch.bfloat16, device=shard_out.device)
    if lse is None and return_lse:
        lse = torch.empty(lead, dtype=torch.float32, device=shard_out.device)
    _check(shard_out, "shard_out", (torch.bfloat16,))
    _check(shard_lse, "shard_lse", (torch.float32,))
    _check(out, "out", (torch.bfloat16,), shape=lead + (D,))
    _check(lse, "lse", (torch.float32,), shape=lead, optional=True)
    _on_device([("shard_out", shard_out), ("shard_lse", shard_lse), ("out", out), ("lse", lse)])
    rc = lib.mqa_lse_merge(_ptr(shard_out), _ptr(shard_lse), _ptr(out), _ptr(lse), int(G), rows, int(D),
                           _stream(stream))
    if rc != OK:
        raise MqaError(rc, "mqa_lse_merge")
    return out, lse


DCP_LAYOUTS = {"round_robin": 0, "contiguous": 1}


def _dcp_layout(layout):
    if layout not in DCP_LAYOUTS:
        raise ValueError(f"layout must be one of {sorted(DCP_LAYOUTS)}, got {layout!r}")
    return DCP_LAYOUTS[layout]


def dcp_shard_max_blocks(max_blocks: int, num_ranks: int) -> int:
    n = int(lib.mqa_dcp_shard_max_blocks(int(max_blocks), int(num_ranks)))
    if n < 0:
        raise ValueError("max_blocks and num_ranks must be >= 1")
    return n


def dcp_shard(block_table, seq_lens, page_size, num_ranks, rank, layout="round_robin"):
    """Pages of rank `rank` of `num_ranks` under decode context parallelism
    (host arrays, C ABI ``mqa_dcp_shard``): block_table int32 [B, max_blocks]
    and seq_lens int32 [B] (numpy or CPU tensors) give the whole sequences;
    returns numpy (shard_block_table int32 [B, ceil(max_blocks / num_ranks)],
    shard_seq_lens int32 [B]) for the decode entry points."""
    import numpy as np
    bt = np.ascontiguousarray(np.asarray(block_table), dtype=np.int32)
    sl = np.ascontiguousarray(np.asarray(seq_lens), dtype=np.int32)
    if bt.ndim != 2 or sl.shape != (bt.shape[0],):
        raise ValueError("block_table must be [B, max_blocks] and seq_lens [B]")
    B, mb = bt.shape
    width = dcp_shard_max_blocks(mb, num_ranks)
    table = np.empty((B, width), dtype=np.int32)
    lens = np.empty(B, dtype=np.int32)
    rc = lib.mqa_dcp_shard(bt.ctypes.data, sl.ctypes.data, B, mb, int(page_size), int(num_ranks), int(rank),
                           _dcp_layout(layout), table.ctypes.data, width, lens.ctypes.data)
    if rc != OK:
        raise MqaError(rc, "mqa_dcp_shard")
    return table, lens


def dcp_locate(pos, seq_len, page_size, num_ranks, layout="round_robin"):
    """(rank, position in that rank's shard) of token `pos` of a sequence of
    seq_len tokens (C ABI ``mqa_dcp_locate``)."""
    r, p = ctypes.c_int(), ctypes.c_int()
    rc = lib.mqa_dcp_locate(int(pos), int(seq_len), int(page_size), int(num_ranks), _dcp_layout(layout),
                            ctypes.byref(r), ctypes.byref(p))
    if rc != OK:
        raise MqaError(rc, "mqa_dcp_locate")
    return r.value, p.value


def dcp_scale_shard(shard_out, gathered_lse, rank, *, scaled=None, lse=None, scaled_fp32=True, stream=None,
                    return_lse=True):
    """This rank's share of the merged output, laid out for a sum
    reduce-scatter over the ranks (C ABI ``mqa_dcp_scale_shard``):
    shard_out bf16 [B, H, D], gathered_lse fp32 [G, B, H]; returns (scaled
    [G, B, H / G, D] fp32 or bf16, merged lse [B, H] fp32)."""
    import torch
    B, H, D = shard_out.shape
    G = gathered_lse.shape[0]
    if H % G != 0:
        raise ValueError("the head count must be a multiple of the number of ranks")
    sdt = torch.float32 if scaled_fp32 else torch.bfloat16
    if scaled is None:
        scaled = torch.empty((G, B, H // G, D), dtype=sdt, device=shard_out.device)
    if lse is None and return_lse:
        lse = torch.empty((B, H), dtype=torch.float32, device=shard_out.device)
    _check(shard_out, "shard_out", (torch.bfloat16,))
    _check(gathered_lse, "gathered_lse", (torch.float32,), shape=(G, B, H))
    _check(scaled, "scaled", (sdt,), shape=(G, B, H // G, D))
    _check(lse, "lse", (torch.float32,), shape=(B, H), optional=True)
    _on_device([("shard_out", shard_out), ("gathered_lse", gathered_lse), ("scaled", scaled), ("lse", lse)])
    rc = lib.mqa_dcp_scale_shard(_ptr(shard_out), _ptr(gathered_lse), _ptr(scaled), _ptr(lse), int(G), int(rank),
                                 int(B), int(H), int(D), int(bool(scaled_fp32)), _stream(stream))
    if rc != OK:
        raise MqaError(rc, "mqa_dcp_scale_shard")
    return scaled, lse


NOALLOC_SCRATCH_BYTES = 64 << 20


def mla_decode_noalloc(q, kv_cache, block_table, seq_lens, scale, k_scale=1.0, *, out, lse=None,
                       num_kv_splits=1, kv_lora_rank=None, kv_dtype=None, device_status=None,
                       stream=None):
    """MLA decode without a caller workspace, for callers that cannot allocate
    device memory: the split partials go to the library's own fixed 64 MiB
    device array, so `out` (and `lse`, if wanted) must already exist.  Calls
    share that array: do not let two of them overlap on the GPU."""
    B, H, D = q.shape
    nb, page, _ = kv_cache.shape
    R = (D - 64) if kv_lora_rank is None else int(kv_lora_rank)
    code = _kv_code(kv_cache, kv_dtype)
    _check_common(q, kv_cache, code, block_table, seq_lens, out, (B, H, R), lse, (B, H), None, device_status)
    rc = lib.mla_decode_noalloc(_ptr(q), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
                                float(scale), float(k_scale), _ptr(out), _ptr(lse), B, H, D, R, nb,
                                page, block_table.shape[1], code,
                                int(num_kv_splits), _ptr(device_status), _stream(stream))
    if rc != OK:
        raise MqaError(rc, "mla_decode_noalloc")
    return out, lse
