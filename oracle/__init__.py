"""CPU fp64 oracle for single-query paged decode attention (MLA and GQA).

TEST INFRASTRUCTURE ONLY.  The test suite, the package smoke check and the
CPU-baseline leg of ``bench.py`` are the only callers.  The library's product
path (``mqa_decode_attention_paged_gb300``) never imports this package, and the
two share no code: the arithmetic lives in ``oracle.c`` (plain C, fp64,
OpenMP over (request, head) pairs), written from the pages' statement of the
method; see the header of ``oracle.c`` for the passages each part follows.

Every function takes host numpy arrays in the same raw encodings the GPU
library consumes (bf16 as uint16 bit patterns, e4m3 as uint8 codes) and
returns float64 arrays.

Parity status: every function here is pinned by tests under ``tests/``
(brute force, closed forms, invariants, exhaustive decoder checks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

KV_BF16 = 0
KV_FP8_E4M3 = 1

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``oracle/_build/liboracle.so`` with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int
        D = ctypes.c_double
        I64 = ctypes.c_int64
        lib.oracle_bf16_value.restype = D
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_value.restype = D
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_bf16_values.argtypes = [P, P, I64]
        lib.oracle_e4m3_values.argtypes = [P, P, I64]
        lib.oracle_num_kv_splits.restype = I
        lib.oracle_num_kv_splits.argtypes = [I, I, I]
        lib.oracle_physical_slot.restype = I64
        lib.oracle_physical_slot.argtypes = [P, I, I, I64, I]
        lib.oracle_max_threads.restype = I
        lib.oracle_set_threads.argtypes = [I]
        mla = [P, P, I, P, P, D, D, P, P, I, I, I, I, I, I, I]
        lib.oracle_mla_decode.restype = I
        lib.oracle_mla_decode.argtypes = mla
        lib.oracle_mla_decode_streaming.restype = I
        lib.oracle_mla_decode_streaming.argtypes = mla + [I]
        lib.oracle_mla_decode_split.restype = I
        lib.oracle_mla_decode_split.argtypes = mla + [I]
        lib.oracle_mla_decode_multi.restype = I
        lib.oracle_mla_decode_multi.argtypes = [P, P, I, P, P, D, D, P, P, I, I, I, I, I, I, I, I]
        lib.oracle_mla_decode_sparse.restype = I
        lib.oracle_mla_decode_sparse.argtypes = [P, P, I, P, P, P, I, D, D, P, P, I, I, I, I, I, I, I]
        lib.oracle_gqa_paged_decode.restype = I
        lib.oracle_gqa_paged_decode.argtypes = [P, P, I, P, P, D, D, D, P, P, I, I, I, I, I, I, I]
        lib.oracle_gqa_paged_decode_pth.restype = I
        lib.oracle_gqa_paged_decode_pth.argtypes = [P, P, I, P, P, D, P, P, I, I, I, I, I, I, I]
        lib.oracle_int8_values.argtypes = [P, P, I64]
        lib.oracle_lse_merge.argtypes = [P, P, P, P, I, I, I, I]
        lib.oracle_lse_share.argtypes = [P, P, I, P, P, I, I, I, I]
        lib.oracle_int4_values.argtypes = [P, P, I64]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _kv_code(kv: np.ndarray, kv_dtype: str) -> int:
    if kv_dtype == "bf16":
        if kv.dtype != np.uint16:
            raise TypeError("bf16 cache must be given as uint16 bit patterns")
        return KV_BF16
    if kv_dtype == "fp8_e4m3":
        if kv.dtype != np.uint8:
            raise TypeError("e4m3 cache must be given as uint8 codes")
        return KV_FP8_E4M3
    raise ValueError(f"unknown kv dtype {kv_dtype!r}")


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def bf16_values(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_bf16_values(_ptr(b), _ptr(out), b.size)
    return out


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_values(_ptr(c), _ptr(out), c.size)
    return out


def num_kv_splits(max_seq_len: int, sm_count: int, batch_invariant: bool) -> int:
    return int(_load().oracle_num_kv_splits(int(max_seq_len), int(sm_count), int(bool(batch_invariant))))


def physical_slot(block_table: np.ndarray, req: int, pos: int, page_size: int) -> int:
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    return int(_load().oracle_physical_slot(_ptr(bt), bt.shape[1], int(req), int(pos), int(page_size)))


def _mla_args(q, kv, kv_dtype, block_table, seq_lens):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kv = np.ascontiguousarray(kv)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    code = _kv_code(kv, kv_dtype)
    B, H, D = q.shape
    nb, P, D2 = kv.shape
    if D2 != D:
        raise ValueError("q and kv head sizes differ")
    return q, kv, bt, sl, code, B, H, D, nb, P


def _run_mla(fn_name, q, kv, kv_dtype, block_table, seq_lens, scale, k_scale, kv_lora_rank, extra):
    q, kv, bt, sl, code, B, H, D, nb, P = _mla_args(q, kv, kv_dtype, block_table, seq_lens)
    R = int(kv_lora_rank)
    out = np.zeros((B, H, R), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    fn = getattr(_load(), fn_name)
    args = [_ptr(q), _ptr(kv), code, _ptr(bt), _ptr(sl), float(scale), float(k_scale),
            _ptr(out), _ptr(lse), B, H, D, R, nb, P, bt.shape[1]] + list(extra)
    rc = fn(*args)
    if rc != 0:
        raise ValueError("oracle: block table entry out of range or too short for a sequence")
    return out, lse


def mla_decode(q, kv, kv_dtype, block_table, seq_lens, scale, k_scale=1.0, kv_lora_rank=None):
    """Direct definition: out[b,h] = sum_t softmax_t(s) V_t, lse = log sum_t exp(s_t)."""
    D = q.shape[-1]
    R = D - 64 if kv_lora_rank is None else kv_lora_rank
    return _run_mla("oracle_mla_decode", q, kv, kv_dtype, block_table, seq_lens, scale, k_scale, R, [])


def mla_decode_streaming(q, kv, kv_dtype, block_table, seq_lens, scale, k_scale=1.0, tile=16,
                         kv_lora_rank=None):
    """Online-softmax formulation over tiles of `tile` tokens."""
    D = q.shape[-1]
    R = D - 64 if kv_lora_rank is None else kv_lora_rank
    return _run_mla("oracle_mla_decode_streaming", q, kv, kv_dtype, block_table, seq_lens, scale,
                    k_scale, R, [int(tile)])


def mla_decode_split(q, kv, kv_dtype, block_table, seq_lens, scale, k_scale=1.0, num_splits=1,
                     kv_lora_rank=None):
    """Split-KV formulation: page-aligned segments merged by LogSumExp."""
    D = q.shape[-1]
    R = D - 64 if kv_lora_rank is None else kv_lora_rank
    return _run_mla("oracle_mla_decode_split", q, kv, kv_dtype, block_table, seq_lens, scale,
                    k_scale, R, [int(num_splits)])


def mla_decode_sparse(q, kv, kv_dtype, block_table, seq_lens, indices, scale, k_scale=1.0, kv_lora_rank=None):
    """Sparse decode: each query of request b attends the positions indices[b, :]
    (entries outside [0, seq_lens[b]) select nothing).  Returns (out [B, H, R], lse [B, H])."""
    q, kv, bt, sl, code, B, H, D, nb, P = _mla_args(q, kv, kv_dtype, block_table, seq_lens)
    idx = np.ascontiguousarray(indices, dtype=np.int32)
    if idx.ndim != 2 or idx.shape[0] != B:
        raise ValueError("indices must be [batch, topk]")
    R = D - 64 if kv_lora_rank is None else int(kv_lora_rank)
    out = np.zeros((B, H, R), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    rc = _load().oracle_mla_decode_sparse(_ptr(q), _ptr(kv), code, _ptr(bt), _ptr(sl), _ptr(idx), idx.shape[1],
                                          float(scale), float(k_scale), _ptr(out), _ptr(lse), B, H, D, R, nb,
                                          P, bt.shape[1])
    if rc != 0:
        raise ValueError("oracle: block table entry out of range for a selected position")
    return out, lse


def mla_decode_multi(q, kv, kv_dtype, block_table, seq_lens, scale, k_scale=1.0, kv_lora_rank=None):
    """Multi-token decode: q [B, q_len, H, D]; query i of request b sees the
    first seq_lens[b] - q_len + i + 1 tokens.  Returns (out [B, q_len, H, R],
    lse [B, q_len, H])."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    if q.ndim != 4:
        raise ValueError("q must be [batch, q_len, heads, head_size]")
    B, Lq, H, D = q.shape
    R = D - 64 if kv_lora_rank is None else int(kv_lora_rank)
    _, kv, bt, sl, code, _, _, _, nb, P = _mla_args(q.reshape(B, Lq * H, D), kv, kv_dtype, block_table,
                                                     seq_lens)
    out = np.zeros((B, Lq, H, R), dtype=np.float64)
    lse = np.zeros((B, Lq, H), dtype=np.float64)
    rc = _load().oracle_mla_decode_multi(_ptr(q), _ptr(kv), code, _ptr(bt), _ptr(sl), float(scale),
                                         float(k_scale), _ptr(out), _ptr(lse), B, Lq, H, D, R, nb, P,
                                         bt.shape[1])
    if rc != 0:
        raise ValueError("oracle: block table entry out of range or too short for a sequence")
    return out, lse


PTH_KINDS = {"fp8_e4m3_pth": 0, "int8_pth": 1, "int4_pth": 2}


def int4_values(packed: np.ndarray) -> np.ndarray:
    """Values of packed int4 codes (uint8, element 2i in the low nibble of byte
    i, two's complement): n bytes -> 2n values."""
    b = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.float64)
    _load().oracle_int4_values(_ptr(b), _ptr(out), b.size)
    return out


def int8_values(codes: np.ndarray) -> np.ndarray:
    """Two's-complement values of int8 codes given as uint8."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_int8_values(_ptr(c), _ptr(out), c.size)
    return out


def gqa_paged_decode(q, kv, kv_dtype, block_table, seq_lens, scale, k_scale=1.0, v_scale=1.0):
    """q [B,Hq,D] bf16 bits; kv [num_blocks, 2, P, Hkv, D] (bf16 bits or e4m3
    codes with per-tensor k_scale / v_scale), or, for kv_dtype "fp8_e4m3_pth"
    / "int8_pth", uint8 [num_blocks, 2, P, Hkv, D + 4] rows of D codes plus
    their inline fp32 scale, or "int4_pth", rows of D / 2 bytes of packed
    4-bit codes plus the scale (k_scale / v_scale unused); returns
    (out [B,Hq,D], lse [B,Hq])."""
    if kv_dtype in PTH_KINDS:
        return _gqa_pth(q, kv, kv_dtype, block_table, seq_lens, scale)
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kv = np.ascontiguousarray(kv)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    code = _kv_code(kv, kv_dtype)
    B, Hq, D = q.shape
    nb, two, P, Hkv, D2 = kv.shape
    if two != 2 or D2 != D:
        raise ValueError("kv cache must be [num_blocks, 2, page, num_kv_heads, head_size]")
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    rc = _load().oracle_gqa_paged_decode(_ptr(q), _ptr(kv), code, _ptr(bt), _ptr(sl), float(scale),
                                         float(k_scale), float(v_scale), _ptr(out), _ptr(lse),
                                         B, Hq, Hkv, D, nb, P, bt.shape[1])
    if rc != 0:
        raise ValueError("oracle: bad block table or head counts")
    return out, lse


def _gqa_pth(q, kv, kv_dtype, block_table, seq_lens, scale):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kv = np.ascontiguousarray(kv)
    if kv.dtype != np.uint8:
        raise TypeError("per-token-head cache must be given as uint8 bytes")
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    B, Hq, D = q.shape
    nb, two, P, Hkv, Dp = kv.shape
    code_bytes = D // 2 if kv_dtype == "int4_pth" else D
    if two != 2 or Dp != code_bytes + 4:
        raise ValueError(f"per-token-head cache must be [num_blocks, 2, page, num_kv_heads, {code_bytes + 4}]")
    out = np.zeros((B, Hq, D), dtype=np.float64)
    lse = np.zeros((B, Hq), dtype=np.float64)
    rc = _load().oracle_gqa_paged_decode_pth(_ptr(q), _ptr(kv), PTH_KINDS[kv_dtype], _ptr(bt), _ptr(sl),
                                             float(scale), _ptr(out), _ptr(lse), B, Hq, Hkv, D, nb, P,
                                             bt.shape[1])
    if rc != 0:
        raise ValueError("oracle: bad block table or head counts")
    return out, lse


def lse_share(out_g, lses, g):
    """Shard g's share of the merged output for an exchange that all-gathers
    the lse and sums the outputs: out_g [B, H, R] (shard g's normalised
    output), lses [G, B, H]; returns (share [B, H, R], merged lse [B, H]) with
    share = e^{lse_g - lse} out_g.  The shares of all shards sum to
    ``lse_merge``'s output."""
    o = np.ascontiguousarray(out_g, dtype=np.float64)
    l = np.ascontiguousarray(lses, dtype=np.float64)
    G, B, H = l.shape
    if o.ndim != 3 or o.shape[:2] != (B, H):
        raise ValueError("out_g must be [B, H, R] with lses [G, B, H]")
    if not 0 <= g < G:
        raise ValueError("g must be a shard index")
    R = o.shape[2]
    share = np.zeros((B, H, R), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    _load().oracle_lse_share(_ptr(o), _ptr(l), int(g), _ptr(share), _ptr(lse), G, B, H, R)
    return share, lse


def lse_merge(outs, lses):
    """Merge shard results: outs [G, B, H, R] (normalised), lses [G, B, H]
    (natural log, -inf for an empty shard); returns (out [B, H, R], lse [B, H])."""
    o = np.ascontiguousarray(outs, dtype=np.float64)
    l = np.ascontiguousarray(lses, dtype=np.float64)
    G, B, H, R = o.shape
    if l.shape != (G, B, H):
        raise ValueError("lses must be [G, B, H]")
    out = np.zeros((B, H, R), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    _load().oracle_lse_merge(_ptr(o), _ptr(l), _ptr(out), _ptr(lse), G, B, H, R)
    return out, lse
