"""Seeded synthetic inputs for paged decode attention.

This module is shared by the tests, the smoke check and the benchmark, and it
holds none of the attention arithmetic: it only draws random numbers, encodes
them (bf16 with round-to-nearest-even, OCP e4m3fn through torch's cast), draws
sequence lengths and builds permuted block tables.  Both the CUDA path and the
CPU oracle consume its arrays unchanged.

Encodings (the same bytes the C-ABI takes):
  * q            uint16 bf16 bit patterns, [B, H, D]
  * MLA cache    [num_blocks, page, D], uint16 (bf16) or uint8 (e4m3 codes)
  * GQA cache    [num_blocks, 2, page, Hkv, D], same element encodings; or,
                 per-token-head quantised ("fp8_e4m3_pth", "int8_pth"), uint8
                 [num_blocks, 2, page, Hkv, D + 4]: each (token, KV head) row
                 holds D codes then its scale (little-endian float32),
                 scale = max|row| / 448 (e4m3) or / 127 (int8)
  * block_table  int32 [B, max_blocks]; entries past a sequence's last page = -1
  * seq_lens     int32 [B]

Named workloads (shapes and distributions of the decode configurations this
library is measured on):
  tiny_mla     B=2, H=16, D=576 (R=512), page 16, bf16, seq_lens [37, 100],
               exact pool of 3 + 7 blocks, randomly permuted.
  mla_v2lite   B=64, H=16, D=576, page 64, bf16, seq_lens uniform in
               [1024, 8192], 1.5x oversized pool, random block sample.
  mla_v3_fp8   B=128, H=128, D=576, page 64, e4m3 cache with k_scale 0.05
               (values N(0,1)/0.05 clamped to +-448), seq_lens uniform in
               [4096, 32768], exact permuted pool.
  mla_longctx  B=4, H=128, D=576, page 64, bf16,
               seq_lens [131072, 98304, 65536, 120000].
  gqa          B=256, Hq=32, Hkv=8, D=128, page 16, bf16, seq_lens
               ceil(exp(N(ln 2048, 1))) clipped to [1, 16384].
  gqa_fp8_pth  the gqa batch with a per-token-head e4m3 cache.
  gqa_int8_pth the gqa batch with a per-token-head int8 cache.
  gqa_int4_pth the gqa batch with a per-token-head int4 cache (two codes per
               byte).
  mla_mtp      the mla_v2lite batch with 8 query tokens x 16 heads per request.
  mla_sparse   B=64, H=16, D=576, page 64, bf16, seq_lens uniform in
               [16384, 40960], 2048 distinct random positions per request
               (meta["indices"], drawn with seed + 7919).
All q and KV values are N(0, 1) (before the fp8 division), from
numpy.random.default_rng(seed); MLA scale is 1/sqrt(192), GQA 1/sqrt(128).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace  # noqa: F401 (replace is re-exported)

import numpy as np
import torch

BF16_NAN = np.uint16(0x7FC0)
E4M3_NAN = np.uint8(0x7F)
E4M3_MAX = 448.0


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round-to-nearest-even); return the bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def to_e4m3_codes(x: np.ndarray) -> np.ndarray:
    """Clamp to +-448 and round to OCP e4m3fn (torch's cast); return the byte codes."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).clamp_(-E4M3_MAX, E4M3_MAX)
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@dataclass
class PagedCase:
    """One decode batch: query, paged cache, block table and lengths (host arrays)."""

    kind: str  # "mla" or "gqa"
    q: np.ndarray
    kv: np.ndarray
    block_table: np.ndarray
    seq_lens: np.ndarray
    kv_dtype: str  # "bf16" or "fp8_e4m3"
    scale: float
    k_scale: float = 1.0
    v_scale: float = 1.0
    page: int = 16
    num_kv_heads: int = 1
    kv_lora_rank: int = 0  # MLA only
    name: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def head_size(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_blocks(self) -> int:
        return int(self.kv.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_table.shape[1])

    @property
    def total_tokens(self) -> int:
        return int(self.seq_lens.astype(np.int64).sum())


def draw_seq_lens(rng: np.random.Generator, B: int, spec) -> np.ndarray:
    """spec: explicit list, ("uniform", lo, hi) inclusive, or
    ("lognormal", median, sigma, max)."""
    if isinstance(spec, (list, tuple, np.ndarray)) and (len(spec) == 0 or not isinstance(spec[0], str)):
        out = np.asarray(spec, dtype=np.int64)
        if out.shape != (B,):
            raise ValueError("explicit seq_lens must have B entries")
        return out.astype(np.int32)
    kind = spec[0]
    if kind == "uniform":
        return rng.integers(int(spec[1]), int(spec[2]) + 1, size=B).astype(np.int32)
    if kind == "lognormal":
        median, sigma, mx = float(spec[1]), float(spec[2]), int(spec[3])
        x = np.ceil(np.exp(rng.normal(math.log(median), sigma, size=B)))
        return np.clip(x, 1, mx).astype(np.int32)
    raise ValueError(f"unknown seq_len spec {spec!r}")


def build_block_table(rng: np.random.Generator, seq_lens: np.ndarray, page: int,
                      pool_factor: float = 1.0, extra_cols: int = 0):
    """Random physical placement: sequence b owns ceil(seq_b/page) blocks drawn
    without replacement from a pool of ceil(pool_factor * total) blocks.
    Returns (block_table int32 [B, max_blocks], num_blocks, used_block_ids)."""
    n_pages = (seq_lens.astype(np.int64) + page - 1) // page
    total = int(n_pages.sum())
    num_blocks = max(1, int(math.ceil(pool_factor * total)), total)
    ids = rng.permutation(num_blocks)[:total].astype(np.int32)
    max_blocks = max(1, int(n_pages.max()) if len(n_pages) else 1) + int(extra_cols)
    table = np.full((len(seq_lens), max_blocks), -1, dtype=np.int32)
    pos = 0
    for b, n in enumerate(n_pages):
        table[b, :n] = ids[pos:pos + n]
        pos += n
    return table, num_blocks, ids


def _fill_blocks(rng, kv: np.ndarray, ids: np.ndarray, kv_dtype: str, k_scale: float,
                 chunk_elems: int = 1 << 26):
    """Draw N(0,1) values for the used blocks `ids` (in order) and encode them."""
    per_block = int(np.prod(kv.shape[1:]))
    step = max(1, chunk_elems // max(per_block, 1))
    for i in range(0, len(ids), step):
        sel = ids[i:i + step]
        x = rng.standard_normal(size=(len(sel),) + kv.shape[1:], dtype=np.float32)
        if kv_dtype == "bf16":
            kv[sel] = to_bf16_bits(x)
        else:
            x /= np.float32(k_scale)
            kv[sel] = to_e4m3_codes(x)


# Per-token-head quantised GQA caches: code range each row is scaled into.
PTH_DTYPES = {"fp8_e4m3_pth": E4M3_MAX, "int8_pth": 127.0, "int4_pth": 7.0}


def pth_code_bytes(D: int, kv_dtype: str) -> int:
    """Bytes of codes per (token, KV head) row: D, or D / 2 for packed int4."""
    return D // 2 if kv_dtype == "int4_pth" else D


def encode_pth_rows(x: np.ndarray, kv_dtype: str) -> np.ndarray:
    """Quantise rows x[..., D] (float32) per row: scale = max|x| / code range
    (1 for an all-zero row), codes = x / scale encoded as e4m3 (torch's cast),
    as int8 (round half to even, clipped to +-127) or as int4 (the same,
    clipped to [-8, 7], two per byte: element 2i in the low nibble of byte i);
    returns uint8 [..., C + 4]: the C code bytes followed by the scale as
    little-endian binary32."""
    top = PTH_DTYPES[kv_dtype]
    amax = np.abs(x).max(axis=-1, keepdims=True)
    sc = np.where(amax > 0, amax / np.float32(top), np.float32(1.0)).astype(np.float32)
    y = x / sc
    if kv_dtype == "fp8_e4m3_pth":
        codes = to_e4m3_codes(y)
    elif kv_dtype == "int4_pth":
        n = np.clip(np.rint(y), -8, 7).astype(np.int16) & 15
        codes = (n[..., 0::2] | (n[..., 1::2] << 4)).astype(np.uint8)
    else:
        codes = np.clip(np.rint(y), -127, 127).astype(np.int8).view(np.uint8)
    out = np.empty(x.shape[:-1] + (codes.shape[-1] + 4,), dtype=np.uint8)
    out[..., :-4] = codes
    out[..., -4:] = sc.astype("<f4").view(np.uint8).reshape(x.shape[:-1] + (4,))
    return out


def _fill_blocks_pth(rng, kv: np.ndarray, ids: np.ndarray, kv_dtype: str, chunk_elems: int = 1 << 26):
    """Draw N(0,1) rows for the used blocks `ids` and quantise each (token, KV
    head) row of each plane with its own scale."""
    D = 2 * (kv.shape[-1] - 4) if kv_dtype == "int4_pth" else kv.shape[-1] - 4
    shape = kv.shape[1:-1] + (D,)
    per_block = int(np.prod(shape))
    step = max(1, chunk_elems // max(per_block, 1))
    for i in range(0, len(ids), step):
        sel = ids[i:i + step]
        x = rng.standard_normal(size=(len(sel),) + shape, dtype=np.float32)
        kv[sel] = encode_pth_rows(x, kv_dtype)


def draw_topk_indices(rng: np.random.Generator, seq_lens: np.ndarray, topk: int,
                      pad: float = 0.0) -> np.ndarray:
    """Sparse-decode index lists, int32 [B, topk]: min(topk, seq_len) distinct
    positions of each request in random order, -1 in the remaining entries,
    and a share `pad` of all entries replaced by -1."""
    out = np.full((len(seq_lens), topk), -1, dtype=np.int32)
    for b, n in enumerate(seq_lens):
        k = min(topk, int(n))
        if k > 0:
            out[b, :k] = rng.choice(int(n), size=k, replace=False)
        if pad > 0:
            out[b, rng.random(topk) < pad] = -1
    return out


def make_mla_case(seq_lens, B=None, H=16, D=576, R=None, page=16, kv_dtype="bf16",
                  k_scale=1.0, pool_factor=1.0, seed=0, scale=None, name="",
                  extra_cols=0) -> PagedCase:
    rng = np.random.default_rng(seed)
    if B is None:
        B = len(seq_lens)
    sl = draw_seq_lens(rng, B, seq_lens)
    R = D - 64 if R is None else R
    scale = 1.0 / math.sqrt(192.0) if scale is None else scale
    table, nb, ids = build_block_table(rng, sl, page, pool_factor, extra_cols)
    q = to_bf16_bits(rng.standard_normal(size=(B, H, D), dtype=np.float32))
    kv = np.zeros((nb, page, D), dtype=np.uint16 if kv_dtype == "bf16" else np.uint8)
    _fill_blocks(rng, kv, ids, kv_dtype, k_scale)
    return PagedCase("mla", q, kv, table, sl, kv_dtype, float(scale),
                     k_scale=float(k_scale) if kv_dtype != "bf16" else 1.0,
                     v_scale=float(k_scale) if kv_dtype != "bf16" else 1.0,
                     page=page, num_kv_heads=1, kv_lora_rank=R, name=name)


def make_gqa_case(seq_lens, B=None, Hq=32, Hkv=8, D=128, page=16, kv_dtype="bf16",
                  k_scale=1.0, v_scale=1.0, pool_factor=1.0, seed=0, scale=None, name="",
                  extra_cols=0) -> PagedCase:
    rng = np.random.default_rng(seed)
    if B is None:
        B = len(seq_lens)
    sl = draw_seq_lens(rng, B, seq_lens)
    scale = 1.0 / math.sqrt(float(D)) if scale is None else scale
    table, nb, ids = build_block_table(rng, sl, page, pool_factor, extra_cols)
    q = to_bf16_bits(rng.standard_normal(size=(B, Hq, D), dtype=np.float32))
    if kv_dtype in PTH_DTYPES:
        kv = np.zeros((nb, 2, page, Hkv, pth_code_bytes(D, kv_dtype) + 4), dtype=np.uint8)
        _fill_blocks_pth(rng, kv, ids, kv_dtype)
        return PagedCase("gqa", q, kv, table, sl, kv_dtype, float(scale), page=page, num_kv_heads=Hkv,
                         kv_lora_rank=0, name=name)
    kv = np.zeros((nb, 2, page, Hkv, D), dtype=np.uint16 if kv_dtype == "bf16" else np.uint8)
    _fill_blocks(rng, kv, ids, kv_dtype, k_scale)
    return PagedCase("gqa", q, kv, table, sl, kv_dtype, float(scale),
                     k_scale=float(k_scale) if kv_dtype != "bf16" else 1.0,
                     v_scale=float(v_scale) if kv_dtype != "bf16" else 1.0,
                     page=page, num_kv_heads=Hkv, kv_lora_rank=0, name=name)


WORKLOADS = {
    "tiny_mla": dict(kind="mla", seq_lens=[37, 100], H=16, D=576, page=16, kv_dtype="bf16",
                     seed=1001),
    "mla_v2lite": dict(kind="mla", B=64, seq_lens=("uniform", 1024, 8192), H=16, D=576, page=64,
                       kv_dtype="bf16", pool_factor=1.5, seed=1002),
    "mla_v3_fp8": dict(kind="mla", B=128, seq_lens=("uniform", 4096, 32768), H=128, D=576,
                       page=64, kv_dtype="fp8_e4m3", k_scale=0.05, seed=1003),
    "mla_longctx": dict(kind="mla", seq_lens=[131072, 98304, 65536, 120000], H=128, D=576,
                        page=64, kv_dtype="bf16", seed=1004),
    "gqa": dict(kind="gqa", B=256, seq_lens=("lognormal", 2048, 1.0, 16384), Hq=32, Hkv=8, D=128,
                page=16, kv_dtype="bf16", seed=1005),
    # per-token-head quantised GQA caches (same batch as "gqa", own seeds)
    "gqa_fp8_pth": dict(kind="gqa", B=256, seq_lens=("lognormal", 2048, 1.0, 16384), Hq=32, Hkv=8, D=128,
                        page=16, kv_dtype="fp8_e4m3_pth", seed=1008),
    "gqa_int8_pth": dict(kind="gqa", B=256, seq_lens=("lognormal", 2048, 1.0, 16384), Hq=32, Hkv=8, D=128,
                         page=16, kv_dtype="int8_pth", seed=1009),
    "gqa_int4_pth": dict(kind="gqa", B=256, seq_lens=("lognormal", 2048, 1.0, 16384), Hq=32, Hkv=8, D=128,
                         page=16, kv_dtype="int4_pth", seed=1011),
    # multi-token decode (speculative verification): the V2-Lite-like batch
    # with 8 new positions per request, 16 heads -> 128 query rows (q is
    # [B, q_len, H, D], stored here as its [B, q_len * H, D] view)
    "mla_mtp": dict(kind="mla", B=64, seq_lens=("uniform", 1024, 8192), H=128, D=576, page=64,
                    kv_dtype="bf16", pool_factor=1.5, seed=1006, q_len=8),
    # sparse (top-k) decode: 2048 selected positions per request out of
    # 16k..40k-token contexts, 16 heads (128 heads split 8 ways); the index
    # lists are in case.meta["indices"]
    "mla_sparse": dict(kind="mla", B=64, seq_lens=("uniform", 16384, 40960), H=16, D=576, page=64,
                       kv_dtype="bf16", seed=1007, topk=2048),
}


def workload(name: str, **overrides) -> PagedCase:
    """Build a named workload; keyword overrides replace its parameters."""
    spec = dict(WORKLOADS[name])
    spec.update(overrides)
    kind = spec.pop("kind")
    q_len = spec.pop("q_len", 1)
    topk = spec.pop("topk", 0)
    spec.setdefault("name", name)
    if kind == "mla":
        case = make_mla_case(**spec)
        case.meta["q_len"] = q_len  # query rows are q_len x heads, token-major
        if topk:
            rng = np.random.default_rng(int(spec["seed"]) + 7919)
            case.meta["indices"] = draw_topk_indices(rng, case.seq_lens, topk)
        return case
    return make_gqa_case(**spec)


def shard_case(case: PagedCase, num_shards: int) -> list:
    """Cut every sequence of `case` into `num_shards` page-aligned shards, as
    decode context parallelism places a request's KV pages on several ranks:
    shard g of a sequence with n tokens (np pages) holds pages
    [g L, min((g + 1) L, np)), L = ceil(np / num_shards).  Returns one case
    per shard with the same q and cache, the shard's block-table columns and
    its token count (0 for a shard past the end)."""
    P = case.page
    n = case.seq_lens.astype(np.int64)
    npg = (n + P - 1) // P
    L = np.maximum((npg + num_shards - 1) // num_shards, 1)
    width = int(L.max()) if len(L) else 1
    shards = []
    for g in range(num_shards):
        table = np.full((case.batch, width), -1, dtype=np.int32)
        sl = np.zeros(case.batch, dtype=np.int32)
        for b in range(case.batch):
            j0 = int(g * L[b])
            j1 = int(min((g + 1) * L[b], npg[b]))
            if j1 > j0:
                table[b, :j1 - j0] = case.block_table[b, j0:j1]
                sl[b] = int(min(j1 * P, n[b]) - j0 * P)
        shards.append(replace(case, block_table=table, seq_lens=sl))
    return shards


def poison(case: PagedCase, table_fill: int = -1) -> PagedCase:
    """Copy of `case` with NaN in every cache slot no valid token owns (tail
    slots of last pages and unreferenced blocks) and `table_fill` in every
    block-table entry past a sequence's last page."""
    kv = case.kv.copy()
    nan = BF16_NAN if kv.dtype == np.uint16 else E4M3_NAN
    if case.kv_dtype in PTH_DTYPES:
        # codes 0x7F (NaN for e4m3, 127 for int8) and a NaN scale
        nan = np.array([0x7F] * (kv.shape[-1] - 4) + [0x00, 0x00, 0xC0, 0x7F], dtype=np.uint8)
    used = np.zeros(case.num_blocks, dtype=bool)
    table = case.block_table.copy()
    P = case.page
    for b, n in enumerate(case.seq_lens):
        npg = (int(n) + P - 1) // P
        blocks = table[b, :npg]
        used[blocks] = True
        table[b, npg:] = table_fill
        tail = int(n) - (npg - 1) * P
        if npg > 0 and tail < P:
            last = blocks[-1]
            if case.kind == "mla":
                kv[last, tail:, :] = nan
            else:
                kv[last, :, tail:, :, :] = nan
    kv[~used] = nan
    return replace(case, kv=kv, block_table=table)
