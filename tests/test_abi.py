"""C-ABI checks that need no GPU: the library loads, exports every function the
header declares, its pure host helpers agree with the pages' rules, and host
validation rejects bad arguments before anything touches the device.

Every call below that passes fake device pointers is built to FAIL validation,
so nothing is ever enqueued with them, on any machine.
"""
import ctypes
import json
import os
import re

import pytest

from mqa_decode_attention_paged_gb300 import _binding as mqa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FAKE = 0x10000  # aligned, never dereferenced (validation fails first)


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in {"defined"}))


def test_header_symbols_are_exported():
    names = _declared_functions()
    # the test hooks sit in their own header, not in the product interface
    product = open(os.path.join(ROOT, "include", "mqa_decode.h")).read()
    assert "mqa_test_" not in product
    assert {"mqa_test_gqa_withheld_arrive", "mqa_test_mla_withheld_arrive",
            "mqa_test_mla_warp_gives_up"} <= set(names)
    assert {"mla_decode", "mla_decode_fixed_splits", "mla_decode_multi", "mla_decode_sparse", "gqa_paged_decode", "mqa_lse_merge",
            "mqa_num_kv_splits", "mla_decode_workspace_bytes",
            "gqa_paged_decode_workspace_bytes", "mqa_status_string", "mqa_abi_version",
            "mqa_device_sm_count", "mqa_dcp_shard_max_blocks", "mqa_dcp_shard", "mqa_dcp_locate",
            "mqa_dcp_scale_shard"} <= set(names)
    lib = ctypes.CDLL(mqa.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_abi_version_and_status_strings():
    assert mqa.abi_version() == 1
    for code in range(7):
        assert mqa.status_string(code) and mqa.status_string(code) != "unknown status"
    assert mqa.status_string(99) == "unknown status"


def test_num_kv_splits_matches_golden():
    with open(os.path.join(ROOT, "tests", "golden", "num_kv_splits.json")) as f:
        g = json.load(f)
    for c in g["cases"]:
        assert mqa.num_kv_splits(c["max_seq_len"], c["sm_count"], c["batch_invariant"]) == c["splits"], c


def test_workspace_bytes():
    # [B, H, S, R + 1] fp32, nothing for a single split.
    assert mqa.mla_decode_workspace_bytes(64, 16, 512, 16) == 64 * 16 * 16 * 513 * 4
    assert mqa.mla_decode_workspace_bytes(4, 128, 512, 1) == 0
    assert mqa.gqa_paged_decode_workspace_bytes(256, 32, 128, 32) == 256 * 32 * 32 * 129 * 4
    assert mqa.mla_decode_workspace_bytes(0, 16, 512, 2) == 0


def _mla(**kw):
    a = dict(q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, scale=0.07, k_scale=1.0, out=FAKE, lse=None,
             B=2, H=16, D=576, R=512, nb=10, P=16, maxb=8, kvd=0, S=1, ws=None, wsb=0,
             status=None, stream=None)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731
    return mqa.lib.mla_decode(P(a["q"]), P(a["kv"]), P(a["bt"]), P(a["sl"]), a["scale"], a["k_scale"],
                              P(a["out"]), P(a["lse"]), a["B"], a["H"], a["D"], a["R"], a["nb"],
                              a["P"], a["maxb"], a["kvd"], a["S"], P(a["ws"]), a["wsb"],
                              P(a["status"]), P(a["stream"]))


def _mla_multi(**kw):
    a = dict(q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, scale=0.07, k_scale=1.0, out=FAKE, lse=None,
             B=2, L=4, H=16, D=576, R=512, nb=10, P=16, maxb=8, kvd=0, S=1, ws=None, wsb=0)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731
    return mqa.lib.mla_decode_multi(P(a["q"]), P(a["kv"]), P(a["bt"]), P(a["sl"]), a["scale"], a["k_scale"],
                                    P(a["out"]), P(a["lse"]), a["B"], a["L"], a["H"], a["D"], a["R"], a["nb"],
                                    a["P"], a["maxb"], a["kvd"], a["S"], P(a["ws"]), a["wsb"], None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(L=0), mqa.ERR_INVALID_ARG),
    (dict(H=0), mqa.ERR_INVALID_ARG),
    (dict(L=9, H=16), mqa.ERR_UNSUPPORTED),            # q_len x heads rows at most 128
    (dict(L=129, H=1), mqa.ERR_UNSUPPORTED),
    (dict(q=None), mqa.ERR_INVALID_ARG),               # then the checks of mla_decode on the rows
    (dict(D=512, R=448), mqa.ERR_UNSUPPORTED),
    (dict(S=4, ws=FAKE, wsb=mqa.mla_decode_workspace_bytes(2, 64, 512, 4) - 1), mqa.ERR_WORKSPACE_TOO_SMALL),
])
def test_mla_multi_validation(kw, code):
    assert _mla_multi(**kw) == code


def _mla_sparse(**kw):
    a = dict(q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, idx=FAKE, scale=0.07, k_scale=1.0, out=FAKE, lse=None,
             B=2, H=16, D=576, R=512, nb=10, P=16, maxb=8, topk=2048, kvd=0, S=1, ws=None, wsb=0)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731
    return mqa.lib.mla_decode_sparse(P(a["q"]), P(a["kv"]), P(a["bt"]), P(a["sl"]), P(a["idx"]), a["scale"],
                                     a["k_scale"], P(a["out"]), P(a["lse"]), a["B"], a["H"], a["D"], a["R"],
                                     a["nb"], a["P"], a["maxb"], a["topk"], a["kvd"], a["S"], P(a["ws"]),
                                     a["wsb"], None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(idx=None), mqa.ERR_INVALID_ARG),
    (dict(idx=FAKE + 2), mqa.ERR_INVALID_ARG),         # indices are int32
    (dict(topk=0), mqa.ERR_INVALID_ARG),
    (dict(topk=(1 << 24) + 1), mqa.ERR_UNSUPPORTED),
    (dict(q=None), mqa.ERR_INVALID_ARG),
    (dict(bt=None), mqa.ERR_INVALID_ARG),
    (dict(H=0), mqa.ERR_INVALID_ARG),
    (dict(H=129), mqa.ERR_UNSUPPORTED),
    (dict(B=4097), mqa.ERR_UNSUPPORTED),
    (dict(D=512, R=448), mqa.ERR_UNSUPPORTED),
    (dict(kvd=7), mqa.ERR_UNSUPPORTED),
    (dict(scale=float("inf")), mqa.ERR_INVALID_ARG),
    (dict(S=4, ws=None), mqa.ERR_WORKSPACE_TOO_SMALL),
    (dict(S=4, ws=FAKE, wsb=mqa.mla_decode_workspace_bytes(2, 16, 512, 4) - 1), mqa.ERR_WORKSPACE_TOO_SMALL),
])
def test_mla_sparse_validation(kw, code):
    assert _mla_sparse(**kw) == code


def _gqa(**kw):
    a = dict(q=FAKE, kv=FAKE, bt=FAKE, sl=FAKE, scale=0.09, ks=1.0, vs=1.0, out=FAKE, lse=None, B=2, Hq=32,
             Hkv=8, D=128, nb=10, P=16, maxb=8, kvd=0, S=1, ws=None, wsb=0)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731
    return mqa.lib.gqa_paged_decode(P(a["q"]), P(a["kv"]), P(a["bt"]), P(a["sl"]), a["scale"], a["ks"],
                                    a["vs"], P(a["out"]), P(a["lse"]), a["B"], a["Hq"], a["Hkv"], a["D"],
                                    a["nb"], a["P"], a["maxb"], a["kvd"], a["S"], P(a["ws"]), a["wsb"],
                                    None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), mqa.ERR_INVALID_ARG),
    (dict(kv=None), mqa.ERR_INVALID_ARG),
    (dict(bt=None), mqa.ERR_INVALID_ARG),
    (dict(sl=None), mqa.ERR_INVALID_ARG),
    (dict(out=None), mqa.ERR_INVALID_ARG),
    (dict(q=FAKE + 8), mqa.ERR_INVALID_ARG),          # not 16-byte aligned
    (dict(kv=FAKE + 4), mqa.ERR_INVALID_ARG),
    (dict(B=0), mqa.ERR_INVALID_ARG),
    (dict(H=0), mqa.ERR_INVALID_ARG),
    (dict(S=0), mqa.ERR_INVALID_ARG),
    (dict(scale=float("nan")), mqa.ERR_INVALID_ARG),
    (dict(D=512, R=448), mqa.ERR_UNSUPPORTED),         # head sizes 320 / 576 only
    (dict(D=576, R=256), mqa.ERR_UNSUPPORTED),
    (dict(P=24), mqa.ERR_UNSUPPORTED),                 # page must be a multiple of 16
    (dict(P=8), mqa.ERR_UNSUPPORTED),
    (dict(kvd=7), mqa.ERR_UNSUPPORTED),
    (dict(kvd=2), mqa.ERR_UNSUPPORTED),                # per-token-head formats are GQA-only
    (dict(kvd=3), mqa.ERR_UNSUPPORTED),
    (dict(kvd=4), mqa.ERR_UNSUPPORTED),
    (dict(H=129), mqa.ERR_UNSUPPORTED),
    (dict(B=4097), mqa.ERR_UNSUPPORTED),
    (dict(S=4, ws=None, wsb=0), mqa.ERR_WORKSPACE_TOO_SMALL),
    (dict(S=4, ws=FAKE, wsb=2 * 16 * 4 * 513 * 4 - 1), mqa.ERR_WORKSPACE_TOO_SMALL),
])
def test_mla_validation(kw, code):
    assert _mla(**kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), mqa.ERR_INVALID_ARG),
    (dict(Hq=30, Hkv=8), mqa.ERR_INVALID_ARG),         # Hq must be a multiple of Hkv
    (dict(D=96), mqa.ERR_UNSUPPORTED),
    (dict(Hkv=16, Hq=32), mqa.ERR_UNSUPPORTED),
    (dict(Hkv=1, Hq=32), mqa.ERR_UNSUPPORTED),         # at most 16 query heads per KV head
    (dict(kvd=5), mqa.ERR_UNSUPPORTED),                # bf16, e4m3 and the per-token-head formats only
    (dict(kvd=-1), mqa.ERR_UNSUPPORTED),
    (dict(kvd=1, ks=float("nan")), mqa.ERR_INVALID_ARG),  # per-tensor fp8 needs finite scales
    (dict(kvd=1, vs=float("inf")), mqa.ERR_INVALID_ARG),
    (dict(kvd=1, S=2), mqa.ERR_WORKSPACE_TOO_SMALL),   # each accepted format reaches the workspace check
    (dict(kvd=2, S=2), mqa.ERR_WORKSPACE_TOO_SMALL),
    (dict(kvd=3, S=2, ks=float("nan")), mqa.ERR_WORKSPACE_TOO_SMALL),  # scales unused by per-token-head
    (dict(kvd=4, S=2), mqa.ERR_WORKSPACE_TOO_SMALL),
    (dict(P=40), mqa.ERR_UNSUPPORTED),
    (dict(S=2), mqa.ERR_WORKSPACE_TOO_SMALL),
])
def test_gqa_validation(kw, code):
    assert _gqa(**kw) == code


def _merge(**kw):
    a = dict(outs=FAKE, lses=FAKE, out=FAKE, lse=None, G=4, rows=64, D=512)
    a.update(kw)
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731
    return mqa.lib.mqa_lse_merge(P(a["outs"]), P(a["lses"]), P(a["out"]), P(a["lse"]), a["G"], a["rows"], a["D"],
                                 None)


@pytest.mark.parametrize("kw,code", [
    (dict(outs=None), mqa.ERR_INVALID_ARG),
    (dict(lses=None), mqa.ERR_INVALID_ARG),
    (dict(out=None), mqa.ERR_INVALID_ARG),
    (dict(outs=FAKE + 8), mqa.ERR_INVALID_ARG),         # 16-byte alignment
    (dict(lses=FAKE + 4), mqa.ERR_INVALID_ARG),
    (dict(lse=FAKE + 4), mqa.ERR_INVALID_ARG),
    (dict(G=0), mqa.ERR_INVALID_ARG),
    (dict(rows=0), mqa.ERR_INVALID_ARG),
    (dict(D=4), mqa.ERR_INVALID_ARG),                   # head_dim a multiple of 8 in [8, 4096]
    (dict(D=100), mqa.ERR_INVALID_ARG),
    (dict(D=4104), mqa.ERR_INVALID_ARG),
    (dict(rows=1 << 40), mqa.ERR_UNSUPPORTED),
])
def test_lse_merge_validation(kw, code):
    assert _merge(**kw) == code


def test_withheld_arrive_hook_validation(monkeypatch):
    fn = mqa.lib.mqa_test_gqa_withheld_arrive
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fn.restype = I
    fn.argtypes = [P, P, P, P, F, P, P, I, I, I, I, I, I, I, I, P, SZ, P, P, I]
    f = ctypes.c_void_p(FAKE)
    args = [f, f, f, f, 0.09, f, None, 2, 8, 2, 128, 10, 16, 8, 1, None, 0, None, None]
    # without the gate the hook refuses before looking at anything
    monkeypatch.delenv("MQA_ENABLE_TEST_HOOKS", raising=False)
    assert fn(*args, 0) == mqa.ERR_UNSUPPORTED
    monkeypatch.setenv("MQA_ENABLE_TEST_HOOKS", "0")
    assert fn(*args, 0) == mqa.ERR_UNSUPPORTED
    monkeypatch.setenv("MQA_ENABLE_TEST_HOOKS", "1")
    assert fn(*args, -1) == mqa.ERR_INVALID_ARG          # a unit to withhold is required
    assert fn(*(args[:7] + [0] + args[8:]), 0) == mqa.ERR_INVALID_ARG  # the usual validation runs first
    assert fn(*(args[:14] + [2] + args[15:]), 0) == mqa.ERR_WORKSPACE_TOO_SMALL


def test_mla_withheld_arrive_hook_validation(monkeypatch):
    fn = mqa.lib.mqa_test_mla_withheld_arrive
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fn.restype = I
    fn.argtypes = [P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, I, I, P, SZ, P, P, I]
    f = ctypes.c_void_p(FAKE)
    args = [f, f, f, f, 0.07, 1.0, f, None, 2, 16, 576, 512, 10, 16, 8, 0, 1, None, 0, None, None]
    monkeypatch.delenv("MQA_ENABLE_TEST_HOOKS", raising=False)
    assert fn(*args, 0) == mqa.ERR_UNSUPPORTED          # gated
    monkeypatch.setenv("MQA_ENABLE_TEST_HOOKS", "1")
    assert fn(*args, -1) == mqa.ERR_INVALID_ARG         # a unit to withhold is required
    assert fn(*(args[:8] + [0] + args[9:]), 0) == mqa.ERR_INVALID_ARG   # the usual validation runs first
    assert fn(*(args[:10] + [320] + args[11:]), 0) == mqa.ERR_UNSUPPORTED
    assert fn(*(args[:16] + [2] + args[17:]), 0) == mqa.ERR_WORKSPACE_TOO_SMALL


def test_dcp_scale_shard_validation():
    # argument errors come back before anything is enqueued (no GPU needed)
    f = mqa.lib.mqa_dcp_scale_shard
    P = lambda v: None if v is None else ctypes.c_void_p(v)  # noqa: E731

    def call(so=FAKE, gl=FAKE, dst=FAKE, lse=None, G=2, r=0, B=3, H=16, D=512, f32=1):
        return f(P(so), P(gl), P(dst), P(lse), G, r, B, H, D, f32, None)

    assert call(so=None) == mqa.ERR_INVALID_ARG
    assert call(dst=None) == mqa.ERR_INVALID_ARG
    assert call(so=FAKE + 8) == mqa.ERR_INVALID_ARG        # unaligned
    assert call(lse=FAKE + 4) == mqa.ERR_INVALID_ARG
    assert call(r=2) == mqa.ERR_INVALID_ARG
    assert call(r=-1) == mqa.ERR_INVALID_ARG
    assert call(G=3) == mqa.ERR_INVALID_ARG                # 16 heads over 3 ranks
    assert call(G=0) == mqa.ERR_INVALID_ARG
    assert call(D=12) == mqa.ERR_INVALID_ARG
    assert call(D=8192) == mqa.ERR_INVALID_ARG
    assert call(B=0) == mqa.ERR_INVALID_ARG


def test_mla_warp_gives_up_hook_validation(monkeypatch):
    fn = mqa.lib.mqa_test_mla_warp_gives_up
    P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    fn.restype = I
    fn.argtypes = [P, P, P, P, F, F, P, P, I, I, I, I, I, I, I, I, P, SZ, P, P, I, I]
    f = ctypes.c_void_p(FAKE)
    args = [f, f, f, f, 0.07, 1.0, f, None, 2, 128, 576, 512, 10, 64, 8, 1, None, 0, None, None]
    monkeypatch.delenv("MQA_ENABLE_TEST_HOOKS", raising=False)
    assert fn(*args, 0, 3) == mqa.ERR_UNSUPPORTED          # gated
    monkeypatch.setenv("MQA_ENABLE_TEST_HOOKS", "1")
    assert fn(*args, -1, 3) == mqa.ERR_INVALID_ARG
    assert fn(*args, 0, 1) == mqa.ERR_INVALID_ARG          # not a softmax warp
    assert fn(*args, 0, 10) == mqa.ERR_INVALID_ARG
    assert fn(*(args[:9] + [32] + args[10:]), 0, 3) == mqa.ERR_INVALID_ARG   # no tensor-core kernel
    assert fn(*(args[:8] + [0] + args[9:]), 0, 3) == mqa.ERR_INVALID_ARG    # the usual validation runs
