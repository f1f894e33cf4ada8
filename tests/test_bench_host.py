"""Host-side logic of bench.py for N > 1 ranks, on the CPU with gloo.

The GPU bench runs one replica of the workload per rank (weak scaling) and
reports the slowest rank's step time; these tests cover that reduction with
two gloo processes, the whole-job throughput, and the reference arm's rank
handling (only rank 0 runs the oracle and prints)."""
import json
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms per step and 10 - r ms end to end
        got = bench.max_over_ranks([rank + 1.0, 10.0 - rank], dist)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump(got, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_processes(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        with open(tmp_path / f"rank{r}.json") as f:
            assert json.load(f) == [2.0, 10.0]


def test_max_over_ranks_without_a_group_is_identity():
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]


def test_whole_job_throughput_scales_with_ranks():
    one = bench.job_throughput_gbs(1, 1e9, 10.0)
    assert one == pytest.approx(100.0)
    assert bench.job_throughput_gbs(4, 1e9, 10.0) == pytest.approx(4 * one)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")

    class Args:
        workload = "tiny_mla"
        splits = 0
        steps = 1
        warmup = 0
        gpus = 2
        ref_budget = 0.05

    assert bench.run_reference(Args()) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_rank_zero_prints_one_line(monkeypatch, capsys):
    pytest.importorskip("numpy")
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("LOCAL_RANK", "0")

    class Args:
        workload = "tiny_mla"
        splits = 0
        steps = 1
        warmup = 0
        gpus = 1
        ref_budget = 0.05

    bench.run_reference(Args())
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["gpu_launches"] == 0


def test_algorithmic_bytes_and_flops_per_workload():
    # The roofline's numerator: cache bytes of the valid (or selected) tokens
    # plus q, out and lse, in each cache format; FLOPs 2 H tokens (D + R) for
    # MLA and 4 Hq tokens D for GQA.
    import numpy as np
    import synth
    mla = synth.make_mla_case([37, 100], H=16, D=576, page=16, seed=1)
    st = bench.workload_stats(mla, 1)
    assert st["tokens"] == 137
    assert st["kv_bytes"] == 137 * 576 * 2
    assert st["alg_bytes"] == st["kv_bytes"] + 2 * 16 * 576 * 2 + 2 * 16 * 512 * 2 + 2 * 16 * 4
    assert st["flops"] == 2.0 * 16 * 137 * (576 + 512)
    fp8 = synth.make_mla_case([37, 100], H=16, D=576, page=16, kv_dtype="fp8_e4m3", k_scale=0.05, seed=1)
    assert bench.workload_stats(fp8, 1)["kv_bytes"] == 137 * 576
    for kv_dtype, row, elt in (("bf16", 128, 2), ("fp8_e4m3", 128, 1), ("fp8_e4m3_pth", 132, 1),
                               ("int8_pth", 132, 1), ("int4_pth", 68, 1)):
        g = synth.make_gqa_case([19, 40], Hq=8, Hkv=2, D=128, page=16, kv_dtype=kv_dtype, seed=2)
        st = bench.workload_stats(g, 1)
        assert st["kv_bytes"] == 59 * 2 * 2 * row * elt, kv_dtype
        assert st["flops"] == 2.0 * 8 * 59 * 2 * 128
    # sparse: only the selected entries count, plus the index lists and one
    # block-table entry per selected row
    sp = synth.make_mla_case([50, 10], H=16, D=576, page=16, seed=3)
    idx = np.array([[0, 49, -1, 50], [3, 9, 9, 12]], dtype=np.int32)
    sp.meta["indices"] = idx
    st = bench.workload_stats(sp, 1)
    assert st["tokens"] == 5  # 0, 49 | 3, 9, 9 (positions >= seq_len and -1 select nothing)
    assert st["alg_bytes"] == 5 * 576 * 2 + 2 * 16 * 576 * 2 + 2 * 16 * 512 * 2 + 2 * 16 * 4 + idx.size * 4 + 5 * 4


def test_merge_workload_bytes():
    spec = bench.MERGE_WORKLOADS["dcp_merge_v3"]
    st = bench.merge_stats(spec)
    rows = spec["B"] * spec["H"]
    assert st["alg_bytes"] == spec["G"] * rows * spec["R"] * 2 + spec["G"] * rows * 4 + rows * spec["R"] * 2 + rows * 4
    assert st["in_bytes"] + st["out_bytes"] == st["alg_bytes"]


def test_clock_reason_bits_and_summary():
    # NVML clock-event reason bits (nvml.h): sw power cap 0x4, hw slowdown 0x8,
    # sw thermal 0x20, hw thermal 0x40, hw power brake 0x80; idle (0x1) and
    # application clocks (0x2) are not among the judged reasons
    assert bench.decode_reasons(0) == []
    assert bench.decode_reasons(0x1 | 0x2) == []
    assert bench.decode_reasons(0x4) == ["sw_power_cap"]
    assert bench.decode_reasons(0x8 | 0x40) == ["hw_slowdown", "hw_thermal_slowdown"]
    assert bench.decode_reasons(0x20 | 0x80) == ["hw_power_brake_slowdown", "sw_thermal_slowdown"]
    s = bench.summarize_clocks([(2070.0, []), (1980.0, ["sw_power_cap"]), (2070.0, [])], 2070.0, "test")
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                 "source": "test"}
    assert bench.summarize_clocks([], 2070.0, "test")["samples"] == 0
