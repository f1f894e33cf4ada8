"""Benchmark: paged MLA/GQA decode on GB300 through the C ABI.

One step = one decode call (split-KV stage 1 + LSE merge) over one batch of the
chosen workload, inputs resident in HBM.  Default workload: the MLA V3-like
batch (B=128, H=128, head 576 = 512 + 64, bf16 query, e4m3 KV cache with
k_scale 0.05, seq_lens uniform in [4096, 32768], page 64, random block
permutation), the largest of the MLA configurations and one that the 70 %
roofline target is set on; `--workload` picks the others (mla_longctx,
mla_v2lite, gqa, ...).

Prints ONE JSON line (rank 0).  `value` is KV GB/s (algorithmic KV bytes of the
valid tokens / device time, summed over ranks); `ms_per_step` gives the
per-call latency; `roofline` compares the decode call against the measured HBM
or bf16 tensor peak; `e2e` is the same metric with the per-step host<->device
copies (query, block table and lengths in; output and lse out) inside the
timed region; `cpu_baseline` times the fp64 CPU oracle on the host cores.

Timing: W untimed warm-up steps, then K steps.  Before every step a 256 MiB
buffer (> the 129 MB L2) is overwritten and then read back, so no KV line is
L2-resident and the flush's own dirty lines are written back before the timed
region instead of during it; each step is bracketed by CUDA events on the
launching stream (the flush is outside the events).  Under torchrun every rank runs an independent replica (the path
has no cross-GPU exchange), the timed region is bracketed by a barrier and
synchronize on both sides, and rank 0 reports the max over ranks.

`--split-mode fixed` times the dense MLA workloads with one work unit per
request and split (every request cut into num_kv_splits equal page ranges,
`mla_decode_fixed_splits`) instead of the page-balanced units of `mla_decode`.

`--impl reference` times the CPU oracle instead (no GPU work), on the same
workload, with a bounded sample of requests per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MLA decode µs/call, KV GB/s and % of roofline at B×H×seq_len (1 GB300)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one stage-1
# launch from an ncu capture (summaries under profiles/), keyed by workload;
# valid only while the sources that kernel is built from hash to `src_sha`.
MMA_FILES = ("mla_mma.cu", "common.cuh", "plan.cuh", "args.cuh")
TC_FILES = ("mla_tc.cu", "tc_ptx.cuh", "common.cuh", "plan.cuh", "args.cuh")
Q8_FILES = ("gqa_q8.cu", "gqa_q8.cuh", "common.cuh", "plan.cuh", "args.cuh")
MERGE_FILES = ("shard_merge.cu", "shard_merge.cuh", "common.cuh")
GQA_FILES = ("gqa_mma.cu", "common.cuh", "plan.cuh", "args.cuh")
SPARSE_FILES = MMA_FILES + ("api.cu",)  # the gather's tensor map is encoded there
NCU_TRAFFIC = {
    "mla_v2lite": {"files": MMA_FILES, "src_sha": "0a3a858fdff4ea58", "splits": 16, "bytes": 329795328 + 3672832,
                   "kernel": "mla_decode_mma_kernel<576,512,0,64,0,0,0>"},
    "mla_longctx": {"files": TC_FILES, "src_sha": "e5b65c697f1f6c69", "splits": 256, "bytes": 484526848 + 3496704,
                    "kernel": "mla_decode_tc_kernel<576,512,0,0,2>"},
    "mla_v3_fp8": {"files": TC_FILES, "src_sha": "e5b65c697f1f6c69", "splits": 64, "bytes": 1423863552 + 25623040,
                   "kernel": "mla_decode_tc_kernel<576,512,1,0,0>"},
    "mla_mtp": {"files": TC_FILES, "src_sha": "e5b65c697f1f6c69", "splits": 16, "bytes": 362287360 + 6680320,
                "kernel": "mla_decode_tc_kernel<576,512,0,1,2>"},
    "gqa": {"files": GQA_FILES, "src_sha": "5279abc033f1ca5a", "splits": 32, "bytes": 3241169152 + 4573696,
            "kernel": "gqa_decode_mma_kernel<128>"},
    "gqa_fp8_pth": {"files": Q8_FILES, "src_sha": "dba3282edc657b61", "splits": 32, "bytes": 1535350272 + 5330944,
                    "kernel": "gqa_decode_q8_kernel<128,2,1>"},
    "gqa_int8_pth": {"files": Q8_FILES, "src_sha": "dba3282edc657b61", "splits": 32, "bytes": 1689822464 + 5506560,
                     "kernel": "gqa_decode_q8_kernel<128,3,1>"},
    "gqa_int4_pth": {"files": Q8_FILES, "src_sha": "dba3282edc657b61", "splits": 32, "bytes": 843228416 + 4604160,
                     "kernel": "gqa_decode_q8_kernel<128,4,1>"},
    "dcp_merge_v3": {"files": MERGE_FILES, "src_sha": "8c157f962d4da4f4", "bytes": 126340608 + 7121920,
                     "kernel": "shard_merge_kernel"},
    "mla_sparse": {"files": SPARSE_FILES, "src_sha": "4949d7ed343be6ee", "splits": 4, "bytes": 152941056 + 3016192,
                   "kernel": "mla_decode_mma_kernel<576,512,0,64,0,1,0>"},
}


def kernel_sources_sha(files=None) -> str:
    h = hashlib.sha256()
    d = os.path.join(ROOT, "mqa_decode_attention_paged_gb300", "csrc")
    for fn in sorted(files if files is not None else os.listdir(d)):
        with open(os.path.join(d, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def workload_stats(case, splits):
    """Algorithmic bytes and flops of one decode call.  Sparse decode reads
    the selected rows only (plus the index lists and one block-table entry per
    selected row)."""
    idx = case.meta.get("indices")
    if idx is not None:
        sel = (idx >= 0) & (idx < case.seq_lens[:, None])
        tokens = int(sel.sum())
    else:
        tokens = int(case.seq_lens.astype(np.int64).sum())
    elt = 2 if case.kv_dtype == "bf16" else 1
    B, H, D = case.q.shape
    if case.kind == "mla":
        R = case.kv_lora_rank
        kv_bytes = tokens * D * elt
        flops = 2.0 * H * tokens * (D + R)
        out_w = R
    else:
        Hkv = case.num_kv_heads
        # per-token-head rows carry their 4-byte scale after the codes
        row = {"fp8_e4m3_pth": D + 4, "int8_pth": D + 4, "int4_pth": D // 2 + 4}.get(case.kv_dtype, D)
        kv_bytes = tokens * 2 * Hkv * row * elt
        flops = 2.0 * H * tokens * 2 * D
        out_w = D
    io_bytes = B * H * D * 2 + B * H * out_w * 2 + B * H * 4
    if idx is not None:
        io_bytes += idx.size * 4 + tokens * 4
    return dict(tokens=tokens, kv_bytes=kv_bytes, alg_bytes=kv_bytes + io_bytes, flops=flops,
                q_bytes=B * H * D * 2, out_bytes=B * H * out_w * 2, lse_bytes=B * H * 4)


def load_workload(synth, args):
    """The named workload, with its batch overridden by --batch (a smaller
    case of the same shape, e.g. for a profiler capture)."""
    if not getattr(args, "batch", 0):
        return synth.workload(args.workload)
    if "B" not in synth.WORKLOADS[args.workload]:
        raise SystemExit(f"--batch: workload {args.workload} has explicit sequence lengths")
    return synth.workload(args.workload, B=args.batch)


def workload_config(case, name, splits):
    import synth
    spec = synth.WORKLOADS[name]
    cfg = {"workload": name, "kind": case.kind, "batch": case.batch, "num_heads": case.num_heads,
           "head_size": case.head_size, "page_size": case.page, "kv_dtype": case.kv_dtype,
           "seq_lens": spec["seq_lens"] if not isinstance(spec["seq_lens"], tuple) else list(spec["seq_lens"]),
           "total_tokens": int(case.seq_lens.astype(np.int64).sum()),
           "num_kv_splits": splits, "seed": spec["seed"],
           "l2": "flushed before every timed step: 256 MiB written then read back (cold, clean L2), "
                 "outside the timed events"}
    if case.kind == "mla":
        cfg["kv_lora_rank"] = case.kv_lora_rank
        if case.meta.get("q_len", 1) > 1:
            cfg["q_len"] = case.meta["q_len"]
            cfg["num_heads"] = case.num_heads // case.meta["q_len"]
            cfg["query_rows"] = case.num_heads
        if case.meta.get("indices") is not None:
            cfg["topk"] = int(case.meta["indices"].shape[1])
            cfg["selected_tokens"] = workload_stats(case, splits)["tokens"]
    else:
        cfg["num_kv_heads"] = case.num_kv_heads
    return cfg


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*): the ones a
# run is judged by.
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def decode_reasons(mask: int):
    """Names of the judged NVML clock-event reasons set in `mask`."""
    return sorted(n for bit, n in NVML_REASONS.items() if mask & bit)


def summarize_clocks(samples, max_mhz, source):
    """samples: [(sm_mhz, reason names)] taken while the timed region ran."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": max_mhz, "reasons": [], "samples": 0, "source": source}
    reasons = sorted(set(r for _, rs in samples for r in rs))
    return {"sm_mhz": statistics.median(m for m, _ in samples), "sm_max_mhz": max_mhz, "reasons": reasons,
            "samples": len(samples), "source": source}


class NvmlPoller:
    """Reads the SM clock and the clock-event reasons of one GPU through NVML
    (libnvidia-ml, part of the driver) every `period_s` on a background
    thread.  Read-only: it changes no setting of the GPU."""

    def __init__(self, pci_bus_id: str | None, index: int, period_s: float = 0.001):
        import ctypes
        import threading
        self.ct = ctypes
        self.period = period_s
        self.samples = []
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.h = ctypes.c_void_p()
        ok = False
        if pci_bus_id:
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:  # 1 = NVML_CLOCK_SM
            self.max_mhz = float(mx.value)

    def read(self):
        c = self.ct
        mhz, rs = c.c_uint(), c.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.h, 1, c.byref(mhz)) != 0:
            return None
        if self.reason_fn(self.h, c.byref(rs)) != 0:
            return None
        return float(mhz.value), decode_reasons(int(rs.value))

    def _run(self):
        while not self._stop.is_set():
            r = self.read()
            if r is not None:
                self.samples.append(r)
            self._stop.wait(self.period)

    def start(self):
        import threading
        self._thread = threading.Thread(target=self._run, daemon=True)
        self._thread.start()

    def stop(self):
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=5)
        r = self.read()  # one reading at the end of the region as well
        if r is not None:
            self.samples.append(r)
        self.lib.nvmlShutdown()


def device_pci_bus_id(dev_index: int):
    try:
        import torch
        p = torch.cuda.get_device_properties(dev_index)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:
        return None


class ClockSampler:
    """SM clocks and clock-event reasons of the GPU while the timed region
    runs: NVML read every millisecond (so that even a timed region of a few
    milliseconds is sampled), else nvidia-smi every 50 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.nvml = None
        self.out = ""

    def __enter__(self):
        try:
            self.nvml = NvmlPoller(device_pci_bus_id(self.index), self.index)
            self.nvml.start()
            return self
        except (OSError, AttributeError):
            self.nvml = None
        try:
            bus = device_pci_bus_id(self.index)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", bus or str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.nvml.stop()
            return
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        if self.nvml is not None:
            return summarize_clocks(self.nvml.samples, self.nvml.max_mhz, "nvml, 1 ms")
        samples, mx = [], None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm = float(parts[0])
                mx = float(parts[1])
            except ValueError:
                continue
            samples.append((sm, [n for n, v in zip(names, parts[3:7]) if v.lower().startswith("active")]))
        return summarize_clocks(samples, mx, "nvidia-smi, 50 ms")


def time_oracle(case, budget_s=12.0, min_reps=1):
    """Time the fp64 oracle on bounded request samples; returns (GB/s, cores, sample text)."""
    import oracle
    import synth
    cores = oracle.max_threads()
    rng = np.random.default_rng(0)
    order = rng.permutation(case.batch)
    stats_full = workload_stats(case, 1)
    per_tok = stats_full["kv_bytes"] / max(stats_full["tokens"], 1)
    done_tokens, elapsed, reps, rows_used = 0, 0.0, 0, 0
    n = 1
    while elapsed < budget_s and rows_used < case.batch:
        rows = order[rows_used:rows_used + n]
        sub = synth.replace(case, q=case.q[rows], block_table=case.block_table[rows],
                            seq_lens=case.seq_lens[rows])
        idx = case.meta.get("indices")
        t0 = time.perf_counter()
        q_len = case.meta.get("q_len", 1)
        if idx is not None:
            oracle.mla_decode_sparse(sub.q, sub.kv, sub.kv_dtype, sub.block_table, sub.seq_lens,
                                     np.ascontiguousarray(idx[rows]), sub.scale, k_scale=sub.k_scale,
                                     kv_lora_rank=sub.kv_lora_rank)
        elif case.kind == "mla" and q_len > 1:
            nb_, rows_, d_ = sub.q.shape
            oracle.mla_decode_multi(sub.q.reshape(nb_, q_len, rows_ // q_len, d_), sub.kv, sub.kv_dtype,
                                    sub.block_table, sub.seq_lens, sub.scale, k_scale=sub.k_scale,
                                    kv_lora_rank=sub.kv_lora_rank)
        elif case.kind == "mla":
            oracle.mla_decode(sub.q, sub.kv, sub.kv_dtype, sub.block_table, sub.seq_lens, sub.scale,
                              k_scale=sub.k_scale, kv_lora_rank=sub.kv_lora_rank)
        else:
            oracle.gqa_paged_decode(sub.q, sub.kv, sub.kv_dtype, sub.block_table, sub.seq_lens,
                                    sub.scale, k_scale=sub.k_scale, v_scale=sub.v_scale)
        dt = time.perf_counter() - t0
        elapsed += dt
        if idx is not None:
            sel = idx[rows]
            done_tokens += int(((sel >= 0) & (sel < sub.seq_lens[:, None])).sum())
        else:
            done_tokens += int(sub.seq_lens.astype(np.int64).sum())
        rows_used += len(rows)
        reps += 1
        n = min(case.batch - rows_used, max(1, len(rows) * 2))
        if n <= 0:
            break
    gbs = done_tokens * per_tok / elapsed / 1e9
    sample = (f"{rows_used} of {case.batch} requests (all heads, {done_tokens} tokens) in {elapsed:.1f} s "
              f"of fp64 oracle work on {cores} host threads")
    return gbs, cores, sample, elapsed, done_tokens


def max_over_ranks(values, dist=None, device="cpu"):
    """Each value's maximum over all ranks (the values themselves without a
    process group): step times are reported as the slowest rank's."""
    import torch
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput_gbs(world, bytes_per_rank, ms):
    """Whole-job throughput in GB/s: every rank decodes its own replica of the
    workload (weak scaling), all within the slowest rank's `ms`."""
    return world * bytes_per_rank / (ms * 1e-3) / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import synth
    case = load_workload(synth, args)
    # The oracle computes the direct definition whatever the split count; the
    # line names the split count the GPU arm uses on this machine (the heuristic
    # with the device's SM count, 152 on a GB300 when no device is visible)
    # so that both arms describe the same workload.
    idx = case.meta.get("indices")
    split_len = idx.shape[1] if idx is not None else int(case.seq_lens.max())
    try:
        import torch
        sms = torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152
    except Exception:
        sms = 152
    splits = args.splits or oracle.num_kv_splits(split_len, sms, False)
    st = workload_stats(case, splits)
    times = []
    tokens = 0
    total_gb = 0.0
    # each step is a bounded sample so that the whole run stays within minutes
    budget = max(0.05, min(args.ref_budget, 150.0 / (args.steps + args.warmup)))
    for i in range(args.warmup + args.steps):
        gbs, cores, sample, elapsed, tok = time_oracle(case, budget_s=budget)
        if i >= args.warmup:
            times.append(elapsed)
            tokens += tok
            total_gb += gbs
    value = total_gb / max(len(times), 1)
    per_tok_ms = 1e3 * sum(times) / max(tokens, 1)
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_tok_ms * st["tokens"], 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(case, args.workload, splits),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample + " per step"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


# Merge of sequence-shard results (decode context parallelism): the shards'
# (output, lse) of the V3-like batch (B=128, H=128, R=512) spread over 8 ranks,
# gathered on one GPU and merged.  Shard outputs ~ N(0,1) in bf16, lse ~
# N(10, 3) with 1/16 of the (shard, row) pairs empty (lse = -inf).
MERGE_WORKLOADS = {"dcp_merge_v3": dict(G=8, B=128, H=128, R=512, seed=1010)}


def merge_inputs(spec):
    rng = np.random.default_rng(spec["seed"])
    G, rows, R = spec["G"], spec["B"] * spec["H"], spec["R"]
    import synth
    outs = synth.to_bf16_bits(rng.standard_normal((G, rows, R), dtype=np.float32))
    lses = (10.0 + 3.0 * rng.standard_normal((G, rows))).astype(np.float32)
    lses[rng.random((G, rows)) < 1.0 / 16] = -np.inf
    return outs, lses


def merge_stats(spec):
    G, rows, R = spec["G"], spec["B"] * spec["H"], spec["R"]
    alg = G * rows * R * 2 + G * rows * 4 + rows * R * 2 + rows * 4
    return dict(alg_bytes=alg, in_bytes=G * rows * R * 2 + G * rows * 4, out_bytes=rows * R * 2 + rows * 4)


def merge_config(name, spec):
    return {"workload": name, "kind": "lse_merge", "num_shards": spec["G"], "batch": spec["B"],
            "num_heads": spec["H"], "head_dim": spec["R"], "seed": spec["seed"],
            "l2": "flushed before every timed step: 256 MiB written then read back (cold, clean L2), "
                  "outside the timed events"}


def run_merge(args):
    """Time mqa_lse_merge (ours) or the oracle's merge (reference) on a
    merge workload; same JSON contract as the decode workloads."""
    spec = MERGE_WORKLOADS[args.workload]
    world, rank, local = dist_env()
    st = merge_stats(spec)
    outs_np, lses_np = merge_inputs(spec)
    G, rows, R = spec["G"], spec["B"] * spec["H"], spec["R"]

    def time_cpu(budget_s):
        import oracle
        n, done, t = 64, 0, 0.0
        while t < budget_s and done < rows:
            sel = slice(done, min(rows, done + n))
            o = oracle.bf16_values(outs_np[:, sel])[:, :, None, :]
            t0 = time.perf_counter()
            oracle.lse_merge(o, lses_np[:, sel, None].astype(np.float64))
            t += time.perf_counter() - t0
            done = sel.stop
            n *= 2
        gbs = st["alg_bytes"] * done / rows / t / 1e9
        return gbs, oracle.max_threads(), f"{done} of {rows} rows (all {G} shards)"

    if args.impl == "reference":
        if rank != 0:
            return
        vals = [time_cpu(args.ref_budget / max(1, args.steps)) for _ in range(max(1, args.steps))]
        gbs = statistics.median(v[0] for v in vals)
        line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
                "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": round(st["alg_bytes"] / gbs / 1e6, 3), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                "config": merge_config(args.workload, spec),
                "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": vals[0][1], "kind": "oracle",
                                 "sample": vals[0][2] + " per step"},
                "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                "gpu_launches": 0}
        print(json.dumps(line), flush=True)
        return

    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())
    from mqa_decode_attention_paged_gb300 import _binding as mqa
    so = torch.from_numpy(outs_np.view(np.int16)).view(torch.bfloat16).to(dev)
    sl = torch.from_numpy(lses_np).to(dev)
    out = torch.empty((rows, R), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((rows,), dtype=torch.float32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush32 = flush.view(torch.int32)
    stream = torch.cuda.current_stream()

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        flush32.max()

    for i in range(args.warmup):
        flush_l2(i)
        mqa.lse_merge(so, sl, out=out, lse=lse, stream=stream)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if world == 1 else local)
    with sampler:
        for i in range(args.steps):
            flush_l2(i)
            starts[i].record(stream)
            mqa.lse_merge(so, sl, out=out, lse=lse, stream=stream)
            ends[i].record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    mean_ms = sum(s_.elapsed_time(e) for s_, e in zip(starts, ends)) / args.steps

    # end to end: the gathered shard results copied in from pinned host
    # memory, the merged output and lse copied back, every step
    so_h = torch.from_numpy(outs_np.view(np.int16)).view(torch.bfloat16).pin_memory()
    sl_h = torch.from_numpy(lses_np).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    so_d, sl_d = torch.empty_like(so), torch.empty_like(sl)
    e2e_steps = max(3, min(args.steps, 100))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps + 2):
        flush_l2(i)
        j = i - 2
        if j >= 0:
            es[j].record(stream)
        so_d.copy_(so_h, non_blocking=True)
        sl_d.copy_(sl_h, non_blocking=True)
        mqa.lse_merge(so_d, sl_d, out=out, lse=lse, stream=stream)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        if j >= 0:
            ee[j].record(stream)
        stream.synchronize()
    e2e_ms = sum(s_.elapsed_time(e) for s_, e in zip(es, ee)) / e2e_steps
    mean_ms, e2e_ms = max_over_ranks([mean_ms, e2e_ms], dist, dev)

    peaks, peak_src = load_peaks()
    gbs = st["alg_bytes"] / (mean_ms * 1e-3) / 1e9
    tr = NCU_TRAFFIC.get(args.workload)
    traffic = tr["bytes"] if tr and tr.get("src_sha") == kernel_sources_sha(tr["files"]) else None
    roof = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
            "traffic_kernel": "shard_merge_kernel" if traffic else None,
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
            "kernel": "shard_merge_kernel (the whole call)", "alg_bytes_per_call": st["alg_bytes"],
            "ideal_us": round(1e6 * st["alg_bytes"] / (peaks["hbm_gbs"] * 1e9), 2)}
    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        v, cores, sample = time_cpu(args.ref_budget)
        cpu = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    line = {
        "metric": METRIC, "value": round(job_throughput_gbs(world, st["alg_bytes"], mean_ms), 2), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_ms, 5),
        "us_per_call": round(mean_ms * 1e3, 2), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (fp32 sums)", "data": "synthetic (seeded N(0,1) shard outputs, N(10,3) lse, 1/16 empty)",
        "config": merge_config(args.workload, spec), "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": round(job_throughput_gbs(world, st["alg_bytes"], e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": st["in_bytes"],
                "d2h_bytes_per_step": st["out_bytes"],
                "note": "per step: the gathered shard outputs and lse host->device, the merged out and lse "
                        "device->host (pinned host buffers)"},
        "gpu_launches": args.steps, "clocks": sampler.summary(), "kernel_src_sha": kernel_sources_sha(),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", torch.cuda.current_device())

    from mqa_decode_attention_paged_gb300 import _binding as mqa
    import synth

    case = load_workload(synth, args)
    if args.split_mode == "fixed" and (case.kind != "mla" or case.meta.get("indices") is not None
                                       or case.meta.get("q_len", 1) > 1):
        raise SystemExit("--split-mode fixed serves the dense single-token MLA workloads")
    st = workload_stats(case, 1)
    sms = mqa.device_sm_count()
    idx_np = case.meta.get("indices")
    # sparse decode splits the topk entries, dense decode the context
    split_len = idx_np.shape[1] if idx_np is not None else int(case.seq_lens.max())
    splits = args.splits or mqa.num_kv_splits(split_len, sms, False)

    # inputs resident in HBM
    q = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).to(dev)
    pth = case.kv_dtype in synth.PTH_DTYPES
    if case.kv_dtype == "bf16":
        kv = torch.from_numpy(case.kv.view(np.int16)).view(torch.bfloat16).to(dev)
    elif pth:
        kv = torch.from_numpy(case.kv).to(dev)  # uint8 rows: codes + inline scale
    else:
        kv = torch.from_numpy(case.kv).view(torch.float8_e4m3fn).to(dev)
    bt = torch.from_numpy(case.block_table).to(dev)
    sl = torch.from_numpy(case.seq_lens).to(dev)
    idx = torch.from_numpy(idx_np).to(dev) if idx_np is not None else None
    B, H, D = q.shape
    R = case.kv_lora_rank if case.kind == "mla" else D
    out = torch.empty((B, H, R), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H), dtype=torch.float32, device=dev)
    if case.kind == "mla":
        need = mqa.mla_decode_workspace_bytes(B, H, R, splits)
    else:
        need = mqa.gqa_paged_decode_workspace_bytes(B, H, D, splits)
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush32 = flush.view(torch.int32)

    def flush_l2(i):
        flush.fill_(i & 0xFF)
        flush32.max()  # read back: the dirty lines leave L2 before the timed call

    stream = torch.cuda.current_stream()
    launches_per_call = 1 if splits == 1 else 2

    q_len = case.meta.get("q_len", 1)

    def call(qq=q, btt=bt, sll=sl, oo=out, ll=lse, ii=idx):
        if ii is not None:
            mqa.mla_decode_sparse(qq, kv, btt, sll, ii, case.scale, case.k_scale, out=oo, lse=ll,
                                  num_kv_splits=splits, workspace=ws, kv_lora_rank=R, stream=stream)
        elif case.kind == "mla" and q_len > 1:  # rows are q_len x heads, token-major
            hh = H // q_len
            mqa.mla_decode_multi(qq.view(B, q_len, hh, D), kv, btt, sll, case.scale, case.k_scale,
                                 out=oo.view(B, q_len, hh, R), lse=ll.view(B, q_len, hh),
                                 num_kv_splits=splits, workspace=ws, kv_lora_rank=R, stream=stream)
        elif case.kind == "mla":
            fn = mqa.mla_decode_fixed_splits if args.split_mode == "fixed" else mqa.mla_decode
            fn(qq, kv, btt, sll, case.scale, case.k_scale, out=oo, lse=ll, num_kv_splits=splits, workspace=ws,
               kv_lora_rank=R, stream=stream)
        else:
            mqa.gqa_paged_decode(qq, kv, btt, sll, case.scale, case.k_scale, case.v_scale, out=oo,
                                 lse=ll, num_kv_splits=splits, workspace=ws, stream=stream,
                                 kv_dtype=case.kv_dtype if pth else None)

    for i in range(args.warmup):
        flush_l2(i)
        call()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index if world == 1 else local)
    with sampler:
        for i in range(args.steps):
            flush_l2(i)
            starts[i].record(stream)
            call()
            ends[i].record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    mean_ms = sum(step_ms) / len(step_ms)

    # ---- end to end: host buffers, copies inside the timed region
    q_h = torch.from_numpy(case.q.view(np.int16)).view(torch.bfloat16).pin_memory()
    bt_h = torch.from_numpy(case.block_table).pin_memory()
    sl_h = torch.from_numpy(case.seq_lens).pin_memory()
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    q_d, bt_d, sl_d = torch.empty_like(q), torch.empty_like(bt), torch.empty_like(sl)
    idx_h = torch.from_numpy(idx_np).pin_memory() if idx_np is not None else None
    idx_d = torch.empty_like(idx) if idx is not None else None
    e2e_steps = max(3, min(args.steps, 200))
    es = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps + 2):
        flush_l2(i)
        j = i - 2
        if j >= 0:
            es[j].record(stream)
        q_d.copy_(q_h, non_blocking=True)
        bt_d.copy_(bt_h, non_blocking=True)
        sl_d.copy_(sl_h, non_blocking=True)
        if idx_d is not None:
            idx_d.copy_(idx_h, non_blocking=True)
        call(q_d, bt_d, sl_d, out, lse, idx_d)
        out_h.copy_(out, non_blocking=True)
        lse_h.copy_(lse, non_blocking=True)
        if j >= 0:
            ee[j].record(stream)
        stream.synchronize()
    e2e_ms = sum(s.elapsed_time(e) for s, e in zip(es, ee)) / e2e_steps
    h2d = q_h.numel() * 2 + bt_h.numel() * 4 + sl_h.numel() * 4 + (idx_h.numel() * 4 if idx_h is not None else 0)
    d2h = out_h.numel() * 2 + lse_h.numel() * 4

    # ---- max over ranks
    mean_ms, e2e_ms = max_over_ranks([mean_ms, e2e_ms], dist, dev)

    peaks, peak_src = load_peaks()
    kv_gbs = job_throughput_gbs(world, st["kv_bytes"], mean_ms)
    alg_gbs = st["alg_bytes"] / (mean_ms * 1e-3) / 1e9
    tflops = st["flops"] / (mean_ms * 1e-3) / 1e12
    t_hbm = st["alg_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = st["flops"] / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    traffic = None
    tr = NCU_TRAFFIC.get(args.workload)
    traffic_kernel = None
    if (tr and tr.get("src_sha") == kernel_sources_sha(tr["files"]) and tr.get("splits") == splits
            and args.split_mode == "balanced" and not getattr(args, "batch", 0)):
        traffic = tr["bytes"]
        traffic_kernel = tr["kernel"] + " (stage 1 only)"
    if bound == "hbm":
        roof = {"bound": "hbm", "achieved": round(alg_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(alg_gbs / peaks["hbm_gbs"], 4)}
    else:
        roof = {"bound": "tensor", "achieved": round(tflops, 2), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(tflops / peaks["bf16_tflops"], 4)}
    roof["traffic"] = traffic
    roof["traffic_kernel"] = traffic_kernel
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback"
    roof["kernel"] = "decode call: split-KV stage-1 kernel + LSE merge"
    roof["alg_bytes_per_call"] = st["alg_bytes"]
    roof["alg_flops_per_call"] = st["flops"]
    roof["ideal_us"] = round(1e6 * max(t_hbm, t_tc), 2)

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        gbs, cores, sample, _, _ = time_oracle(case, budget_s=args.ref_budget)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    line = {
        "metric": METRIC, "value": round(kv_gbs, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_ms, 5),
        "us_per_call": round(mean_ms * 1e3, 2), "tflops": round(tflops, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "fp8_e4m3": "bf16 (fp8-e4m3 KV)",
                  "fp8_e4m3_pth": "bf16 (fp8-e4m3 KV, per-token-head scales)",
                  "int8_pth": "bf16 (int8 KV, per-token-head scales)",
                  "int4_pth": "bf16 (int4 KV, per-token-head scales)"}[case.kv_dtype],
        "data": "synthetic (seeded N(0,1) q/KV, random block permutation)",
        "config": dict(workload_config(case, args.workload, splits), split_mode=args.split_mode),
        "roofline": roof, "cpu_baseline": cpu,
        "e2e": {"value": round(job_throughput_gbs(world, st["kv_bytes"], e2e_ms), 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "note": "per step: q, block_table, seq_lens (and sparse indices) host->device and out, "
                        "lse device->host "
                        "(pinned host buffers); the KV cache is decode state resident in HBM"},
        "gpu_launches": args.steps * launches_per_call,
        "clocks": sampler.summary(),
        "kernel_src_sha": kernel_sources_sha(),
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mla_v3_fp8")
    ap.add_argument("--splits", type=int, default=0, help="num_kv_splits (0 = heuristic)")
    ap.add_argument("--split-mode", default="balanced", choices=["balanced", "fixed"],
                    help="balanced: num_kv_splits is a partial budget over page-balanced units (mla_decode); "
                         "fixed: one unit per request and split, equal page ranges (mla_decode_fixed_splits)")
    ap.add_argument("--batch", type=int, default=0,
                    help="override the workload's batch size (same shape otherwise; 0 = as defined)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget", type=float, default=12.0, help="seconds of oracle work per sample")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.workload in MERGE_WORKLOADS:
        run_merge(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
