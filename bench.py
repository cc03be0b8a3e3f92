#!/usr/bin/env python
"""Paged decode attention benchmark on GB300.

One step = one decode attention call through libpa's public API (the V1/V2
choice, Phase 1 and, for V2, the Phase 2 reduce) over one batch of synthetic
inputs already resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c4_batch256] [--variant auto|v1|v2]
                  [--math auto|tensor|simt] [--stages S]

Metric: KV-read GB/s = (sum_s L_s * Hkv * D * elt * 2) / device time per step,
and decode tokens/s = num_seqs / device time per step.

Timed region (``value``): K consecutive steps, as a decode pass runs them,
one per layer: the steps cycle through ``layers`` copies of the workload
(each its own K/V cache, queries and output; the block tables and lengths
are shared, as across the layers of a model), enough copies that the cycle
reads at least 4x the L2 size, so every step finds its K/V cold in L2 without
a flush between steps.  Workloads too small for that (the tiny fp32 case)
are timed step by step with an L2 flush before each step instead.
``isolated`` reports the single-step latency too: the L2 flushed (a write
and a read of 2x L2, outside the events) before every step, CUDA events
around each step.

Under torchrun (N > 1) every rank runs its own batch of the same shape on its
own GPU (weak scaling; sequences are independent, there is no collective on
the data path); the step time is the max over ranks and `value` counts the
bytes of all ranks.

`--impl reference` times the CPU fp64 oracle (the only other implementation:
the method's pages publish no runnable kernel) on a bounded sample of the same
workload, on the host cores, rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "paged decode attention KV-read GB/s (% of GB300 HBM peak) and decode tokens/s"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
CHUNK_TOKENS = 4
LONG_CHUNK_TOKENS = 64
MAX_LAYERS = 64
# the other workloads reported beside the headline, each timed like it
SECONDARY = [("c3_long_100k", None), ("c2_gqa_batch8", None), ("c5_mixed_d256", 512),
             ("c5_mixed_d256", 256), ("c1_tiny_fp32", None), ("gqa16_c4", None)]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c4_batch256",
                    choices=sorted(workloads.CONFIGS) + ["gqa16_c4"])
    ap.add_argument("--variant", choices=["auto", "v1", "v2"], default="auto")
    ap.add_argument("--math", choices=["auto", "tensor", "simt"], default="auto")
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--ctas-per-sm", type=int, default=0)
    ap.add_argument("--fuse-partitions", type=int, default=0,
                    help="V2: combine sequences of at most this many partitions inside "
                         "Phase 1 (0: never, the library default)")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the other workloads, the query chunks and the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# ranks

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_over_ranks(value: float, op: str, world: int, device=None) -> float:
    """max or sum of a scalar over all ranks (host-side bookkeeping only)."""
    if world <= 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region

CLOCK_FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index: int):
        self.proc = None
        self.uuid = None
        try:
            u = str(torch.cuda.get_device_properties(device_index).uuid)
            self.uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        if self.uuid:
            mine = [r for r in rows if r[0].strip() == self.uuid]
            rows = mine or rows
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.strip() == "Active":
                    reasons.add(name)
        loaded = [x for x in sm if x > 0.5 * (max(mx) if mx else 0)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ---------------------------------------------------------------------------

def measured_hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C++ source without its comments and with whitespace collapsed: what the
    compiler sees, up to formatting."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_digest(csrc: str = None) -> str:
    """Digest of the kernel sources' code (comments and formatting ignored), so
    that a traffic record stays attached to the code it was measured on."""
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "paged_decode_attention_v2_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                h.update(name.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, kernel: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("kernel_source_digest") != kernel_source_digest() or rec.get("kernel") != kernel:
        return None
    return rec.get("dram_bytes_per_launch")


def bench_case(name: str, partition_size=None, seed_offset: int = 0):
    """A named workload: the five configurations, plus ``gqa16_c4`` (the
    256-sequence lengths and cache shape with 32 query / 2 KV heads, groups
    of 16 query heads per KV head)."""
    if name == "gqa16_c4":
        c = dict(workloads.CONFIGS["c4_batch256"])
        c.pop("index")
        c["num_kv_heads"] = 2
        if partition_size:
            c["partition_size"] = partition_size
        return workloads.make_case("gqa16_c4", workloads.SEED_BASE + 77 + 1000 * seed_offset, **c)
    return workloads.config_case(name, partition_size, seed_offset=seed_offset)


def describe(name: str) -> str:
    if name == "gqa16_c4":
        return "256 seqs, L~U[512,3584], 32 q / 2 kv heads (G=16), D128, bf16, bs16"
    return workloads.DESCRIPTIONS[name]


def algorithmic_bytes(case, phase2_separate: bool) -> dict:
    """Bytes the dominant kernel must move: K and V of every token, the
    queries, the block-table entries it dereferences and seq_lens, and the
    output unless a separate Phase 2 kernel writes it (workspace partials are
    implementation overhead and not counted)."""
    elt = case.query.element_size()
    kv = case.kv_bytes()
    q = case.query.numel() * elt
    pages = int(((case.seq_lens.to(torch.int64) + case.block_size - 1)
                 // case.block_size).sum().item())
    table = pages * 4 + case.num_seqs * 4
    out = 0 if phase2_separate else q
    return {"kv": kv, "kernel": kv + q + table + out}


def layers_for(kv_bytes: int, l2_bytes: int) -> int:
    """Layer copies to cycle through so that one cycle reads >= 4x L2 of K/V;
    0 when that would take more than MAX_LAYERS copies (timed with a flush)."""
    n = max(2, math.ceil(4 * l2_bytes / max(kv_bytes, 1)))
    return n if n <= MAX_LAYERS else 0


def workload_config(name: str, case, world: int, l2_note: str) -> dict:
    """The `config` object: what the workload is, identical in both arms."""
    return {
        "workload": name, "description": describe(name),
        "num_seqs": case.num_seqs, "num_heads": case.num_heads,
        "num_kv_heads": case.num_kv_heads, "head_size": case.head_size,
        "block_size": case.block_size, "partition_size": case.partition_size,
        "dtype": dtype_name(case.dtype),
        "mean_seq_len": round(float(case.seq_lens.double().mean()), 1),
        "kv_bytes_per_step": case.kv_bytes(),
        "l2": l2_note,
        "parallelism": f"dp{world} (independent batches per GPU)",
    }


def l2_note_for(kv_bytes: int, l2_bytes: int) -> str:
    n = layers_for(kv_bytes, l2_bytes)
    if n:
        return (f"inputs larger than L2: consecutive steps cycle through {n} layers' K/V caches "
                f"({n * kv_bytes / 1e9:.2f} GB a cycle, L2 {l2_bytes / 1e6:.0f} MB); no flush "
                "between steps")
    return "flushed before every timed step (write then read of 2x L2 each, outside the events)"


def dtype_name(dt) -> str:
    return {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}[dt]


class Runner:
    """A workload resident on the GPU, in `layers` copies (each its own K/V
    cache, queries and output), plus the call that runs one step."""

    def __init__(self, case, device, variant="auto", math="auto", stages=0, ctas_per_sm=0,
                 fuse_partitions=0, layers=1):
        import paged_decode_attention_v2_gb300 as pa
        self.pa = pa
        self.case = case
        self.device = device
        q = case.query.to(device)
        kc = case.key_cache.to(device)
        vc = case.value_cache.to(device)
        self.bt = case.block_tables.to(device)
        self.sl = case.seq_lens.to(device)
        self.layer = [(q, kc, vc, torch.empty_like(q))]
        for _ in range(1, max(1, layers)):
            self.layer.append((q.clone(), kc.clone(), vc.clone(), torch.empty_like(q)))
        self.q, self.kc, self.vc, self.out = self.layer[0]
        self.max_seq_len = case.max_seq_len
        self.variant = {"auto": pa.PA_VARIANT_AUTO, "v1": pa.PA_VARIANT_V1,
                        "v2": pa.PA_VARIANT_V2}[variant]
        self.math = {"auto": pa.PA_MATH_AUTO, "tensor": pa.PA_MATH_TENSOR,
                     "simt": pa.PA_MATH_SIMT}[math]
        self.stages = stages
        self.ctas_per_sm = ctas_per_sm
        self.fuse_partitions = fuse_partitions
        self.ws = pa.alloc_workspace(case.num_seqs, case.num_heads, case.head_size,
                                     self.max_seq_len, case.partition_size, device=device)
        sm = torch.cuda.get_device_properties(device).multi_processor_count
        if self.variant == pa.PA_VARIANT_AUTO:
            self.is_v2 = bool(pa.pa_choose_v2(case.num_seqs, case.num_kv_heads,
                                              self.max_seq_len, case.partition_size, sm))
        else:
            self.is_v2 = self.variant == pa.PA_VARIANT_V2
        # With fusion asked for, V2 sequences of at most min(n, 16) partitions
        # get their combine inside the Phase 1 kernel, and a Phase 2 kernel
        # runs only if longer ones can occur.
        fuse = min(fuse_partitions, 16) if fuse_partitions > 0 else 0
        self.has_phase2 = self.is_v2 and -(-self.max_seq_len // case.partition_size) > fuse
        self.kernels_per_step = 2 if self.has_phase2 else 1

    @property
    def layers(self) -> int:
        return len(self.layer)

    def step(self, layer=0, phase1_event=None):
        q, kc, vc, out = self.layer[layer % len(self.layer)]
        self.pa.pa_forward(out, q, kc, vc, self.bt, self.sl,
                           self.case.scale, self.case.partition_size, self.ws,
                           max_seq_len=self.max_seq_len, variant=self.variant, math=self.math,
                           num_stages=self.stages, phase1_event=phase1_event,
                           ctas_per_sm=self.ctas_per_sm, fuse_partitions=self.fuse_partitions)

    def check_status(self):
        st = self.pa.pa_read_device_status(self.ws)
        if st != self.pa.PA_OK:
            raise RuntimeError(f"device status {st}: {self.pa.pa_status_string(st)}")


class ChunkRunner:
    """The same cache as a Runner, queried with chunks of `tokens` tokens per
    sequence (pa_chunks_forward), in `layers` copies."""

    def __init__(self, case, device, tokens, layers=1, share_kv=0):
        import paged_decode_attention_v2_gb300 as pa
        self.pa = pa
        self.case = case
        self.share_kv = share_kv
        q, qs = workloads.chunk_queries(case, tokens)
        q = q.to(device)
        self.q_start = qs.to(device)
        kc = case.key_cache.to(device)
        vc = case.value_cache.to(device)
        self.bt = case.block_tables.to(device)
        self.sl = case.seq_lens.to(device)
        self.layer = [(q, kc, vc, torch.empty_like(q))]
        for _ in range(1, max(1, layers)):
            self.layer.append((q.clone(), kc.clone(), vc.clone(), torch.empty_like(q)))
        self.q = q
        self.tokens = tokens
        sm = torch.cuda.get_device_properties(device).multi_processor_count
        self.is_v2 = bool(pa.pa_choose_v2_chunks(case.num_seqs, case.num_heads,
                                                 case.num_kv_heads, case.head_size, tokens,
                                                 case.max_seq_len, case.partition_size, sm))
        self.has_phase2 = self.is_v2
        self.kernels_per_step = 2 if self.is_v2 else 1
        self.ws = pa.alloc_workspace(q.shape[0], case.num_heads, case.head_size,
                                     case.max_seq_len, case.partition_size, device=device)

    @property
    def layers(self) -> int:
        return len(self.layer)

    def step(self, layer=0, phase1_event=None):
        q, kc, vc, out = self.layer[layer % len(self.layer)]
        self.pa.pa_chunks_forward(out, q, kc, vc, self.bt, self.sl,
                                  self.q_start, self.case.scale, self.case.partition_size,
                                  self.ws, max_seq_len=self.case.max_seq_len,
                                  max_chunk=self.tokens, phase1_event=phase1_event,
                                  share_kv=self.share_kv)

    def check_status(self):
        st = self.pa.pa_read_device_status(self.ws)
        if st != self.pa.PA_OK:
            raise RuntimeError(f"device status {st}: {self.pa.pa_status_string(st)}")


class L2Flush:
    """Evicts the workload from L2: writes a buffer of twice the L2 size, then
    reads a second one, so that the dirty lines of the write are written back
    here and not during the timed kernel."""

    def __init__(self, device):
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        self.r = torch.zeros(n, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)

    def zero_(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def l2_flush_buffer(device):
    return L2Flush(device)


def _event():
    return torch.cuda.Event(enable_timing=True)


def time_consecutive(runner, steps, flush):
    """K consecutive steps (cycling through the runner's layers) between one
    pair of CUDA events on the launching stream; the L2 is flushed once
    before the first.  Returns total ms."""
    flush.zero_()
    start, end = _event(), _event()
    start.record()
    for i in range(steps):
        runner.step(layer=i)
    end.record()
    torch.cuda.synchronize()
    return start.elapsed_time(end)


def time_steps(runner, steps, flush, with_phase=False):
    """Per-step device times (ms) with CUDA events on the launching stream;
    the L2 flush runs before each step's start event."""
    starts, ends = [_event() for _ in range(steps)], [_event() for _ in range(steps)]
    mids = [_event() for _ in range(steps)] if with_phase else None
    if mids:
        # torch creates the CUDA event at its first record(); do that here so
        # the handle handed to the library is live
        for m in mids:
            m.record()
        torch.cuda.synchronize()
    for i in range(steps):
        flush.zero_()
        starts[i].record()
        runner.step(phase1_event=mids[i] if mids else None)
        ends[i].record()
    torch.cuda.synchronize()
    total = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    phase1 = [s.elapsed_time(m) for s, m in zip(starts, mids)] if mids else None
    return total, phase1


def time_e2e(runner, steps, flush):
    """The same steps through the library's host-buffer C-ABI call
    (pa_forward_host) from pinned HOST buffers: the query, block table and
    lengths are copied in and the output copied out by the call itself,
    every step, inside the timed region.  Steps cycle through the runner's
    layers like the device-resident steps."""
    c = runner.case
    pa = runner.pa
    hq = c.query.pin_memory()
    hbt = c.block_tables.pin_memory()
    hsl = c.seq_lens.pin_memory()
    hout = torch.empty(c.query.shape, dtype=c.query.dtype).pin_memory()
    staging = pa.alloc_staging(hq, hbt, device=runner.device)

    def call(i):
        _, kc, vc, _ = runner.layer[i % runner.layers]
        pa.pa_forward_host(hout, hq, kc, vc, hbt, hsl, c.scale, c.partition_size, staging,
                           runner.ws, max_seq_len=runner.max_seq_len, variant=runner.variant,
                           math=runner.math, num_stages=runner.stages,
                           ctas_per_sm=runner.ctas_per_sm,
                           fuse_partitions=runner.fuse_partitions)
    for i in range(3):
        call(i)
    torch.cuda.synchronize()
    h2d = hq.numel() * hq.element_size() + hbt.numel() * 4 + hsl.numel() * 4
    d2h = hout.numel() * hout.element_size()
    if runner.layers > 1:
        flush.zero_()
        start, end = _event(), _event()
        start.record()
        for i in range(steps):
            call(i)
        end.record()
        torch.cuda.synchronize()
        return start.elapsed_time(end) / steps, h2d, d2h
    ms = []
    for i in range(steps):
        flush.zero_()
        start, end = _event(), _event()
        start.record()
        call(i)
        end.record()
        torch.cuda.synchronize()
        ms.append(start.elapsed_time(end))
    return statistics.mean(ms), h2d, d2h


def measure(name, case, runner, flush, peak, steps, iso_steps):
    """One workload as a `secondary` entry: consecutive steps (or flushed
    steps when it is too small to cycle through L2), the isolated flushed
    step, and the Phase 1 kernel's share of it."""
    for _ in range(5):
        runner.step()
    if runner.layers > 1:
        ms = time_consecutive(runner, steps, flush) / steps
    else:
        ms = None
    iso, _ = time_steps(runner, iso_steps, flush)
    p1 = None
    if runner.has_phase2:
        _, p1 = time_steps(runner, max(iso_steps // 2, 20), flush, with_phase=True)
    runner.check_status()
    iso_ms = statistics.median(iso)
    step_ms = ms if ms is not None else iso_ms
    kv = case.kv_bytes()
    gbs = kv / (step_ms / 1e3) / 1e9
    alg = algorithmic_bytes(case, runner.has_phase2)
    entry = {
        "value": round(gbs, 2), "unit": UNIT, "frac_of_peak": round(gbs / peak, 4),
        "ms_per_step": round(step_ms, 5),
        "tokens_per_s": round(case.num_seqs / (step_ms / 1e3), 1),
        "timing": (f"{steps} consecutive steps over {runner.layers} layers' caches"
                   if ms is not None else "flushed steps (too small to cycle through L2)"),
        "isolated": {"ms_per_step": round(iso_ms, 5),
                     "value": round(kv / (iso_ms / 1e3) / 1e9, 2),
                     "frac_of_peak": round(kv / (iso_ms / 1e3) / 1e9 / peak, 4)},
        "variant": "v2" if runner.is_v2 else "v1",
        "kv_bytes_per_step": kv,
        "description": describe(name),
    }
    if p1:
        p1m = statistics.median(p1)
        entry["phase1_ms"] = round(p1m, 5)
        entry["phase1_frac_of_peak"] = round(alg["kernel"] / (p1m / 1e3) / 1e9 / peak, 4)
    return entry


# ---------------------------------------------------------------------------
# CPU baseline (the oracle, as it stands)

def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def cpu_oracle_sample(case, target_s=3.0, nthreads=0):
    """The first n sequences of the case, n sized for about target_s of
    oracle wall time on nthreads host threads (0: all)."""
    import oracle
    n = 1
    while True:
        sub = workloads.sub_batch(case, n)
        t0 = time.perf_counter()
        oracle.attention(sub.query, sub.key_cache, sub.value_cache, sub.block_tables,
                         sub.seq_lens, sub.scale, nthreads=nthreads)
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= case.num_seqs:
            break
        n = min(case.num_seqs, max(n + 1, int(n * min(8.0, 1.2 * target_s / max(dt, 1e-3)))))
    return sub


def time_oracle(sub, runs=3, nthreads=0):
    """Median wall time (steady clock) of `runs` oracle calls on sub."""
    import oracle
    ts = []
    for _ in range(runs):
        t0 = time.perf_counter()
        oracle.attention(sub.query, sub.key_cache, sub.value_cache, sub.block_tables,
                         sub.seq_lens, sub.scale, nthreads=nthreads)
        ts.append(time.perf_counter() - t0)
    return statistics.median(ts)


def cpu_baseline(name, case, target_s=3.0):
    """The oracle on all host cores, median of 3, on a bounded sample of the
    headline workload, plus one thread on the three small configurations."""
    import oracle
    oracle.build()
    nt = oracle.max_threads()
    sub = cpu_oracle_sample(case, target_s)
    dt = time_oracle(sub, 3)
    single = {}
    for cname in ("c1_tiny_fp32", "c2_gqa_batch8", "c3_long_100k"):
        c = case if cname == name else workloads.config_case(cname)
        s1 = cpu_oracle_sample(c, 1.0, nthreads=1)
        d1 = time_oracle(s1, 3, nthreads=1)
        single[cname] = {"value": round(s1.kv_bytes() / d1 / 1e9, 4), "unit": UNIT,
                         "tokens_per_s": round(s1.num_seqs / d1, 2),
                         "sample": f"first {s1.num_seqs} of {c.num_seqs} sequences, "
                                   f"median of 3 runs of {d1:.3f} s"}
    return {
        "value": round(sub.kv_bytes() / dt / 1e9, 4), "unit": UNIT, "cores": nt, "kind": "oracle",
        "sample": f"first {sub.num_seqs} of {case.num_seqs} sequences of {name} "
                  f"({sub.kv_bytes()} KV bytes), fp64 C oracle, median of 3 runs of {dt:.3f} s",
        "tokens_per_s": round(sub.num_seqs / dt, 2),
        "cpu_model": cpu_model(), "nproc": os.cpu_count(),
        "single_thread": single,
    }


# ---------------------------------------------------------------------------

def run_ours(args):
    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    from paged_decode_attention_v2_gb300 import build_lib
    if rank == 0 or world == 1:
        build_lib.build()
    barrier(world)

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    P = args.partition_size or None
    case = bench_case(args.workload, P, seed_offset=rank)
    runner = Runner(case, device, args.variant, args.math, args.stages, args.ctas_per_sm,
                    args.fuse_partitions, layers=max(1, layers_for(case.kv_bytes(), l2)))
    flush = l2_flush_buffer(device)
    for i in range(args.warmup):
        runner.step(layer=i)
    runner.check_status()

    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    # ---- the timed region: K consecutive steps (or K flushed steps)
    if runner.layers > 1:
        flush.zero_()
        torch.cuda.synchronize()
        barrier(world)
        start, end = _event(), _event()
        start.record()
        for i in range(args.steps):
            runner.step(layer=i)
        end.record()
        torch.cuda.synchronize()
        barrier(world)
        total_ms = start.elapsed_time(end)
        step_ms = [total_ms / args.steps] * args.steps
    else:
        step_ms, _ = time_steps(runner, args.steps, flush)
        total_ms = sum(step_ms)
        torch.cuda.synchronize()
        barrier(world)
    # per-kernel breakdown, isolated steps and end-to-end timing, still under load
    brk_steps = min(max(args.steps, 50), 500)
    iso_ms, phase1_ms = time_steps(runner, brk_steps, flush, with_phase=runner.has_phase2)
    e2e_ms, h2d, d2h = time_e2e(runner, min(max(args.steps, 50), 500), flush)
    clocks = sampler.stop()
    runner.check_status()

    total_s_max = reduce_over_ranks(total_ms / 1e3, "max", world, device)
    kv_all = reduce_over_ranks(float(case.kv_bytes()), "sum", world, device)
    seqs_all = reduce_over_ranks(float(case.num_seqs), "sum", world, device)
    e2e_s_max = reduce_over_ranks(e2e_ms / 1e3, "max", world, device)
    value = kv_all * args.steps / total_s_max / 1e9
    if rank != 0:
        return None

    peak, peak_kind = measured_hbm_peak()
    alg = algorithmic_bytes(case, runner.has_phase2)
    dom_ms = statistics.mean(phase1_ms) if phase1_ms else statistics.mean(iso_ms)
    achieved = alg["kernel"] / (dom_ms / 1e3) / 1e9
    kernel_name = ("pa_attn_kernel(phase1)" if runner.has_phase2 else
                   "pa_attn_kernel(v2, combine fused)" if runner.is_v2 else "pa_attn_kernel(v1)")
    iso_med = statistics.median(iso_ms)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_s_max * 1e3 / args.steps, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": dtype_name(case.dtype),
        "data": "synthetic (seeded N(0,1) Q/K/V, shuffled paged pool)",
        "config": workload_config(args.workload, case, world, l2_note_for(case.kv_bytes(), l2)),
        "implementation": {"variant": "v2" if runner.is_v2 else "v1", "math": args.math,
                           "layers": runner.layers},
        "tokens_per_s": round(seqs_all * args.steps / total_s_max, 1),
        "frac_of_peak": round(value / peak / world, 4),
        "frac_of_nominal_8tbs": round(value / NOMINAL_HBM_GBS / world, 4),
        "isolated": {"ms_per_step": round(iso_med, 5),
                     "value": round(case.kv_bytes() / (iso_med / 1e3) / 1e9, 2),
                     "frac_of_peak": round(case.kv_bytes() / (iso_med / 1e3) / 1e9 / peak, 4),
                     "step_ms_p10_p50_p90": [round(x, 5) for x in
                                             statistics.quantiles(iso_ms, n=10)[::4]],
                     "how": "L2 flushed before every step, CUDA events around each step "
                            "(includes the launch latency of an isolated call)"},
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(args.workload, kernel_name),
            "kernel": kernel_name, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "alg_bytes_per_launch": alg["kernel"], "kernel_ms": round(dom_ms, 5),
            "kernel_ms_how": "isolated flushed steps: CUDA event before the step to the event "
                             "the library records between Phase 1 and Phase 2",
        },
        "e2e": {"value": round(kv_all / e2e_s_max / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": runner.kernels_per_step * args.steps,
        "clocks": clocks,
    }
    if phase1_ms:
        line["phase_ms"] = {"phase1": round(statistics.mean(phase1_ms), 5),
                            "phase2_incl_gap": round(statistics.mean(iso_ms)
                                                     - statistics.mean(phase1_ms), 5)}
    del runner
    torch.cuda.empty_cache()
    if world == 1 and not args.no_secondary:
        sec = {}
        for name, Ps in SECONDARY:
            if name == args.workload and (Ps or None) == P:
                continue
            c2 = bench_case(name, Ps)
            r2 = Runner(c2, device, layers=max(1, layers_for(c2.kv_bytes(), l2)))
            key = name if Ps is None else f"{name}_P{Ps}"
            sec[key] = measure(name, c2, r2, flush, peak, 200, 200)
            del r2
            torch.cuda.empty_cache()
        line["secondary"] = sec
        # query chunks (speculative-decoding verification shape): the headline
        # cache with 4-token chunks per sequence
        cr = ChunkRunner(case, device, CHUNK_TOKENS,
                         layers=max(1, layers_for(case.kv_bytes(), l2)))
        ce = measure(args.workload, case, cr, flush, peak, 200, 200)
        ce["workload"] = f"{args.workload}, {CHUNK_TOKENS}-token query chunks"
        ce["query_rows_per_s"] = round(cr.q.shape[0] / (ce["ms_per_step"] / 1e3), 1)
        ce.pop("tokens_per_s", None)
        line["chunks"] = ce
        del cr
        torch.cuda.empty_cache()
        # long chunks (a prefill chunk whose keys and values are already cached):
        # 64 tokens per sequence, 512 (token, head) rows per KV head
        cr = ChunkRunner(case, device, LONG_CHUNK_TOKENS,
                         layers=max(1, layers_for(case.kv_bytes(), l2)))
        ce = measure(args.workload, case, cr, flush, peak, 20, 20)
        ce["workload"] = f"{args.workload}, {LONG_CHUNK_TOKENS}-token query chunks"
        ce["query_rows_per_s"] = round(cr.q.shape[0] / (ce["ms_per_step"] / 1e3), 1)
        ce.pop("tokens_per_s", None)
        rows = cr.q.shape[0] * case.num_heads
        vis = float(case.seq_lens.double().sum()) - case.num_seqs * (LONG_CHUNK_TOKENS - 1) / 2
        flops = 4.0 * case.num_heads * LONG_CHUNK_TOKENS * vis * case.head_size
        ce["attention_tflops"] = round(flops / (ce["ms_per_step"] / 1e3) / 1e12, 1)
        ce["rows"] = rows
        # the same step with the row groups of each (sequence, KV head) in a
        # thread-block cluster sharing every K/V stage (share_kv): K/V cross
        # HBM once instead of once per row group
        cr.share_kv = 1
        se = measure(args.workload, case, cr, flush, peak, 20, 20)
        ce["shared_kv"] = {"ms_per_step": se["ms_per_step"],
                           "attention_tflops": round(flops / (se["ms_per_step"] / 1e3) / 1e12, 1),
                           "isolated_ms_per_step": se["isolated"]["ms_per_step"]}
        line["long_chunks"] = ce
        del cr
        torch.cuda.empty_cache()
    if world == 1 and not args.no_cpu_baseline and not args.no_secondary:
        line["cpu_baseline"] = cpu_baseline(args.workload, case)
    return line


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    P = args.partition_size or None
    case = bench_case(args.workload, P)
    l2 = 0
    try:
        if torch.cuda.is_available():
            l2 = torch.cuda.get_device_properties(0).L2_cache_size
    except Exception:
        l2 = 0
    l2 = l2 or 126 * 1024 * 1024
    nt = oracle.max_threads()
    # size the per-step sample so that warmup + steps end within ~2 minutes
    probe = cpu_oracle_sample(case, target_s=0.05)
    dt = time_oracle(probe, 1)
    budget = 120.0
    per_step = budget / max(1, args.steps + args.warmup)
    n = max(1, min(case.num_seqs, int(probe.num_seqs * per_step / max(dt, 1e-6))))
    sample = workloads.sub_batch(case, n)
    run = lambda: oracle.attention(sample.query, sample.key_cache, sample.value_cache,  # noqa
                                   sample.block_tables, sample.seq_lens, sample.scale)
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        run()
        times.append(time.perf_counter() - t0)
    mean_s = statistics.mean(times)
    value = sample.kv_bytes() / mean_s / 1e9
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(mean_s * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded N(0,1) Q/K/V, shuffled paged pool)",
        "config": workload_config(args.workload, case, world, l2_note_for(case.kv_bytes(), l2)),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": nt, "kind": "oracle",
                         "sample": f"first {n} of {case.num_seqs} sequences per step",
                         "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)
    _, world, _ = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
