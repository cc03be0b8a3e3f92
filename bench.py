#!/usr/bin/env python
"""Paged decode attention benchmark on GB300.

One step = one decode attention call through libpa's public API (the V1/V2
choice, Phase 1 and, for V2, the Phase 2 reduce) over one batch of synthetic
inputs already resident in HBM.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c4_batch256] [--variant auto|v1|v2]
                  [--math auto|tensor|simt] [--stages S]

Metric: KV-read GB/s = (sum_s L_s * Hkv * D * elt * 2) / device time per step,
and decode tokens/s = num_seqs / device time per step.  The L2 is flushed
(a write larger than L2) before every timed step, outside the timed events.

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
import os
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
SECONDARY = "c3_long_100k"


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c4_batch256", choices=sorted(workloads.CONFIGS))
    ap.add_argument("--variant", choices=["auto", "v1", "v2"], default="auto")
    ap.add_argument("--math", choices=["auto", "tensor", "simt"], default="auto")
    ap.add_argument("--stages", type=int, default=0)
    ap.add_argument("--ctas-per-sm", type=int, default=0)
    ap.add_argument("--fuse-partitions", type=int, default=0,
                    help="V2: combine sequences of at most this many partitions inside "
                         "Phase 1 (0: never, the library default)")
    ap.add_argument("--partition-size", type=int, default=0)
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the extra long-context measurement")
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


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_decode_attention_v2_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + f.read())
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


class Runner:
    """A workload resident on the GPU plus the call that runs one step."""

    def __init__(self, case, device, variant, math, stages, ctas_per_sm=0, fuse_partitions=0):
        import paged_decode_attention_v2_gb300 as pa
        self.pa = pa
        self.case = case
        self.device = device
        self.q = case.query.to(device)
        self.kc = case.key_cache.to(device)
        self.vc = case.value_cache.to(device)
        self.bt = case.block_tables.to(device)
        self.sl = case.seq_lens.to(device)
        self.out = torch.empty_like(self.q)
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

    def step(self, q=None, bt=None, sl=None, out=None, phase1_event=None):
        self.pa.pa_forward(out if out is not None else self.out,
                           q if q is not None else self.q, self.kc, self.vc,
                           bt if bt is not None else self.bt,
                           sl if sl is not None else self.sl,
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
    sequence (pa_chunks_forward)."""

    def __init__(self, case, device, tokens):
        import paged_decode_attention_v2_gb300 as pa
        self.pa = pa
        self.case = case
        q, qs = workloads.chunk_queries(case, tokens)
        self.q = q.to(device)
        self.q_start = qs.to(device)
        self.kc = case.key_cache.to(device)
        self.vc = case.value_cache.to(device)
        self.bt = case.block_tables.to(device)
        self.sl = case.seq_lens.to(device)
        self.out = torch.empty_like(self.q)
        self.tokens = tokens
        self.ws = pa.alloc_workspace(self.q.shape[0], case.num_heads, case.head_size,
                                     case.max_seq_len, case.partition_size, device=device)

    def step(self, phase1_event=None, **_):
        self.pa.pa_chunks_forward(self.out, self.q, self.kc, self.vc, self.bt, self.sl,
                                  self.q_start, self.case.scale, self.case.partition_size,
                                  self.ws, max_seq_len=self.case.max_seq_len,
                                  max_chunk=self.tokens)

    def check_status(self):
        st = self.pa.pa_read_device_status(self.ws)
        if st != self.pa.PA_OK:
            raise RuntimeError(f"device status {st}: {self.pa.pa_status_string(st)}")


class L2Flush:
    """Evicts the workload from L2 before a timed step: writes a buffer of
    twice the L2 size, then reads a second one, so that the dirty lines of the
    write are written back here (outside the timed events) and not during
    the timed kernel."""

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


def time_steps(runner, steps, flush, with_phase=False):
    """Per-step device times (ms) with CUDA events on the launching stream;
    the L2 flush runs before each step's start event."""
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    starts, ends = [E() for _ in range(steps)], [E() for _ in range(steps)]
    mids = [E() for _ in range(steps)] if with_phase else None
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
    """The same step through the library's host-buffer C-ABI call
    (pa_forward_host) from pinned HOST buffers: the query, block table and
    lengths are copied in and the output copied out inside the timed region,
    by the call itself."""
    c = runner.case
    pa = runner.pa
    hq = c.query.pin_memory()
    hbt = c.block_tables.pin_memory()
    hsl = c.seq_lens.pin_memory()
    hout = torch.empty(c.query.shape, dtype=c.query.dtype).pin_memory()
    staging = pa.alloc_staging(hq, hbt, device=runner.device)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    starts, ends = [E() for _ in range(steps)], [E() for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record()
        pa.pa_forward_host(hout, hq, runner.kc, runner.vc, hbt, hsl, c.scale,
                           c.partition_size, staging, runner.ws,
                           max_seq_len=runner.max_seq_len, variant=runner.variant,
                           math=runner.math, num_stages=runner.stages,
                           ctas_per_sm=runner.ctas_per_sm,
                           fuse_partitions=runner.fuse_partitions)
        ends[i].record()
    torch.cuda.synchronize()
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    h2d = hq.numel() * hq.element_size() + hbt.numel() * 4 + hsl.numel() * 4
    d2h = hout.numel() * hout.element_size()
    return ms, h2d, d2h


def cpu_oracle_sample(case, target_s=3.0):
    """Time the oracle, as it stands, on the first n sequences of the case,
    n sized for a few seconds of wall time on all host cores."""
    import oracle
    nt = oracle.max_threads()
    n = 1
    while True:
        sub = workloads.sub_batch(case, n)
        t0 = time.perf_counter()
        oracle.attention(sub.query, sub.key_cache, sub.value_cache, sub.block_tables,
                         sub.seq_lens, sub.scale)
        dt = time.perf_counter() - t0
        if dt >= target_s or n >= case.num_seqs:
            break
        n = min(case.num_seqs, max(n + 1, int(n * min(8.0, 1.2 * target_s / max(dt, 1e-3)))))
    return sub, dt, nt


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

    P = args.partition_size or None
    case = workloads.config_case(args.workload, P, seed_offset=rank)
    runner = Runner(case, device, args.variant, args.math, args.stages, args.ctas_per_sm,
                    args.fuse_partitions)
    flush = l2_flush_buffer(device)
    for _ in range(args.warmup):
        runner.step()
    runner.check_status()

    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    step_ms, _ = time_steps(runner, args.steps, flush)
    torch.cuda.synchronize()
    barrier(world)
    # per-kernel breakdown and end-to-end timing, still under load
    brk_steps = min(args.steps, 500)
    brk_ms, phase1_ms = time_steps(runner, brk_steps, flush, with_phase=runner.has_phase2)
    e2e_ms, h2d, d2h = time_e2e(runner, min(args.steps, 500), flush)
    clocks = sampler.stop()
    runner.check_status()

    total_s = sum(step_ms) / 1e3
    total_s_max = reduce_over_ranks(total_s, "max", world, device)
    kv_all = reduce_over_ranks(float(case.kv_bytes()), "sum", world, device)
    seqs_all = reduce_over_ranks(float(case.num_seqs), "sum", world, device)
    e2e_s_max = reduce_over_ranks(sum(e2e_ms) / 1e3, "max", world, device)
    value = kv_all * args.steps / total_s_max / 1e9
    if rank != 0:
        return None

    peak, peak_kind = measured_hbm_peak()
    alg = algorithmic_bytes(case, runner.has_phase2)
    dom_ms = statistics.mean(phase1_ms) if phase1_ms else statistics.mean(brk_ms)
    achieved = alg["kernel"] / (dom_ms / 1e3) / 1e9
    kernel_name = ("pa_attn_kernel(phase1)" if runner.has_phase2 else
                   "pa_attn_kernel(v2, combine fused)" if runner.is_v2 else "pa_attn_kernel(v1)")
    mean_ms = statistics.mean(step_ms)
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
        "dtype": {torch.bfloat16: "bf16", torch.float16: "f16",
                  torch.float32: "f32"}[case.dtype],
        "data": "synthetic (seeded N(0,1) Q/K/V, shuffled paged pool)",
        "config": {
            "workload": args.workload,
            "description": workloads.DESCRIPTIONS[args.workload],
            "num_seqs": case.num_seqs, "num_heads": case.num_heads,
            "num_kv_heads": case.num_kv_heads, "head_size": case.head_size,
            "block_size": case.block_size, "partition_size": case.partition_size,
            "mean_seq_len": round(float(case.seq_lens.double().mean()), 1),
            "kv_bytes_per_step": case.kv_bytes(),
            "variant": "v2" if runner.is_v2 else "v1", "math": args.math,
            "l2": "flushed before every timed step (write then read of 2x L2 each, outside the events)",
            "parallelism": f"dp{world} (independent batches per GPU)",
        },
        "tokens_per_s": round(seqs_all * args.steps / total_s_max, 1),
        "frac_of_nominal_8tbs": round(value / NOMINAL_HBM_GBS / world, 4),
        "step_ms_p10_p50_p90": [round(x, 5) for x in statistics.quantiles(step_ms, n=10)[::4]]
        if len(step_ms) >= 10 else None,
        "roofline": {
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": recorded_traffic(args.workload, kernel_name),
            "kernel": kernel_name, "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "alg_bytes_per_launch": alg["kernel"], "kernel_ms": round(dom_ms, 5),
        },
        "e2e": {"value": round(kv_all * len(e2e_ms) / e2e_s_max / 1e9, 2), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": round(statistics.mean(e2e_ms), 5)},
        "gpu_launches": runner.kernels_per_step * args.steps,
        "clocks": clocks,
    }
    if phase1_ms:
        line["phase_ms"] = {"phase1": round(statistics.mean(phase1_ms), 5),
                            "phase2_incl_gap": round(statistics.mean(brk_ms)
                                                     - statistics.mean(phase1_ms), 5)}
    if world == 1 and not args.no_secondary and args.workload != SECONDARY:
        sec = workloads.config_case(SECONDARY)
        r2 = Runner(sec, device, "auto", "auto", 0)
        for _ in range(max(args.warmup, 3)):
            r2.step()
        # the step as a whole (Phase 2 chained to Phase 1), then a second pass
        # with an event between the phases for the split
        ms2, _ = time_steps(r2, min(args.steps, 500), flush)
        p1 = None
        if r2.has_phase2:
            _, p1 = time_steps(r2, min(args.steps, 200), flush, with_phase=True)
        r2.check_status()
        gbs = sec.kv_bytes() / (statistics.mean(ms2) / 1e3) / 1e9
        line["secondary"] = {SECONDARY: {
            "value": round(gbs, 2), "unit": UNIT, "frac_of_peak": round(gbs / peak, 4),
            "ms_per_step": round(statistics.mean(ms2), 5),
            "variant": "v2" if r2.is_v2 else "v1",
            "phase1_ms": round(statistics.mean(p1), 5) if p1 else None}}
        del r2
    if world == 1 and not args.no_secondary:
        # query chunks (speculative-decoding verification shape): the headline
        # cache with 4-token chunks per sequence
        cr = ChunkRunner(case, device, CHUNK_TOKENS)
        for _ in range(max(args.warmup, 3)):
            cr.step()
        msc, _ = time_steps(cr, min(args.steps, 500), flush)
        cr.check_status()
        mc = statistics.mean(msc)
        line["chunks"] = {
            "workload": f"{args.workload}, {CHUNK_TOKENS}-token query chunks",
            "value": round(case.kv_bytes() / (mc / 1e3) / 1e9, 2), "unit": UNIT,
            "frac_of_peak": round(case.kv_bytes() / (mc / 1e3) / 1e9 / peak, 4),
            "ms_per_step": round(mc, 5),
            "query_rows_per_s": round(cr.q.shape[0] / (mc / 1e3), 1)}
        del cr
    if world == 1 and not args.no_cpu_baseline:
        sub, dt, nt = cpu_oracle_sample(case)
        line["cpu_baseline"] = {
            "value": round(sub.kv_bytes() / dt / 1e9, 4), "unit": UNIT, "cores": nt,
            "kind": "oracle",
            "sample": f"first {sub.num_seqs} of {case.num_seqs} sequences of {args.workload} "
                      f"({sub.kv_bytes()} KV bytes), fp64 C oracle, one run, {dt:.2f} s wall"}
    return line


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    oracle.build()
    P = args.partition_size or None
    case = workloads.config_case(args.workload, P)
    # size the per-step sample so that warmup + steps end within ~2 minutes
    sub, dt, nt = cpu_oracle_sample(case, target_s=0.05)
    budget = 120.0
    per_step = budget / max(1, args.steps + args.warmup)
    n = max(1, min(case.num_seqs, int(sub.num_seqs * per_step / max(dt, 1e-6))))
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
        "config": {"workload": args.workload,
                   "description": workloads.DESCRIPTIONS[args.workload],
                   "sample_seqs": n, "num_seqs": case.num_seqs},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": nt, "kind": "oracle",
                         "sample": f"first {n} of {case.num_seqs} sequences per step"},
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
