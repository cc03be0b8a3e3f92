"""GPU parity: libpa (through its C ABI) against the CPU fp64 oracle, element
by element, on the five decode workloads at full size and on small ragged
cases that cover every supported dtype, head size, block size and GQA group.
"""
import functools

import numpy as np
import pytest
import torch

import paged_decode_attention_v2_gb300 as pa
import workloads
from gpu_helpers import DeviceCase, assert_close, config_case, reference

pytestmark = pytest.mark.gpu

CONFIGS = [("c1_tiny_fp32", None), ("c2_gqa_batch8", None), ("c3_long_100k", None),
           ("c4_batch256", None), ("c5_mixed_d256", 512), ("c5_mixed_d256", 256)]


@functools.lru_cache(maxsize=4)
def device_config(name, P):
    return DeviceCase(config_case(name, P))


@pytest.mark.parametrize("name,P", CONFIGS, ids=[f"{n}-P{p or 'def'}" for n, p in CONFIGS])
@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2, pa.PA_VARIANT_AUTO],
                         ids=["v1", "v2", "auto"])
def test_config_parity(name, P, variant):
    dc = device_config(name, P)
    ref = reference(dc.case)
    out = dc.run(variant=variant)
    assert_close(out, ref, dc.case.dtype, f"{name} P={dc.case.partition_size} v{variant}")


def test_gqa16_full_size_parity():
    """Groups of 16 query heads (the 16-row kernel, two CTAs per SM of three
    stages) at full size: c4_batch256's lengths and cache shape with 32 q / 2
    kv heads, every output against the oracle, V2 and auto."""
    c = dict(workloads.CONFIGS["c4_batch256"])
    c.pop("index")
    c["num_kv_heads"] = 2
    case = workloads.make_case("gqa16", workloads.SEED_BASE + 77, **c)
    ref = reference(case)
    dc = DeviceCase(case)
    for variant in (pa.PA_VARIANT_V2, pa.PA_VARIANT_AUTO):
        assert_close(dc.run(variant=variant), ref, case.dtype, f"G=16 v{variant}")


@pytest.mark.parametrize("name", ["c2_gqa_batch8", "c5_mixed_d256"])
def test_config_parity_simt_math(name):
    """The CUDA-core path on 16-bit inputs (forced) meets the same bar."""
    dc = device_config(name, None if name != "c5_mixed_d256" else 512)
    ref = reference(dc.case)
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        out = dc.run(variant=variant, math=pa.PA_MATH_SIMT)
        assert_close(out, ref, dc.case.dtype, f"{name} simt v{variant}")


# ---- small ragged cases ------------------------------------------------------

def _ragged_lengths(bs, P):
    return [1, 2, bs - 1, bs, bs + 1, 15, 16, 17, 63, 64, 65, P - 1, P, P + 1, 2 * P + 17,
            3 * P - 5]


SMALL = []
for dtype in (torch.float32, torch.bfloat16, torch.float16):
    for D in (64, 128, 256):
        for G, bs in ((1, 8), (4, 16), (8, 32), (16, 64), (2, 16)):
            SMALL.append((dtype, D, G, bs))


@pytest.mark.parametrize("dtype,D,G,bs", SMALL,
                         ids=[f"{str(d)[6:]}-D{D}-G{G}-bs{bs}" for d, D, G, bs in SMALL])
def test_small_ragged(dtype, D, G, bs):
    P = 256
    lens = _ragged_lengths(bs, P)
    Hkv = 2
    case = workloads.make_case("ragged", 1000 + D + 10 * G + bs, len(lens), G * Hkv, Hkv, D,
                               dtype, bs, lens, partition_size=P, extra_blocks=5, k_mult=2.0)
    ref = reference(case)
    dc = DeviceCase(case)
    maths = [pa.PA_MATH_AUTO] if dtype == torch.float32 else [pa.PA_MATH_TENSOR, pa.PA_MATH_SIMT]
    for math in maths:
        for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
            out = dc.run(variant=variant, math=math)
            assert_close(out, ref, dtype, f"math {math} v{variant}")


@pytest.mark.parametrize("fuse", [-1, 0, 1, 4, 16, 64])
@pytest.mark.parametrize("name", ["c2_gqa_batch8", "c5_mixed_d256"])
def test_fused_combine_limits(name, fuse):
    """The cross-partition combine inside Phase 1 for sequences of at most
    min(`fuse`, 16) partitions (0, the default, and -1: never): same result."""
    dc = device_config(name, 512 if name == "c5_mixed_d256" else None)
    for _ in range(2):  # twice: the combine counters must be left at zero
        out = dc.run(variant=pa.PA_VARIANT_V2, fuse_partitions=fuse)
        assert_close(out, reference(dc.case), dc.case.dtype, f"fuse={fuse}")


@pytest.mark.parametrize("P", [64, 128, 512, 1024, 2048, 8192])
def test_partition_sizes(P):
    lens = [1, P - 1, P, P + 1, 5 * P + 3, 1000]
    case = workloads.make_case("psweep", 77 + P, len(lens), 8, 1, 128, torch.bfloat16, 16, lens,
                               partition_size=P, extra_blocks=3)
    ref = reference(case)
    dc = DeviceCase(case)
    out = dc.run(variant=pa.PA_VARIANT_V2)
    assert_close(out, ref, torch.bfloat16, f"P={P}")


@pytest.mark.parametrize("stages", [2, 3, 4, 6])
def test_pipeline_depths(stages):
    case = workloads.make_case("stages", 5, 4, 32, 4, 128, torch.bfloat16, 16,
                               [3000, 517, 4096, 77], partition_size=512)
    ref = reference(case)
    dc = DeviceCase(case)
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        out = dc.run(variant=variant, num_stages=stages)
        assert_close(out, ref, torch.bfloat16, f"stages={stages} v{variant}")


def test_stages_beyond_shared_memory_are_rejected():
    """8 stages of 32 KB exceed the 227 KB a CTA may use: refused on the host."""
    case = workloads.make_case("stages8", 6, 1, 8, 1, 128, torch.bfloat16, 16, [1000],
                               partition_size=512)
    dc = DeviceCase(case)
    with pytest.raises(pa.PAError) as e:
        dc.run(variant=pa.PA_VARIANT_V2, num_stages=8)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


def test_empty_sequences_give_zeros():
    lens = [0, 5, 0, 300]
    case = workloads.make_case("empty", 9, 4, 8, 2, 64, torch.bfloat16, 16, lens,
                               partition_size=128, max_blocks_per_seq=20)
    ref = reference(case)
    dc = DeviceCase(case)
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        out = dc.run(variant=variant)
        assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
        assert_close(out, ref, torch.bfloat16, f"v{variant}")


def test_all_sequences_empty():
    case = workloads.make_case("allempty", 10, 3, 4, 1, 128, torch.float16, 16, [0, 0, 0],
                               partition_size=512, max_blocks_per_seq=4, extra_blocks=2)
    dc = DeviceCase(case)
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        out = dc.run(variant=variant)
        assert torch.all(out == 0)


def test_max_seq_len_above_actual_lengths():
    """max_seq_len is a bound, not the maximum: extra V2 partitions stay idle."""
    case = workloads.make_case("bound", 11, 3, 16, 2, 128, torch.bfloat16, 16, [100, 900, 33],
                               partition_size=256, max_blocks_per_seq=300)
    ref = reference(case)
    dc = DeviceCase(case)
    dc.max_seq_len = 300 * 16
    dc.ws = pa.alloc_workspace(3, 16, 128, dc.max_seq_len, 256)
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        out = dc.run(variant=variant)
        assert_close(out, ref, torch.bfloat16, f"v{variant}")


def test_non_default_stream_and_graph_capture():
    case = workloads.make_case("graph", 12, 4, 32, 4, 128, torch.bfloat16, 16,
                               [2000, 3000, 700, 5000], partition_size=512)
    ref = reference(case)
    dc = DeviceCase(case)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = dc.run(variant=pa.PA_VARIANT_V2, stream=s)
    assert_close(out, ref, torch.bfloat16, "side stream")
    # capture one V2 step (both kernels) in a CUDA graph and replay it
    out = torch.zeros_like(dc.q)
    warm = torch.cuda.Stream()
    with torch.cuda.stream(warm):
        pa.pa_forward(out, dc.q, dc.kc, dc.vc, dc.bt, dc.sl, case.scale, 512, dc.ws,
                      max_seq_len=dc.max_seq_len, variant=pa.PA_VARIANT_V2)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    out.zero_()
    with torch.cuda.graph(g):
        pa.pa_forward(out, dc.q, dc.kc, dc.vc, dc.bt, dc.sl, case.scale, 512, dc.ws,
                      max_seq_len=dc.max_seq_len, variant=pa.PA_VARIANT_V2)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert pa.pa_read_device_status(dc.ws) == pa.PA_OK
    assert_close(out, ref, torch.bfloat16, "graph replay")


def test_sampled_outputs_at_full_size_long_context():
    """The 100K-token workload also checked on sampled (seq, head) pairs computed
    one by one by the oracle (independent of the whole-batch reference)."""
    import oracle
    dc = device_config("c3_long_100k", None)
    out = dc.run(variant=pa.PA_VARIANT_AUTO).double().cpu().numpy()
    pairs = [(0, h) for h in (0, 7, 8, 31)]
    ref = oracle.attention_pairs(pairs, dc.case.query, dc.case.key_cache, dc.case.value_cache,
                                 dc.case.block_tables, dc.case.seq_lens, dc.case.scale)
    for i, (s, h) in enumerate(pairs):
        assert_close(torch.from_numpy(out[s, h]), ref[i], torch.bfloat16, f"pair {(s, h)}")


def test_shared_prefix_blocks():
    """Block tables that share physical blocks, as prefix caching leaves them:
    sequences 1-3 start with sequence 0's first 40 blocks (640 tokens), and
    sequence 3 also repeats one block inside its own table."""
    import dataclasses
    lens = [2000, 1500, 900, 3000]
    base = workloads.make_case("shared", 17, len(lens), 32, 4, 128, torch.bfloat16, 16, lens,
                               partition_size=512, extra_blocks=4)
    bt = base.block_tables.clone()
    for s in (1, 2, 3):
        bt[s, :40] = bt[0, :40]
    bt[3, 100] = bt[3, 50]
    case = dataclasses.replace(base, block_tables=bt)
    ref = reference(case)
    dc = DeviceCase(case)
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        assert_close(dc.run(variant=variant), ref, torch.bfloat16, f"v{variant}")


def test_very_long_sequences_sampled():
    """Two sequences of 300K tokens (586 partitions each) and a short one:
    Phase 2 at its widest; checked on sampled (seq, head) pairs computed one
    by one by the oracle."""
    import oracle
    lens = [300000, 299999, 77]
    case = workloads.make_case("verylong", 23, len(lens), 16, 2, 128, torch.bfloat16, 16, lens,
                               partition_size=512)
    dc = DeviceCase(case)
    pairs = [(0, 0), (0, 15), (1, 3), (1, 8), (2, 9)]
    ref = oracle.attention_pairs(pairs, case.query, case.key_cache, case.value_cache,
                                 case.block_tables, case.seq_lens, case.scale)
    for variant in (pa.PA_VARIANT_V2, pa.PA_VARIANT_V1):
        out = dc.run(variant=variant).double().cpu().numpy()
        for i, (s_, h) in enumerate(pairs):
            assert_close(torch.from_numpy(out[s_, h]), ref[i], torch.bfloat16,
                         f"v{variant} pair {(s_, h)}")
