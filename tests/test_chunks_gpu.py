"""Multi-token queries over the paged cache (pa_chunks_forward) against the
oracle's query_chunks, element by element: chunks of the last n tokens of
each sequence, causal among themselves, over V1 / V2 / auto, every tensor
dtype, head size and a spread of group sizes (which set how many chunk
tokens an item holds: 16 / G on the two-n-tile kernel, 64 / G on the
row-owning one (D 64), 128 / G on the tcgen05 one, which takes chunks of
more than 16 rows per KV head at D 128)."""
import pytest
import torch

import oracle
import paged_decode_attention_v2_gb300 as pa
import workloads
from gpu_helpers import assert_close

pytestmark = pytest.mark.gpu


def _chunk_case(seed, lens, qlens, H, Hkv, D, dtype, bs, P):
    c = workloads.make_case("chunks", seed, len(lens), H, Hkv, D, dtype, bs, lens,
                            partition_size=P, extra_blocks=3, k_mult=2.0)
    g = torch.Generator().manual_seed(seed + 7)
    q = torch.randn(sum(qlens), H, D, generator=g).to(dtype)
    qs = [0]
    for n in qlens:
        qs.append(qs[-1] + n)
    return c, q, torch.tensor(qs, dtype=torch.int32)


CASES = [  # dtype, D, G, Hkv, bs, P, lens, qlens
    (torch.bfloat16, 128, 8, 2, 16, 512, [100, 700, 2000, 40, 300, 5], [1, 2, 5, 17, 0, 3]),
    (torch.bfloat16, 128, 8, 4, 16, 256, [1500, 33], [33, 33]),          # whole-sequence chunk
    (torch.float16, 64, 4, 2, 8, 256, [900, 1700, 64], [7, 16, 9]),
    (torch.bfloat16, 256, 2, 2, 32, 512, [3000, 1200], [12, 8]),
    (torch.float16, 128, 1, 8, 16, 512, [2500, 600, 17], [20, 3, 17]),  # 16 tokens an item
    (torch.bfloat16, 64, 16, 1, 64, 256, [5000, 260], [2, 1]),           # one token an item
    # tcgen05 kernel (> 16 rows per KV head at D 128): f16, pages of 32, 8 and 64 tokens,
    # a chunk that is its whole sequence, ragged row groups
    (torch.float16, 128, 4, 2, 32, 512, [1000, 2100, 70], [40, 64, 70]),
    (torch.bfloat16, 128, 16, 1, 8, 256, [600, 1300], [9, 13]),
    (torch.bfloat16, 128, 2, 4, 64, 512, [3000, 129], [64, 129]),
]


@pytest.mark.parametrize("dtype,D,G,Hkv,bs,P,lens,qlens", CASES,
                         ids=[f"{str(c[0])[6:]}-D{c[1]}-G{c[2]}-bs{c[4]}-P{c[5]}" for c in CASES])
@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2, pa.PA_VARIANT_AUTO],
                         ids=["v1", "v2", "auto"])
def test_chunks_match_oracle(dtype, D, G, Hkv, bs, P, lens, qlens, variant):
    H = G * Hkv
    c, q, qs = _chunk_case(4000 + D + G + P, lens, qlens, H, Hkv, D, dtype, bs, P)
    ref = oracle.query_chunks(q, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, qs,
                              c.scale)
    dev = "cuda"
    R = q.shape[0]
    ws = pa.alloc_workspace(R, H, D, c.max_seq_len, P)
    out = torch.full((R, H, D), float("nan"), dtype=dtype, device=dev)
    args = (q.to(dev), c.key_cache.to(dev), c.value_cache.to(dev), c.block_tables.to(dev),
            c.seq_lens.to(dev), qs.to(dev))
    for _ in range(2):
        pa.pa_chunks_forward(out, *args, c.scale, P, ws, max_seq_len=c.max_seq_len,
                             max_chunk=max(qlens), variant=variant)
        assert pa.pa_read_device_status(ws) == pa.PA_OK
        assert_close(out, ref, dtype, f"chunks v{variant}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16], ids=["bf16", "f16"])
def test_tcgen05_and_mma_sync_kernels_agree_with_the_oracle(dtype):
    """The same chunks (136 and 264 rows per KV head) on the tcgen05 kernel and,
    with PA_DEBUG_NO_TCGEN05, on the row-owning mma.sync kernel: both within
    the bar of the oracle, V1 and V2."""
    H, Hkv, D, P = 16, 2, 128, 256
    c, q, qs = _chunk_case(4242, [700, 1800, 40, 2500], [17, 33, 40, 1], H, Hkv, D, dtype, 16, P)
    ref = oracle.query_chunks(q, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, qs,
                              c.scale)
    dev = "cuda"
    R = q.shape[0]
    ws = pa.alloc_workspace(R, H, D, c.max_seq_len, P)
    args = (q.to(dev), c.key_cache.to(dev), c.value_cache.to(dev), c.block_tables.to(dev),
            c.seq_lens.to(dev), qs.to(dev))
    for flags in (0, pa.PA_DEBUG_NO_TCGEN05):
        for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
            out = torch.full((R, H, D), float("nan"), dtype=dtype, device=dev)
            pa.pa_chunks_forward(out, *args, c.scale, P, ws, max_seq_len=c.max_seq_len,
                                 max_chunk=40, variant=variant, debug_flags=flags)
            assert pa.pa_read_device_status(ws) == pa.PA_OK
            assert_close(out, ref, dtype, f"chunks flags {flags} v{variant}")


def test_single_token_chunks_equal_decode():
    """Chunks of one token are decode: the chunk path and pa_forward agree."""
    lens = [700, 1300, 1, 4097]
    c = workloads.make_case("chunk1", 4100, len(lens), 32, 4, 128, torch.bfloat16, 16, lens,
                            partition_size=512)
    dev = "cuda"
    q, kc, vc = c.query.to(dev), c.key_cache.to(dev), c.value_cache.to(dev)
    bt, sl = c.block_tables.to(dev), c.seq_lens.to(dev)
    qs = torch.arange(len(lens) + 1, dtype=torch.int32, device=dev)
    ws = pa.alloc_workspace(len(lens), 32, 128, c.max_seq_len, 512)
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        a = torch.empty_like(q)
        b = torch.empty_like(q)
        pa.pa_forward(a, q, kc, vc, bt, sl, c.scale, 512, ws, max_seq_len=c.max_seq_len,
                      variant=variant)
        pa.pa_chunks_forward(b, q, kc, vc, bt, sl, qs, c.scale, 512, ws,
                             max_seq_len=c.max_seq_len, max_chunk=1, variant=variant)
        assert pa.pa_read_device_status(ws) == pa.PA_OK
        assert_close(b, a.double().cpu().numpy(), torch.bfloat16, f"v{variant}")


def test_chunk_longer_than_its_sequence_is_reported():
    lens, qlens = [50, 300], [51, 2]
    c, q, qs = _chunk_case(4200, lens, qlens, 8, 1, 64, torch.bfloat16, 16, 256)
    dev = "cuda"
    ws = pa.alloc_workspace(q.shape[0], 8, 64, c.max_seq_len, 256)
    out = torch.zeros(q.shape, dtype=torch.bfloat16, device=dev)
    pa.pa_chunks_forward(out, q.to(dev), c.key_cache.to(dev), c.value_cache.to(dev),
                         c.block_tables.to(dev), c.seq_lens.to(dev), qs.to(dev), c.scale, 256,
                         ws, max_seq_len=c.max_seq_len, max_chunk=51, variant=pa.PA_VARIANT_V2)
    assert pa.pa_read_device_status(ws) == pa.PA_ERR_DEVICE_BAD_INPUT
    # the valid sequence's rows are still right
    ref = oracle.query_chunks(q[51:], c.key_cache, c.value_cache, c.block_tables, c.seq_lens,
                              torch.tensor([0, 0, 2], dtype=torch.int32), c.scale)
    assert_close(out[51:], ref[0:2], torch.bfloat16, "valid rows")


def test_chunks_refuse_f32():
    c, q, qs = _chunk_case(4300, [100], [3], 4, 1, 64, torch.float32, 16, 256)
    ws = pa.alloc_workspace(3, 4, 64, c.max_seq_len, 256)
    out = torch.zeros(q.shape, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_chunks_forward(out, q.cuda(), c.key_cache.cuda(), c.value_cache.cuda(),
                             c.block_tables.cuda(), c.seq_lens.cuda(), qs.cuda(), c.scale, 256,
                             ws, max_seq_len=c.max_seq_len, max_chunk=3)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED


def test_bench_chunk_workload_full_size():
    """The benchmark's query-chunk step at full size: the c4_batch256 cache
    (256 sequences, 32 q / 4 kv heads, D 128, bf16) with a 4-token chunk per
    sequence from the workload generator, every output against the oracle."""
    c = workloads.config_case("c4_batch256")
    q, qs = workloads.chunk_queries(c, 4)
    ref = oracle.query_chunks(q, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, qs,
                              c.scale)
    dev = "cuda"
    R, H, D = q.shape
    ws = pa.alloc_workspace(R, H, D, c.max_seq_len, c.partition_size)
    out = torch.full((R, H, D), float("nan"), dtype=c.dtype, device=dev)
    pa.pa_chunks_forward(out, q.to(dev), c.key_cache.to(dev), c.value_cache.to(dev),
                         c.block_tables.to(dev), c.seq_lens.to(dev), qs.to(dev), c.scale,
                         c.partition_size, ws, max_seq_len=c.max_seq_len, max_chunk=4)
    assert pa.pa_read_device_status(ws) == pa.PA_OK
    assert_close(out, ref, c.dtype, "c4 cache, 4-token chunks")


def test_long_chunk_workload_full_size():
    """Long chunks at full size: the c4_batch256 cache with a 64-token causal
    chunk per sequence (16384 query rows, 512 (token, head) rows per KV head,
    run as 128-row items on the tcgen05 kernel), V2 and V1, every output
    against the oracle; the benchmark's `long_chunks` entry runs this step."""
    c = workloads.config_case("c4_batch256")
    q, qs = workloads.chunk_queries(c, 64)
    ref = oracle.query_chunks(q, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, qs,
                              c.scale)
    dev = "cuda"
    R, H, D = q.shape
    ws = pa.alloc_workspace(R, H, D, c.max_seq_len, c.partition_size)
    args = (q.to(dev), c.key_cache.to(dev), c.value_cache.to(dev), c.block_tables.to(dev),
            c.seq_lens.to(dev), qs.to(dev))
    for variant in (pa.PA_VARIANT_V2, pa.PA_VARIANT_V1):
        outs = []
        for share in (0, 1):  # 1: clusters of 4 CTAs share each K/V stage
            out = torch.full((R, H, D), float("nan"), dtype=c.dtype, device=dev)
            pa.pa_chunks_forward(out, *args, c.scale, c.partition_size, ws,
                                 max_seq_len=c.max_seq_len, max_chunk=64, variant=variant,
                                 share_kv=share)
            assert pa.pa_read_device_status(ws) == pa.PA_OK
            assert_close(out, ref, c.dtype, f"c4 cache, 64-token chunks, v{variant}, share {share}")
            outs.append(out)
        # each CTA does the same arithmetic either way; stages past a row
        # group's own limit add exact zeros
        assert torch.equal(outs[0], outs[1])


TCGEN05_CASES = [c for c in CASES if c[1] == 128 and c[2] * max(c[7]) > 16]


@pytest.mark.parametrize("dtype,D,G,Hkv,bs,P,lens,qlens", TCGEN05_CASES,
                         ids=[f"{str(c[0])[6:]}-G{c[2]}-bs{c[4]}-P{c[5]}" for c in TCGEN05_CASES])
@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2], ids=["v1", "v2"])
def test_shared_kv_clusters_equal_separate_loads(dtype, D, G, Hkv, bs, P, lens, qlens, variant):
    """share_kv (the CTAs of a (sequence, KV head)'s row groups as a cluster
    sharing each K/V stage by multicast, row groups past a short chunk left
    empty) gives the same bits as separate loads, on every tcgen05 case."""
    H = G * Hkv
    c, q, qs = _chunk_case(4000 + D + G + P, lens, qlens, H, Hkv, D, dtype, bs, P)
    R = q.shape[0]
    ws = pa.alloc_workspace(R, H, D, c.max_seq_len, P)
    args = (q.cuda(), c.key_cache.cuda(), c.value_cache.cuda(), c.block_tables.cuda(),
            c.seq_lens.cuda(), qs.cuda())
    outs = []
    for share in (0, 1):
        out = torch.full((R, H, D), float("nan"), dtype=dtype, device="cuda")
        pa.pa_chunks_forward(out, *args, c.scale, P, ws, max_seq_len=c.max_seq_len,
                             max_chunk=max(qlens), variant=variant, share_kv=share)
        assert pa.pa_read_device_status(ws) == pa.PA_OK
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
