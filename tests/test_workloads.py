"""The seeded input generators (CPU): the length distributions of the five
decode workloads, the paged layout they produce (shapes, scattered pool,
unused table entries), determinism, the K scaling of the peaky workload,
the query-chunk generator and the pool permutation used by the invariance
tests.  The large caches (c3-c5, up to ~1 GB) are not materialised: their
length draws are checked with the generator seeded as config_case seeds it."""
import math

import pytest
import torch

import workloads


def _lengths(name):
    c = workloads.CONFIGS[name]
    g = torch.Generator(device="cpu")
    g.manual_seed(workloads.SEED_BASE + c["index"])
    return c["seq_lens"](g)


def test_length_distributions():
    assert _lengths("c1_tiny_fp32") == [1000]
    assert _lengths("c3_long_100k") == [100000]
    c2 = _lengths("c2_gqa_batch8")
    assert len(c2) == 8 and all(1024 <= x <= 8192 for x in c2)
    c4 = _lengths("c4_batch256")
    assert len(c4) == 256 and all(512 <= x <= 3584 for x in c4)
    assert 1700 < sum(c4) / len(c4) < 2400  # U[512, 3584] has mean 2048
    c5 = _lengths("c5_mixed_d256")
    assert len(c5) == 64 and all(16 <= x < 131072 for x in c5)
    # log-uniform: about half the lengths fall below the geometric midpoint
    mid = math.sqrt(16 * 131072)
    below = sum(x < mid for x in c5) / len(c5)
    assert 0.25 < below < 0.75


def test_config_case_matches_its_draws():
    case = workloads.config_case("c1_tiny_fp32")
    assert case.seq_lens.tolist() == _lengths("c1_tiny_fp32")
    assert case.query.shape == (1, 4, 64) and case.dtype == torch.float32
    assert case.key_cache.shape == (64, 1, 16, 64) == case.value_cache.shape
    assert case.scale == 1.0 / 8.0 and case.partition_size == 512
    # 1000 tokens in 63 blocks of a 64-block pool
    row = case.block_tables[0]
    assert int((row >= 0).sum()) == 63 and row.numel() == 63
    assert case.meta["config_index"] == 1


@pytest.mark.parametrize("bs,extra", [(8, 0), (16, 5), (32, 2)])
def test_paged_layout(bs, extra):
    lens = [1, bs - 1, bs, bs + 1, 10 * bs + 3, 0]
    case = workloads.make_case("layout", 3, len(lens), 8, 2, 64, torch.bfloat16, bs, lens,
                               extra_blocks=extra)
    nblk = [(L + bs - 1) // bs for L in lens]
    assert case.num_blocks == sum(nblk) + extra
    assert case.block_tables.shape == (len(lens), max(nblk))
    assert case.block_tables.dtype == torch.int32 and case.seq_lens.dtype == torch.int32
    used = []
    for s, n in enumerate(nblk):
        row = case.block_tables[s]
        assert bool((row[:n] >= 0).all()) and bool((row[n:] == -1).all())
        used += row[:n].tolist()
    # every used block is a distinct slot of the pool
    assert len(set(used)) == len(used) and all(0 <= b < case.num_blocks for b in used)
    # the pool is shuffled, not dealt out in order
    assert used != sorted(used)
    assert case.scale == pytest.approx(1.0 / 8.0)  # 1 / sqrt(64) by default
    assert case.kv_bytes() == sum(lens) * 2 * 64 * 2 * 2


def test_seeded_and_distinct_per_rank():
    a = workloads.config_case("c2_gqa_batch8")
    b = workloads.config_case("c2_gqa_batch8")
    for x, y in ((a.query, b.query), (a.key_cache, b.key_cache), (a.value_cache, b.value_cache),
                 (a.block_tables, b.block_tables), (a.seq_lens, b.seq_lens)):
        assert torch.equal(x, y)
    c = workloads.config_case("c2_gqa_batch8", seed_offset=1)
    assert not torch.equal(a.query, c.query)
    assert a.query.dtype == torch.bfloat16 and a.query.shape == (8, 32, 128)


def test_k_scaling_makes_the_softmax_peaky():
    case = workloads.make_case("peaky", 5, 2, 4, 2, 64, torch.float32, 16, [300, 200],
                               k_mult=4.0)
    assert 3.6 < float(case.key_cache.std()) < 4.4
    assert 0.9 < float(case.value_cache.std()) < 1.1
    assert 0.8 < float(case.query.std()) < 1.2


def test_chunk_queries():
    case = workloads.make_case("chunks", 9, 3, 8, 2, 64, torch.bfloat16, 16, [40, 5, 77])
    q, qs = workloads.chunk_queries(case, 5)
    assert q.shape == (15, 8, 64) and q.dtype == torch.bfloat16
    assert qs.dtype == torch.int32 and qs.tolist() == [0, 5, 10, 15]
    q2, _ = workloads.chunk_queries(case, 5)
    assert torch.equal(q, q2)
    with pytest.raises(ValueError):
        workloads.chunk_queries(case, 6)  # the second sequence holds 5 tokens


def test_permute_pool_keeps_every_sequence_content():
    case = workloads.make_case("perm", 11, 3, 4, 2, 32, torch.float32, 8, [17, 3, 40],
                               extra_blocks=4)
    p = workloads.permute_pool(case, 3)
    assert not torch.equal(case.block_tables, p.block_tables)
    for s, L in enumerate(case.seq_lens.tolist()):
        for t in range(L):
            b0 = int(case.block_tables[s, t // 8])
            b1 = int(p.block_tables[s, t // 8])
            assert torch.equal(case.key_cache[b0, :, t % 8], p.key_cache[b1, :, t % 8])
            assert torch.equal(case.value_cache[b0, :, t % 8], p.value_cache[b1, :, t % 8])
    assert torch.equal(p.block_tables == -1, case.block_tables == -1)


def test_sub_batch_shares_the_cache():
    case = workloads.make_case("sub", 13, 4, 4, 1, 32, torch.float32, 8, [9, 20, 1, 33])
    sub = workloads.sub_batch(case, 2)
    assert sub.num_seqs == 2 and sub.seq_lens.tolist() == [9, 20]
    assert sub.key_cache is case.key_cache and sub.value_cache is case.value_cache
    assert torch.equal(sub.query, case.query[:2])
