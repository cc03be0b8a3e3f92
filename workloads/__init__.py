"""Seeded synthetic decode workloads, shared by the tests, the benchmark and
the oracle checks.

This module only draws random inputs and lays them out in the paged-cache
format; it holds none of the attention arithmetic.  Inputs are drawn on the
CPU with one ``torch.Generator`` per case, in a fixed order: sequence lengths,
then the permutation of the physical block pool, then Q, K and V.  Q/K/V are
drawn as float32 N(0, 1) and rounded once to the case's dtype (K is scaled
first when ``k_mult`` != 1, to make the softmax peaky).

Layouts (row-major, contiguous):
  query            [num_seqs, num_heads, head_size]
  key/value_cache  [num_blocks, num_kv_heads, block_size, head_size]
  block_tables     int32 [num_seqs, max_blocks_per_seq], unused entries = -1
  seq_lens         int32 [num_seqs]
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

SEED_BASE = 20261200


@dataclass
class DecodeCase:
    name: str
    query: torch.Tensor
    key_cache: torch.Tensor
    value_cache: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    scale: float
    block_size: int
    partition_size: int
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return self.query.shape[0]

    @property
    def num_heads(self) -> int:
        return self.query.shape[1]

    @property
    def head_size(self) -> int:
        return self.query.shape[2]

    @property
    def num_kv_heads(self) -> int:
        return self.key_cache.shape[1]

    @property
    def num_blocks(self) -> int:
        return self.key_cache.shape[0]

    @property
    def dtype(self) -> torch.dtype:
        return self.query.dtype

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.num_seqs else 0

    def kv_bytes(self) -> int:
        """Bytes of K and V that one decode step must read: sum_s L_s*Hkv*D*elt*2."""
        elt = self.query.element_size()
        return int(self.seq_lens.to(torch.int64).sum().item()) * self.num_kv_heads * \
            self.head_size * elt * 2

    def io_bytes(self) -> int:
        """Bytes of the per-step inputs other than the cache, plus the output."""
        elt = self.query.element_size()
        q = self.query.numel() * elt
        return 2 * q + self.block_tables.numel() * 4 + self.seq_lens.numel() * 4


def _round(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    return x.to(dtype).contiguous()


def make_case(name: str, seed: int, num_seqs: int, num_heads: int,
              num_kv_heads: int, head_size: int, dtype: torch.dtype,
              block_size: int, seq_lens, partition_size: int = 512,
              scale: float | None = None, k_mult: float = 1.0,
              extra_blocks: int = 0, max_blocks_per_seq: int | None = None,
              meta: dict | None = None) -> DecodeCase:
    """Build one paged decode case.

    ``seq_lens`` is a list of ints, or a callable ``f(generator) -> list``
    drawn first from the case's generator.  The physical pool holds
    sum_s ceil(L_s / block_size) + extra_blocks blocks; a random permutation of
    the pool is dealt out to the sequences in order, so the blocks of every
    sequence are scattered across the pool.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if callable(seq_lens):
        seq_lens = seq_lens(g)
    lens = [int(x) for x in seq_lens]
    assert len(lens) == num_seqs
    nblk = [(L + block_size - 1) // block_size for L in lens]
    pool = sum(nblk) + extra_blocks
    pool = max(pool, 1)
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    mb = max_blocks_per_seq if max_blocks_per_seq is not None else max(max(nblk, default=0), 1)
    assert mb >= max(nblk, default=0)
    bt = torch.full((num_seqs, mb), -1, dtype=torch.int32)
    pos = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[pos:pos + n]
        pos += n
    q = torch.randn(num_seqs, num_heads, head_size, generator=g, dtype=torch.float32)
    k = torch.randn(pool, num_kv_heads, block_size, head_size, generator=g,
                    dtype=torch.float32)
    if k_mult != 1.0:
        k.mul_(k_mult)
    v = torch.randn(pool, num_kv_heads, block_size, head_size, generator=g,
                    dtype=torch.float32)
    if scale is None:
        scale = 1.0 / math.sqrt(head_size)
    return DecodeCase(
        name=name, query=_round(q, dtype), key_cache=_round(k, dtype),
        value_cache=_round(v, dtype), block_tables=bt,
        seq_lens=torch.tensor(lens, dtype=torch.int32), scale=float(scale),
        block_size=block_size, partition_size=partition_size,
        meta=dict(meta or {}, seed=seed))


# ---------------------------------------------------------------------------
# The five decode workloads.  C1 is the tiny fp32 case; C2-C5 are bf16.

def _c1(g):
    return [1000]


def _c2(g):
    return torch.randint(1024, 8193, (8,), generator=g).tolist()


def _c3(g):
    return [100000]


def _c4(g):
    return torch.randint(512, 3585, (256,), generator=g).tolist()


def _c5(g):
    u = torch.rand(64, generator=g, dtype=torch.float64)
    lo, hi = math.log(16.0), math.log(131072.0)
    return [int(math.floor(math.exp(lo + float(x) * (hi - lo)))) for x in u]


CONFIGS = {
    "c1_tiny_fp32": dict(index=1, num_seqs=1, num_heads=4, num_kv_heads=1,
                         head_size=64, dtype=torch.float32, block_size=16,
                         seq_lens=_c1, partition_size=512, scale=1.0 / 8.0,
                         extra_blocks=1),
    "c2_gqa_batch8": dict(index=2, num_seqs=8, num_heads=32, num_kv_heads=4,
                          head_size=128, dtype=torch.bfloat16, block_size=16,
                          seq_lens=_c2, partition_size=512),
    "c3_long_100k": dict(index=3, num_seqs=1, num_heads=32, num_kv_heads=4,
                         head_size=128, dtype=torch.bfloat16, block_size=16,
                         seq_lens=_c3, partition_size=512),
    "c4_batch256": dict(index=4, num_seqs=256, num_heads=32, num_kv_heads=4,
                        head_size=128, dtype=torch.bfloat16, block_size=16,
                        seq_lens=_c4, partition_size=512),
    "c5_mixed_d256": dict(index=5, num_seqs=64, num_heads=16, num_kv_heads=2,
                          head_size=256, dtype=torch.bfloat16, block_size=32,
                          seq_lens=_c5, partition_size=512, k_mult=4.0),
}

DESCRIPTIONS = {
    "c1_tiny_fp32": "1 seq x 1000 tokens, 4 q / 1 kv heads, D64, fp32, bs16, 64-block pool",
    "c2_gqa_batch8": "8 seqs, L~U[1024,8192], 32 q / 4 kv heads, D128, bf16, bs16",
    "c3_long_100k": "1 seq x 100000 tokens, 32 q / 4 kv heads, D128, bf16, bs16",
    "c4_batch256": "256 seqs, L~U[512,3584], 32 q / 4 kv heads, D128, bf16, bs16",
    "c5_mixed_d256": "64 seqs, L log-uniform [16,131072], 16 q / 2 kv heads, D256, bf16, K x4, bs32",
}


def chunk_queries(case: DecodeCase, tokens: int, seed: int = 7):
    """Query chunks of `tokens` tokens for every sequence of a case (its last
    tokens, so each sequence must hold at least that many): q [B * tokens, H,
    D] drawn N(0, 1) and rounded to the case's dtype, and q_start [B + 1]."""
    B, H, D = case.query.shape
    if int(case.seq_lens.min()) < tokens:
        raise ValueError("a sequence is shorter than its chunk")
    g = torch.Generator(device="cpu")
    g.manual_seed(SEED_BASE + 5000 + seed)
    q = _round(torch.randn(B * tokens, H, D, generator=g), case.dtype)
    q_start = torch.arange(0, B * tokens + 1, tokens, dtype=torch.int32)
    return q, q_start


def config_case(name: str, partition_size: int | None = None,
                seed_offset: int = 0) -> DecodeCase:
    """One of the five named workloads, drawn from seed SEED_BASE + index
    (+ 1000 * seed_offset: another batch of the same shape, e.g. per rank)."""
    c = dict(CONFIGS[name])
    idx = c.pop("index")
    if partition_size is not None:
        c["partition_size"] = partition_size
    return make_case(name, SEED_BASE + idx + 1000 * seed_offset,
                     meta={"config_index": idx}, **c)


def sub_batch(case: DecodeCase, num_seqs: int) -> DecodeCase:
    """The first num_seqs sequences of a case (same cache and pool)."""
    return replace(case, query=case.query[:num_seqs].contiguous(),
                   block_tables=case.block_tables[:num_seqs].contiguous(),
                   seq_lens=case.seq_lens[:num_seqs].contiguous(),
                   name=f"{case.name}[:{num_seqs}]")


def with_partition_size(case: DecodeCase, partition_size: int) -> DecodeCase:
    return replace(case, partition_size=partition_size)


def permute_pool(case: DecodeCase, seed: int) -> DecodeCase:
    """The same logical case with the physical pool shuffled: block b moves to
    slot perm[b] and every table entry is remapped, so each sequence still
    sees the same keys and values in the same order."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    nb = case.num_blocks
    perm = torch.randperm(nb, generator=g)
    k = torch.empty_like(case.key_cache)
    v = torch.empty_like(case.value_cache)
    k[perm] = case.key_cache
    v[perm] = case.value_cache
    bt = case.block_tables.clone()
    used = bt >= 0
    bt[used] = perm.to(torch.int32)[bt[used].long()]
    return replace(case, key_cache=k, value_cache=v, block_tables=bt,
                   name=case.name + f"_perm{seed}")
