"""Context parallelism for long decode sequences over several GPUs.

The partitions of every sequence are split into contiguous ranges, one per
rank.  Each rank runs Phase 1 over its own range (``pa_v2_partials``) into
its own workspace, holding only the K/V pages of that range; one exchange
(an all-gather of each rank's max_logits, exp_sums and tmp_out slots) gives
every rank all the slots; Phase 2 (``pa_v2_combine``) then writes the output
that a single-GPU ``pa_v2_forward`` would.  The "paged_attention_v2" commit
note (project_6, commit 96f4baf "Dockerfile", section "Implementation")
defines the two phases; the split is possible because the partitions are
independent until the Phase 2 reduction.

The exchange only moves bytes (torch.distributed: NCCL between GPUs, gloo
for CPU tensors); the arithmetic of both phases runs in libpa's kernels.
"""
from __future__ import annotations

import torch

from . import pa_v2_combine, pa_v2_partials, pa_workspace_layout


def partition_ranges(max_parts: int, world: int) -> list[tuple[int, int]]:
    """Contiguous ranges [begin, end) covering partitions 0 .. max_parts-1,
    one per rank, their sizes differing by at most one."""
    if world < 1 or max_parts < 0:
        raise ValueError("world >= 1 and max_parts >= 0")
    base, extra = divmod(max_parts, world)
    out, b = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((b, b + n))
        b += n
    return out


def partials_views(workspace: torch.Tensor, num_seqs: int, num_heads: int, head_size: int,
                   max_seq_len: int, partition_size: int):
    """(max_logits [B, H, Np], exp_sums [B, H, Np], tmp_out [B, H, Np, D]):
    float32 views of a workspace's Phase 1 slots, Np = ceil(max_seq_len / P)."""
    off = pa_workspace_layout(num_seqs, num_heads, head_size, max_seq_len, partition_size)
    n = max(-(-max_seq_len // partition_size), 1)
    B, H, D = num_seqs, num_heads, head_size
    w = workspace.view(torch.uint8)

    def view(o, count, shape):
        return w[o:o + count * 4].view(torch.float32).view(shape)
    return (view(off[1], B * H * n, (B, H, n)), view(off[2], B * H * n, (B, H, n)),
            view(off[3], B * H * n * D, (B, H, n, D)))


def exchange_partials(workspace: torch.Tensor, num_seqs: int, num_heads: int, head_size: int,
                      max_seq_len: int, partition_size: int, ranges, group=None) -> None:
    """All-gather: rank r contributes the slots of its range ranges[r]; on
    return every rank's workspace holds the slots of every range.  Ranges of
    unequal length are padded to the longest for the collective."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    world = dist.get_world_size(group)
    if len(ranges) != world:
        raise ValueError("one partition range per rank")
    width = max((e - b for b, e in ranges), default=0)
    if width == 0:
        return
    # gloo moves host tensors: device slots go through host copies there
    via_host = workspace.is_cuda and dist.get_backend(group) == "gloo"
    for v in partials_views(workspace, num_seqs, num_heads, head_size, max_seq_len,
                            partition_size):
        b, e = ranges[rank]
        dev = torch.device("cpu") if via_host else v.device
        mine = torch.zeros(v.shape[:2] + (width,) + v.shape[3:], dtype=v.dtype, device=dev)
        mine[:, :, :e - b] = v[:, :, b:e].to(dev)
        parts = [torch.empty_like(mine) for _ in range(world)]
        dist.all_gather(parts, mine, group=group)
        for r, (rb, re_) in enumerate(ranges):
            if r != rank and re_ > rb:
                v[:, :, rb:re_] = parts[r][:, :, :re_ - rb].to(v.device)


def context_parallel_forward(out, query, key_cache, value_cache, block_tables, seq_lens, scale,
                             partition_size, workspace, max_seq_len, group=None,
                             stream=None) -> None:
    """Decode attention for sequences split over the ranks of `group` by
    partition ranges: Phase 1 over this rank's range, the exchange, then
    Phase 2.  Every rank passes the whole lengths and a block table whose
    entries are valid at least for its own range; every rank gets `out`."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    B, H, D = query.shape
    ranges = partition_ranges(-(-max_seq_len // partition_size), world)
    b, e = ranges[rank]
    pa_v2_partials(query, key_cache, value_cache, block_tables, seq_lens, scale, partition_size,
                   workspace, b, e, max_seq_len=max_seq_len, stream=stream)
    exchange_partials(workspace, B, H, D, max_seq_len, partition_size, ranges, group)
    pa_v2_combine(out, seq_lens, partition_size, workspace, max_seq_len, stream=stream)
