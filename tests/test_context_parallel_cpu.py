"""Context parallelism on CPU: sequences split over gloo ranks by partition
ranges.  Each rank computes the Phase 1 partials of its own range with the
oracle, writes them into a workspace laid out by libpa's pa_workspace_layout
(host arithmetic only, no GPU), and the exchange of
``paged_decode_attention_v2_gb300.context_parallel`` gathers every rank's
slots.  The gathered workspace must hold exactly the single-rank partials,
and the oracle's Phase 2 combine of them must equal the unpartitioned
softmax (the "paged_attention_v2" commit note, project_6 commit 96f4baf,
section "Implementation": partitions are independent until Phase 2)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case():
    import workloads
    lens = [1, 40, 64, 65, 200, 131]
    return workloads.make_case("cp", 41, len(lens), 8, 2, 64, torch.float32, 16, lens,
                               partition_size=64, extra_blocks=3, k_mult=2.0)


def _workspace(case):
    import paged_decode_attention_v2_gb300 as pa
    n = pa.pa_workspace_bytes(case.num_seqs, case.num_heads, case.head_size, case.max_seq_len,
                              case.partition_size)
    return torch.full((n,), 0xFF, dtype=torch.uint8)  # NaN in every float slot


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    import paged_decode_attention_v2_gb300 as pa
    from paged_decode_attention_v2_gb300 import context_parallel as cp
    pa.load_library()
    c = _case()
    P = c.partition_size
    np_max = -(-c.max_seq_len // P)
    ranges = cp.partition_ranges(np_max, world)
    ml, es, to = oracle.partials(c.query, c.key_cache, c.value_cache, c.block_tables,
                                 c.seq_lens, c.scale, P, max_parts=np_max)
    ws = _workspace(c)
    vml, ves, vto = cp.partials_views(ws, c.num_seqs, c.num_heads, c.head_size, c.max_seq_len, P)
    b, e = ranges[rank]
    # this rank's own range only: the oracle's partials of partitions [b, e)
    vml[:, :, b:e] = torch.from_numpy(ml[:, :, b:e]).float()
    ves[:, :, b:e] = torch.from_numpy(es[:, :, b:e]).float()
    vto[:, :, b:e] = torch.from_numpy(to[:, :, b:e]).float()
    cp.exchange_partials(ws, c.num_seqs, c.num_heads, c.head_size, c.max_seq_len, P, ranges)
    q.put((rank, ranges, ws.numpy().copy()))
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_exchange_gathers_every_range(world):
    import oracle
    import paged_decode_attention_v2_gb300 as pa
    from paged_decode_attention_v2_gb300 import context_parallel as cp
    pa.load_library()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    c = _case()
    P = c.partition_size
    np_max = -(-c.max_seq_len // P)
    assert res[0][1] == cp.partition_ranges(np_max, world)
    assert all(e > b for b, e in res[0][1]), "every rank owns some partitions here"
    ml, es, to = oracle.partials(c.query, c.key_cache, c.value_cache, c.block_tables,
                                 c.seq_lens, c.scale, P, max_parts=np_max)
    npt = oracle.num_partitions(c.seq_lens.numpy(), P)
    ref = oracle.attention(c.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens,
                           c.scale)
    for rank, _, raw in res:
        ws = torch.from_numpy(raw)
        vml, ves, vto = cp.partials_views(ws, c.num_seqs, c.num_heads, c.head_size,
                                          c.max_seq_len, P)
        for s in range(c.num_seqs):
            n = int(npt[s])
            # every slot of every partition holds the single-rank partial, bit for bit
            assert torch.equal(vml[s, :, :n], torch.from_numpy(ml[s, :, :n]).float()), (rank, s)
            assert torch.equal(ves[s, :, :n], torch.from_numpy(es[s, :, :n]).float()), (rank, s)
            assert torch.equal(vto[s, :, :n], torch.from_numpy(to[s, :, :n]).float()), (rank, s)
        # the combine of the gathered slots is the unpartitioned softmax
        out = oracle.combine(vml.double().numpy(), ves.double().numpy(), vto.double().numpy(),
                             npt)
        assert np.allclose(out, ref, rtol=1e-6, atol=1e-6), rank


def test_partition_ranges_cover_once():
    from paged_decode_attention_v2_gb300 import context_parallel as cp
    for n in (0, 1, 5, 196, 586):
        for w in (1, 2, 3, 4, 8):
            r = cp.partition_ranges(n, w)
            assert len(r) == w and r[0][0] == 0 and r[-1][1] == n
            assert all(r[i][1] == r[i + 1][0] for i in range(w - 1))
            sizes = [e - b for b, e in r]
            assert max(sizes) - min(sizes) <= 1
