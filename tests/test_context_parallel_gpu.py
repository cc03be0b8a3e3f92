"""V2's phases as separate C-ABI calls (pa_v2_partials / pa_v2_combine) and
the context-parallel split of long sequences built on them, on one GPU.

The "paged_attention_v2" commit note (project_6, commit 96f4baf, section
"Implementation") defines Phase 1 per partition and Phase 2 as the
reduction over a sequence's partitions; a split of the partitions over
ranks therefore needs one exchange of partials between the phases.  Here the
ranks' Phase 1 runs on this GPU, the exchange goes through two gloo
processes on the CPU, and Phase 2 runs on this GPU again."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import paged_decode_attention_v2_gb300 as pa
from paged_decode_attention_v2_gb300 import context_parallel as cp
import workloads
from gpu_helpers import DeviceCase, assert_close, config_case, reference

pytestmark = pytest.mark.gpu


def _canary_ws(case):
    n = pa.pa_workspace_bytes(case.num_seqs, case.num_heads, case.head_size, case.max_seq_len,
                              case.partition_size)
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
    ws[:256] = 0  # the status block starts at zero, as after pa_workspace_init
    return ws


def _views(ws, case):
    return cp.partials_views(ws, case.num_seqs, case.num_heads, case.head_size,
                             case.max_seq_len, case.partition_size)


def _partials(dc, ws, b, e, bt=None):
    c = dc.case
    pa.pa_v2_partials(dc.q, dc.kc, dc.vc, dc.bt if bt is None else bt, dc.sl, c.scale,
                      c.partition_size, ws, b, e, max_seq_len=dc.max_seq_len)
    st = pa.pa_read_device_status(ws)
    assert st == pa.PA_OK, pa.pa_status_string(st)


@pytest.mark.parametrize("rng", [(0, 3), (2, 9), (5, 2 ** 31 - 1), (0, 2 ** 31 - 1)])
def test_partials_range_writes_only_its_slots(rng):
    """Slots of partitions in the range equal pa_v2_forward's Phase 1 bit for
    bit; every other byte of the partials keeps the canary."""
    dc = DeviceCase(config_case("c2_gqa_batch8"))
    c = dc.case
    dc.run(variant=pa.PA_VARIANT_V2)
    ref = [v.clone() for v in _views(dc.ws, c)]
    ws = _canary_ws(c)
    b, e = rng
    _partials(dc, ws, b, e)
    np_s = (c.seq_lens.to(torch.int64) + c.partition_size - 1) // c.partition_size
    for got, want in zip(_views(ws, c), ref):
        raw = got.view(torch.int32)
        for s in range(c.num_seqs):
            hi = min(int(np_s[s]), e)
            if hi > b:
                assert torch.equal(got[s, :, b:hi], want[s, :, b:hi]), (s, rng)
            outside = torch.ones(got.shape[2], dtype=torch.bool, device="cuda")
            outside[b:max(hi, b)] = False
            assert torch.all(raw[s][:, outside] == -1), (s, rng)


def test_combine_alone_equals_forward():
    """Phase 1 over every partition, then Phase 2 alone: bit-identical to
    pa_v2_forward, on the mixed-length D = 256 workload at P = 256."""
    dc = DeviceCase(config_case("c5_mixed_d256", 256))
    c = dc.case
    want = dc.run(variant=pa.PA_VARIANT_V2)
    ws = _canary_ws(c)
    _partials(dc, ws, 0, 2 ** 31 - 1)
    out = torch.full_like(dc.q, float("nan"))
    pa.pa_v2_combine(out, dc.sl, c.partition_size, ws, dc.max_seq_len)
    torch.cuda.synchronize()
    assert torch.equal(out, want)
    assert_close(out, reference(c), c.dtype, "combine alone")


def test_combine_rejects_bad_arguments():
    dc = DeviceCase(config_case("c1_tiny_fp32"))
    c = dc.case
    out = torch.empty_like(dc.q)
    small = torch.zeros(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_v2_combine(out, dc.sl, c.partition_size, small, dc.max_seq_len)
    assert e.value.status == pa.PA_ERR_WORKSPACE_TOO_SMALL
    with pytest.raises(pa.PAError) as e:
        pa.pa_v2_combine(out, dc.sl, 100, dc.ws, dc.max_seq_len)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    with pytest.raises(pa.PAError) as e:
        pa.pa_v2_partials(dc.q, dc.kc, dc.vc, dc.bt, dc.sl, c.scale, c.partition_size, dc.ws,
                          3, 2, max_seq_len=dc.max_seq_len)
    assert e.value.status == pa.PA_ERR_INVALID_ARG


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _exchange_worker(rank, world, port, raw, shape, ranges, q):
    """One rank of the exchange, on the CPU: its workspace bytes in, the
    gathered workspace bytes out (rank 0)."""
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import paged_decode_attention_v2_gb300 as pa_
    from paged_decode_attention_v2_gb300 import context_parallel as cp_
    pa_.load_library()
    ws = torch.from_numpy(raw)
    B, H, D, L, P = shape
    cp_.exchange_partials(ws, B, H, D, L, P, ranges)
    q.put((rank, ws.numpy().copy()))
    dist.destroy_process_group()


def _gloo_exchange(workspaces, case, ranges):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    shape = (case.num_seqs, case.num_heads, case.head_size, case.max_seq_len,
             case.partition_size)
    procs = [ctx.Process(target=_exchange_worker,
                         args=(r, len(workspaces), port, w.cpu().numpy(), shape, ranges, q))
             for r, w in enumerate(workspaces)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return [torch.from_numpy(res[r]) for r in range(len(workspaces))]


@pytest.mark.parametrize("sharded", [False, True], ids=["full-table", "sharded-table"])
def test_split_over_two_ranks_equals_single_gpu(sharded):
    """The 100K-token workload split into two partition ranges: each range's
    Phase 1 into its own workspace, the slots exchanged through two gloo
    processes, Phase 2 on each rank's gathered workspace.  Both ranks' outputs
    equal pa_v2_forward bit for bit and the oracle at the bf16 bar.  With
    `sharded`, each rank's block table keeps only the pages of its own range
    (-1 elsewhere), as a GPU that holds only its shard of the cache would."""
    dc = DeviceCase(config_case("c3_long_100k"))
    c = dc.case
    want = dc.run(variant=pa.PA_VARIANT_V2)
    np_max = -(-c.max_seq_len // c.partition_size)
    ranges = cp.partition_ranges(np_max, 2)
    pages_per_part = c.partition_size // c.block_size
    workspaces = []
    for b, e in ranges:
        bt = None
        if sharded:
            bt = torch.full_like(dc.bt, -1)
            lo, hi = b * pages_per_part, min(e * pages_per_part, dc.bt.shape[1])
            bt[:, lo:hi] = dc.bt[:, lo:hi]
        ws = _canary_ws(c)
        _partials(dc, ws, b, e, bt)
        workspaces.append(ws)
    gathered = _gloo_exchange(workspaces, c, ranges)
    ref = reference(c)
    for r, g in enumerate(gathered):
        ws = g.to("cuda")
        out = torch.full_like(dc.q, float("nan"))
        pa.pa_v2_combine(out, dc.sl, c.partition_size, ws, dc.max_seq_len)
        torch.cuda.synchronize()
        assert torch.equal(out, want), r
        assert_close(out, ref, c.dtype, f"rank {r}")


def test_context_parallel_forward_single_rank():
    """context_parallel_forward in a group of one (gloo, this process): the
    whole range, an exchange that moves nothing, then the combine."""
    import torch.distributed as dist
    dc = DeviceCase(config_case("c2_gqa_batch8"))
    c = dc.case
    want = dc.run(variant=pa.PA_VARIANT_V2)
    port = _free_port()
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    group_made = False
    if not dist.is_initialized():
        dist.init_process_group("gloo", rank=0, world_size=1)
        group_made = True
    try:
        out = torch.full_like(dc.q, float("nan"))
        cp.context_parallel_forward(out, dc.q, dc.kc, dc.vc, dc.bt, dc.sl, c.scale,
                                    c.partition_size, dc.ws, dc.max_seq_len)
        torch.cuda.synchronize()
        assert torch.equal(out, want)
    finally:
        if group_made:
            dist.destroy_process_group()
