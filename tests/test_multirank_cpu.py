"""The N > 1 path of bench.py on CPU: two gloo ranks.  Each rank draws its
own batch of the same shape (weak scaling, no data-path collective) and the
timing bookkeeping takes the max of the step time and the sum of the work
over ranks."""
import os
import socket

import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import workloads
    r, w, local = bench.dist_env()
    assert (r, w, local) == (rank, world, rank)
    bench.init_dist(w, "gloo")
    case = workloads.config_case("c1_tiny_fp32", seed_offset=r)
    t = 1.0 + r  # rank r "took" 1 + r seconds
    mx = bench.reduce_over_ranks(t, "max", w)
    sm = bench.reduce_over_ranks(float(case.kv_bytes()), "sum", w)
    bench.barrier(w)
    q.put((r, mx, sm, case.query[0, 0, :4].tolist(), tuple(case.key_cache.shape)))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=300) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, mx0, sm0, q0, sh0), (r1, mx1, sm1, q1, sh1) = res
    assert mx0 == mx1 == 2.0
    one = 1000 * 1 * 64 * 4 * 2  # L * Hkv * D * elt * 2 for the tiny fp32 workload
    assert sm0 == sm1 == 2 * one
    assert sh0 == sh1            # same shape on every rank
    assert q0 != q1              # but a different batch


def test_single_rank_bookkeeping_is_identity():
    import bench
    assert bench.reduce_over_ranks(3.5, "max", 1) == 3.5
    assert bench.reduce_over_ranks(3.5, "sum", 1) == 3.5
    assert torch.tensor(0).item() == 0
