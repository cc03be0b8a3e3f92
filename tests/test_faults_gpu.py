"""Device-side failure reporting, exercised without faulting or hanging the
GPU: bad data is caught by the kernels' own checks and reported through the
workspace status word; a bounded wait on a barrier that nothing releases runs
out, reports PA_ERR_DEVICE_TIMEOUT, and the context stays usable."""
import pytest
import torch

import paged_decode_attention_v2_gb300 as pa
import workloads
from gpu_helpers import DeviceCase, assert_close, reference

pytestmark = pytest.mark.gpu


def _case():
    return workloads.make_case("faults", 81, 4, 16, 2, 128, torch.bfloat16, 16,
                               [100, 1000, 2500, 7], partition_size=512, extra_blocks=8)


@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2])
def test_out_of_range_block_id_is_reported(variant):
    case = _case()
    dc = DeviceCase(case)
    bad = dc.bt.clone()
    bad[1, 10] = case.num_blocks + 5      # past the pool
    bad[2, 3] = -7                        # negative
    out = torch.empty_like(dc.q)
    pa.pa_forward(out, dc.q, dc.kc, dc.vc, bad, dc.sl, case.scale, 512, dc.ws,
                  max_seq_len=dc.max_seq_len, variant=variant)
    assert pa.pa_read_device_status(dc.ws) == pa.PA_ERR_DEVICE_BAD_INPUT
    # the status word was cleared by the read; a good call reports OK
    out = dc.run(variant=variant)
    assert_close(out, reference(case), torch.bfloat16)


def test_sequence_length_above_bound_is_reported():
    case = _case()
    dc = DeviceCase(case)
    sl = dc.sl.clone()
    sl[0] = dc.max_seq_len + 1
    out = torch.empty_like(dc.q)
    pa.pa_forward(out, dc.q, dc.kc, dc.vc, dc.bt, sl, case.scale, 512, dc.ws,
                  max_seq_len=dc.max_seq_len, variant=pa.PA_VARIANT_V2)
    assert pa.pa_read_device_status(dc.ws) == pa.PA_ERR_DEVICE_BAD_INPUT
    sl[0] = -3
    pa.pa_forward(out, dc.q, dc.kc, dc.vc, dc.bt, sl, case.scale, 512, dc.ws,
                  max_seq_len=dc.max_seq_len, variant=pa.PA_VARIANT_V1)
    assert pa.pa_read_device_status(dc.ws) == pa.PA_ERR_DEVICE_BAD_INPUT


@pytest.mark.parametrize("math", [pa.PA_MATH_TENSOR, pa.PA_MATH_SIMT])
@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2])
def test_bounded_wait_runs_out_and_context_survives(variant, math):
    case = _case()
    dc = DeviceCase(case)
    out = torch.zeros_like(dc.q)
    pa.pa_forward(out, dc.q, dc.kc, dc.vc, dc.bt, dc.sl, case.scale, 512, dc.ws,
                  max_seq_len=dc.max_seq_len, variant=variant, math=math,
                  debug_flags=pa.PA_DEBUG_STALL_CONSUMERS, wait_limit_ns=200_000)
    assert pa.pa_read_device_status(dc.ws) == pa.PA_ERR_DEVICE_TIMEOUT
    torch.cuda.synchronize()  # the context is still usable
    out = dc.run(variant=variant, math=math)
    assert_close(out, reference(case), torch.bfloat16)


@pytest.mark.parametrize("share_kv", [0, 1], ids=["own", "cluster"])
@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2])
def test_bounded_wait_runs_out_in_the_tcgen05_chunk_kernel(variant, share_kv):
    """Query chunks of 40 tokens x 8 heads (320 rows per KV head: the tcgen05
    kernel) with every softmax warp waiting on a barrier nothing releases: the
    MMA thread and the producer give up in turn, the MMA thread waits for its
    own MMAs, the tensor memory is freed, PA_ERR_DEVICE_TIMEOUT is reported,
    and the next call on the same context matches the oracle; also with the
    CTAs in clusters sharing K/V, where every CTA still meets the cluster's
    last barrier."""
    import oracle
    c = workloads.make_case("faults_chunks", 83, 3, 16, 2, 128, torch.bfloat16, 16,
                            [900, 2000, 40], partition_size=512, extra_blocks=4)
    qlens = [40, 17, 40]
    g = torch.Generator().manual_seed(84)
    q = torch.randn(sum(qlens), 16, 128, generator=g).to(torch.bfloat16)
    qs = torch.tensor([0, 40, 57, 97], dtype=torch.int32)
    ref = oracle.query_chunks(q, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, qs,
                              c.scale)
    args = (q.cuda(), c.key_cache.cuda(), c.value_cache.cuda(), c.block_tables.cuda(),
            c.seq_lens.cuda(), qs.cuda())
    ws = pa.alloc_workspace(q.shape[0], 16, 128, c.max_seq_len, 512)
    out = torch.zeros(q.shape, dtype=torch.bfloat16, device="cuda")
    pa.pa_chunks_forward(out, *args, c.scale, 512, ws, max_seq_len=c.max_seq_len, max_chunk=40,
                         variant=variant, debug_flags=pa.PA_DEBUG_STALL_CONSUMERS,
                         wait_limit_ns=200_000, share_kv=share_kv)
    assert pa.pa_read_device_status(ws) == pa.PA_ERR_DEVICE_TIMEOUT
    torch.cuda.synchronize()  # the context is still usable
    pa.pa_chunks_forward(out, *args, c.scale, 512, ws, max_seq_len=c.max_seq_len, max_chunk=40,
                         variant=variant, share_kv=share_kv)
    assert pa.pa_read_device_status(ws) == pa.PA_OK
    assert_close(out, ref, torch.bfloat16, "chunks after a timed-out call")


def test_status_keeps_first_error_until_read():
    case = _case()
    dc = DeviceCase(case)
    out = torch.empty_like(dc.q)
    pa.pa_forward(out, dc.q, dc.kc, dc.vc, dc.bt, dc.sl, case.scale, 512, dc.ws,
                  max_seq_len=dc.max_seq_len, variant=pa.PA_VARIANT_V2,
                  debug_flags=pa.PA_DEBUG_STALL_CONSUMERS, wait_limit_ns=100_000)
    bad = dc.bt.clone()
    bad[0, 0] = 1 << 30
    pa.pa_forward(out, dc.q, dc.kc, dc.vc, bad, dc.sl, case.scale, 512, dc.ws,
                  max_seq_len=dc.max_seq_len, variant=pa.PA_VARIANT_V2)
    assert pa.pa_read_device_status(dc.ws) == pa.PA_ERR_DEVICE_TIMEOUT
    assert pa.pa_read_device_status(dc.ws) == pa.PA_OK


def test_host_errors_do_not_launch():
    case = _case()
    dc = DeviceCase(case)
    out = torch.full_like(dc.q, 7.0)
    with pytest.raises(pa.PAError) as e:
        pa.pa_forward(out, dc.q, dc.kc, dc.vc, dc.bt, dc.sl, case.scale, 500, dc.ws,
                      max_seq_len=dc.max_seq_len, variant=pa.PA_VARIANT_V2)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    small = dc.ws[:1024]
    with pytest.raises(pa.PAError) as e:
        pa.pa_forward(out, dc.q, dc.kc, dc.vc, dc.bt, dc.sl, case.scale, 512, small,
                      max_seq_len=dc.max_seq_len, variant=pa.PA_VARIANT_V2)
    assert e.value.status == pa.PA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
