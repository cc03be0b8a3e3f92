"""pa_forward_host: the per-step data (query, block tables, lengths, output)
in host memory, copied by the library's own C-ABI call.  Its output equals
the device-pointer call's bit for bit (same kernels, same inputs) and meets
the oracle bar; argument errors come back before anything is enqueued."""
import pytest
import torch

import paged_decode_attention_v2_gb300 as pa
import workloads
from gpu_helpers import DeviceCase, assert_close, reference

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2, pa.PA_VARIANT_AUTO])
def test_host_buffers_match_device_call(variant, pinned):
    case = workloads.make_case("host", 31, 5, 32, 4, 128, torch.bfloat16, 16,
                               [1, 700, 2048, 5000, 129], partition_size=512, extra_blocks=3)
    dc = DeviceCase(case)
    dev_out = dc.run(variant=variant)

    def host(t):
        t = t.contiguous()
        return t.pin_memory() if pinned else t.clone()
    hq, hbt, hsl = host(case.query), host(case.block_tables), host(case.seq_lens)
    hout = host(torch.full_like(case.query, float("nan")))
    staging = pa.alloc_staging(hq, hbt)
    for _ in range(2):
        pa.pa_forward_host(hout, hq, dc.kc, dc.vc, hbt, hsl, case.scale, 512, staging, dc.ws,
                           max_seq_len=dc.max_seq_len, variant=variant)
        torch.cuda.synchronize()
        assert pa.pa_read_device_status(dc.ws) == pa.PA_OK
        assert torch.equal(hout.view(torch.int16), dev_out.cpu().view(torch.int16))
    assert_close(hout, reference(case), torch.bfloat16, "host buffers")


def test_host_call_rejects_bad_staging_before_enqueueing():
    case = workloads.make_case("host_bad", 32, 2, 8, 1, 64, torch.float16, 16, [100, 300],
                               partition_size=256)
    dc = DeviceCase(case)
    hq, hbt, hsl = case.query.pin_memory(), case.block_tables.pin_memory(), \
        case.seq_lens.pin_memory()
    hout = torch.full_like(case.query, 7.0).pin_memory()
    need = pa.pa_host_staging_bytes(2, 8, 64, hbt.shape[1], torch.float16)
    small = torch.zeros(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PAError) as e:
        pa.pa_forward_host(hout, hq, dc.kc, dc.vc, hbt, hsl, case.scale, 256, small, dc.ws,
                           max_seq_len=dc.max_seq_len)
    assert e.value.status == pa.PA_ERR_INVALID_ARG
    staging = pa.alloc_staging(hq, hbt)
    with pytest.raises(pa.PAError) as e:  # partition size 100: refused on the host
        pa.pa_forward_host(hout, hq, dc.kc, dc.vc, hbt, hsl, case.scale, 100, staging, dc.ws,
                           max_seq_len=dc.max_seq_len, variant=pa.PA_VARIANT_V2)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert torch.all(hout == 7.0)
