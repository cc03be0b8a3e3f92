"""pa_v2_forward_noalloc: the V2 entry point for callers that cannot allocate
device memory (for example a plug-in whose host framework owns all device
memory, or a serving loop that must not pay cudaMalloc's synchronisation).
Its scratch is the library's own fixed device array, so the caller passes
only inputs and outputs.

Called here straight through the C ABI (ctypes), twice in a row, and compared
on each call both with the ordinary pa_v2_forward (caller-owned workspace)
and with the CPU fp64 oracle, at the tests' bf16 tolerance: the second
comparison would also catch a fault shared by the two entry points' kernels.  This file sorts last so that a run stopping at the first failure
has run every other test before it; it also passes on its own in a fresh
process.
"""
import ctypes

import pytest
import torch

import paged_decode_attention_v2_gb300 as pa
import workloads
from gpu_helpers import DeviceCase, assert_close, reference

pytestmark = pytest.mark.gpu


def _noalloc(lib, dc, out, max_seq_len=None, partition_size=None):
    c = dc.case
    return lib.pa_v2_forward_noalloc(
        out.data_ptr(), dc.q.data_ptr(), dc.kc.data_ptr(), dc.vc.data_ptr(),
        dc.bt.data_ptr(), dc.sl.data_ptr(), c.num_seqs, c.num_heads, c.num_kv_heads,
        c.head_size, c.num_blocks, c.block_size, dc.bt.shape[1],
        max_seq_len if max_seq_len is not None else dc.max_seq_len, ctypes.c_float(c.scale),
        partition_size or c.partition_size, pa.PA_DTYPE_BF16,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_the_workspace_entry_point_twice():
    lib = pa.load_library()
    case = workloads.make_case("noalloc", 91, 6, 32, 4, 128, torch.bfloat16, 16,
                               [1, 300, 513, 2048, 4096, 3001], partition_size=512,
                               extra_blocks=7)
    dc = DeviceCase(case)
    ref = torch.empty_like(dc.q)
    pa.pa_v2_forward(ref, dc.q, dc.kc, dc.vc, dc.bt, dc.sl, case.scale, 512, dc.ws,
                     max_seq_len=dc.max_seq_len)
    assert pa.pa_read_device_status(dc.ws) == pa.PA_OK
    ref_np = ref.double().cpu().numpy()
    exact = reference(case)
    for _ in range(2):
        out = torch.full_like(dc.q, float("nan"))
        assert _noalloc(lib, dc, out) == pa.PA_OK
        torch.cuda.synchronize()
        assert_close(out, ref_np, torch.bfloat16, "noalloc vs pa_v2_forward")
        assert_close(out, exact, torch.bfloat16, "noalloc vs the fp64 oracle")


def test_noalloc_refuses_requests_beyond_its_scratch():
    lib = pa.load_library()
    case = workloads.make_case("noalloc_big", 92, 2, 32, 4, 128, torch.bfloat16, 16,
                               [100, 200], partition_size=64, max_blocks_per_seq=8192)
    dc = DeviceCase(case)
    out = torch.zeros_like(dc.q)
    # 2 seqs x 32 heads x 2048 partitions x (128 + 2) floats is ~68 MB > 32 MiB
    assert _noalloc(lib, dc, out, max_seq_len=8192 * 16, partition_size=64) == \
        pa.PA_ERR_WORKSPACE_TOO_SMALL
    torch.cuda.synchronize()
    assert torch.all(out == 0)
