"""Python binding of libpa, the GB300 paged decode attention library.

Argument marshalling only: every step of the computation runs in libpa's
CUDA kernels.  The functions carry the C ABI's names (``include/pa.h``) and
take torch tensors for the buffers; the torch stream is passed through as a
raw ``cudaStream_t``.  There is no fallback: if ``_lib/libpa.so`` is missing
(build it with ``python -m paged_decode_attention_v2_gb300.build_lib``) the
first call raises.

Layouts: query/out [num_seqs, num_heads, head_size]; key/value cache
[num_blocks, num_kv_heads, block_size, head_size]; block_tables int32
[num_seqs, max_blocks_per_seq]; seq_lens int32 [num_seqs].
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_WORKSPACE_TOO_SMALL = 3
PA_ERR_CUDA = 4
PA_ERR_DEVICE_BAD_INPUT = 5
PA_ERR_DEVICE_TIMEOUT = 6

PA_DTYPE_F32, PA_DTYPE_BF16, PA_DTYPE_F16 = 0, 1, 2
PA_VARIANT_AUTO, PA_VARIANT_V1, PA_VARIANT_V2 = 0, 1, 2
PA_MATH_AUTO, PA_MATH_SIMT, PA_MATH_TENSOR = 0, 1, 2
PA_DEBUG_STALL_CONSUMERS = 1
PA_DEBUG_NO_TCGEN05 = 2
PA_DEBUG_TCGEN05_KEYS = 4

_DTYPES = {torch.float32: PA_DTYPE_F32, torch.bfloat16: PA_DTYPE_BF16,
           torch.float16: PA_DTYPE_F16}

# Every function the header declares (checked against include/pa.h by tests).
EXPORTS = ("pa_workspace_bytes", "pa_workspace_layout", "pa_workspace_init",
           "pa_v1_forward", "pa_v2_forward", "pa_forward", "pa_choose_v2", "pa_choose_v2_chunks",
           "pa_read_device_status", "pa_status_string", "pa_last_cuda_error",
           "pa_version", "pa_v2_forward_noalloc", "pa_host_staging_bytes", "pa_forward_host",
           "pa_chunks_forward", "pa_v2_partials", "pa_v2_combine")


class PAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_text(status)} (status {status})")


class pa_options_t(ctypes.Structure):
    _fields_ = [("variant", ctypes.c_int32), ("math", ctypes.c_int32),
                ("num_stages", ctypes.c_int32), ("debug_flags", ctypes.c_int32),
                ("wait_limit_ns", ctypes.c_uint64), ("phase1_event", ctypes.c_void_p),
                ("ctas_per_sm", ctypes.c_int32), ("fuse_partitions", ctypes.c_int32),
                ("share_kv", ctypes.c_int32)]


_lib = None
_lock = threading.Lock()

_FWD_ARGS = [ctypes.c_void_p] * 6 + [ctypes.c_int] * 8 + [ctypes.c_float, ctypes.c_int,
                                                           ctypes.c_int, ctypes.c_void_p,
                                                           ctypes.c_size_t, ctypes.c_void_p]


def load_library(path: str = LIB_PATH):
    """Load libpa (no fallback: raises if the shared library is absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libpa.so not found at {path}; build it with "
                "`python -m paged_decode_attention_v2_gb300.build_lib`")
        lib = ctypes.CDLL(path)
        ci, cs, vp = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
        lib.pa_workspace_bytes.restype = cs
        lib.pa_workspace_bytes.argtypes = [ci] * 5
        lib.pa_workspace_layout.restype = ci
        lib.pa_workspace_layout.argtypes = [ci] * 5 + [ctypes.POINTER(cs)]
        lib.pa_workspace_init.restype = ci
        lib.pa_workspace_init.argtypes = [vp, cs, vp]
        for name in ("pa_v1_forward", "pa_v2_forward"):
            f = getattr(lib, name)
            f.restype = ci
            f.argtypes = _FWD_ARGS
        lib.pa_v2_partials.restype = ci
        lib.pa_v2_partials.argtypes = (_FWD_ARGS[1:17] + [ci, ci] + _FWD_ARGS[17:])
        lib.pa_v2_combine.restype = ci
        lib.pa_v2_combine.argtypes = [vp, vp] + [ci] * 6 + [vp, cs, vp]
        lib.pa_v2_forward_noalloc.restype = ci
        lib.pa_v2_forward_noalloc.argtypes = _FWD_ARGS[:17] + [vp]
        lib.pa_forward.restype = ci
        lib.pa_forward.argtypes = _FWD_ARGS + [ctypes.POINTER(pa_options_t)]
        lib.pa_chunks_forward.restype = ci
        lib.pa_chunks_forward.argtypes = ([vp] * 7 + [ci] * 10 +
                                          [ctypes.c_float, ci, ci, vp, cs, vp,
                                           ctypes.POINTER(pa_options_t)])
        lib.pa_host_staging_bytes.restype = cs
        lib.pa_host_staging_bytes.argtypes = [ci] * 5
        lib.pa_forward_host.restype = ci
        lib.pa_forward_host.argtypes = (_FWD_ARGS[:17] + [vp, cs] + _FWD_ARGS[17:] +
                                        [ctypes.POINTER(pa_options_t)])
        lib.pa_choose_v2.restype = ci
        lib.pa_choose_v2.argtypes = [ci] * 5
        lib.pa_choose_v2_chunks.restype = ci
        lib.pa_choose_v2_chunks.argtypes = [ci] * 8
        lib.pa_read_device_status.restype = ci
        lib.pa_read_device_status.argtypes = [vp, vp]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_status_string.argtypes = [ci]
        lib.pa_last_cuda_error.restype = ctypes.c_char_p
        lib.pa_last_cuda_error.argtypes = []
        lib.pa_version.restype = ci
        lib.pa_version.argtypes = []
        _lib = lib
        return lib


def status_text(status: int) -> str:
    return load_library().pa_status_string(int(status)).decode()


def _check(status: int, what: str) -> int:
    if status != PA_OK:
        if status == PA_ERR_CUDA:
            what = f"{what} [{load_library().pa_last_cuda_error().decode()}]"
        raise PAError(status, what)
    return status


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None) -> int:
    if t is None:
        return 0
    if not t.is_contiguous():
        raise ValueError("libpa takes contiguous tensors")
    return t.data_ptr()


# ---------------------------------------------------------------------------
# Workspace

def pa_workspace_bytes(num_seqs: int, num_heads: int, head_size: int, max_seq_len: int,
                       partition_size: int) -> int:
    return int(load_library().pa_workspace_bytes(num_seqs, num_heads, head_size,
                                                 max_seq_len, partition_size))


def pa_workspace_layout(num_seqs: int, num_heads: int, head_size: int, max_seq_len: int,
                        partition_size: int) -> tuple[int, int, int, int, int]:
    off = (ctypes.c_size_t * 5)()
    _check(load_library().pa_workspace_layout(num_seqs, num_heads, head_size, max_seq_len,
                                              partition_size, off), "pa_workspace_layout")
    return tuple(int(x) for x in off)


def pa_workspace_init(workspace: torch.Tensor, stream=None) -> None:
    _check(load_library().pa_workspace_init(_ptr(workspace), workspace.numel() *
                                            workspace.element_size(),
                                            _stream_handle(stream)), "pa_workspace_init")


def alloc_workspace(num_seqs: int, num_heads: int, head_size: int, max_seq_len: int,
                    partition_size: int, device=None, stream=None) -> torch.Tensor:
    """A zero-status workspace large enough for V2 (and so for V1)."""
    n = max(pa_workspace_bytes(num_seqs, num_heads, head_size, max_seq_len, partition_size), 256)
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    pa_workspace_init(ws, stream)
    return ws


# ---------------------------------------------------------------------------
# Forward calls

def _fwd_args(out, query, key_cache, value_cache, block_tables, seq_lens, scale,
              partition_size, workspace, max_seq_len, stream):
    if query.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {query.dtype}")
    B, H, D = query.shape
    nb, hkv, bs, d2 = key_cache.shape
    if max_seq_len is None:
        max_seq_len = block_tables.shape[1] * bs
    return (_ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
            _ptr(seq_lens), B, H, hkv, D, nb, bs, block_tables.shape[1], int(max_seq_len),
            float(scale), int(partition_size), _DTYPES[query.dtype], _ptr(workspace),
            workspace.numel() * workspace.element_size(), _stream_handle(stream))


def pa_v1_forward(out, query, key_cache, value_cache, block_tables, seq_lens, scale,
                  partition_size, workspace, max_seq_len=None, stream=None) -> None:
    """V1: one pass over each whole sequence (see include/pa.h)."""
    _check(load_library().pa_v1_forward(*_fwd_args(
        out, query, key_cache, value_cache, block_tables, seq_lens, scale, partition_size,
        workspace, max_seq_len, stream)), "pa_v1_forward")


def pa_v2_forward(out, query, key_cache, value_cache, block_tables, seq_lens, scale,
                  partition_size, workspace, max_seq_len=None, stream=None) -> None:
    """V2: partition kernel + log-sum-exp reduce (see include/pa.h)."""
    _check(load_library().pa_v2_forward(*_fwd_args(
        out, query, key_cache, value_cache, block_tables, seq_lens, scale, partition_size,
        workspace, max_seq_len, stream)), "pa_v2_forward")


def pa_v2_partials(query, key_cache, value_cache, block_tables, seq_lens, scale,
                   partition_size, workspace, part_begin=0, part_end=2 ** 31 - 1,
                   max_seq_len=None, stream=None) -> None:
    """Phase 1 of V2 over partitions [part_begin, part_end) of every sequence,
    into their workspace slots (see include/pa.h)."""
    a = _fwd_args(query, query, key_cache, value_cache, block_tables, seq_lens, scale,
                  partition_size, workspace, max_seq_len, stream)
    _check(load_library().pa_v2_partials(*a[1:17], int(part_begin), int(part_end), *a[17:]),
           "pa_v2_partials")


def pa_v2_combine(out, seq_lens, partition_size, workspace, max_seq_len, num_kv_heads=None,
                  stream=None) -> None:
    """Phase 2 of V2 alone: out [B, H, D] from the partials in the workspace
    (see include/pa.h).  ``num_kv_heads`` is unused (Phase 2 works per query
    head) and accepted for symmetry with the forward calls."""
    if out.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {out.dtype}")
    B, H, D = out.shape
    _check(load_library().pa_v2_combine(
        _ptr(out), _ptr(seq_lens), B, H, D, int(max_seq_len), int(partition_size),
        _DTYPES[out.dtype], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream_handle(stream)), "pa_v2_combine")


def pa_v2_forward_noalloc(out, query, key_cache, value_cache, block_tables, seq_lens, scale,
                          partition_size, max_seq_len=None, stream=None) -> None:
    """V2 without a caller workspace, for callers that cannot allocate device
    memory: scratch comes from the library's fixed 32 MiB device array (one
    per GPU, shared by all calls; overlapping calls race)."""
    args = _fwd_args(out, query, key_cache, value_cache, block_tables, seq_lens, scale,
                     partition_size, torch.empty(0, dtype=torch.uint8), max_seq_len, stream)
    _check(load_library().pa_v2_forward_noalloc(*args[:17], args[19]),
           "pa_v2_forward_noalloc")


def _event_handle(ev):
    """The cudaEvent_t of a torch.cuda.Event (or a raw handle), or None."""
    if ev is None:
        return None
    h = ev.cuda_event if hasattr(ev, "cuda_event") else int(ev)
    if not h:
        raise ValueError("phase1_event has no CUDA event yet (torch creates it at the "
                         "first record(); record it once before passing it)")
    return h


def pa_forward(out, query, key_cache, value_cache, block_tables, seq_lens, scale,
               partition_size, workspace, max_seq_len=None, stream=None, variant=PA_VARIANT_AUTO,
               math=PA_MATH_AUTO, num_stages=0, debug_flags=0, wait_limit_ns=0,
               phase1_event=None, ctas_per_sm=0, fuse_partitions=0) -> None:
    """V1 or V2 chosen by pa_choose_v2, or forced through the options.
    ``phase1_event`` (a torch.cuda.Event) is recorded between V2's two kernels."""
    opts = pa_options_t(variant, math, num_stages, debug_flags, wait_limit_ns,
                        _event_handle(phase1_event), ctas_per_sm, fuse_partitions)
    _check(load_library().pa_forward(*_fwd_args(
        out, query, key_cache, value_cache, block_tables, seq_lens, scale, partition_size,
        workspace, max_seq_len, stream), ctypes.byref(opts)), "pa_forward")


def pa_chunks_forward(out, query, key_cache, value_cache, block_tables, seq_lens, q_start,
                      scale, partition_size, workspace, max_seq_len=None, max_chunk=None,
                      stream=None, variant=PA_VARIANT_AUTO, num_stages=0, ctas_per_sm=0,
                      phase1_event=None, debug_flags=0, wait_limit_ns=0,
                      share_kv=0) -> None:
    """Multi-token queries over the paged cache (see include/pa.h): query and
    out [num_rows, H, D]; the chunk of sequence s is rows q_start[s] ..
    q_start[s+1]-1 (int32 on the device), its last tokens.  max_chunk bounds
    the chunk lengths (default: max_seq_len)."""
    if query.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {query.dtype}")
    R, H, D = query.shape
    nb, hkv, bs, d2 = key_cache.shape
    B = seq_lens.numel()
    if q_start.numel() != B + 1 or q_start.dtype != torch.int32:
        raise ValueError("q_start must be int32 [num_seqs + 1]")
    if max_seq_len is None:
        max_seq_len = block_tables.shape[1] * bs
    mc = int(max_chunk) if max_chunk is not None else int(max_seq_len)
    opts = pa_options_t(variant, PA_MATH_AUTO, num_stages, debug_flags, wait_limit_ns,
                        _event_handle(phase1_event), ctas_per_sm, 0, share_kv)
    _check(load_library().pa_chunks_forward(
        _ptr(out), _ptr(query), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        _ptr(seq_lens), _ptr(q_start), B, R, mc, H, hkv, D, nb, bs, block_tables.shape[1],
        int(max_seq_len), float(scale), int(partition_size), _DTYPES[query.dtype],
        _ptr(workspace), workspace.numel() * workspace.element_size(), _stream_handle(stream),
        ctypes.byref(opts)), "pa_chunks_forward")


def pa_host_staging_bytes(num_seqs: int, num_heads: int, head_size: int,
                          max_blocks_per_seq: int, dtype) -> int:
    """Device bytes pa_forward_host stages the per-step data in."""
    code = _DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load_library().pa_host_staging_bytes(num_seqs, num_heads, head_size,
                                                    max_blocks_per_seq, code))


def alloc_staging(query, block_tables, device=None) -> torch.Tensor:
    """A device staging buffer for pa_forward_host calls of this shape."""
    B, H, D = query.shape
    n = pa_host_staging_bytes(B, H, D, block_tables.shape[1], query.dtype)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def pa_forward_host(out_host, query_host, key_cache, value_cache, block_tables_host,
                    seq_lens_host, scale, partition_size, staging, workspace, max_seq_len=None,
                    stream=None, variant=PA_VARIANT_AUTO, math=PA_MATH_AUTO, num_stages=0,
                    ctas_per_sm=0, fuse_partitions=0) -> None:
    """pa_forward with the query, block tables, lengths and output in host
    memory (pinned for asynchronous copies): one C-ABI call enqueues the
    host-to-device copies into ``staging``, the kernels and the copy of the
    output back to ``out_host``.  Synchronise the stream before reading it."""
    for t in (out_host, query_host, block_tables_host, seq_lens_host):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("pa_forward_host takes contiguous host tensors for "
                             "out, query, block_tables and seq_lens")
    opts = pa_options_t(variant, math, num_stages, 0, 0, None, ctas_per_sm, fuse_partitions)
    args = _fwd_args(out_host, query_host, key_cache, value_cache, block_tables_host,
                     seq_lens_host, scale, partition_size, workspace, max_seq_len, stream)
    _check(load_library().pa_forward_host(
        *args[:17], _ptr(staging), staging.numel() * staging.element_size(), *args[17:],
        ctypes.byref(opts)), "pa_forward_host")


def pa_choose_v2(num_seqs: int, num_kv_heads: int, max_seq_len: int, partition_size: int,
                 sm_count: int) -> int:
    return int(load_library().pa_choose_v2(num_seqs, num_kv_heads, max_seq_len,
                                           partition_size, sm_count))


def pa_choose_v2_chunks(num_seqs: int, num_heads: int, num_kv_heads: int, head_size: int,
                        max_chunk: int, max_seq_len: int, partition_size: int,
                        sm_count: int) -> int:
    return int(load_library().pa_choose_v2_chunks(num_seqs, num_heads, num_kv_heads, head_size,
                                                  max_chunk, max_seq_len, partition_size,
                                                  sm_count))


def pa_read_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise the stream, return and clear the kernels' status word."""
    return int(load_library().pa_read_device_status(_ptr(workspace), _stream_handle(stream)))


def pa_status_string(status: int) -> str:
    return status_text(status)


def pa_last_cuda_error() -> str:
    return load_library().pa_last_cuda_error().decode()


def pa_version() -> int:
    return int(load_library().pa_version())
