"""CPU fp64 oracle for paged decode attention (ctypes wrapper over pa_oracle.c).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product path (``libpa`` and ``paged_decode_attention_v2_gb300``)
never imports it, and it imports nothing from the product.

Every function here follows the "paged_attention_v2" commit note (project_6,
commit 96f4baf "Dockerfile", section "Implementation"):

* ``attention``         the exact result the method reaches: one softmax over
                        all L tokens of each sequence, gathered through the
                        block table (no partitioning);
* ``partials``          "Phase 1: Per-partition attention" (max_logits,
                        exp_sums, normalised tmp_output per partition);
* ``combine``           "Phase 2: Cross-partition reduction (log-sum-exp)".

Parity pins: every function is pinned by ``tests/test_oracle_pins.py`` against
closed forms, library special cases, brute force on tiny inputs and the
partition-combine invariant; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

ORC_F64, ORC_F32, ORC_BF16, ORC_F16 = 0, 1, 2, 3
_DTYPE_CODE = {
    torch.float64: ORC_F64,
    torch.float32: ORC_F32,
    torch.bfloat16: ORC_BF16,
    torch.float16: ORC_F16,
}

_lock = threading.Lock()
_lib = None


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile ``src`` (plain C, OpenMP) into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           *extra_flags, src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build liboracle.so in-tree if missing or older than its source."""
    with _lock:
        if (force or not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            compile_oracle()
    return _LIB_PATH


def _declare(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    vp = ctypes.c_void_p
    i32p = ctypes.c_void_p
    ci, cd = ctypes.c_int, ctypes.c_double
    lib.pa_oracle_max_threads.restype = ci
    lib.pa_oracle_max_threads.argtypes = []
    lib.pa_oracle_widen.restype = None
    lib.pa_oracle_widen.argtypes = [dp, vp, ci, ctypes.c_size_t]
    lib.pa_oracle_attention.restype = None
    lib.pa_oracle_attention.argtypes = [
        dp, vp, vp, vp, ci, i32p, i32p, ci, ci, ci, ci, ci, ci, cd, ci, dp, ci]
    lib.pa_oracle_attention_pairs.restype = None
    lib.pa_oracle_attention_pairs.argtypes = [
        dp, i32p, ci, vp, vp, vp, ci, i32p, i32p, ci, ci, ci, ci, ci, ci, cd,
        ci, dp, ci]
    lib.pa_oracle_partials.restype = None
    lib.pa_oracle_partials.argtypes = [
        dp, dp, dp, vp, vp, vp, ci, i32p, i32p, ci, ci, ci, ci, ci, ci, cd, ci,
        ci, ci, dp]
    lib.pa_oracle_combine.restype = None
    lib.pa_oracle_combine.argtypes = [dp, dp, dp, dp, i32p, ci, ci, ci, ci]
    lib.pa_oracle_query_chunks.restype = None
    lib.pa_oracle_query_chunks.argtypes = [
        dp, vp, vp, vp, ci, i32p, i32p, i32p, ci, ci, ci, ci, ci, ci, cd, ci, dp, ci]
    return lib


def load_library(path: str):
    """Load an oracle shared library (the real one or a test-built variant)."""
    return _declare(ctypes.CDLL(path))


def _get_lib():
    global _lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _cpu_contig(t: torch.Tensor) -> torch.Tensor:
    if t.device.type != "cpu":
        raise ValueError("the oracle takes CPU tensors only")
    return t.contiguous()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPE_CODE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DTYPE_CODE[t.dtype]


def _common(q, k_cache, v_cache, block_tables, seq_lens):
    q, k_cache, v_cache = (_cpu_contig(x) for x in (q, k_cache, v_cache))
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise ValueError("q, k_cache and v_cache must share one dtype")
    bt = _cpu_contig(block_tables).to(torch.int32)
    sl = _cpu_contig(seq_lens).to(torch.int32)
    B, H, D = q.shape
    nb, Hkv, bs, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes do not match the query")
    if H % Hkv:
        raise ValueError("num_heads must be a multiple of num_kv_heads")
    if bt.shape[0] != B or sl.shape[0] != B:
        raise ValueError("block_tables / seq_lens batch mismatch")
    return q, k_cache, v_cache, bt, sl, (B, H, Hkv, D, bs, bt.shape[1])


def max_threads(nthreads: int = 0) -> int:
    lib = _get_lib()
    return nthreads if nthreads > 0 else lib.pa_oracle_max_threads()


def widen(t: torch.Tensor, lib=None) -> np.ndarray:
    """Exact widening of f64/f32/bf16/f16 elements to float64 (flat)."""
    lib = lib or _get_lib()
    t = _cpu_contig(t)
    out = np.empty(t.numel(), dtype=np.float64)
    lib.pa_oracle_widen(_dptr(out), ctypes.c_void_p(t.data_ptr()),
                        _dtype_code(t), t.numel())
    return out


def attention(q, k_cache, v_cache, block_tables, seq_lens, scale: float,
              nthreads: int = 0, lib=None) -> np.ndarray:
    """Exact paged softmax attention, fp64: returns out [B, H, D]."""
    lib = lib or _get_lib()
    q, kc, vc, bt, sl, (B, H, Hkv, D, bs, mb) = _common(
        q, k_cache, v_cache, block_tables, seq_lens)
    maxL = max(int(sl.max().item()) if B else 0, 1)
    nt = nthreads if nthreads > 0 else lib.pa_oracle_max_threads()
    scratch = np.empty(nt * maxL, dtype=np.float64)
    out = np.zeros((B, H, D), dtype=np.float64)
    lib.pa_oracle_attention(
        _dptr(out), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(vc.data_ptr()), _dtype_code(q),
        ctypes.c_void_p(bt.data_ptr()), ctypes.c_void_p(sl.data_ptr()),
        B, H, Hkv, D, bs, mb, float(scale), nt, _dptr(scratch), maxL)
    return out


def attention_pairs(pairs, q, k_cache, v_cache, block_tables, seq_lens,
                    scale: float, nthreads: int = 0, lib=None) -> np.ndarray:
    """The same definition for selected (seq, head) pairs: out [n, D]."""
    lib = lib or _get_lib()
    q, kc, vc, bt, sl, (B, H, Hkv, D, bs, mb) = _common(
        q, k_cache, v_cache, block_tables, seq_lens)
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    if pr.size and (pr[:, 0].min() < 0 or pr[:, 0].max() >= B
                    or pr[:, 1].min() < 0 or pr[:, 1].max() >= H):
        raise ValueError("pair out of range")
    maxL = max(int(sl.max().item()) if B else 0, 1)
    nt = nthreads if nthreads > 0 else lib.pa_oracle_max_threads()
    scratch = np.empty(nt * maxL, dtype=np.float64)
    out = np.zeros((pr.shape[0], D), dtype=np.float64)
    lib.pa_oracle_attention_pairs(
        _dptr(out), ctypes.c_void_p(pr.ctypes.data), pr.shape[0],
        ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(vc.data_ptr()), _dtype_code(q),
        ctypes.c_void_p(bt.data_ptr()), ctypes.c_void_p(sl.data_ptr()),
        B, H, Hkv, D, bs, mb, float(scale), nt, _dptr(scratch), maxL)
    return out


def query_chunks(q, k_cache, v_cache, block_tables, seq_lens, q_start, scale: float,
                 nthreads: int = 0, lib=None) -> np.ndarray:
    """Multi-token queries over the paged cache (the causal reading in
    pa_oracle.c): q [rows, H, D], the chunk of sequence s being rows
    q_start[s] .. q_start[s+1]-1, its last tokens.  Returns out [rows, H, D]."""
    lib = lib or _get_lib()
    q, kc, vc = (_cpu_contig(x) for x in (q, k_cache, v_cache))
    if not (q.dtype == kc.dtype == vc.dtype):
        raise ValueError("q, k_cache and v_cache must share one dtype")
    bt = _cpu_contig(block_tables).to(torch.int32)
    sl = _cpu_contig(seq_lens).to(torch.int32)
    qs = _cpu_contig(torch.as_tensor(q_start)).to(torch.int32)
    R, H, D = q.shape
    nb, Hkv, bs, D2 = kc.shape
    B = sl.numel()
    if D2 != D or qs.numel() != B + 1 or int(qs[-1]) != R or H % Hkv:
        raise ValueError("inconsistent shapes")
    maxL = max(int(sl.max().item()) if B else 0, 1)
    nt = nthreads if nthreads > 0 else lib.pa_oracle_max_threads()
    scratch = np.empty(nt * maxL, dtype=np.float64)
    out = np.zeros((R, H, D), dtype=np.float64)
    lib.pa_oracle_query_chunks(
        _dptr(out), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(kc.data_ptr()),
        ctypes.c_void_p(vc.data_ptr()), _dtype_code(q), ctypes.c_void_p(bt.data_ptr()),
        ctypes.c_void_p(sl.data_ptr()), ctypes.c_void_p(qs.data_ptr()), B, H, Hkv, D, bs,
        bt.shape[1], float(scale), nt, _dptr(scratch), maxL)
    return out


def num_partitions(seq_lens, partition_size: int) -> np.ndarray:
    sl = np.asarray(seq_lens, dtype=np.int64)
    return ((sl + partition_size - 1) // partition_size).astype(np.int32)


def partials(q, k_cache, v_cache, block_tables, seq_lens, scale: float,
             partition_size: int, max_parts: int | None = None,
             nthreads: int = 0, lib=None):
    """Phase 1 partials: (max_logits [B,H,Np], exp_sums [B,H,Np],
    tmp_out [B,H,Np,D]); entries of partitions past a sequence's end are NaN."""
    lib = lib or _get_lib()
    q, kc, vc, bt, sl, (B, H, Hkv, D, bs, mb) = _common(
        q, k_cache, v_cache, block_tables, seq_lens)
    if max_parts is None:
        max_parts = int(num_partitions(sl.numpy(), partition_size).max()) if B else 0
    max_parts = max(int(max_parts), 1)
    ml = np.full((B, H, max_parts), np.nan)
    es = np.full((B, H, max_parts), np.nan)
    to = np.full((B, H, max_parts, D), np.nan)
    nt = nthreads if nthreads > 0 else lib.pa_oracle_max_threads()
    scratch = np.empty(nt * partition_size, dtype=np.float64)
    lib.pa_oracle_partials(
        _dptr(ml), _dptr(es), _dptr(to), ctypes.c_void_p(q.data_ptr()),
        ctypes.c_void_p(kc.data_ptr()), ctypes.c_void_p(vc.data_ptr()),
        _dtype_code(q), ctypes.c_void_p(bt.data_ptr()),
        ctypes.c_void_p(sl.data_ptr()), B, H, Hkv, D, bs, mb, float(scale),
        int(partition_size), max_parts, nt, _dptr(scratch))
    return ml, es, to


def combine(max_logits, exp_sums, tmp_out, num_parts, lib=None) -> np.ndarray:
    """Phase 2 log-sum-exp combine: out [B, H, D]."""
    lib = lib or _get_lib()
    ml = np.ascontiguousarray(max_logits, dtype=np.float64)
    es = np.ascontiguousarray(exp_sums, dtype=np.float64)
    to = np.ascontiguousarray(tmp_out, dtype=np.float64)
    npt = np.ascontiguousarray(num_parts, dtype=np.int32)
    B, H, max_parts, D = to.shape
    out = np.zeros((B, H, D), dtype=np.float64)
    lib.pa_oracle_combine(_dptr(out), _dptr(ml), _dptr(es), _dptr(to),
                          ctypes.c_void_p(npt.ctypes.data), B, H, D, max_parts)
    return out
