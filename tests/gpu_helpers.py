"""Helpers for the GPU tests: run a workload through libpa's C ABI (via the
binding) and compare with the CPU fp64 oracle element by element."""
from __future__ import annotations

import functools

import numpy as np
import torch

import oracle
import paged_decode_attention_v2_gb300 as pa
import workloads

# The parity bar: bf16/f16 max |err| <= 4e-3 + 1e-2 |ref|; f32 max |err| <= 1e-5.
TOL = {torch.float32: (1e-5, 0.0), torch.bfloat16: (4e-3, 1e-2), torch.float16: (4e-3, 1e-2)}


@functools.lru_cache(maxsize=8)
def config_case(name, partition_size=None):
    return workloads.config_case(name, partition_size)


_REF_CACHE = {}


def reference(case):
    key = id(case)
    if key not in _REF_CACHE:
        _REF_CACHE[key] = (case, oracle.attention(case.query, case.key_cache, case.value_cache,
                                                  case.block_tables, case.seq_lens, case.scale))
    return _REF_CACHE[key][1]


class DeviceCase:
    """A DecodeCase copied to the GPU, with a V2-sized workspace."""

    def __init__(self, case, device="cuda"):
        self.case = case
        self.q = case.query.to(device)
        self.kc = case.key_cache.to(device)
        self.vc = case.value_cache.to(device)
        self.bt = case.block_tables.to(device)
        self.sl = case.seq_lens.to(device)
        self.max_seq_len = case.max_seq_len
        self.ws = pa.alloc_workspace(case.num_seqs, case.num_heads, case.head_size,
                                     self.max_seq_len, case.partition_size, device=device)

    def run(self, variant=pa.PA_VARIANT_AUTO, math=pa.PA_MATH_AUTO, partition_size=None,
            num_stages=0, stream=None, fill=float("nan"), check_status=True, **kw):
        P = partition_size or self.case.partition_size
        if pa.pa_workspace_bytes(self.case.num_seqs, self.case.num_heads, self.case.head_size,
                                 self.max_seq_len, P) > self.ws.numel():
            self.ws = pa.alloc_workspace(self.case.num_seqs, self.case.num_heads,
                                         self.case.head_size, self.max_seq_len, P)
        out = torch.full_like(self.q, fill)
        pa.pa_forward(out, self.q, self.kc, self.vc, self.bt, self.sl, self.case.scale, P,
                      self.ws, max_seq_len=self.max_seq_len, stream=stream, variant=variant,
                      math=math, num_stages=num_stages, **kw)
        if check_status:
            st = pa.pa_read_device_status(self.ws, stream)
            assert st == pa.PA_OK, pa.pa_status_string(st)
        return out

    def partials(self, partition_size=None):
        """(max_logits, exp_sums, tmp_out) of the last V2 run, as float64."""
        c = self.case
        P = partition_size or c.partition_size
        off = pa.pa_workspace_layout(c.num_seqs, c.num_heads, c.head_size, self.max_seq_len, P)
        n = -(-self.max_seq_len // P)
        B, H, D = c.num_seqs, c.num_heads, c.head_size
        f = self.ws.view(torch.uint8)

        def view(o, count, shape):
            return f[o:o + count * 4].view(torch.float32).reshape(shape).double().cpu().numpy()
        return (view(off[1], B * H * n, (B, H, n)), view(off[2], B * H * n, (B, H, n)),
                view(off[3], B * H * n * D, (B, H, n, D)))


def assert_close(got, ref, dtype, what=""):
    atol, rtol = TOL[dtype]
    g = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; worst at {idx}: "
            f"got {g[idx]!r} ref {ref[idx]!r} (|err| {err[idx]:.3e} > {bound[idx]:.3e})")
    return float(err.max()) if err.size else 0.0
