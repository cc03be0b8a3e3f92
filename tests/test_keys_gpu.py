"""The tcgen05 kernel of small items (the keys on the MMA's M, at most 16
query rows an item, D 128, 16-bit; taken with PA_DEBUG_TCGEN05_KEYS) against
the oracle, element by element: decode with groups of 1-16 query heads and
short query chunks; V1 and V2, page sizes
8-64, partition sizes that are and are not multiples of its 128-key stage,
empty, one-token and stage-edge lengths; Phase 1's partials; keys whose
logits grow along the sequence, so that the lazily raised row maxima move
in the middle of items; bit-identical results under a shuffled pool; the
same inputs on the mma.sync kernels within the same bar."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_v2_gb300 as pa
import workloads
from gpu_helpers import DeviceCase, assert_close, reference

pytestmark = pytest.mark.gpu

KEYS = pa.PA_DEBUG_TCGEN05_KEYS

DECODE_CASES = [  # dtype, G, Hkv, bs, P, lens, flags
    (torch.bfloat16, 16, 2, 16, 512, [1, 127, 128, 129, 700, 2000, 4097, 0], KEYS),
    (torch.float16, 12, 1, 8, 192, [300, 1, 1000, 65, 0], KEYS),
    (torch.bfloat16, 9, 3, 64, 256, [5000, 64, 128, 3], KEYS),
    (torch.float16, 16, 1, 32, 64, [1500, 63, 257], KEYS),
    (torch.bfloat16, 8, 4, 32, 512, [1, 513, 2048, 777], KEYS),
    (torch.float16, 1, 8, 16, 64, [100, 1000, 0], KEYS),
    (torch.bfloat16, 4, 2, 16, 512, [3000, 17, 384], KEYS),
]


def _ids(cases):
    return [f"{str(c[0])[6:]}-G{c[1]}-bs{c[3]}-P{c[4]}" for c in cases]


@pytest.mark.parametrize("dtype,G,Hkv,bs,P,lens,flags", DECODE_CASES, ids=_ids(DECODE_CASES))
@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2, pa.PA_VARIANT_AUTO],
                         ids=["v1", "v2", "auto"])
def test_keys_decode_matches_oracle(dtype, G, Hkv, bs, P, lens, flags, variant):
    case = workloads.make_case("keys", 5000 + G * 7 + bs + P, len(lens), G * Hkv, Hkv, 128, dtype,
                               bs, lens, partition_size=P, extra_blocks=5, k_mult=2.0)
    ref = reference(case)
    dc = DeviceCase(case)
    for _ in range(2):  # the work counters return to zero for the next launch
        assert_close(dc.run(variant=variant, debug_flags=flags), ref, dtype,
                     f"keys kernel v{variant}")


@pytest.mark.parametrize("dtype,G,Hkv,bs,P,lens,flags", DECODE_CASES[:3], ids=_ids(DECODE_CASES[:3]))
def test_keys_and_mma_sync_kernels_agree_with_the_oracle(dtype, G, Hkv, bs, P, lens, flags):
    case = workloads.make_case("keys_vs", 5100 + G, len(lens), G * Hkv, Hkv, 128, dtype, bs, lens,
                               partition_size=P, extra_blocks=5)
    ref = reference(case)
    dc = DeviceCase(case)
    for f in (flags, pa.PA_DEBUG_NO_TCGEN05):
        for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
            assert_close(dc.run(variant=variant, debug_flags=f), ref, dtype, f"flags {f} v{variant}")


@pytest.mark.parametrize("dtype,G,P,flags", [(torch.bfloat16, 16, 512, KEYS),
                                             (torch.float16, 12, 192, KEYS),
                                             (torch.bfloat16, 8, 256, KEYS)])
def test_keys_phase1_partials_match_oracle(dtype, G, P, flags):
    """Phase 1's records (the true maximum in natural-log units, the sum of
    exponentials relative to it, the normalised partial output) against the
    oracle's partials, at the bounds the mma.sync kernels are held to: a
    logit differs by the fp32 accumulation of D products, a weight by its
    rounding to the input type before the PV product."""
    D = 128
    lens = [1, P - 3, P, P + 1, 3 * P + 100, 129]
    case = workloads.make_case("keys_partials", 5200 + G, len(lens), 2 * G, 2, D, dtype, 16, lens,
                               partition_size=P, k_mult=3.0)
    dc = DeviceCase(case)
    dc.run(variant=pa.PA_VARIANT_V2, debug_flags=flags)
    ml, es, to = dc.partials()
    rml, res, rto = oracle.partials(case.query, case.key_cache, case.value_cache,
                                    case.block_tables, case.seq_lens, case.scale, P)
    live = ~np.isnan(rml)
    u = 2.0 ** -24
    qn = case.query.double().norm(dim=-1).numpy()
    kn = float(case.key_cache.double().norm(dim=-1).max())
    eb = (D * u * case.scale * qn * kn)[:, :, None] * np.ones_like(rml)
    assert np.all(np.abs(ml[live] - rml[live]) <= eb[live] + 8 * u * np.abs(rml[live]))
    rho = {torch.bfloat16: 2.0 ** -9, torch.float16: 2.0 ** -11}[dtype]
    bound_es = res[live] * (rho + 2 * eb[live] + P * u)
    assert np.all(np.abs(es[live] - res[live]) <= bound_es)
    assert_close(torch.from_numpy(to[live]), rto[live], dtype, "tmp_out")


def _ramped(case, rate):
    """The case with every key of sequence s scaled by 1 + rate * j / L_s at
    its position j: logits that grow along the sequence, so that a row's
    maximum keeps rising from stage to stage."""
    k = case.key_cache.double().clone()
    bs = case.block_size
    for s, L in enumerate(case.seq_lens.tolist()):
        for j in range(L):
            blk = int(case.block_tables[s, j // bs])
            k[blk, :, j % bs, :] *= 1.0 + rate * j / max(L, 1)
    return dataclasses.replace(case, key_cache=k.to(case.key_cache.dtype))


@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2], ids=["v1", "v2"])
def test_keys_rising_maxima_rescale_in_the_middle_of_items(variant):
    base = workloads.make_case("keys_ramp", 5300, 4, 32, 2, 128, torch.bfloat16, 16,
                               [3000, 1800, 640, 4097], partition_size=1024, k_mult=2.5)
    case = _ramped(base, 4.0)
    ref = reference(case)
    assert_close(DeviceCase(case).run(variant=variant, debug_flags=KEYS), ref, torch.bfloat16,
                 f"ramp v{variant}")


def test_keys_pool_permutation_is_bit_identical():
    lens = [9, 600, 2000, 4097, 777, 0]
    case = workloads.make_case("keys_perm", 5400, len(lens), 32, 2, 128, torch.bfloat16, 16, lens,
                               partition_size=512, extra_blocks=20)
    a, b = DeviceCase(case), DeviceCase(workloads.permute_pool(case, 9))
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        assert torch.equal(a.run(variant=variant, debug_flags=KEYS).view(torch.int16),
                           b.run(variant=variant, debug_flags=KEYS).view(torch.int16))


CHUNK_CASES = [  # dtype, G, Hkv, bs, P, lens, qlens
    (torch.bfloat16, 8, 2, 16, 512, [100, 700, 2000, 40, 300, 5], [1, 2, 2, 1, 0, 2]),
    (torch.float16, 16, 1, 8, 256, [900, 1700, 64], [1, 1, 1]),
    (torch.bfloat16, 4, 2, 32, 512, [1500, 33, 2600], [4, 3, 4]),
    (torch.float16, 2, 4, 64, 192, [3000, 129, 8], [8, 5, 8]),
]


@pytest.mark.parametrize("dtype,G,Hkv,bs,P,lens,qlens", CHUNK_CASES,
                         ids=[f"{str(c[0])[6:]}-G{c[1]}-bs{c[3]}-P{c[4]}" for c in CHUNK_CASES])
@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2], ids=["v1", "v2"])
def test_keys_chunks_match_oracle(dtype, G, Hkv, bs, P, lens, qlens, variant):
    """Query chunks of up to 16 rows per KV head on the kernel of small items
    (forced): causal rows, a row's keys ending inside a stage, row groups of
    16 / G tokens."""
    H = G * Hkv
    c = workloads.make_case("keys_chunks", 5500 + G + P, len(lens), H, Hkv, 128, dtype, bs, lens,
                            partition_size=P, extra_blocks=3, k_mult=2.0)
    g = torch.Generator().manual_seed(5500 + G)
    q = torch.randn(sum(qlens), H, 128, generator=g).to(dtype)
    qs = torch.tensor(np.concatenate([[0], np.cumsum(qlens)]), dtype=torch.int32)
    ref = oracle.query_chunks(q, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, qs,
                              c.scale)
    R = q.shape[0]
    ws = pa.alloc_workspace(R, H, 128, c.max_seq_len, P)
    out = torch.full((R, H, 128), float("nan"), dtype=dtype, device="cuda")
    args = (q.cuda(), c.key_cache.cuda(), c.value_cache.cuda(), c.block_tables.cuda(),
            c.seq_lens.cuda(), qs.cuda())
    for _ in range(2):
        pa.pa_chunks_forward(out, *args, c.scale, P, ws, max_seq_len=c.max_seq_len,
                             max_chunk=max(qlens), variant=variant, debug_flags=KEYS)
        assert pa.pa_read_device_status(ws) == pa.PA_OK
        assert_close(out, ref, dtype, f"keys chunks v{variant}")


def _g16_case():
    return workloads.make_case("keys_faults", 5600, 4, 32, 2, 128, torch.bfloat16, 16,
                               [100, 1000, 2500, 7], partition_size=512, extra_blocks=8)


@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2], ids=["v1", "v2"])
def test_keys_bounded_wait_runs_out_and_context_survives(variant):
    """Every softmax warp waits on a barrier that nothing releases: the MMA
    thread and the producer give up in turn, the tensor memory is freed,
    PA_ERR_DEVICE_TIMEOUT is reported and the next call is right."""
    case = _g16_case()
    dc = DeviceCase(case)
    out = torch.zeros_like(dc.q)
    pa.pa_forward(out, dc.q, dc.kc, dc.vc, dc.bt, dc.sl, case.scale, 512, dc.ws,
                  max_seq_len=dc.max_seq_len, variant=variant,
                  debug_flags=pa.PA_DEBUG_STALL_CONSUMERS | KEYS, wait_limit_ns=200_000)
    assert pa.pa_read_device_status(dc.ws) == pa.PA_ERR_DEVICE_TIMEOUT
    torch.cuda.synchronize()
    assert_close(dc.run(variant=variant, debug_flags=KEYS), reference(case), torch.bfloat16,
                 "after a timeout")


@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V1, pa.PA_VARIANT_V2], ids=["v1", "v2"])
def test_keys_out_of_range_block_id_is_reported(variant):
    case = _g16_case()
    dc = DeviceCase(case)
    bad = dc.bt.clone()
    bad[1, 10] = case.num_blocks + 5
    bad[2, 3] = -7
    out = torch.empty_like(dc.q)
    pa.pa_forward(out, dc.q, dc.kc, dc.vc, bad, dc.sl, case.scale, 512, dc.ws,
                  max_seq_len=dc.max_seq_len, variant=variant, debug_flags=KEYS)
    assert pa.pa_read_device_status(dc.ws) == pa.PA_ERR_DEVICE_BAD_INPUT
    assert_close(dc.run(variant=variant, debug_flags=KEYS), reference(case), torch.bfloat16,
                 "after bad input")


@pytest.mark.parametrize("variant", [pa.PA_VARIANT_V2, pa.PA_VARIANT_V1], ids=["v2", "v1"])
def test_keys_gqa16_full_size(variant):
    """At full size on the 16-head-group decode workload (the 256-sequence
    lengths and cache shape with 32 query / 2 KV heads): every output against
    the oracle, V2 and V1."""
    c = dict(workloads.CONFIGS["c4_batch256"])
    c.pop("index")
    c["num_kv_heads"] = 2
    case = workloads.make_case("gqa16", workloads.SEED_BASE + 77, **c)
    assert_close(DeviceCase(case).run(variant=variant, debug_flags=KEYS), reference(case),
                 case.dtype, f"G=16 full size v{variant}")
