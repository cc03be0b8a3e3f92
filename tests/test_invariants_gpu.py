"""GPU invariants: Phase 1 partials against the oracle's partials, Phase 2
alone, bit-identical results under a shuffled block pool, V1 == V2 and
P=256 == P=512 within tolerance, GQA heads == the same heads run as MHA."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_decode_attention_v2_gb300 as pa
import workloads
from gpu_helpers import DeviceCase, assert_close, reference

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,D,bs,P", [(torch.bfloat16, 128, 16, 512),
                                          (torch.float32, 64, 16, 256),
                                          (torch.float16, 256, 32, 256)])
def test_phase1_partials_match_oracle(dtype, D, bs, P):
    lens = [1, P - 3, P, P + 1, 3 * P + 100]
    case = workloads.make_case("partials", 31, len(lens), 16, 2, D, dtype, bs, lens,
                               partition_size=P, k_mult=3.0)
    dc = DeviceCase(case)
    dc.run(variant=pa.PA_VARIANT_V2)
    ml, es, to = dc.partials()
    rml, res, rto = oracle.partials(case.query, case.key_cache, case.value_cache,
                                    case.block_tables, case.seq_lens, case.scale, P)
    live = ~np.isnan(rml)
    # Both sides use the same dtype-rounded inputs, so a logit differs only by
    # the kernel's fp32 accumulation of the D products (each exact in fp32 for
    # 16-bit inputs): |d logit| <= D u scale |q| max_t |k_t| with u = 2^-24
    # (Cauchy-Schwarz on sum |q_d k_d|), plus a few roundings of |m| itself.
    u = 2.0 ** -24
    qn = case.query.double().norm(dim=-1).numpy()                         # [B, H]
    kn = float(case.key_cache.double().norm(dim=-1).max())
    eb = (D * u * case.scale * qn * kn)[:, :, None] * np.ones_like(rml)   # [B, H, Np]
    assert np.all(np.abs(ml[live] - rml[live]) <= eb[live] + 8 * u * np.abs(rml[live]))
    # exp_sums: the tensor path rounds each weight exp(logit - m) to the
    # input type before it is summed (2^-9 relative for bf16, 2^-11 for f16;
    # the fp32 path keeps it), and the logit error enters twice (logit and
    # max); the fp32 sum of up to P terms adds P u.
    rho = {torch.bfloat16: 2.0 ** -9, torch.float16: 2.0 ** -11, torch.float32: 4 * u}[dtype]
    bound_es = res[live] * (rho + 2 * eb[live] + P * u)
    assert np.all(np.abs(es[live] - res[live]) <= bound_es)
    assert_close(torch.from_numpy(to[live]), rto[live], dtype, "tmp_out")
    # Phase 2 alone: the oracle's combine of the GPU's partials equals the
    # GPU's final output within rounding of the output dtype
    npt = oracle.num_partitions(case.seq_lens.numpy(), P)
    comb = oracle.combine(np.nan_to_num(ml), np.nan_to_num(es), np.nan_to_num(to), npt)
    out = dc.run(variant=pa.PA_VARIANT_V2)
    assert_close(out, comb, dtype, "phase 2 vs oracle combine of GPU partials")


@pytest.mark.parametrize("math", [pa.PA_MATH_TENSOR, pa.PA_MATH_SIMT])
def test_pool_permutation_is_bit_identical(math):
    case = workloads.make_case("perm", 41, 6, 32, 4, 128, torch.bfloat16, 16,
                               [1, 100, 513, 2000, 4097, 777], partition_size=512,
                               extra_blocks=20)
    a = DeviceCase(case)
    b = DeviceCase(workloads.permute_pool(case, 3))
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        oa = a.run(variant=variant, math=math)
        ob = b.run(variant=variant, math=math)
        assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))



def test_pool_permutation_is_bit_identical_16_rows():
    """The 16-row kernels too: groups of 16 query heads (V1 and V2) and query
    chunks of 4 tokens, each bit-identical after the physical pool is
    shuffled (the arithmetic follows the logical token order only)."""
    lens = [9, 600, 2000, 4097, 777]
    g16 = workloads.make_case("perm16", 42, len(lens), 32, 2, 128, torch.bfloat16, 16, lens,
                              partition_size=512, extra_blocks=20)
    a, b = DeviceCase(g16), DeviceCase(workloads.permute_pool(g16, 5))
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        assert torch.equal(a.run(variant=variant).view(torch.int16),
                           b.run(variant=variant).view(torch.int16))
    ch = workloads.make_case("permch", 43, len(lens), 32, 4, 128, torch.bfloat16, 16, lens,
                             partition_size=512, extra_blocks=20)
    q, qs = workloads.chunk_queries(ch, 4)
    outs = []
    for c in (ch, workloads.permute_pool(ch, 6)):
        dc = DeviceCase(c)
        qd, qsd = q.cuda(), qs.cuda()
        ws = pa.alloc_workspace(q.shape[0], c.num_heads, c.head_size, c.max_seq_len,
                                c.partition_size)
        out = torch.full_like(qd, float("nan"))
        pa.pa_chunks_forward(out, qd, dc.kc, dc.vc, dc.bt, dc.sl, qsd, c.scale,
                             c.partition_size, ws, max_seq_len=c.max_seq_len, max_chunk=4)
        assert pa.pa_read_device_status(ws) == pa.PA_OK
        outs.append(out)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))

def test_v1_equals_v2_and_partition_sizes_agree():
    case = workloads.config_case("c5_mixed_d256", 512)
    small = dataclasses.replace(
        case, query=case.query[:16], block_tables=case.block_tables[:16],
        seq_lens=case.seq_lens[:16])
    dc = DeviceCase(small)
    ref = reference(small)
    o1 = dc.run(variant=pa.PA_VARIANT_V1)
    o2 = dc.run(variant=pa.PA_VARIANT_V2, partition_size=512)
    o3 = dc.run(variant=pa.PA_VARIANT_V2, partition_size=256)
    for o in (o1, o2, o3):
        assert_close(o, ref, torch.bfloat16)
    # the three differ only by rounding: compare to each other at the same bar
    assert_close(o2, o1.double().cpu().numpy(), torch.bfloat16, "V2 P512 vs V1")
    assert_close(o3, o2.double().cpu().numpy(), torch.bfloat16, "P256 vs P512")


def test_gqa_equals_mha_with_repeated_kv():
    """Query heads of a GQA group give the same result as MHA with each KV
    head repeated G times (the kernel's group batching changes nothing)."""
    G, Hkv = 8, 2
    case = workloads.make_case("gqa", 51, 3, G * Hkv, Hkv, 128, torch.bfloat16, 16,
                               [700, 1500, 64], partition_size=512)
    mha = dataclasses.replace(case, key_cache=case.key_cache.repeat_interleave(G, dim=1),
                              value_cache=case.value_cache.repeat_interleave(G, dim=1))
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        og = DeviceCase(case).run(variant=variant)
        om = DeviceCase(mha).run(variant=variant)
        assert_close(og, om.double().cpu().numpy(), torch.bfloat16, "GQA vs MHA")


def test_constant_v_gives_v():
    case = workloads.make_case("constv", 61, 4, 16, 2, 128, torch.bfloat16, 16,
                               [1, 33, 1000, 5000], partition_size=512, k_mult=4.0)
    case.value_cache.fill_(0.375)
    out = DeviceCase(case).run(variant=pa.PA_VARIANT_V2)
    assert torch.all(out == 0.375)


def test_one_hot_logit_selects_one_value():
    """A key aligned with the query and 30x larger makes one token's weight 1
    to well within bf16: out == that token's V (after rounding to bf16)."""
    case = workloads.make_case("onehot", 71, 1, 8, 1, 128, torch.bfloat16, 16, [3000],
                               partition_size=512)
    q = case.query[0, 0]
    blk = int(case.block_tables[0, 1234 // 16])
    case.query[0, :] = q
    case.key_cache[blk, 0, 1234 % 16] = (q.float() * 30).to(torch.bfloat16)
    out = DeviceCase(case).run(variant=pa.PA_VARIANT_V2)
    v = case.value_cache[blk, 0, 1234 % 16]
    assert torch.equal(out[0].cpu(), v.expand(8, -1))


def test_fused_combine_reads_every_partition():
    """Regression: the CTA that finishes a sequence's last partition must see
    every other CTA's partials.  A bf16 batch warms the GPU first (the
    failure showed with that timing); then a 4-partition f32 sequence runs
    through the fused combine repeatedly and must match the oracle to 1e-5."""
    warm = workloads.make_case("warm", 7, 3, 16, 2, 128, torch.bfloat16, 16, [1, 700, 1300],
                               partition_size=512, extra_blocks=4)
    DeviceCase(warm).run(variant=pa.PA_VARIANT_V2, fuse_partitions=16)
    case = workloads.make_case("fused", 8, 2, 4, 1, 64, torch.float32, 16, [37, 1000],
                               partition_size=256, extra_blocks=2)
    ref = reference(case)
    dc = DeviceCase(case)
    for _ in range(8):
        assert_close(dc.run(variant=pa.PA_VARIANT_V2, fuse_partitions=16), ref, torch.float32,
                     "fused combine")


@pytest.mark.parametrize("variant,fuse", [(pa.PA_VARIANT_V1, 0), (pa.PA_VARIANT_V2, 0),
                                          (pa.PA_VARIANT_V2, 1), (pa.PA_VARIANT_V2, 16)])
def test_work_counters_return_to_zero(variant, fuse):
    """After every call the work-queue counters (words 1 and 2 of the status
    block) are zero again, whoever resets them: Phase 1's last CTA (V1, or V2
    with every sequence combined inside Phase 1) or the Phase 2 kernel after
    its wait.  Repeated calls give the oracle's result each time."""
    case = workloads.make_case("counters", 12, 3, 16, 2, 128, torch.bfloat16, 16, [5, 300, 1100],
                               partition_size=256, extra_blocks=2)
    ref = reference(case)
    dc = DeviceCase(case)
    for _ in range(3):
        assert_close(dc.run(variant=variant, fuse_partitions=fuse), ref, torch.bfloat16,
                     f"variant {variant}, fuse {fuse}")
        words = dc.ws[:12].view(torch.int32).cpu().tolist()
        assert words == [0, 0, 0], words


@pytest.mark.parametrize("fuse", [16, 0])
@pytest.mark.parametrize("dtype,H,Hkv,D", [(torch.float32, 4, 1, 64), (torch.bfloat16, 16, 2, 128)])
def test_writes_stay_inside_out_and_workspace(dtype, H, Hkv, D, fuse):
    """Regression: every write lands inside `out` and the workspace.  Both are
    views at the head of larger buffers whose tails hold a canary, and the
    inputs are unchanged afterwards.  The batch has fewer sequences than a
    warp scans at once and an empty one."""
    lens = [0, 37, 1000]
    case = workloads.make_case("bounds", 91, len(lens), H, Hkv, D, dtype, 16, lens,
                               partition_size=256, extra_blocks=2)
    ref = reference(case)
    host = [case.query, case.key_cache, case.value_cache, case.block_tables, case.seq_lens]
    q, kc, vc, bt, sl = (t.cuda() for t in host)
    canary = 1 << 16
    nbytes = pa.pa_workspace_bytes(case.num_seqs, H, D, case.max_seq_len, 256)
    wsbuf = torch.full((nbytes + canary,), 0xAB, dtype=torch.uint8, device="cuda")
    ws = wsbuf[:nbytes]
    pa.pa_workspace_init(ws)
    n = case.query.numel()
    for variant in (pa.PA_VARIANT_V1, pa.PA_VARIANT_V2):
        obuf = torch.full((n + canary,), float("nan"), dtype=dtype, device="cuda")
        out = obuf[:n].view(case.query.shape)
        pa.pa_forward(out, q, kc, vc, bt, sl, case.scale, 256, ws, max_seq_len=case.max_seq_len,
                      variant=variant, fuse_partitions=fuse)
        assert pa.pa_read_device_status(ws) == pa.PA_OK
        assert_close(out, ref, dtype, f"v{variant}")
        assert torch.all(torch.isnan(obuf[n:])), "write past the end of out"
        assert torch.all(wsbuf[nbytes:] == 0xAB), "write past the end of the workspace"
        for dev_t, host_t in zip((q, kc, vc, bt, sl), host):
            assert torch.equal(dev_t.cpu(), host_t), "an input was modified"
