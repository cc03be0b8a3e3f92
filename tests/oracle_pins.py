"""Pins for the CPU oracle: checks that tie it to something other than itself.

Each ``pin_*`` function takes an oracle library handle (the real one, or a
variant with a planted mistake built by ``test_oracle_mutants.py``) and raises
``AssertionError`` when the oracle disagrees with

* the hand-derived worked examples in ``golden/hand_examples.json``;
* library special cases (``torch.softmax`` / ``scaled_dot_product_attention``
  in float64 after an explicit Python gather; numpy / torch dtype casts);
* closed forms (L = 1, constant V, q = 0, one-hot logits, linearity in V);
* the invariants of the method: the Phase 1 / Phase 2 log-sum-exp combine
  ("paged_attention_v2" commit note, project_6 commit 96f4baf, section
  "Implementation") equals one softmax over all tokens, and the result does
  not depend on where the blocks sit in the physical pool.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import dataclasses

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "hand_examples.json")


def _case_from_json(ex):
    t = lambda x, dt=torch.float64: torch.tensor(x, dtype=dt)
    return (t(ex["query"]), t(ex["k_cache"]), t(ex["v_cache"]),
            t(ex["block_tables"], torch.int32), t(ex["seq_lens"], torch.int32),
            ex["scale"])


def gather_contiguous(case_q, kc, vc, bt, sl, s, kvh):
    """K and V of one sequence and KV head as contiguous [L, D] tensors, by an
    explicit Python walk over the block table (independent of the oracle's
    own indexing)."""
    bs = kc.shape[2]
    L = int(sl[s])
    ks, vs = [], []
    for t in range(L):
        blk = int(bt[s, t // bs])
        ks.append(kc[blk, kvh, t % bs].to(torch.float64))
        vs.append(vc[blk, kvh, t % bs].to(torch.float64))
    return torch.stack(ks), torch.stack(vs)


def small_case(seed, B=3, H=4, Hkv=2, D=4, bs=4, lens=(1, 5, 17),
               dtype=torch.float64, k_mult=1.0, extra_blocks=3):
    return workloads.make_case("pin", seed, B, H, Hkv, D, dtype, bs, list(lens),
                               partition_size=8, k_mult=k_mult,
                               extra_blocks=extra_blocks)


def _run(lib, c, **kw):
    return oracle.attention(c.query, c.key_cache, c.value_cache, c.block_tables,
                            c.seq_lens, c.scale, lib=lib, **kw)


# ---------------------------------------------------------------------------

def pin_hand_examples(lib):
    data = json.load(open(GOLDEN))
    for ex in data["examples"]:
        q, kc, vc, bt, sl, scale = _case_from_json(ex)
        out = oracle.attention(q, kc, vc, bt, sl, scale, lib=lib)
        exp = np.array(ex["out"])
        assert np.allclose(out, exp, rtol=0, atol=ex["tol"]), (ex["name"], out, exp)
        if "partition_size" in ex:
            ml, es, to = oracle.partials(q, kc, vc, bt, sl, scale,
                                         ex["partition_size"], lib=lib)
            assert np.allclose(ml, ex["max_logits"], atol=ex["tol"]), ml
            assert np.allclose(es, ex["exp_sums"], atol=ex["tol"]), es
            assert np.allclose(to, ex["tmp_out"], atol=ex["tol"]), to
            np_ = oracle.num_partitions(sl.numpy(), ex["partition_size"])
            comb = oracle.combine(ml, es, to, np_, lib=lib)
            assert np.allclose(comb, exp, atol=ex["tol"]), comb


def pin_widen_bf16(lib):
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    t = bits.view(torch.bfloat16)
    got = oracle.widen(t, lib=lib)
    ref = t.to(torch.float64).numpy()
    assert np.array_equal(got, ref, equal_nan=True)


def pin_widen_f16(lib):
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    t = torch.from_numpy(bits.view(np.int16).copy()).view(torch.float16)
    got = oracle.widen(t, lib=lib)
    assert np.array_equal(got, ref, equal_nan=True)


def pin_brute_force_softmax(lib):
    """Tiny cases against torch.softmax in float64 after a Python gather."""
    for seed, (D, bs, lens, H, Hkv) in enumerate([
            (1, 2, (1, 2, 3), 2, 1), (4, 4, (17, 3, 1), 4, 2),
            (4, 1, (2, 5, 3), 2, 2), (1, 4, (17, 16, 15), 6, 3)]):
        c = small_case(100 + seed, B=len(lens), H=H, Hkv=Hkv, D=D, bs=bs, lens=lens)
        out = _run(lib, c)
        G = H // Hkv
        for s in range(c.num_seqs):
            for h in range(H):
                K, V = gather_contiguous(c.query, c.key_cache, c.value_cache,
                                         c.block_tables, c.seq_lens, s, h // G)
                logits = (K @ c.query[s, h].to(torch.float64)) * c.scale
                ref = torch.softmax(logits, dim=0) @ V
                assert np.allclose(out[s, h], ref.numpy(), rtol=1e-13, atol=1e-13), \
                    (s, h, out[s, h], ref)


def pin_sdpa_identity_table(lib):
    """With an identity block table and one sequence, the paged cache is a
    contiguous [Hkv, L, D] tensor: compare with torch SDPA (GQA expanded)."""
    B, H, Hkv, D, bs, L = 1, 8, 2, 16, 8, 37
    g = torch.Generator().manual_seed(7)
    nb = (L + bs - 1) // bs
    kc = torch.randn(nb, Hkv, bs, D, generator=g, dtype=torch.float64)
    vc = torch.randn(nb, Hkv, bs, D, generator=g, dtype=torch.float64)
    q = torch.randn(B, H, D, generator=g, dtype=torch.float64)
    bt = torch.arange(nb, dtype=torch.int32).reshape(1, nb)
    sl = torch.tensor([L], dtype=torch.int32)
    scale = 0.3
    out = oracle.attention(q, kc, vc, bt, sl, scale, lib=lib)
    K = kc.permute(1, 0, 2, 3).reshape(Hkv, nb * bs, D)[:, :L]
    V = vc.permute(1, 0, 2, 3).reshape(Hkv, nb * bs, D)[:, :L]
    G = H // Hkv
    K = K.repeat_interleave(G, dim=0)
    V = V.repeat_interleave(G, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q[0].unsqueeze(1), K, V, scale=scale).squeeze(1)
    assert np.allclose(out[0], ref.numpy(), rtol=1e-12, atol=1e-12)


def pin_single_token(lib):
    """L = 1: the softmax weight is exactly 1, so out == v_0 exactly."""
    c = small_case(11, B=2, H=4, Hkv=2, D=8, bs=4, lens=(1, 1), k_mult=3.0)
    out = _run(lib, c)
    for s in range(2):
        for h in range(4):
            blk = int(c.block_tables[s, 0])
            assert np.array_equal(out[s, h], c.value_cache[blk, h // 2, 0].numpy())


def pin_constant_v(lib):
    c = small_case(12, lens=(7, 16, 33), k_mult=2.0)
    c.value_cache[:] = 0.625
    out = _run(lib, c)
    assert np.allclose(out, 0.625, rtol=0, atol=1e-15)


def pin_zero_query_is_mean(lib):
    """q = 0: every logit is 0, the weights are uniform, out = mean of V."""
    c = small_case(13, lens=(3, 9, 20))
    c.query.zero_()
    out = _run(lib, c)
    G = c.num_heads // c.num_kv_heads
    for s in range(c.num_seqs):
        for h in range(c.num_heads):
            _, V = gather_contiguous(c.query, c.key_cache, c.value_cache,
                                     c.block_tables, c.seq_lens, s, h // G)
            assert np.allclose(out[s, h], V.numpy().mean(axis=0), rtol=0, atol=1e-14)


def pin_one_hot_logit(lib):
    """Key j = c * q with c large: logit_j exceeds the others by > 700, so
    out equals v_j to double precision (exp(-700) underflows relative to 1).
    The large logits also make a softmax without max-subtraction overflow."""
    B, H, Hkv, D, bs, L = 1, 2, 1, 4, 4, 11
    g = torch.Generator().manual_seed(3)
    nb = 3
    q = torch.zeros(B, H, D, dtype=torch.float64)
    q[0, :, 0] = 1.0
    kc = torch.randn(nb, Hkv, bs, D, generator=g, dtype=torch.float64) * 0.1
    vc = torch.randn(nb, Hkv, bs, D, generator=g, dtype=torch.float64)
    bt = torch.tensor([[2, 0, 1]], dtype=torch.int32)
    sl = torch.tensor([L], dtype=torch.int32)
    j = 6  # token 6 -> block bt[0][1] = 0, offset 2
    kc[0, 0, 2, 0] = 800.0
    out = oracle.attention(q, kc, vc, bt, sl, 1.0, lib=lib)
    for h in range(H):
        assert np.allclose(out[0, h], vc[0, 0, 2].numpy(), rtol=0, atol=1e-15), out


def pin_linearity_in_v(lib):
    c = small_case(14, lens=(5, 12, 30), k_mult=1.5)
    a, b = -2.5, 0.75
    out = _run(lib, c)
    c2 = dataclasses.replace(c, value_cache=c.value_cache * a + b)
    out2 = _run(lib, c2)
    assert np.allclose(out2, a * out + b, rtol=1e-13, atol=1e-13)


def pin_scale_folds_into_query(lib):
    c = small_case(15, lens=(4, 9, 21), k_mult=2.0)
    c.scale = 0.37
    out = _run(lib, c)
    c2 = dataclasses.replace(c, query=c.query * 0.37, scale=1.0)
    out2 = _run(lib, c2)
    assert np.allclose(out, out2, rtol=1e-12, atol=1e-12)


def pin_gqa_head_map(lib):
    """Each KV head carries a constant V equal to its index: out[h] must be
    h // G for every head (contiguous groups)."""
    c = small_case(16, B=2, H=8, Hkv=4, D=4, bs=4, lens=(6, 13))
    for kvh in range(4):
        c.value_cache[:, kvh] = float(kvh)
    out = _run(lib, c)
    for h in range(8):
        assert np.allclose(out[:, h], float(h // 2), atol=1e-15), (h, out[:, h])


def pin_tail_masking(lib):
    """Entries after L in the last block, and whole unused blocks, must not
    contribute: poison them and the output must not move."""
    c = small_case(17, lens=(5, 13, 2), bs=4, extra_blocks=2)
    out = _run(lib, c)
    used = {}
    for s in range(c.num_seqs):
        L = int(c.seq_lens[s])
        for t in range(L):
            used[(int(c.block_tables[s, t // 4]), t % 4)] = True
    kc, vc = c.key_cache.clone(), c.value_cache.clone()
    for blk in range(c.num_blocks):
        for off in range(4):
            if (blk, off) not in used:
                kc[blk, :, off] = 1e3
                vc[blk, :, off] = 1e6
    c2 = dataclasses.replace(c, key_cache=kc, value_cache=vc)
    out2 = _run(lib, c2)
    assert np.array_equal(out, out2)


def pin_pool_permutation(lib):
    """Moving blocks around the pool (and remapping the table) changes
    nothing: same values in the same logical order -> identical bits."""
    c = small_case(18, lens=(9, 31, 4), bs=4, extra_blocks=5, k_mult=2.0)
    out = _run(lib, c)
    for seed in (1, 2):
        out2 = _run(lib, workloads.permute_pool(c, seed))
        assert np.array_equal(out, out2)


def pin_partition_combine_equals_softmax(lib):
    """Phase 1 partials + Phase 2 log-sum-exp combine == unpartitioned
    softmax, for partition sizes at, below and above the sequence lengths."""
    lens = (1, 15, 16, 17, 31, 32, 33, 64, 70)
    c = small_case(19, B=len(lens), H=4, Hkv=2, D=8, bs=4, lens=lens, k_mult=3.0)
    ref = _run(lib, c)
    for P in (4, 8, 16, 32, 64, 128):
        ml, es, to = oracle.partials(c.query, c.key_cache, c.value_cache,
                                     c.block_tables, c.seq_lens, c.scale, P, lib=lib)
        npt = oracle.num_partitions(c.seq_lens.numpy(), P)
        out = oracle.combine(ml, es, to, npt, lib=lib)
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-12), P


def pin_partials_closed_form(lib):
    """q = 0: every logit is 0, so each partition has max 0, exp-sum equal to
    its token count and tmp_out equal to the mean V of its tokens."""
    lens = (10, 3)
    P = 4
    c = small_case(20, B=2, H=2, Hkv=1, D=3, bs=2, lens=lens)
    c.query.zero_()
    ml, es, to = oracle.partials(c.query, c.key_cache, c.value_cache,
                                 c.block_tables, c.seq_lens, c.scale, P, lib=lib)
    for s, L in enumerate(lens):
        K, V = gather_contiguous(c.query, c.key_cache, c.value_cache,
                                 c.block_tables, c.seq_lens, s, 0)
        for p in range(math.ceil(L / P)):
            n = min(P, L - p * P)
            for h in range(2):
                assert ml[s, h, p] == 0.0
                assert es[s, h, p] == float(n)
                assert np.allclose(to[s, h, p], V[p * P:p * P + n].numpy().mean(0),
                                   atol=1e-15)


def pin_empty_sequence(lib):
    c = small_case(21, B=2, lens=(0, 5))
    out = _run(lib, c)
    assert np.array_equal(out[0], np.zeros_like(out[0]))


def pin_attention_pairs_match_attention(lib):
    """The (seq, head) pair entry point gives, for every pair in any order,
    the row the whole-batch definition gives for that sequence and head:
    the same arithmetic, so the same bits.  B = 5 and H = 4 differ, so a pair
    decoded as (h, s) instead of (s, h) lands on another row (or out of the
    batch), and the shuffled order catches an output written to the wrong
    slot."""
    c = small_case(22, B=5, H=4, Hkv=2, D=4, bs=4, lens=(3, 9, 1, 14, 6), k_mult=2.0)
    ref = _run(lib, c)
    pairs = [(s, h) for s in range(5) for h in range(4)]
    order = np.random.default_rng(5).permutation(len(pairs))
    pairs = [pairs[i] for i in order]
    got = oracle.attention_pairs(pairs, c.query, c.key_cache, c.value_cache,
                                 c.block_tables, c.seq_lens, c.scale, lib=lib)
    for i, (s, h) in enumerate(pairs):
        assert np.array_equal(got[i], ref[s, h]), ((s, h), got[i], ref[s, h])


def _chunks_case(seed, lens, qlens, H=4, Hkv=2, D=4, bs=4, dtype=torch.float64):
    """A cache case plus query chunks: rows = sum(qlens) query vectors."""
    c = small_case(seed, B=len(lens), H=H, Hkv=Hkv, D=D, bs=bs, lens=lens, dtype=dtype)
    g = torch.Generator().manual_seed(seed + 1000)
    q = torch.randn(sum(qlens), H, D, generator=g, dtype=torch.float64).to(dtype)
    q_start = [0]
    for n in qlens:
        q_start.append(q_start[-1] + n)
    return c, q, q_start


def pin_query_chunks_single_token_is_decode(lib):
    """One query token per sequence: the chunk definition is the decode one
    (computed by the separately pinned attention function)."""
    c = small_case(31, lens=(1, 6, 17))
    out = oracle.query_chunks(c.query, c.key_cache, c.value_cache, c.block_tables,
                              c.seq_lens, [0, 1, 2, 3], c.scale, lib=lib)
    assert np.allclose(out, _run(lib, c), rtol=0, atol=1e-13)


def pin_query_chunks_causal_brute_force(lib):
    """Chunks of 1, 2, 3 and L tokens against a Python gather and
    torch.softmax in float64: row i of a chunk of n over L cached tokens
    sees tokens [0, L - n + i]."""
    lens, qlens = (5, 7, 9, 4), (1, 2, 3, 4)
    c, q, qs = _chunks_case(32, lens, qlens)
    out = oracle.query_chunks(q, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, qs,
                              c.scale, lib=lib)
    G = 4 // 2
    for s, (L, n) in enumerate(zip(lens, qlens)):
        for i in range(n):
            for h in range(4):
                K, V = gather_contiguous(None, c.key_cache, c.value_cache, c.block_tables,
                                         c.seq_lens, s, h // G)
                vis = L - n + i + 1
                w = torch.softmax(c.scale * (K[:vis] @ q[qs[s] + i, h].to(torch.float64)), 0)
                ref = (w[:, None] * V[:vis]).sum(0)
                assert torch.allclose(torch.from_numpy(out[qs[s] + i, h]), ref, atol=1e-13)


def pin_query_chunks_first_token_sees_itself(lib):
    """A chunk that is the whole sequence (no prefix): its first token sees
    only itself, so its output is V_0 exactly; its last token sees all."""
    lens = (6, 3)
    c, q, qs = _chunks_case(33, lens, lens)
    out = oracle.query_chunks(q, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, qs,
                              c.scale, lib=lib)
    for s in range(2):
        for h in range(4):
            K, V = gather_contiguous(None, c.key_cache, c.value_cache, c.block_tables,
                                     c.seq_lens, s, h // 2)
            assert np.array_equal(out[qs[s], h], V[0].numpy())


ALL_PINS = [
    pin_hand_examples, pin_widen_bf16, pin_widen_f16, pin_brute_force_softmax,
    pin_sdpa_identity_table, pin_single_token, pin_constant_v,
    pin_zero_query_is_mean, pin_one_hot_logit, pin_linearity_in_v,
    pin_scale_folds_into_query, pin_gqa_head_map, pin_tail_masking,
    pin_pool_permutation, pin_partition_combine_equals_softmax,
    pin_partials_closed_form, pin_empty_sequence, pin_attention_pairs_match_attention,
    pin_query_chunks_single_token_is_decode, pin_query_chunks_causal_brute_force,
    pin_query_chunks_first_token_sees_itself,
]
