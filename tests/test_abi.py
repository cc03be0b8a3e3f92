"""libpa's C ABI on the host: the library loads, exports every function the
header declares, and the host-only entry points (workspace sizing, the V1/V2
heuristic, status text, argument checks) behave as documented.  CPU only: no
call here reaches a CUDA API."""
import ctypes
import os
import re

import pytest

import paged_decode_attention_v2_gb300 as pa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return pa.load_library()


def header_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_header_lists_the_forward_calls():
    names = header_functions()
    for n in ("pa_v1_forward", "pa_v2_forward", "pa_forward", "pa_workspace_bytes"):
        assert n in names


def test_library_exports_every_header_function(lib):
    names = header_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(lib, n), f"libpa.so does not export {n}"
    assert sorted(pa.EXPORTS) == names


def test_version_and_status_text(lib):
    assert pa.pa_version() >= 100
    for code in range(7):
        assert pa.pa_status_string(code) and pa.pa_status_string(code) != "unknown status"
    assert pa.pa_status_string(99) == "unknown status"


def test_workspace_layout_and_size(lib):
    B, H, D, L, P = 3, 32, 128, 100000, 512
    off = pa.pa_workspace_layout(B, H, D, L, P)
    parts = -(-L // P)
    assert parts == 196  # ceil(100000 / 512)
    assert off[0] == 0 and off[1] == 256
    assert all(o % 256 == 0 for o in off)
    stats = B * H * parts * 4
    assert off[2] - off[1] >= stats and off[2] - off[1] < stats + 256
    assert off[3] - off[2] == off[2] - off[1]
    assert len(off) == 5 and off[4] - off[3] >= B * H * parts * D * 4
    size = pa.pa_workspace_bytes(B, H, D, L, P)
    assert size >= off[4] + B * H * 4 and size % 256 == 0
    # no partitions: the status block and the combine counters
    assert pa.pa_workspace_bytes(4, 8, 64, 0, 512) == 256 + 256
    assert pa.pa_workspace_bytes(-1, 8, 64, 10, 512) == 0
    assert pa.pa_workspace_bytes(1, 8, 64, 10, 0) == 0


# The rule's cells as measured on GB300 (152 SMs, P = 512, 4 KV heads): the
# V1/V2 sweep over (sequences x KV heads) in {1, 2, 4, 8, 16} x 152 and
# max length in {512 .. 16384}.
CHOOSE_V2_MEASURED = {
    # (B*Hkv, max L): faster variant
    (152, 512): 0, (152, 1024): 1, (152, 2048): 1, (152, 4096): 1, (152, 8192): 1,
    (152, 16384): 1,
    (304, 512): 0, (304, 1024): 0, (304, 2048): 0, (304, 4096): 1, (304, 8192): 1,
    (304, 16384): 1,
    (608, 512): 0, (608, 1024): 1, (608, 2048): 1, (608, 4096): 1, (608, 8192): 1,
    (608, 16384): 1,
    (1216, 512): 0, (1216, 1024): 0, (1216, 2048): 1, (1216, 4096): 1, (1216, 8192): 1,
    (1216, 16384): 1,
    (2432, 512): 0, (2432, 1024): 0, (2432, 2048): 0, (2432, 4096): 0, (2432, 8192): 0,
    (2432, 16384): 0,
}


@pytest.mark.parametrize("cell", sorted(CHOOSE_V2_MEASURED))
def test_choose_v2_matches_the_measured_crossover(lib, cell):
    bh, L = cell
    assert pa.pa_choose_v2(bh // 4, 4, L, 512, 152) == CHOOSE_V2_MEASURED[cell]


# Query chunks, measured on GB300 (bf16, D 128, consecutive steps): (workload,
# tokens a chunk): faster variant.  c4: 256 sequences of up to 3584 tokens, 32 q /
# 4 kv heads; c2: 8 sequences of up to 8192; c3: one of 100,000.
CHUNK_SHAPES = {"c4": (256, 32, 4, 128, 3584), "c2": (8, 32, 4, 128, 8192),
                "c3": (1, 32, 4, 128, 100000)}
CHOOSE_V2_CHUNKS_MEASURED = {
    ("c4", 2): 1, ("c4", 4): 0, ("c4", 8): 0, ("c4", 16): 0, ("c4", 32): 0, ("c4", 64): 0,
    ("c2", 4): 1, ("c2", 16): 1, ("c2", 64): 1, ("c3", 16): 1, ("c3", 64): 1,
}


@pytest.mark.parametrize("cell", sorted(CHOOSE_V2_CHUNKS_MEASURED))
def test_choose_v2_chunks_matches_the_measured_cells(lib, cell):
    B, H, Hkv, D, L = CHUNK_SHAPES[cell[0]]
    got = pa.pa_choose_v2_chunks(B, H, Hkv, D, cell[1], L, 512, 152)
    assert got == CHOOSE_V2_CHUNKS_MEASURED[cell]


def test_choose_v2_chunks_small_rows_follow_decode(lib):
    # up to 8 rows per KV head (1 token of 8 heads, 2 of 4): the decode rule
    for B, L in ((256, 3584), (8, 8192), (4096, 1024), (1, 100000)):
        assert pa.pa_choose_v2_chunks(B, 32, 4, 128, 1, L, 512, 152) == \
            pa.pa_choose_v2(B, 4, L, 512, 152)
        assert pa.pa_choose_v2_chunks(B, 16, 4, 128, 2, L, 512, 152) == \
            pa.pa_choose_v2(B, 4, L, 512, 152)
    assert pa.pa_choose_v2_chunks(256, 32, 4, 128, 16, 500, 512, 152) == 0  # one partition


@pytest.mark.parametrize("args,expect", [
    ((1, 4, 100000, 512, 152), 1),   # one long sequence: V2 spreads it over the GPU
    ((8, 4, 8192, 512, 152), 1),     # few (seq, kv head) items: V2
    ((64, 4, 512, 512, 152), 0),     # every sequence in one partition: V1
    ((4096, 8, 4096, 512, 152), 0),  # 32K items of short sequences: V1 fills the GPU
    ((4096, 8, 20000, 512, 152), 0), # 32K items: V1 balances at any length
    ((256, 4, 3584, 512, 152), 1),   # 1024 items (6.7 per SM) of up to 7 partitions: V2
    ((1, 1, 0, 512, 152), 0),
    ((76, 4, 1024, 512, 0), 1),      # unknown SM count: V2 unless one partition
])
def test_choose_v2(lib, args, expect):
    assert pa.pa_choose_v2(*args) == expect


# ---- argument checks (rejected on the host before any CUDA call) ----------

FAKE = 1 << 20  # aligned, never dereferenced by the host checks


def _call(lib, variant=pa.PA_VARIANT_V2, **over):
    a = dict(out=FAKE, query=FAKE, key_cache=FAKE, value_cache=FAKE, block_tables=FAKE,
             seq_lens=FAKE, num_seqs=2, num_heads=8, num_kv_heads=2, head_size=128,
             num_blocks=64, block_size=16, max_blocks_per_seq=8, max_seq_len=128,
             scale=0.1, partition_size=512, dtype=pa.PA_DTYPE_BF16, workspace=FAKE,
             workspace_bytes=1 << 30, stream=0)
    a.update(over)
    opts = pa.pa_options_t(variant, 0, 0, 0, 0, None, 0, 0)
    return lib.pa_forward(a["out"], a["query"], a["key_cache"], a["value_cache"],
                          a["block_tables"], a["seq_lens"], a["num_seqs"], a["num_heads"],
                          a["num_kv_heads"], a["head_size"], a["num_blocks"], a["block_size"],
                          a["max_blocks_per_seq"], a["max_seq_len"], a["scale"],
                          a["partition_size"], a["dtype"], a["workspace"],
                          a["workspace_bytes"], a["stream"], ctypes.byref(opts))


@pytest.mark.parametrize("over,expect", [
    (dict(out=0), pa.PA_ERR_INVALID_ARG),
    (dict(query=0), pa.PA_ERR_INVALID_ARG),
    (dict(key_cache=FAKE + 8), pa.PA_ERR_INVALID_ARG),      # not 16-byte aligned
    (dict(workspace=FAKE + 16), pa.PA_ERR_INVALID_ARG),     # not 256-byte aligned
    (dict(block_tables=FAKE + 2), pa.PA_ERR_INVALID_ARG),
    (dict(num_heads=6, num_kv_heads=4), pa.PA_ERR_INVALID_ARG),
    (dict(num_heads=64, num_kv_heads=2), pa.PA_ERR_UNSUPPORTED),  # group of 32
    (dict(head_size=96), pa.PA_ERR_UNSUPPORTED),
    (dict(block_size=12, max_seq_len=96), pa.PA_ERR_UNSUPPORTED),
    (dict(block_size=128), pa.PA_ERR_UNSUPPORTED),
    (dict(partition_size=500), pa.PA_ERR_UNSUPPORTED),
    (dict(partition_size=16384), pa.PA_ERR_UNSUPPORTED),
    (dict(partition_size=0), pa.PA_ERR_INVALID_ARG),
    (dict(dtype=7), pa.PA_ERR_INVALID_ARG),
    (dict(max_seq_len=129), pa.PA_ERR_INVALID_ARG),         # > max_blocks * block_size
    (dict(max_seq_len=-1), pa.PA_ERR_INVALID_ARG),
    (dict(num_seqs=-1), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), pa.PA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), pa.PA_ERR_INVALID_ARG),
    (dict(workspace_bytes=255), pa.PA_ERR_WORKSPACE_TOO_SMALL),
    (dict(num_blocks=1 << 27, num_kv_heads=8, num_heads=8), pa.PA_ERR_UNSUPPORTED),
])
def test_argument_errors(lib, over, expect):
    assert _call(lib, **over) == expect


def test_v2_needs_the_partials_workspace(lib):
    need = pa.pa_workspace_bytes(2, 8, 128, 128, 512)
    assert _call(lib, workspace_bytes=need - 1) == pa.PA_ERR_WORKSPACE_TOO_SMALL
    # V1 only needs the status block
    assert _call(lib, variant=pa.PA_VARIANT_V1, workspace_bytes=255) == \
        pa.PA_ERR_WORKSPACE_TOO_SMALL


def test_empty_batch_is_a_noop(lib):
    assert _call(lib, num_seqs=0) == pa.PA_OK
    assert _call(lib, variant=pa.PA_VARIANT_V1, num_seqs=0) == pa.PA_OK


def test_bad_variant(lib):
    assert _call(lib, variant=9) == pa.PA_ERR_INVALID_ARG


def test_workspace_init_rejects_bad_buffers(lib):
    assert lib.pa_workspace_init(0, 256, 0) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_workspace_init(FAKE, 128, 0) == pa.PA_ERR_INVALID_ARG
    assert lib.pa_read_device_status(FAKE + 4, 0) == pa.PA_ERR_INVALID_ARG


def test_host_staging_bytes(lib):
    # query and out (B*H*D*elt each), block tables, seq_lens; 256-byte parts
    assert pa.pa_host_staging_bytes(3, 8, 128, 10, pa.PA_DTYPE_BF16) == 6144 * 2 + 256 + 256
    assert pa.pa_host_staging_bytes(3, 8, 128, 100, pa.PA_DTYPE_F32) == \
        12288 * 2 + 1280 + 256
    assert pa.pa_host_staging_bytes(-1, 8, 128, 10, pa.PA_DTYPE_BF16) == 0
    assert pa.pa_host_staging_bytes(3, 8, 128, 10, 7) == 0


# ---- the split phases (context parallelism) --------------------------------

def _partials(lib, part_begin, part_end, **over):
    a = dict(query=FAKE, key_cache=FAKE, value_cache=FAKE, block_tables=FAKE, seq_lens=FAKE,
             num_seqs=2, num_heads=8, num_kv_heads=2, head_size=128, num_blocks=64,
             block_size=16, max_blocks_per_seq=8, max_seq_len=128, scale=0.1,
             partition_size=512, dtype=pa.PA_DTYPE_BF16, workspace=FAKE,
             workspace_bytes=1 << 30, stream=0)
    a.update(over)
    return lib.pa_v2_partials(a["query"], a["key_cache"], a["value_cache"], a["block_tables"],
                              a["seq_lens"], a["num_seqs"], a["num_heads"], a["num_kv_heads"],
                              a["head_size"], a["num_blocks"], a["block_size"],
                              a["max_blocks_per_seq"], a["max_seq_len"], a["scale"],
                              a["partition_size"], a["dtype"], part_begin, part_end,
                              a["workspace"], a["workspace_bytes"], a["stream"])


def _combine(lib, **over):
    a = dict(out=FAKE, seq_lens=FAKE, num_seqs=2, num_heads=8, head_size=128, max_seq_len=128,
             partition_size=512, dtype=pa.PA_DTYPE_BF16, workspace=FAKE,
             workspace_bytes=1 << 30, stream=0)
    a.update(over)
    return lib.pa_v2_combine(a["out"], a["seq_lens"], a["num_seqs"], a["num_heads"],
                             a["head_size"], a["max_seq_len"], a["partition_size"], a["dtype"],
                             a["workspace"], a["workspace_bytes"], a["stream"])


@pytest.mark.parametrize("rng,over,expect", [
    ((-1, 4), {}, pa.PA_ERR_INVALID_ARG),             # negative start
    ((3, 2), {}, pa.PA_ERR_INVALID_ARG),              # empty-backwards range
    ((0, 1), dict(query=0), pa.PA_ERR_INVALID_ARG),
    ((0, 1), dict(workspace=FAKE + 64), pa.PA_ERR_INVALID_ARG),
    ((0, 1), dict(head_size=96), pa.PA_ERR_UNSUPPORTED),
    ((0, 1), dict(workspace_bytes=pa.pa_workspace_bytes(2, 8, 128, 128, 512) - 1),
     pa.PA_ERR_WORKSPACE_TOO_SMALL),
    ((5, 5), {}, pa.PA_OK),                            # empty range: nothing to do
    ((0, 4), dict(num_seqs=0), pa.PA_OK),              # no sequences: nothing to do
])
def test_partials_argument_errors(lib, rng, over, expect):
    assert _partials(lib, *rng, **over) == expect


@pytest.mark.parametrize("over,expect", [
    (dict(out=0), pa.PA_ERR_INVALID_ARG),
    (dict(seq_lens=0), pa.PA_ERR_INVALID_ARG),
    (dict(out=FAKE + 4), pa.PA_ERR_INVALID_ARG),
    (dict(workspace=FAKE + 16), pa.PA_ERR_INVALID_ARG),
    (dict(head_size=96), pa.PA_ERR_UNSUPPORTED),
    (dict(partition_size=100), pa.PA_ERR_UNSUPPORTED),
    (dict(dtype=7), pa.PA_ERR_INVALID_ARG),
    (dict(num_seqs=-1), pa.PA_ERR_INVALID_ARG),
    (dict(workspace_bytes=pa.pa_workspace_bytes(2, 8, 128, 128, 512) - 1),
     pa.PA_ERR_WORKSPACE_TOO_SMALL),
])
def test_combine_argument_errors(lib, over, expect):
    assert _combine(lib, **over) == expect
