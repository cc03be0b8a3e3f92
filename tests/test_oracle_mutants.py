"""Plant plausible mistakes in a copy of the oracle's C source and check that
each one is caught by at least one pin.  This is what shows the pins are
strong enough to trust the oracle.  CPU only; the mutants live in a temp dir
and run in child processes, because an indexing mistake can crash the process
that loads it (a crash also counts as caught)."""
import json
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(os.path.dirname(oracle.__file__), "pa_oracle.c")

# (name, original text, mutated text).  Each original must occur exactly once.
MUTANTS = [
    ("block_and_offset_swapped",
     "block_tables[(size_t)s * max_blocks + t / bs];\n  int off = t % bs;",
     "block_tables[(size_t)s * max_blocks + t % bs];\n  int off = t / bs;"),
    ("kv_head_modulo", "int kvh = h / G;", "int kvh = h % Hkv;"),
    ("scale_dropped", "return scale * dot;", "return dot;"),
    ("scale_squared", "return scale * dot;", "return scale * scale * dot;"),
    ("last_token_dropped", "for (int t = t0; t < t1; ++t) {\n    double w",
     "for (int t = t0; t < t1 - 1; ++t) {\n    double w"),
    ("no_max_subtraction", "double w = exp(logits[t - t0] - m);",
     "double w = exp(logits[t - t0]);"),
    ("partial_not_normalised", "for (int d = 0; d < D; ++d) o[d] /= sum;", ""),
    ("k_used_as_v", "o[d] += w * load_elem(vc,", "o[d] += w * load_elem(kc,"),
    ("query_head_is_kv_head", "load_elem(q, ((size_t)s * H + h) * D + d, dtype)",
     "load_elem(q, ((size_t)s * H + kvh) * D + d, dtype)"),
    ("combine_sign_flipped", "double w = exp(ml[p] - gmax) * es[p] / total;",
     "double w = exp(gmax - ml[p]) * es[p] / total;"),
    ("combine_ignores_exp_sums",
     "total += exp(ml[p] - gmax) * es[p];", "total += exp(ml[p] - gmax);"),
    ("partition_end_off_by_one", "int t1 = t0 + P < L ? t0 + P : L;",
     "int t1 = t0 + P - 1 < L ? t0 + P - 1 : L;"),
    ("chunk_sees_one_token_too_many", "const int pos = L - n + (int)(row - q_start[s]);",
     "const int pos = L - n + (int)(row - q_start[s]) + 1;"),
    ("chunk_row_to_sequence_off", "while (s + 1 < B && q_start[s + 1] <= row) ++s;",
     "while (s + 1 < B && q_start[s + 1] < row) ++s;"),
    ("chunk_query_head_dropped", "dot += load_elem(q, (size_t)i * D + d, dtype) *",
     "dot += load_elem(q, (size_t)row * H * D + d, dtype) *"),
    ("f16_exponent_bias", "e - 25); /* (1 + f/1024)", "e - 24); /* (1 + f/1024)"),
    ("f16_subnormal_scale", "ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    ("bf16_wrong_half", "uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b << 15;"),
    ("pairs_s_h_swapped", "int s = pairs[2 * i], h = pairs[2 * i + 1];",
     "int h = pairs[2 * i], s = pairs[2 * i + 1];"),
    ("dot_drops_last_dim", "for (int d = 0; d < D; ++d)\n    dot +=",
     "for (int d = 0; d < D - 1; ++d)\n    dot +="),
]

RUNNER = r"""
import json, sys
sys.path[:0] = [sys.argv[2], sys.argv[3]]
import oracle, oracle_pins
lib = oracle.load_library(sys.argv[1])
failed = []
for pin in oracle_pins.ALL_PINS:
    try:
        pin(lib)
    except AssertionError:
        failed.append(pin.__name__)
    except Exception as e:
        failed.append(pin.__name__ + ":" + type(e).__name__)
print(json.dumps(failed))
"""


@pytest.fixture(scope="module")
def source():
    return open(SRC).read()


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) == 1, f"mutation site for {name} not found once"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new))
    so = oracle.compile_oracle(str(src), str(tmp_path / "libmutant.so"))
    r = subprocess.run([sys.executable, "-c", RUNNER, so, ROOT, HERE],
                       capture_output=True, text=True, timeout=300)
    if r.returncode != 0:
        return  # the mutant crashed the process: caught
    failed = json.loads(r.stdout.strip().splitlines()[-1])
    assert failed, f"mutant {name} passed every pin"
