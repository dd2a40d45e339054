"""Plant plausible mistakes in copies of the oracle and check the pins catch them.

Each mutant is the oracle's C source with one textual change (a dropped term, a
wrong sign, a wrong index, a transposed operand, an off-by-one), compiled to a
temporary library on the CPU. The pins of oracle_pins must fail on every one.
The pins run on each mutant in a child process: a mutant may index outside its
buffers (an unchecked page number, say), and its writes must not reach the
test process's own memory. A child killed by such an access has shown the
mistake as well.
"""
import json
import os
import subprocess
import sys
import tempfile

import pytest

import oracle
import oracle_pins

SRC = open(oracle._SRC).read()

# (name, original text, replacement). Each original must occur exactly once.
MUTANTS = [
    ("group_index_modulo", "int g = h / (Hq / Hkv);", "int g = h % Hkv;"),
    ("group_index_modulo_batch", "g = h / G;\n                const int L",
     "g = h % Hkv;\n                const int L"),
    ("no_max_subtraction", "w[t] = exp(w[t] - mx);", "w[t] = exp(w[t]);"),
    ("flipped_exponent_sign", "w[t] = exp(w[t] - mx);", "w[t] = exp(mx - w[t]);"),
    ("scale_dropped", "w[t] = scale * dot;", "w[t] = dot;"),
    ("softmax_not_normalised", "for (int t = 0; t < L; ++t) w[t] /= sum;", ""),
    ("cache_index_transposed",
     "return c + (((size_t)b * (size_t)S_max + (size_t)t) * (size_t)Hkv + (size_t)g) * (size_t)D;",
     "return c + (((size_t)b * (size_t)Hkv + (size_t)g) * (size_t)S_max + (size_t)t) * (size_t)D;"),
    ("last_token_dropped", "for (int t = 0; t < L; ++t) {\n                    const uint16_t* vr",
     "for (int t = 0; t < L - 1; ++t) {\n                    const uint16_t* vr"),
    ("merge_rescale_dropped", "const double a = exp(m[j] - M);", "const double a = 1.0;"),
    ("merge_denominator_unscaled", "denom += a * l[j];", "denom += l[j];"),
    ("lse_missing_max", "return mx + log(sum);", "return log(sum);"),
    ("append_wrong_row", "const size_t dst = (((size_t)b * S_max + (size_t)t) * Hkv + h) * (size_t)D;",
     "const size_t dst = (((size_t)b * S_max + (size_t)(t > 0 ? t - 1 : t)) * Hkv + h) * (size_t)D;"),
    ("paged_block_and_row_swapped",
     "const uint16_t* src = pages + ((size_t)page * (size_t)P + (size_t)(t % P)) * row;",
     "const uint16_t* src = pages + ((size_t)page * (size_t)P + (size_t)(t / P) % P) * row;"),
    ("paged_block_index_off_by_one", "const int page = table[(size_t)b * max_blocks + t / P];\n            uint16_t*",
     "const int page = table[(size_t)b * max_blocks + (t + 1) / P];\n            uint16_t*"),
    ("paged_invalid_entry_not_zeroed", "memset(dst, 0, sizeof(uint16_t) * row);", ""),
    ("paged_invalid_entry_wraps", "if (page < 0 || page >= num_pages) {\n                memset",
     "if (page < 0) {\n                memset"),
    ("paged_append_wrong_row", "const size_t dst = (((size_t)page * P + (size_t)(t % P)) * Hkv + h) * (size_t)D;",
     "const size_t dst = (((size_t)page * P + (size_t)((t + 1) % P)) * Hkv + h) * (size_t)D;"),
    ("q8_scale_over_128", "volatile float sc = a / 127.0f;", "volatile float sc = a / 128.0f;"),
    ("q8_truncates", "c = (int)rintf(y);", "c = (int)y;"),
    ("q8_rounds_half_away", "c = (int)rintf(y);", "c = (int)roundf(y);"),
    ("q8_readback_drops_scale", "out[(size_t)r * D + d] = (double)scales[r] * (double)codes[(size_t)r * D + d];",
     "out[(size_t)r * D + d] = (double)codes[(size_t)r * D + d];"),
    ("f64kv_no_max_subtraction", "const double e = exp(w[t] - top);", "const double e = exp(w[t]);"),
    ("f64kv_wrong_kv_head", "const int kvh = h / G;", "const int kvh = h % Hkv;"),
    ("f64kv_scale_dropped", "w[t] = acc * scale;", "w[t] = acc;"),
    ("paged_append_ignores_bad_page", "if (page < 0 || page >= num_pages) { ++skipped; ++bad; continue; }",
     "if (page < 0) { ++skipped; ++bad; continue; }"),
]


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(name, old, new, workdir):
    assert SRC.count(old) == 1, f"mutation site for {name} not unique/absent"
    src = os.path.join(workdir, f"{name}.c")
    with open(src, "w") as f:
        f.write(SRC.replace(old, new))
    lib_path = oracle.build(force=True, src=src, out=os.path.join(workdir, f"{name}.so"))
    here = os.path.dirname(os.path.abspath(__file__))
    code = (
        "import json, sys\n"
        f"sys.path[:0] = [{here!r}, {os.path.dirname(here)!r}]\n"
        "import oracle, oracle_pins\n"
        f"lib = oracle._load({lib_path!r})\n"
        "failed = []\n"
        "for check in oracle_pins.ALL_CHECKS:\n"
        "    try:\n"
        "        check(lib)\n"
        "    except (AssertionError, ValueError, FloatingPointError):\n"
        "        failed.append(check.__name__)\n"
        "print(json.dumps(failed))\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    if r.returncode < 0:
        return  # killed by a signal: the mutant's stray access showed up
    assert r.returncode == 0, r.stderr[-2000:]
    failed = json.loads(r.stdout.strip().splitlines()[-1])
    assert failed, f"no pin caught the planted mistake {name}"
