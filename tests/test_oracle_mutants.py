"""The oracle's pins must catch plausible mistakes.

Each case copies the oracle's C source, plants one mistake by text
substitution, builds the copy in a temporary folder and runs the pins of
``test_oracle`` against it: at least one must fail.  Mistakes are planted only
in a copy of the oracle, on the CPU.  A mutant that crashes its process (an
out-of-bounds access) counts as caught.
"""
import os
import subprocess
import sys
import tempfile

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = os.path.join(os.path.dirname(oracle.__file__), "pkv_oracle.c")

MUTANTS = {
    "gqa_modulo": ("int g = h / group;", "int g = h % num_kv_heads;"),
    "scale_dropped": ("x[t] = scale * dot;", "x[t] = dot;"),
    "exp_sign": ("w[t] = exp(x[t] - m);", "w[t] = exp(m - x[t]);"),
    "max_is_min": ("if (x[t] > m)", "if (x[t] < m)"),
    "no_normalise": ("w[t] /= z;", "w[t] /= 1.0;"),
    "row_from_block": ("kv_head, t % page_tokens, page_tokens, head_dim);",
                       "kv_head, (t / page_tokens) % page_tokens, page_tokens, head_dim);"),
    "head_row_transposed": ("((int64_t)kv_head * page_tokens + row) * head_dim",
                            "((int64_t)row * page_tokens + kv_head) * head_dim"),
    "last_token_dropped": ("for (int t = 0; t < ctx; ++t) {\n                int64_t page = token_page(row,",
                           "for (int t = 0; t < ctx - 1; ++t) {\n                int64_t page = token_page(row,"),
    "v_from_k_pool": ("o[d] += w[t] * bf16_value(v_pool[v0 + d]);", "o[d] += w[t] * bf16_value(k_pool[v0 + d]);"),
    "block_index_off_by_one": ("int32_t p = table_row[t / page_tokens];", "int32_t p = table_row[(t + 1) / page_tokens];"),
}

@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "pkv_oracle_mut.c")
        with open(path, "w") as f:
            f.write(src.replace(old, new, 1))
        so = os.path.join(d, "libmut.so")
        subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-shared", "-fPIC", "-o", so,
                               path, "-lm"])
        # A mutant may also read or write out of bounds; run it in its own process.
        r = subprocess.run([sys.executable, "-m", "tests._mutant_runner", so], cwd=ROOT,
                           capture_output=True, text=True, timeout=600)
        crashed = r.returncode < 0
        assert crashed or "CAUGHT" in r.stdout, f"no pin caught the planted mistake {name}: {r.stdout}{r.stderr}"
