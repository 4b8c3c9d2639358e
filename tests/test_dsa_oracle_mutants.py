"""Mutation test for the DSA oracle's pins.

Each case copies ``oracle/dsa_oracle.c``, plants one plausible mistake (a
dropped factor, a wrong comparison, a reversed summation order, a wrong tie
rule, contraction into fused multiply-adds), compiles the copy and checks
that at least one pin rejects it.  The real oracle is never modified.  CPU
only.
"""
import os

import pytest

from dsa_oracle_pins import PINS
from oracle import dsa

SRC = os.path.join(os.path.dirname(dsa.__file__), "dsa_oracle.c")

MUTANTS = {
    "allow_at_threshold": ("const int ok = bt > -1e30f;", "const int ok = bt >= -1e30f;"),
    "rows_allow_at_threshold": ("al[t] = (unsigned char)(bt > -1e30f);", "al[t] = (unsigned char)(bt >= -1e30f);"),
    "no_relu": ("scored = scored > 0.0f ? scored : 0.0f;", "scored = scored;"),
    "drop_weights_scale": ("const float wprod = w[h] * weights_scale;", "const float wprod = w[h];"),
    "drop_scale": ("float scored = scale * dot;", "float scored = dot;"),
    "dot_reversed": ("for (int64_t d = 0; d < D; ++d) {", "for (int64_t d = D - 1; d >= 0; --d) {"),
    "heads_reversed": ("for (int64_t h = 0; h < H; ++h) {", "for (int64_t h = H - 1; h >= 0; --h) {"),
    "key_ignores_batch": ("key + (b * T + t) * D, weights + row * H, bt, H, D, scale,\n                            weights_scale)",
                          "key + t * D, weights + row * H, bt, H, D, scale,\n                            weights_scale)"),
    "drop_bias": ("float score = weighted + bias;", "float score = weighted;"),
    "ties_to_highest_index": ("return (a->index > b->index) - (a->index < b->index);",
                              "return (a->index < b->index) - (a->index > b->index);"),
    "output_unsorted": ("qsort(out, (size_t)keep, sizeof(int64_t), index_order);", "(void)index_order;"),
    "pad_with_zero": ("for (int64_t i = keep; i < top_k; ++i) out[i] = -1;",
                      "for (int64_t i = keep; i < top_k; ++i) out[i] = 0;"),
    "no_nan_canonicalisation": ("if (isnan(score)) score = canonical_nan();", "(void)canonical_nan;"),
    "zeros_unordered": ("if (a == 0.0f && sa != sb) return sa ? -1 : 1;", "(void)sb;"),
    "nan_lowest": ("const int ra = na ? (sa ? -2 : 2) : 0;", "const int ra = na ? -2 : 0;"),
    "keep_one_fewer": ("const int64_t keep = n < top_k ? n : top_k;",
                       "const int64_t keep = n < top_k ? n : top_k - 1;"),
    "fused_dot_product": ("const float prod = q[h * D + d] * k[d];\n      dot = dot + prod;",
                          "dot = fmaf(q[h * D + d], k[d], dot);"),
    "fused_head_sum": ("const float term = scored * wprod;\n    weighted = weighted + term;",
                       "weighted = fmaf(scored, wprod, weighted);"),
}


def _check_mutant(path):
    lib = dsa.load(path)
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    return caught


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found in the oracle"
    mutant = tmp_path / "dsa_oracle_mutant.c"
    mutant.write_text(src.replace(old, new, 1))
    lib_path = str(tmp_path / "libmutant.so")
    import subprocess
    subprocess.run(["gcc", *dsa.CFLAGS, "-o", lib_path, str(mutant), "-lm"], check=True)
    assert _check_mutant(lib_path), f"no pin caught the mutant {name}"
