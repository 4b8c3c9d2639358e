"""Mutation test for the oracle's pins.

Each case copies ``oracle/attn_oracle.c``, plants one plausible mistake (a
dropped term, a wrong sign, an off-by-one limit, a wrong index or operand),
compiles the copy with gcc and checks that at least one pin rejects it.  The
real oracle is never modified.  CPU only.
"""
import os
import subprocess

import pytest

import oracle
from oracle_pins import PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_oracle.c")

MUTANTS = {
    "drop_scale": ("double score = p->scale * dot;", "double score = dot;"),
    "causal_off_by_one": ("!(p->causal && j > causal_max)", "!(p->causal && j >= causal_max)"),
    "kv_head_modulo": ("const int64_t kvh = h / group;", "const int64_t kvh = h % p->Hkv;"),
    "mask_before_softcap": (
        "if (p->softcap > 0.0) score = p->softcap * tanh(score / p->softcap);\n"
        "        if (p->mask && p->mask_planes > 0)\n"
        "            score += (double)p->mask[(plane * p->Sq + qi) * p->Sk + j];",
        "if (p->mask && p->mask_planes > 0)\n"
        "            score += (double)p->mask[(plane * p->Sq + qi) * p->Sk + j];\n"
        "        if (p->softcap > 0.0) score = p->softcap * tanh(score / p->softcap);"),
    "mask_plane_per_head_drops_batch": ("plane = b * p->Hq + h;", "plane = h;"),
    "mask_plane_per_batch_uses_head": ("if (p->mask_planes == p->B) plane = b;",
                                       "if (p->mask_planes == p->B) plane = h % p->B;"),
    "mask_row_stride_capacity": ("* p->Sk + j];", "* p->kv_capacity + j];"),
    "window_off_by_one": ("causal_max + 1 - p->local_window", "causal_max - p->local_window"),
    "v_read_from_k": ("const float *vrow = p->v +", "const float *vrow = p->k +"),
    "no_normalisation": ("o[d] /= l;", "o[d] /= 1.0;"),
    "empty_row_not_zero": ("if (m == -INFINITY) return;", "if (m == -INFINITY) m = 0.0;"),
    "ignore_total_lengths": ("p->total_lengths ? (int64_t)p->total_lengths[b] : p->Sk",
                             "p->Sk"),
    "ignore_past_lengths": ("p->past_lengths ? (int64_t)p->past_lengths[b] + qi : lsk - p->Sq + qi",
                            "lsk - p->Sq + qi"),
    "causal_top_left": ("lsk - p->Sq + qi", "qi"),
    "token_major_as_head_major": ("o = t->out + ((b * p->Sq + qi) * p->Hq + h) * p->D;",
                                  "o = t->out + ((b * p->Hq + h) * p->Sq + qi) * p->D;"),
    "exp_sign_flipped": ("exp(s[j] - m)", "exp(m - s[j])"),
    "dot_q_with_q": ("(double)qrow[d] * (double)krow[d]", "(double)qrow[d] * (double)qrow[d]"),
    "softcap_without_inner_divide": ("p->softcap * tanh(score / p->softcap)",
                                     "p->softcap * tanh(score)"),
    "lse_drops_max": ("*lse = m + log(l);", "*lse = log(l);"),
    "lse_log2": ("*lse = m + log(l);", "*lse = m + log2(l);"),
    "kv_plane_ignores_batch": ("const int64_t kv_plane = (b * p->Hkv + kvh) * p->kv_capacity;",
                               "const int64_t kv_plane = kvh * p->kv_capacity;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found in the oracle"
    mutant_src = tmp_path / "attn_oracle_mutant.c"
    mutant_src.write_text(src.replace(old, new))
    lib_path = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O1", "-std=c99", "-fPIC", "-shared", "-o", lib_path,
                    str(mutant_src), "-lm", "-lpthread"], check=True)
    lib = oracle.load(lib_path)
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"no pin detects the planted mistake {name!r}"
