"""The pins must catch plausible mistakes in the oracle.

Each mutant is a copy of the oracle's C source with one deliberate mistake
(a dropped term, a wrong index, a transposed operand, an off-by-one mask),
compiled to a temporary library.  At least one pin must fail on every
mutant.  The mistakes are planted in copies on the CPU; the oracle source
itself is untouched.
"""
import os
import subprocess

import pytest

import oracle
from oracle.build import SRC
from tests.oracle_pins import ALL_PINS

MUTANTS = {
    "causal_off_by_one": ("j <= input_pos + i", "j < input_pos + i"),
    "input_pos_ignored": ("j <= input_pos + i", "j <= i"),
    "gqa_modulo_index": ("const long kvh = h / group;",
                         "const long kvh = h % Hkv;"),
    "scale_dropped": ("score[j] = scale * dot;", "score[j] = dot;"),
    "lse_log2": ("*lse = M + log(L);", "*lse = M + log2(L);"),
    "lse_without_max": ("*lse = M + log(L);", "*lse = log(L);"),
    "scores_use_v": ("dot += q[d] * k[j * D + d];",
                     "dot += q[d] * v[j * D + d];"),
    "output_uses_k": ("out[d] += prob[j] * v[j * D + d];",
                      "out[d] += prob[j] * k[j * D + d];"),
    "no_normalisation": ("prob[j] /= L;", "prob[j] /= 1.0;"),
    "max_not_subtracted": ("exp(score[j] - M)", "exp(score[j])"),
    "max_over_masked_keys": ("if (visible && score[j] > M)",
                             "if (score[j] > M)"),
    "wrong_query_row": ("(b * Hq + h) * Sq + i) * D",
                        "(b * Hq + h) * Sq + 0) * D"),
    "window_off_by_one": ("j > input_pos + i - window",
                          "j >= input_pos + i - window"),
    "window_ignored": ("return window <= 0 || j > input_pos + i - window;",
                       "return 1;"),
    "window_without_offset": ("j > input_pos + i - window",
                              "j > i - window"),
    "bwd_rowsum_dropped": ("const double ds = prob[j] * (dprob[j] - pdp);",
                           "const double ds = prob[j] * dprob[j];"),
    "bwd_dq_scale_dropped": ("dq[d] += scale * ds * k[j * D + d];",
                             "dq[d] += ds * k[j * D + d];"),
    "bwd_dk_uses_k": ("dk[j * D + d] += scale * ds * q[d];",
                      "dk[j * D + d] += scale * ds * k[j * D + d];"),
    "bwd_dv_uses_ds": ("dv[j * D + d] += prob[j] * dout[d];",
                       "dv[j * D + d] += ds * dout[d];"),
    "bwd_dp_uses_k": ("dot += dout[d] * v[j * D + d];",
                      "dot += dout[d] * k[j * D + d];"),
    "bwd_rows_rowsum_dropped": (
        "const double ds = prob[j] * (score[j] - pdp);",
        "const double ds = prob[j] * score[j];"),
    "bwd_keys_rowsum_dropped": ("const double ds = pj * (dp - pdp[rr]);",
                                "const double ds = pj * dp;"),
    "bwd_keys_dv_uses_ds": ("dv[d] += pj * dout[d];", "dv[d] += ds * dout[d];"),
    "bwd_keys_dk_scale_dropped": ("dk[d] += scale * ds * q[d];",
                                  "dk[d] += ds * q[d];"),
    "bwd_keys_wrong_group_head": (
        "const long h = gk * group + rr / Sq, i = rr % Sq;\n        const double* q",
        "const long h = rr / Sq, i = rr % Sq;\n        const double* q"),
    "e4m3_bias_8": ("ldexp((double)(8u + m), (int)e - 10)",
                    "ldexp((double)(8u + m), (int)e - 11)"),
    "e4m3_no_implicit_bit": ("ldexp((double)(8u + m), (int)e - 10)",
                             "ldexp((double)(m), (int)e - 7)"),
    "e4m3_subnormal_as_normal": ("if (e == 0u)\n    v = ldexp((double)m, -9);",
                                 "if (0)\n    v = ldexp((double)m, -9);"),
    "e4m3_sign_dropped": ("return s ? -v : v;", "return v;"),
    "e4m3_nan_whole_binade": ("if (e == 15u && m == 7u) return NAN;",
                              "if (e == 15u) return NAN;"),
    "e4m3_descale_dropped": (
        "out[i] = scale * attn_oracle_e4m3_value(in[i]);",
        "out[i] = attn_oracle_e4m3_value(in[i]);"),
}


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert old in source, "mutation anchor vanished: %r" % old
    mutated = source.replace(old, new)
    src = tmp_path / ("%s.c" % name)
    src.write_text(mutated)
    lib = tmp_path / ("lib%s.so" % name)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    str(src), "-o", str(lib), "-lm"], check=True)
    orc = oracle.Oracle(str(lib))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, "no pin caught mutant %s" % name
