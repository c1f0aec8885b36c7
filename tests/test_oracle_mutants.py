"""Planted mistakes in the oracle must fail at least one pin.

Each mutant is a copy of qoq_oracle.c with one plausible slip (a dropped term,
a wrong sign, index or rounding rule, a transposed operand), compiled on the
CPU into a temporary directory.  The pins of ``oracle_pins`` run against it
and at least one must fail.  Nothing here touches a GPU.
"""
import os

import pytest

import oracle
from tests import oracle_pins

MUTANTS = {
    "tie_half_up": ("if (2 * r == b) return (q & 1) ? q + 1 : q;", "if (2 * r == b) return q + 1;"),
    "s2_floor": ("int64_t scale = (hi - lo + 14) / 15;", "int64_t scale = (hi - lo) / 15;"),
    "dequant_sign": ("return (q - zero) * scale;\n}\n\n/* Same", "return (zero - q) * scale;\n}\n\n/* Same"),
    "no_protective_range": ("symmetric_row(K, wrow, 119, &s1[n], row_q8);",
                            "symmetric_row(K, wrow, 127, &s1[n], row_q8);"),
    "range_without_zero": ("int64_t lo = 0, hi = 0;", "int64_t lo = grp[0], hi = grp[0];"),
    "group_index": ("int64_t w = qoq_oracle_dequant_code(q4row[k], zrow[k / g], s2row[k / g]);",
                    "int64_t w = qoq_oracle_dequant_code(q4row[k], zrow[k % g], s2row[k / g]);"),
    "dropped_s1": ("double y = (double)acc * qoq_oracle_half_to_double(sx) * qoq_oracle_half_to_double(s1);",
                   "double y = (double)acc * qoq_oracle_half_to_double(sx);"),
    "truncate_codes": ("float r = rintf(t);", "float r = truncf(t);"),
    "transposed_operand": ("for (int n = 0; n < N; ++n) {\n      int64_t a = dot_entry(K, g, Xq + (size_t)m * K, q4 + (size_t)n * K,",
                           "for (int n = 0; n < N; ++n) {\n      int64_t a = dot_entry(K, g, Xq + (size_t)(n % M) * K, q4 + (size_t)(m % N) * K,"),
    "half_rounding_floor": ("double r = nearbyint(a / quantum);", "double r = floor(a / quantum);"),
    "zero_point_floor": ("int64_t zero = rne_div(-lo, scale);", "int64_t zero = floor_div(-lo, scale);"),
    "act_scale_127_to_119": ("symmetric_row(K, X + (size_t)m * K, 127, &sx[m], Xq + (size_t)m * K);",
                             "symmetric_row(K, X + (size_t)m * K, 119, &sx[m], Xq + (size_t)m * K);"),
    "norm_square_overflow": ("s2 += (unsigned __int128)mag * mag;", "s2 += (unsigned __int128)(mag * mag);"),
    "norm_missing_eps": ("volatile float den = spread + eps;", "volatile float den = spread;"),
    "layer_no_centering": ("volatile float t = kind == 1 ? x - mu : x;", "volatile float t = x;"),
    "layer_variance_sign": ("(unsigned __int128)K * s2 - a1 * a1;", "(unsigned __int128)K * s2 + a1 * a1;"),
    "rms_mean_divisor": ("spread = s2f / (float)K;", "spread = s2f / (float)(K + 1);"),
    "folded_correction_sign": ("const int64_t a = scaled - corr;", "const int64_t a = scaled + corr;"),
    "folded_zero_without_scale": ("corr += ((int64_t)z[(size_t)n * G + j] * s2[(size_t)n * G + j]) * RS[(size_t)m * G + j];",
                                  "corr += (int64_t)z[(size_t)n * G + j] * RS[(size_t)m * G + j];"),
    "folded_rowsum_range": ("for (int k = j * g; k < (j + 1) * g; ++k) t += Xq[(size_t)m * K + k];",
                            "for (int k = j * g; k < (j + 1) * g - 1; ++k) t += Xq[(size_t)m * K + k];"),
    "w4ax_four_bit_range": ("b < n8 ? 127 : 7, &sxb", "b < n8 ? 127 : 8, &sxb"),
    "w4ax_leading_blocks": ("b < n8 ? 127 : 7, &sxb", "b <= n8 ? 127 : 7, &sxb"),
    "w4ax_block_scale_index": ("y += qoq_oracle_half_to_double(sxb[(size_t)m * B + b]) * (double)a;",
                               "y += qoq_oracle_half_to_double(sxb[(size_t)m * B]) * (double)a;"),
    "norm_unrounded_product": ("volatile float w = u * (float)qoq_oracle_half_to_double(gamma[k]);",
                               "volatile float w = (float)((double)t * (double)r * qoq_oracle_half_to_double(gamma[k]));"),
    "threads_range_gap": ("(int)((int64_t)N * (t + 1) / threads),", "(int)((int64_t)N * (t + 1) / threads) - (t & 1),"),
    "threads_group_index": ("r->s2[(size_t)n * G + k / r->g]);", "r->s2[(size_t)n * G + k % G]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    src = open(oracle.SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found exactly once"
    mpath = os.path.join(tmp_path, f"m_{name}.c")
    with open(mpath, "w") as f:
        f.write(src.replace(old, new))
    lib = oracle.compile_source(mpath, os.path.join(tmp_path, f"lib_{name}.so"))
    o = oracle.Oracle(lib)
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(o)
        except (AssertionError, oracle.OracleError, ValueError, IndexError):
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
