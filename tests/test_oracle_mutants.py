"""Planted mistakes in the oracle are caught by the pins (CPU only).

Each case copies the oracle's C source, changes one expression into a
plausible mistake (a dropped term, a wrong index or sign, a transposed
operand, a wrong rounding), compiles the copy into a temporary library and
runs the pin checks against it: at least one must fail.  The real oracle is
never modified.
"""
import os
import shutil

import pytest

import oracle
import pins

MUTANTS = {
    "window_position": ("(int64_t)(bt - 1 - t) * k", "(int64_t)(bt - t) * k"),
    "no_tail_biting_wrap": ("block_bit(block_words, (p + i) % n)", "block_bit(block_words, (p + i) % (n - 32))"),
    "window_bit_order": ("block_bit(block_words, (p + i) % n) << i", "block_bit(block_words, (p + i) % n) << (L - 1 - i)"),
    "lsb_last_in_word": ("(words[j / 32] >> (j % 32)) & 1u", "(words[j / 32] >> (31 - j % 32)) & 1u"),
    "weight_skips_f32_rounding": ("float prod = (float)((double)value * (double)s);\n    return tcq_oracle_bf16_from_float(prod);",
                                  "return tcq_oracle_bf16_from_double((double)value * (double)s);"),
    "scale_dropped": ("float s = tcq_oracle_bf16_to_float(scales[r]);", "float s = 1.0f;"),
    "ties_away_from_zero": ("double n = nearbyint(r);", "double n = round(r);"),
    "subnormal_spacing": ("if (q < -133) q = -133;", "if (q < -126) q = -126;"),
    "axis1_drops_sample_index": ("(double)tcq_oracle_bf16_to_float(x[m * cols + c]) *\n                           (double)tcq_oracle_bf16_to_float(w[r * cols + c]);\n                s += p;",
                                 "(double)tcq_oracle_bf16_to_float(x[c]) *\n                           (double)tcq_oracle_bf16_to_float(w[r * cols + c]);\n                s += p;"),
    "axis0_transposed_weight": ("(double)tcq_oracle_bf16_to_float(x[m * rows + r]) *\n                           (double)tcq_oracle_bf16_to_float(w[r * cols + c]);\n                s += p;",
                                "(double)tcq_oracle_bf16_to_float(x[m * rows + r]) *\n                           (double)tcq_oracle_bf16_to_float(w[c * rows + r]);\n                s += p;"),
    "abs_dropped": ("sa += fabs(p);", "sa += p;"),
    "split_rows_floor": ("int64_t rp = splits > 0 ? (rows + splits - 1) / splits : rows;",
                         "int64_t rp = splits > 0 ? rows / splits : rows;"),
    "interleave_word_offset": ("+ r * 2 * wpb + (b % 2) * wpb;", "+ r * 2 * wpb + (b % 2);"),
    "rmsnorm_no_mean": ("1.0 / sqrt(ss / (double)D + eps)", "1.0 / sqrt(ss + eps)"),
    "silu_sign": ("gv / (1.0 + exp(-gv)) * uv", "gv / (1.0 + exp(gv)) * uv"),
    "unrounded_weight_rounded": ("w_out[r * cols + c] = (float)((double)lut[win] * (double)s);",
                                 "w_out[r * cols + c] = tcq_oracle_bf16_to_float(tcq_oracle_bf16_from_double((double)lut[win] * (double)s));"),
    "default_splits_floor_log2": ("double s = pow(2.0, ceil(log2(ratio)));", "double s = pow(2.0, floor(log2(ratio)));"),
    "default_splits_no_row_tiles": ("double tiles_k = floor((double)rows / 16.0);", "double tiles_k = floor((double)rows / 32.0);"),
    "unrounded_axis0_transposed": ("(double)tcq_oracle_bf16_to_float(x[m * rows + r]) * (double)w[r * cols + c];",
                                   "(double)tcq_oracle_bf16_to_float(x[m * rows + r]) * (double)w[c * rows + r];"),
}


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc needed to build a mutant")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, source, tmp_path):
    old, new = MUTANTS[name]
    assert source.count(old) >= 1, f"pattern of mutant {name} not in the oracle"
    src = tmp_path / "mutant.c"
    src.write_text(source.replace(old, new, 1) if name != "abs_dropped" else source.replace(old, new))
    lib = oracle.compile_library(str(src), str(tmp_path / "libmutant.so"))
    o = oracle.Oracle(lib)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(o)
        except AssertionError:
            failed.append(check.__name__)
            break
    assert failed, f"no pin caught mutant {name}"
