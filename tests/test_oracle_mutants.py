"""Planted mistakes in a copy of the oracle must each fail at least one pin.

Every mutant is a small textual change to a temporary copy of oracle/q8_oracle.c,
compiled with the same flags; the committed oracle is never modified.
"""
import os
import subprocess

import pytest

import oracle
from oracle_pins import ALL_PINS

SRC = os.path.join(os.path.dirname(oracle.__file__), "q8_oracle.c")

MUTANTS = {
    "reciprocal_multiply": ("float r = roundf(v[i] / d);", "float r = roundf(v[i] * (1.0f / d));"),
    "ties_to_even": ("float r = roundf(v[i] / d);", "float r = rintf(v[i] / d);"),
    "floor_plus_half": ("float r = roundf(v[i] / d);", "float r = floorf(v[i] / d + 0.5f);"),
    "divisor_128": ("float d = amax / 127.0f;", "float d = amax / 128.0f;"),
    "signed_max": ("float a = fabsf(v[i]);", "float a = v[i];"),
    "dropped_last_block": ("for (int64_t b = 0; b < nb; b++) {\n                const uint8_t *blk = block_ptr(w, r, b, nb);\n                int32_t dot",
                           "for (int64_t b = 0; b < nb - 1; b++) {\n                const uint8_t *blk = block_ptr(w, r, b, nb);\n                int32_t dot"),
    "act_scale_of_block0": ("float da = xd[t * nb + b];", "float da = xd[t * nb];"),
    "reversed_operand": ("s += (int32_t)wq[i] * (int32_t)xq[i];", "s += (int32_t)wq[i] * (int32_t)xq[QK - 1 - i];"),
    "negated_dot": ("s += (int32_t)wq[i] * (int32_t)xq[i];", "s -= (int32_t)wq[i] * (int32_t)xq[i];"),
    "f16_truncate": ("if (rem > half || (rem == half && (q & 1u)))", "if (0)"),
    "f16_ties_away": ("if (rem > half || (rem == half && (q & 1u)))", "if (rem >= half)"),
    "f16_decode_bias": ("v = ldexpf((float)(1024 + f), e - 25);", "v = ldexpf((float)(1024 + f), e - 24);"),
    "dequant_unrounded_scale": ("float dw = block_scale(blk);\n            const int8_t *wq",
                                "float dw = block_scale(blk) * 1.0001f;\n            const int8_t *wq"),
    "repack_scales_row_major": ("wdt[b * ldn + r] = block_scale(blk);", "wdt[r * nb + b] = block_scale(blk);"),
    "repack_offset_binary": ("wq16[r * k + b * QK + i] = oracle_f32_to_f16((float)wq[i]);",
                             "wq16[r * k + b * QK + i] = oracle_f32_to_f16((float)(wq[i] + 128));"),
    "q4_nibble_halves_swapped": ("int nib = (i < 16) ? (byte & 0x0f) : (byte >> 4);",
                                 "int nib = (i < 16) ? (byte >> 4) : (byte & 0x0f);"),
    "q4_consecutive_pairs": ("uint8_t byte = blk[2 + (i & 15)];\n    int nib = (i < 16) ? (byte & 0x0f) : (byte >> 4);",
                             "uint8_t byte = blk[2 + (i >> 1)];\n    int nib = (i & 1) ? (byte >> 4) : (byte & 0x0f);"),
    "q4_bias_7": ("return nib - 8;", "return nib - 7;"),
    "q4_writer_divisor_8": ("float d = amax / 7.0f;", "float d = amax / 8.0f;"),
    "q4_dropped_last_block": ("for (int64_t b = 0; b < nb; b++) {\n                const uint8_t *blk = q4_0_block_ptr(w, r, b, nb);\n                int32_t dot",
                              "for (int64_t b = 0; b < nb - 1; b++) {\n                const uint8_t *blk = q4_0_block_ptr(w, r, b, nb);\n                int32_t dot"),
    "q4_dequant_unrounded_scale": ("out[r * k + b * QK + i] = oracle_f32_to_f16(dw * (float)q4_0_value(blk, i));",
                                   "out[r * k + b * QK + i] = oracle_f32_to_f16(dw * 1.0001f * (float)q4_0_value(blk, i));"),
    # K-quant superblocks
    "q6k_scale_per_32": ("int sc = (int)(int8_t)sb[192 + e / 16];", "int sc = (int)(int8_t)sb[192 + e / 32];"),
    "q6k_qh_shift": ("int hi = (sb[128 + 32 * h + l] >> (2 * g)) & 3;", "int hi = (sb[128 + 32 * h + l] >> g) & 3;"),
    "q6k_ql_halves": ("int byte = sb[64 * h + 32 * (g % 2) + l];", "int byte = sb[64 * h + 32 * (g / 2) + l];"),
    "q6k_offset_31": ("return (double)f16_at(sb + 208) * (double)sc * (double)(q - 32);",
                      "return (double)f16_at(sb + 208) * (double)sc * (double)(q - 31);"),
    "q6k_block_scale_pair": ("*E = (int32_t)(int8_t)sb[192 + 2 * i] * d0 + (int32_t)(int8_t)sb[192 + 2 * i + 1] * d1;",
                             "*E = (int32_t)(int8_t)sb[192 + i] * d0 + (int32_t)(int8_t)sb[192 + i + 8] * d1;"),
    "k4_high_bits_swapped": ("*sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);", "*sc = (s[j + 4] & 15) | ((s[j] >> 6) << 4);"),
    "k4_scale_min_nibbles": ("*m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);", "*m = (s[j + 4] & 15) | ((s[j] >> 6) << 4);"),
    "k4_nibble_order": ("int q = u ? (byte >> 4) : (byte & 15);", "int q = u ? (byte & 15) : (byte >> 4);"),
    "k5_qh_bit": ("q += 16 * ((sb[16 + l] >> (2 * g + u)) & 1);", "q += 16 * ((sb[16 + l] >> (g + 4 * u)) & 1);"),
    "k4_min_added": ("return (double)f16_at(sb) * (double)sc * (double)q - (double)f16_at(sb + 2) * (double)m;",
                     "return (double)f16_at(sb) * (double)sc * (double)q + (double)f16_at(sb + 2) * (double)m;"),
    "k4_fold_min_dropped": ("float v = dsc * (float)D - dmm * (float)X;", "float v = dsc * (float)D;"),
    "f64_f16_subnormal_shift": ("int shift = (e >= -14) ? 42 : (28 - e);", "int shift = (e >= -14) ? 42 : (29 - e);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"anchor for {name} not found"
    mutated = src.replace(old, new)
    c = tmp_path / "mut.c"
    so = tmp_path / "libmut.so"
    c.write_text(mutated)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", str(so), str(c), "-lm"], check=True)
    o = oracle.bound(oracle.Oracle(str(so)))
    failed = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
