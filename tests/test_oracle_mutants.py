"""Each plausible mistake planted in a copy of the oracle source must make at
least one pin fail.  The mutants are built on the CPU from a temporary copy of
oracle/tq_oracle.c; the committed oracle is never changed."""
import os
import shutil
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "tq_oracle.c")

# (name, text in tq_oracle.c, replacement): one planted mistake each
MUTANTS = [
    ("butterfly_sign", "v[i + h] = a - b;", "v[i + h] = b - a;"),
    ("stage_order", "for (int h = 1; h < 128; h *= 2) {", "for (int h = 64; h >= 1; h /= 2) {"),
    ("no_normalisation", "out[i] = v[i] * c;", "out[i] = v[i];"),
    ("popcount_bit", "return (ones & 1) ? -1 : 1;", "return (ones & 2) ? -1 : 1;"),
    ("sylvester_block", "h[(i + m) * n + (j + m)] = (int8_t)(-v);", "h[(i + m) * n + (j + m)] = v;"),
    ("f16_round_ties_down", "if (rem > half || (rem == half && (q & 1u))) q += 1;\n    if (q == 0x800u)",
     "if (rem > half) q += 1;\n    if (q == 0x800u)"),
    ("f16_subnormal_scale", "5.9604644775390625e-08f", "1.1920928955078125e-07f"),
    ("sequential_sum", "for (int h = 64; h >= 1; h /= 2)\n    for (int i = 0; i < h; ++i) s[i] = s[i] + s[i + h];",
     "for (int i = 1; i < 128; ++i) s[0] = s[0] + s[i];"),
    ("adjacent_tree", "for (int h = 64; h >= 1; h /= 2)\n    for (int i = 0; i < h; ++i) s[i] = s[i] + s[i + h];",
     "for (int h = 1; h < 128; h *= 2)\n    for (int i = 0; i + h < 128; i += 2 * h) s[i] = s[i] + s[i + h];"),
    ("mean_factor", "s[0] * 0.0078125f", "s[0] * 0.00390625f"),
    ("signed_sum", "s[i] = fabsf(wrot[i]);", "s[i] = wrot[i];"),
    ("divide_by_mean", "float q = wrot[i] / sc;", "float q = wrot[i] / mean;"),
    ("round_half_away", "float r = nearbyintf(q);", "float r = roundf(q);"),
    ("no_clamp", "t[i] = (int8_t)(r > 1.0f ? 1 : (r < -1.0f ? -1 : (int)r));",
     "t[i] = (int8_t)(r > 2.0f ? 1 : (r < -2.0f ? -1 : (int)r));"),
    ("skip_weight_rotation", "tqo_fwht128_f32(grp, rot);", "for (int i = 0; i < 128; ++i) rot[i] = grp[i];"),
    ("pack2_code_map", "unsigned code = (unsigned)(T[n * K + k] + 1);", "unsigned code = (unsigned)(1 - T[n * K + k]);"),
    ("pack2_bit_order", "(code << (2 * (k % 4)))", "(code << (6 - 2 * (k % 4)))"),
    ("pack3_digit_order", "v += d * p;", "v = v * 3 + d;"),
    ("pack3_pad_digit", ": 1u;", ": 0u;"),
    ("gemv_drops_scale", "y[m * nout + r] += (double)tqo_f16_to_f32(S[r * G + g]) * part;",
     "y[m * nout + r] += part;"),
    ("gemv_reversed_x", "blk[i] = (double)x[m * K + g * 128 + i];", "blk[i] = (double)x[m * K + g * 128 + (127 - i)];"),
    ("gemv_no_x_rotation", "tqo_fwht128_f64(blk, rot);\n      for (int64_t r",
     "for (int i = 0; i < 128; ++i) rot[i] = blk[i];\n      for (int64_t r"),
    # transform / group / residual variants
    ("fwhtn_stage_order", "for (int h = 1; h < n; h *= 2) {", "for (int h = n / 2; h >= 1; h /= 2) {"),
    ("fwhtn_norm_1_over_n", "float c = (float)(1.0 / sqrt((double)n));", "float c = (float)(1.0 / (double)n);"),
    ("group_n_mean_factor", "float inv = 1.0f / (float)g;", "float inv = 1.0f / 128.0f;"),
    ("group_n_sequential_sum", "for (int h = g / 2; h >= 1; h /= 2)\n    for (int i = 0; i < h; ++i) s[i] = s[i] + s[i + h];",
     "for (int i = 1; i < g; ++i) s[0] = s[0] + s[i];"),
    ("residual_sign", "wr[g + i] - s1f * (float)t1[g + i]", "wr[g + i] + s1f * (float)t1[g + i]"),
    ("residual_zero_trit_times_scale", "(t1[g + i] == 0) ? wr[g + i] : wr[g + i] - s1f * (float)t1[g + i]",
     "wr[g + i] - s1f * (float)t1[g + i]"),
    ("residual_no_second_rotation", "for (int b = 0; b < u; b += block) tqo_fwht_f32(block, r + b, rr + b);",
     "for (int i = 0; i < u; ++i) rr[i] = r[i];"),
    ("residual_x_not_rotated_twice", "tqo_fwht_f64(block, xr + k0, xrr + k0);",
     "for (int i = 0; i < block; ++i) xrr[k0 + i] = xr[k0 + i];"),
    ("layout_group_stride", "const int8_t *t = T + q * Keff + pass * K + g * group;",
     "const int8_t *t = T + q * Keff + pass * K + g * 128;"),
    # 2:4 sparse format
    ("sp24_tie_to_higher", "if (b > a || (b == a && o < i)) ++beaten;", "if (b > a || (b == a && o > i)) ++beaten;"),
    ("sp24_keep_three", "keep[4 * j + i] = (uint8_t)(beaten < 2);\n      if (beaten < 2)",
     "keep[4 * j + i] = (uint8_t)(beaten < 3);\n      if (beaten < 3 && nk < 64)"),
    ("sp24_signed_select", "float a = fabsf(wrot[4 * j + i]);", "float a = wrot[4 * j + i];"),
    ("sp24_mean_over_128", "float mean = kept[0] * 0.015625f;", "float mean = kept[0] * 0.0078125f;"),
    ("sp24_sequential_sum", "for (int h = 32; h >= 1; h /= 2)\n    for (int i = 0; i < h; ++i) kept[i] = kept[i] + kept[i + h];",
     "for (int i = 1; i < 64; ++i) kept[0] = kept[0] + kept[i];"),
    ("sp24_pruned_not_zeroed", "if (!keep[i] || sc == 0.0f) { t[i] = 0; continue; }", "if (sc == 0.0f) { t[i] = 0; continue; }"),
    ("sp24_pattern_order", "{{0, 1}, {0, 2}, {0, 3}, {1, 2}, {1, 3}, {2, 3}}", "{{0, 1}, {0, 2}, {1, 2}, {0, 3}, {1, 3}, {2, 3}}"),
    ("sp24_trit_order", "unsigned c = (unsigned)(9 * p + 3 * (t[kPat24[p][0]] + 1) + (t[kPat24[p][1]] + 1));",
     "unsigned c = (unsigned)(9 * p + (t[kPat24[p][0]] + 1) + 3 * (t[kPat24[p][1]] + 1));"),
    ("sp24_nibble_order", "grp[j / 2] = (uint8_t)(grp[j / 2] | ((c & 15u) << (4 * (j % 2))));",
     "grp[j / 2] = (uint8_t)(grp[j / 2] | ((c & 15u) << (4 - 4 * (j % 2))));"),
    ("sp24_high_plane_offset", "grp[16 + j / 4] = (uint8_t)(grp[16 + j / 4] | ((c >> 4) << (2 * (j % 4))));",
     "grp[16 + j / 4] = (uint8_t)(grp[16 + j / 4] | ((c >> 4) << (2 * (3 - j % 4))));"),
    ("sp24_unpack_digit_swap", "t[kPat24[p][0]] = (int8_t)(v / 3 - 1);\n        t[kPat24[p][1]] = (int8_t)(v % 3 - 1);",
     "t[kPat24[p][0]] = (int8_t)(v % 3 - 1);\n        t[kPat24[p][1]] = (int8_t)(v / 3 - 1);"),
    ("sp24_unpack_uncounted_bad", "if (c >= 54) { ++bad; continue; }", "if (c >= 54) { continue; }"),
]


# sites that occur more than once: (name, text, replacement, which occurrence)
# (the layout variants of the transform and the quantiser repeat lines of
# the 128-point functions, and the 2:4 quantiser repeats the trit rule and the
# row rotation: occurrence 0 is the 128-point function, 1 the layout variant,
# 2 the 2:4 form)
_REPEATED = ("butterfly_sign", "no_normalisation", "signed_sum", "divide_by_mean", "round_half_away", "no_clamp")
_REPEATED3 = ("divide_by_mean", "round_half_away", "no_clamp")
MUTANTS_NTH = [(*m, 0) for m in MUTANTS if m[0] in _REPEATED] + \
    [("n_" + m[0], m[1], m[2], 1) for m in MUTANTS if m[0] in _REPEATED] + \
    [("sp24_" + m[0], m[1], m[2], 2) for m in MUTANTS if m[0] in _REPEATED3] + \
    [(*m, 0) for m in MUTANTS if m[0] == "skip_weight_rotation"] + \
    [("sp24_" + m[0], m[1], m[2], 1) for m in MUTANTS if m[0] == "skip_weight_rotation"]
MUTANTS = [m for m in MUTANTS if m[0] not in _REPEATED and m[0] != "skip_weight_rotation"]
ALL_MUTANTS = [(*m, None) for m in MUTANTS] + MUTANTS_NTH


def _replace(src: str, old: str, new: str, nth):
    if nth is None:
        assert src.count(old) == 1, "mutation site not unique"
        return src.replace(old, new)
    parts = src.split(old)
    assert len(parts) > nth + 1, "mutation site missing"
    return old.join(parts[:nth + 1]) + new + old.join(parts[nth + 1:])


@pytest.mark.parametrize("name,old,new,nth", ALL_MUTANTS, ids=[m[0] for m in ALL_MUTANTS])
def test_mutant_is_caught(tmp_path, name, old, new, nth):
    src = open(SRC).read()
    mut = tmp_path / "tq_oracle.c"
    mut.write_text(_replace(src, old, new, nth))
    shutil.copy(os.path.join(os.path.dirname(SRC), "tq_oracle.h"), tmp_path / "tq_oracle.h")
    lib = str(tmp_path / f"lib_{name}.so")
    subprocess.run(["gcc", *oracle.CFLAGS, "-I", str(tmp_path), "-o", lib, str(mut), "-lm"], check=True)
    orc = oracle.Oracle(lib)
    failed = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(orc)
        except (AssertionError, ValueError):  # a pin that rejects the mutant's output catches it too
            failed.append(check.__name__)
    assert failed, f"mutant {name} passed every pin"
