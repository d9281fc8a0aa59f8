"""The oracle's pins catch plausible mistakes in it: each mutant below is one
such mistake planted in a copy of cider_oracle.c (a reordered product, a
reciprocal for a division, ties away from zero, a dropped term, swapped
nibbles, a wrong index, a different accumulation order...), built on the
CPU, and the pin suite must fail against it. Two mistakes are not listed
because no input can tell them apart from the oracle: a min-max clamp at
-128 instead of -127 (|x / s| stays below 127.5 for every finite input,
subnormal bf16 scales included), and sending binary32 values above 65520
instead of from 65520 to the fp16 overflow branch (65520 itself rounds to
even on the ordinary path, carries out of the top binade and also gives
infinity). No GPU needed."""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, text in cider_oracle.c, replacement)
M = [
 ("pc_scale_order", "    float t = (float)acc * s_act;\n    t = t * s_weight;", "    float t = (float)acc * (s_act * s_weight);"),
 ("quant_reciprocal", "        float r = rintf(x / scale);", "        float r = rintf(x * (1.0f / scale));"),
 ("quant_ties_away", "        float r = rintf(x / scale);", "        float r = roundf(x / scale);"),
 ("absmax_skips_last", "    for (int64_t k = 0; k < n; ++k) {\n        float a = fabsf(elem_to_float(v[k], dtype));",
                       "    for (int64_t k = 0; k < n - 1; ++k) {\n        float a = fabsf(elem_to_float(v[k], dtype));"),
 ("pack_nibbles_swapped", "            wp[n * (K / 2) + j] = (uint8_t)(lo | (hi << 4));", "            wp[n * (K / 2) + j] = (uint8_t)(hi | (lo << 4));"),
 ("unpack_nibbles_swapped", "            wq[n * K + 2 * j] = (int8_t)((int)(b & 0x0F) - 8);\n            wq[n * K + 2 * j + 1] = (int8_t)((int)(b >> 4) - 8);",
                            "            wq[n * K + 2 * j] = (int8_t)((int)(b >> 4) - 8);\n            wq[n * K + 2 * j + 1] = (int8_t)((int)(b & 0x0F) - 8);"),
 ("int4_offset_7", "            uint8_t lo = (uint8_t)(codes[2 * j] + 8);", "            uint8_t lo = (uint8_t)(codes[2 * j] + 7);"),
 ("pg_descending", "    for (int64_t g = 0; g < G; ++g)\n        f = f + (float)partials[g] * s_weight_row[g];",
                   "    for (int64_t g = G - 1; g >= 0; --g)\n        f = f + (float)partials[g] * s_weight_row[g];"),
 ("pg_sact_per_group", "        f = f + (float)partials[g] * s_weight_row[g];\n    return float_to_elem(f * s_act, y_dtype);",
                       "        f = f + ((float)partials[g] * s_weight_row[g]) * s_act;\n    return float_to_elem(f, y_dtype);"),
 ("pg_fma", "        f = f + (float)partials[g] * s_weight_row[g];", "        f = fmaf((float)partials[g], s_weight_row[g], f);"),
 ("layer_drops_last_k", "                for (int64_t k = g * gs; k < (g + 1) * gs; ++k)\n                    acc += (int32_t)q[k] * (int32_t)wrow[k];",
                        "                for (int64_t k = g * gs; k < (g + 1) * gs - 1; ++k)\n                    acc += (int32_t)q[k] * (int32_t)wrow[k];"),
 ("gemm_drops_last_k", "                for (int64_t k = g * gs; k < (g + 1) * gs; ++k)\n                    acc += (int32_t)q[m * K + k] * (int32_t)wq[n * K + k];",
                       "                for (int64_t k = g * gs; k < (g + 1) * gs - 1; ++k)\n                    acc += (int32_t)q[m * K + k] * (int32_t)wq[n * K + k];"),
 ("half_truncates", "    double n = rint(a / quantum); /* exact quotient; rint rounds ties to even */\n    uint32_t out;\n    if (unbiased == -14",
                    "    double n = floor(a / quantum); /* exact quotient; rint rounds ties to even */\n    uint32_t out;\n    if (unbiased == -14"),
 ("half_ties_away", "    double n = rint(a / quantum); /* exact quotient; rint rounds ties to even */\n    uint32_t out;\n    if (unbiased == -14",
                    "    double n = round(a / quantum); /* exact quotient; rint rounds ties to even */\n    uint32_t out;\n    if (unbiased == -14"),
 ("bf16_truncates", "    double n = rint(a / quantum); /* exact quotient; rint rounds ties to even */\n    uint32_t out;\n    if (unbiased == -126",
                    "    double n = floor(a / quantum); /* exact quotient; rint rounds ties to even */\n    uint32_t out;\n    if (unbiased == -126"),
 ("half_subnormal_step", "        mag = ldexpf((float)frac, -24); /* subnormal: frac * 2^-24 */", "        mag = ldexpf((float)frac, -25); /* subnormal: frac * 2^-24 */"),
 ("pct_position_n", "    double h = (double)(n - 1) * pct / 100.0;", "    double h = (double)n * pct / 100.0;"),
 ("pct_no_interpolation", "    double c = (i + 1 < n) ? (double)q[i] + (h - (double)i) * ((double)q[i + 1] - (double)q[i])",
                          "    double c = (i + 1 < n) ? (double)q[i] + 0.0 * ((double)q[i + 1] - (double)q[i])"),
 ("a16_no_scale", "            total += (double)s_w[n * G + g] * part;", "            total += part;"),
 ("a16_nibbles_swapped", "                    code = (int)((k % 2) ? (b >> 4) : (b & 0x0F)) - 8;", "                    code = (int)((k % 2) ? (b & 0x0F) : (b >> 4)) - 8;"),
 ("pc_scale_index", "                y[m * N + n] = oracle_epilogue_pc_ex(part[0], s_act, s_w[n], y_dtype);", "                y[m * N + n] = oracle_epilogue_pc_ex(part[0], s_act, s_w[0], y_dtype);"),
 ("pg_scale_row", "                y[m * N + n] = oracle_epilogue_pg_ex(part, s_w + n * G, G, s_act, y_dtype);", "                y[m * N + n] = oracle_epilogue_pg_ex(part, s_w + n, G, s_act, y_dtype);"),
 ("act_qmax_128", "        s[m] = quantize_block_t(x + m * K, K, 127.0f, q + m * K, x_dtype);", "        s[m] = quantize_block_t(x + m * K, K, 128.0f, q + m * K, x_dtype);"),
 ("layer_act_qmax_126", "        float s_act = quantize_block_t(x + m * K, K, 127.0f, q, x_dtype);", "        float s_act = quantize_block_t(x + m * K, K, 126.0f, q, x_dtype);"),
 ("int4_qmax_8", "            s_w[n * G + g] = quantize_block(w + n * K + g * gs, gs, 7.0f, codes + g * gs);", "            s_w[n * G + g] = quantize_block(w + n * K + g * gs, gs, 8.0f, codes + g * gs);"),
 ("weight_group_index", "            s_w[n * G + g] = quantize_block(w + n * K + g * gs, gs, 127.0f, wq + n * K + g * gs);", "            s_w[g * N + n] = quantize_block(w + n * K + g * gs, gs, 127.0f, wq + n * K + g * gs);"),
 ("bf16_input_as_half", "    return dtype == ORACLE_BF16 ? oracle_bf16_to_float(v) : oracle_half_to_float(v);", "    return oracle_half_to_float(v);"),
 ("pct_sort_descending", "    return (x > y) - (x < y);", "    return (x < y) - (x > y);"),
 ("pct_no_saturation", "        float r = rintf(elem_to_float(v[k], dtype) / scale);\n        if (r > qmax)\n            r = qmax;", "        float r = rintf(elem_to_float(v[k], dtype) / scale);\n        if (r > 1000.0f)\n            r = qmax;"),
 ("absmax_signed", "        float a = fabsf(elem_to_float(v[k], dtype));\n        if (a > absmax)", "        float a = elem_to_float(v[k], dtype);\n        if (a > absmax)"),
 ("layer_weights_reversed", "                    acc += (int32_t)q[k] * (int32_t)wrow[k];", "                    acc += (int32_t)q[k] * (int32_t)wrow[K - 1 - k];"),
 ("gemm_weight_row_reversed", "                    acc += (int32_t)q[m * K + k] * (int32_t)wq[n * K + k];", "                    acc += (int32_t)q[m * K + k] * (int32_t)wq[(N - 1 - n) * K + k];"),
 ("half_exponent_bias", "        mag = ldexpf((float)(frac | 0x400), expo - 25); /* 1.frac * 2^(expo-15) */", "        mag = ldexpf((float)(frac | 0x400), expo - 24); /* 1.frac * 2^(expo-15) */"),
 ("int4_groups_overwrite", "            s_w[n * G + g] = quantize_block(w + n * K + g * gs, gs, 7.0f, codes + g * gs);", "            s_w[n * G + g] = quantize_block(w + n * K + g * gs, gs, 7.0f, codes);"),
 ("weight_qmax_126", "            s_w[n * G + g] = quantize_block(w + n * K + g * gs, gs, 127.0f, wq + n * K + g * gs);", "            s_w[n * G + g] = quantize_block(w + n * K + g * gs, gs, 126.0f, wq + n * K + g * gs);"),
 ("zero_row_code_one", "    if (absmax == 0.0f) {\n        for (int64_t k = 0; k < n; ++k)\n            out[k] = 0;\n        return 0.0f;\n    }\n    float scale = absmax / qmax;", "    if (absmax == 0.0f) {\n        for (int64_t k = 0; k < n; ++k)\n            out[k] = 1;\n        return 0.0f;\n    }\n    float scale = absmax / qmax;"),
 ("pc_output_always_half", "    t = t * s_weight;\n    return float_to_elem(t, y_dtype);", "    t = t * s_weight;\n    return oracle_float_to_half(t);"),
 ("half_subnormal_floor", "    if (unbiased < -14)\n        unbiased = -14;", "    if (unbiased < -15)\n        unbiased = -15;"),
 ("bf16_carry", "        if (n >= 256.0) {        /* rounding carried into the next binade */\n            n = 128.0;\n            expo += 1;\n        }", "        if (n > 256.0) {        /* rounding carried into the next binade */\n            n = 128.0;\n            expo += 1;\n        }"),
 ("a16_group_scale_index", "            total += (double)s_w[n * G + g] * part;", "            total += (double)s_w[n * G] * part;"),
 ("pct_zero_clip_saturates", "    if (clip == 0.0f) {\n        for (int64_t k = 0; k < n; ++k)\n            out[k] = 0;",
                             "    if (clip == 0.0f) {\n        for (int64_t k = 0; k < n; ++k)\n            out[k] = (int8_t)(elem_to_float(v[k], dtype) > 0.0f ? qmax : elem_to_float(v[k], dtype) < 0.0f ? -qmax : 0.0f);"),
 ("pct_interp_weight", "(h - (double)i) * ((double)q[i + 1] - (double)q[i])", "(1.0 - (h - (double)i)) * ((double)q[i + 1] - (double)q[i])"),
]


def _killed(tmp, name, old, new):
    src = open(oracle._SRC).read()
    assert src.count(old) == 1, f"{name}: the oracle text it mutates has changed"
    c = os.path.join(tmp, f"mut_{name}.c")
    lib = os.path.join(tmp, f"libmut_{name}.so")
    with open(c, "w") as f:
        f.write(src.replace(old, new))
    subprocess.run(["gcc", *oracle._CFLAGS, "-o", lib, c, "-lm"], check=True)
    code = ("import sys\n"
            f"sys.path[:0] = [{ROOT!r}, {os.path.join(ROOT, 'tests')!r}]\n"
            "import oracle\n"
            f"oracle._LIB_PATH = {lib!r}\n"
            "import pytest\n"
            f"sys.exit(pytest.main(['-q', '-x', '-p', 'no:cacheprovider', {PINS!r}]))\n")
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=900)
    return r.returncode != 0


def test_every_planted_mistake_fails_a_pin(tmp_path):
    if subprocess.run(["which", "gcc"], capture_output=True).returncode != 0:
        pytest.skip("no gcc")
    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda m: (m[0], _killed(str(tmp_path), *m)), M))
    survivors = [name for name, killed in results if not killed]
    assert not survivors, f"mutants the pins do not catch: {survivors}"
