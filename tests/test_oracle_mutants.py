"""Planted mistakes: each is a plausible slip in the oracle's C source, built
on the CPU into a separate library, and the pin tests must fail on every one.
This shows the pins constrain each step of the oracle, not just its shape."""
import os
import subprocess
import sys

import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(os.path.dirname(HERE), "oracle", "moe_oracle.c")

MUTANTS = {
    "gate_up_swapped": ("h[n] = g[n] / (1.0 + exp(-g[n])) * u[n];",
                        "h[n] = u[n] / (1.0 + exp(-u[n])) * g[n];"),
    "sigmoid_sign": ("h[n] = g[n] / (1.0 + exp(-g[n])) * u[n];",
                     "h[n] = g[n] / (1.0 + exp(g[n])) * u[n];"),
    "down_transposed": ("                o[m] += hq[n] * bf16_value(wd[m]);",
                        "                o[m] += hq[n] * bf16_value(Wd->b16[e * (long)f * d + (long)m * f + n]);"),
    "weight_dropped": ("yt[m] += wt * jobs[jb].o[m];", "yt[m] += jobs[jb].o[m];"),
    "no_padding": ("offsets[e + 1] = (int32_t)(offsets[e] + tiles * tm);",
                   "offsets[e + 1] = (int32_t)(offsets[e] + counts[e]);"),
    "pad_token_zero": ("            srt_tok[r] = -1;\n            srt_w[r] = 0.0f;",
                       "            srt_tok[r] = 0;\n            srt_w[r] = 0.0f;"),
    "token_from_slot": ("srt_tok[r] = (int32_t)(i / k);", "srt_tok[r] = (int32_t)(i % k);"),
    "unstable_place": ("        r = cursor[id]++;", "        r = offsets[id + 1] - 1 - (cursor[id]++ - offsets[id]) - (offsets[id + 1] - offsets[id] - counts[id]);"),
    "last_slot_dropped": ("        for (j = 0; j < k; j++) {\n            int e = ids[(long)t * k + j];\n            if (e == -1) {",
                          "        for (j = 0; j < k; j++) {\n            int e = (j == k - 1 && k > 1) ? -1 : ids[(long)t * k + j];\n            if (e == -1) {"),
    "f16_exponent_bias": ("v = ldexp((double)(man | 0x400), ex - 25);", "v = ldexp((double)(man | 0x400), ex - 24);"),
    "e4m3_exponent_bias": ("v = ldexp((double)(8 + man), ex - 10);", "v = ldexp((double)(8 + man), ex - 9);"),
    "e4m3_subnormal_step": ("v = ldexp((double)man, -9);", "v = ldexp((double)man, -10);"),
    "e4m3_ties_up": ("best = ((c - 1) & 1) == 0 ? c - 1 : c;", "best = c;"),
    "e4m3_no_saturation": ("    if (a >= 448.0)\n        return (uint8_t)(sign | 0x7e);",
                           "    if (a > 464.0)\n        return (uint8_t)(sign | 0x7e);"),
    "scale_per_expert": ("return e4m3_table[W->q8[i]] * (double)W->scale[e * W->cols + c];",
                         "return e4m3_table[W->q8[i]] * (double)W->scale[e * W->cols];"),
    "scale_divisor": ("s = amax / 448.0f;", "s = amax / 256.0f;"),
    "row_scale_not_minimal": ("        if (amax > ldexp(448.0, e))\n            e++;",
                              "        if (amax >= ldexp(224.0, e))\n            e++;"),
    "row_scale_ignored": ("        x[c] = ldexp(e4m3_value(e4m3_encode((float)ldexp(x[c], -e))), e);",
                          "        x[c] = e4m3_value(e4m3_encode((float)ldexp(x[c], -e)));"),
    "down_input_not_quantized": ("        dequantize_row_e4m3(hq, f);", "        (void)hq;"),
    "down_codes_from_fp64_h": ("        hq[n] = a8 ? to_bf16(h[n]) : h[n];", "        hq[n] = h[n];"),
    "quantize_amax_axis": ("float a = (float)fabs(bf16_value(W[(e * K + k) * M + m]));",
                           "float a = (float)fabs(bf16_value(W[(e * K + m % K) * M + k % M]));"),
    "e2m1_emax": ("#define E2M1_EMAX 2", "#define E2M1_EMAX 3"),
    "e2m1_subnormal_step": ("double v = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);",
                            "double v = ex == 0 ? 0.25 * man : ldexp(1.0 + 0.5 * man, ex - 1);"),
    "e2m1_exponent_bias": ("double v = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex - 1);",
                           "double v = ex == 0 ? 0.5 * man : ldexp(1.0 + 0.5 * man, ex);"),
    "e2m1_ties_up": ("            best = (c & 1) ? c - 1 : c;", "            best = c;"),
    "e2m1_no_saturation": ("    if (a >= 6.0)\n        return (uint8_t)(sign | 0x7);",
                           "    if (a >= 8.0)\n        return (uint8_t)(sign | 0x7);"),
    "mx_scale_bias": ("scales[(e * (K / MX_BLOCK) + b) * M + m] = (uint8_t)(x + 127);",
                      "scales[(e * (K / MX_BLOCK) + b) * M + m] = (uint8_t)(x + 126);"),
    "mx_nibble_order": ("            if ((m & 1) == 0)\n                        *byte",
                        "            if ((m & 1) == 1)\n                        *byte"),
    "mx_block_along_m": ("double a = fabs(bf16_value(W[(e * K + k) * M + m]));",
                         "double a = fabs(bf16_value(W[(e * K + b * MX_BLOCK + (k % MX_BLOCK)) * M + (m / MX_BLOCK) * MX_BLOCK + (k % MX_BLOCK) % M]));"),
    "mx_exponent_from_ceil": ("x = fe - 1 - E2M1_EMAX;", "x = fe - E2M1_EMAX;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, name
    mut = tmp_path / f"{name}.c"
    mut.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", *oracle.GCC_FLAGS, "-o", str(lib), str(mut), "-lm", "-lpthread"],
                   check=True, capture_output=True)
    env = dict(os.environ, MOE_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle_plan.py"),
                        os.path.join(HERE, "test_oracle_layer.py"),
                        os.path.join(HERE, "test_oracle_e4m3.py"),
                        os.path.join(HERE, "test_oracle_mxfp4.py")],
                       env=env, capture_output=True, text=True, cwd=os.path.dirname(HERE))
    assert r.returncode != 0, f"planted mistake {name} passed every pin:\n{r.stdout[-2000:]}"
