"""Plant plausible mistakes in a copy of the oracle and check that the pin
suite (the test_oracle_*.py files other than this one) catches every one.

Each mutant is a one-line edit of pa_oracle.c built on the CPU; the pin suite
then runs in a subprocess against that build and must fail.
"""
import os
import subprocess
import sys

import pytest

from oracle import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pa_oracle.c")

PIN_SUITE = ("test_oracle_quant.py", "test_oracle_decode.py", "test_oracle_fp8.py",
             "test_oracle_multi.py")

MUTANTS = {
    "round_half_away": ("int32_t zp = sat_i32(rintf(zq));", "int32_t zp = sat_i32(roundf(zq));"),
    "code_round_half_away": ("int64_t c = (int64_t)sat_i32(rintf(xq))", "int64_t c = (int64_t)sat_i32(roundf(xq))"),
    "levels_off_by_one": ("volatile float scale = r / (float)L;", "volatile float scale = r / (float)(L + 1);"),
    "zp_sign": ("volatile float zq = -mn / scale;", "volatile float zq = mn / scale;"),
    "zp_clamped": ("int32_t zp = sat_i32(rintf(zq));", "int32_t zp = sat_i32(rintf(zq)); if (zp < 0) zp = 0; if (zp > L) zp = L;"),
    "degenerate_scale_one": ("scale = a / (float)L;", "scale = 1.0f;"),
    "dequant_zp_sign": ("read_code(kv_dtype, codes, page, bs, D, s, c) - old_zp;", "read_code(kv_dtype, codes, page, bs, D, s, c) + old_zp;"),
    "requant_ignores_old": ("const int old_cnt = ctx > first ? (ctx - first < bs ? ctx - first : bs) : 0;", "const int old_cnt = 0;"),
    "nibble_order": ("return (c & 1) ? (byte >> 4) : (byte & 15);", "return (c & 1) ? (byte & 15) : (byte >> 4);"),
    "gqa_head_map": ("j = h / g;", "j = h % Hkv;"),
    "slot_index": ("D, t % bs, c);\n    s[t]", "D, (t + 1) % bs, c);\n    s[t]"),
    "dropped_scale": ("s[t] = softmax_scale * acc;", "s[t] = acc;"),
    "no_normalise": ("const double p = s[t] / denom;", "const double p = s[t];"),
    "dequant_drops_zp": ("return ((double)code - (double)zp[page * D + c]) * (double)scale[page * D + c];", "return ((double)code) * (double)scale[page * D + c];"),
    # E4M3 encoding and the fp8 quantiser
    "fp8_truncates": ("double m = nearbyint(a / q);", "double m = floor(a / q);"),
    "fp8_ties_away": ("double m = nearbyint(a / q);", "double m = round(a / q);"),
    "fp8_exponent_bias": ("return sign | ((ev + 7) << 3) | mant;", "return sign | ((ev + 8) << 3) | mant;"),
    "fp8_overflow_to_nan": ("if (a >= 448.0) return sign | 0x7E;", "if (a >= 464.0) return sign | 0x7F;"),
    "fp8_flushes_subnormals": ("  if (a < ldexp(1.0, -6)) {\n    e = -6;", "  if (a < ldexp(1.0, -6)) {\n    return sign;"),
    "fp8_value_bias": ("ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 11)"),
    "fp8_scale_240": ("volatile float scale = amax / 448.0f;", "volatile float scale = amax / 240.0f;"),
    "fp8_signed_max": ("const float a = fabsf(vals[i]);", "const float a = vals[i];"),
    "fp8_dequant_drops_scale": ("if (kv_dtype == KV_FP8) return oracle_e4m3_value(code) * (double)scale[page * D + c];", "if (kv_dtype == KV_FP8) return oracle_e4m3_value(code);"),
    "fp8_requant_drops_old_scale": ("volatile float x = f * old_scale;\n                vals[s] = x;", "volatile float x = f;\n                vals[s] = x;"),
    # several query tokens per sequence
    "multi_causal_off_by_one": ("const int n_i = seq_lens[b] - (n_q - 1 - i);", "const int n_i = seq_lens[b] - (n_q - i);"),
    "multi_causal_reversed": ("const int n_i = seq_lens[b] - (n_q - 1 - i);", "const int n_i = seq_lens[b] - i;"),
    "multi_no_mask": ("const int n_i = seq_lens[b] - (n_q - 1 - i);", "const int n_i = seq_lens[b] + 0 * i;"),
    "multi_token_major_rows": ("const int h = (int)(r % Hq), b = (int)(bi / n_q), i = (int)(bi % n_q);", "const int h = (int)(r % Hq), b = (int)(bi % (n_rows / n_q / Hq)), i = (int)(bi / (n_rows / n_q / Hq));"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    so = oracle.build_variant(text.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    env = dict(os.environ, PA_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"]
                       + [os.path.join(ROOT, "tests", f) for f in PIN_SUITE],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pin suite:\n{r.stdout[-2000:]}"
