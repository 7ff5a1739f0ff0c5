"""Plant plausible mistakes in a copy of the oracle and check that the pin
suite (test_oracle_quant.py + test_oracle_decode.py) catches every one.

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
    "slot_index": ("D, t % bs, c);\n      s[t]", "D, (t + 1) % bs, c);\n      s[t]"),
    "dropped_scale": ("s[t] = softmax_scale * acc;", "s[t] = acc;"),
    "no_normalise": ("const double p = s[t] / denom;", "const double p = s[t];"),
    "dequant_drops_zp": ("return ((double)code - (double)zp[page * D + c]) * (double)scale[page * D + c];", "return ((double)code) * (double)scale[page * D + c];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    so = oracle.build_variant(text.replace(old, new), str(tmp_path / f"mut_{name}.so"))
    env = dict(os.environ, PA_ORACLE_LIB=so)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_quant.py"),
                        os.path.join(ROOT, "tests", "test_oracle_decode.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pin suite:\n{r.stdout[-2000:]}"
