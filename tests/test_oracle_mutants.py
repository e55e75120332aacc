"""The oracle's pins must catch plausible mistakes.

Each mutant below is a copy of oracle/mx_oracle.c with one planted mistake
(a wrong constant, a dropped clamp, a wrong tie rule, a wrong index).  The pin
suite (tests/test_oracle_pins.py) is run against each mutant in a child
process and must fail.  Mistakes are planted only in the CPU oracle.
"""
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "mx_oracle.c")

MUTANTS = {
    "prescale_constant_255": ("(uint32_t)(254u - (uint32_t)e8m0)", "(uint32_t)(255u - (uint32_t)e8m0)"),
    "no_zero_floor": ("    if (e == 0) e = 1;\n    return e;", "    return e;"),
    "no_clamp_low": ("    if (v < 0) v = 0;\n    uint8_t e", "    uint8_t e"),
    "ties_away_from_zero": ("(fr == 0.5 && (k & 1u))", "(fr == 0.5)"),
    "interleave_stride_16": ("? (i & 3) + 32 * (i >> 2) : i", "? (i & 3) + 16 * (i >> 2) : i"),
    "e4m3_bias_8": ("3, 7, 448.0, 0x7Eu", "3, 8, 448.0, 0x7Eu"),
    "emax_e4m3_7": ("case MXO_E4M3FN: return 8;", "case MXO_E4M3FN: return 7;"),
    "lane_remap_odd_shift": ("if ((index & 1) == 0) result -= 2;", "if ((index & 1) == 1) result -= 2;"),
    "f16_subnormal_scale": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "e8m0_decode_bias_126": ("ldexp(1.0, (int)e - 127)", "ldexp(1.0, (int)e - 126)"),
    "block_8x4_transposed": ("*br = (dim == -2) ? 8 : 4;\n        *bc = (dim == -2) ? 4 : 8;",
                             "*br = (dim == -2) ? 4 : 8;\n        *bc = (dim == -2) ? 8 : 4;"),
    "e5m2_max_code_7c": ("57344.0, 0x7Bu", "57344.0, 0x7Cu"),
    "nan_fp4_not_zero": ("if (isnan(y)) return (uint8_t)(s << 3);", "if (isnan(y)) return (uint8_t)((s << 3) | 7);"),
    "matmul_scale_column": ("sb[n * kb + k / 32]", "sb[n * kb + (k / 32 + 1) % kb]"),
    "nan_e4m3_to_max": ("if (isnan(y)) return (uint8_t)(0x7Fu | (s << 7));\n    return (uint8_t)(nearest_code(fabs((double)y), 3",
                        "if (isnan(y)) return (uint8_t)(0x7Eu | (s << 7));\n    return (uint8_t)(nearest_code(fabs((double)y), 3"),
    "nan_e5m2_to_max": ("if (isnan(y)) return (uint8_t)(0x7Fu | (s << 7));\n    return (uint8_t)(nearest_code(fabs((double)y), 2",
                        "if (isnan(y)) return (uint8_t)(0x7Bu | (s << 7));\n    return (uint8_t)(nearest_code(fabs((double)y), 2"),
    "nan_fp8_sign_dropped": ("if (isnan(y)) return (uint8_t)(0x7Fu | (s << 7));\n    return (uint8_t)(nearest_code(fabs((double)y), 3",
                             "if (isnan(y)) return (uint8_t)(0x7Fu);\n    return (uint8_t)(nearest_code(fabs((double)y), 3"),
}


def _run_mutant(name, tmp):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"{name}: pattern not found exactly once"
    path = os.path.join(tmp, f"{name}.c")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    lib = os.path.join(tmp, f"lib{name}.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-o", lib, path, "-lm"], check=True)
    env = dict(os.environ, MX_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return name, r.returncode


def test_pins_catch_every_planted_mistake():
    with tempfile.TemporaryDirectory() as tmp:
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            results = list(ex.map(lambda n: _run_mutant(n, tmp), sorted(MUTANTS)))
    survivors = [n for n, rc in results if rc == 0]
    assert not survivors, f"pins did not catch: {survivors}"
