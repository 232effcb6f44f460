"""The oracle's pins against planted mistakes: each case copies the oracle's C
source, plants one plausible error (a wrong bit position, divisor, sign, index
or rounding), builds the copy and runs the oracle pins against it in a fresh
interpreter.  Each mutant must fail at least one pin.  This checks the pins,
not the oracle: the oracle itself is never modified, and the mutants are built
in the git-ignored _build/ folder and deleted afterwards.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "w4a16_oracle.c")
WORK = os.path.join(ROOT, "_build", "oracle_mutants")

# name: (original text, replacement, which occurrence (0 = first), pins to run)
MUTANTS = {
    # the 4-bit layer
    "codes high nibble first": ("qrow[k / 8] |= (uint32_t)codes[i] << (4 * (k % 8));",
                                "qrow[k / 8] |= (uint32_t)codes[i] << (4 * (7 - k % 8));", 0, "not q4k"),
    "scale over 16 steps": ("volatile float s32 = range / 15.0f;", "volatile float s32 = range / 16.0f;", 0, "not q4k"),
    "zero point in the next nibble": ("zrow[g / 8] |= (uint32_t)z << (4 * (g % 8));",
                                      "zrow[g / 8] |= (uint32_t)z << (4 * ((g + 1) % 8));", 0, "not q4k"),
    "zero point truncated": ("z = (int)clamp_i64((int64_t)nearbyintf(t), 0, 15);",
                             "z = (int)clamp_i64((int64_t)t, 0, 15);", 0, "not q4k"),
    "zero point added": ("return (float)(q - z) * s;", "return (float)(q + z) * s;", 0, "not q4k"),
    "zero point dropped from codes": ("int64_t q = (int64_t)nearbyintf(t) + z;", "int64_t q = (int64_t)nearbyintf(t);",
                                      0, "not q4k"),
    "activation scale divides": ("double xv = (double)oracle_bf16_to_f32(x_bf16[m * K + k]) * (double)x_scale[k];",
                                 "double xv = (double)oracle_bf16_to_f32(x_bf16[m * K + k]) / (double)x_scale[k];",
                                 0, "act_scale"),
    "8-bit high-plane scale 8 s8": ("srow[g] = oracle_f32_to_f16(16.0f * oracle_f16_to_f32(sb));",
                                    "srow[g] = oracle_f32_to_f16(8.0f * oracle_f16_to_f32(sb));", 0, "pack8 or linear8"),
    # the 8-bit word layout
    "8-bit word: codes high byte first": ("qrow[k / 4] |= (uint32_t)codes[i] << (8 * (k % 4));",
                                          "qrow[k / 4] |= (uint32_t)codes[i] << (8 * (3 - k % 4));", 0, "pack8w"),
    "8-bit word: zero in the next byte": ("zrow[g / 4] |= (uint32_t)z << (8 * (g % 4));",
                                          "zrow[g / 4] |= (uint32_t)z << (8 * ((g + 1) % 4));", 0, "pack8w"),
    "8-bit word: zero point added": ("    return (float)(q - z) * s;\n}\n\nvoid oracle_dequant8w(",
                                     "    return (float)(q + z) * s;\n}\n\nvoid oracle_dequant8w(", 0, "8w"),
    # the super-block layer
    "q4k: m high bits at 2j + 1": ("rec[3] |= (uint32_t)(m[j] >> 4) << (16 + 2 * j);",
                                   "rec[3] |= (uint32_t)(m[j] >> 4) << (2 * j + 1);", 0, "q4k"),
    "q4k: d from max / 64": ("volatile float dq = amax / 63.0f, dmq = bmax / 63.0f;",
                             "volatile float dq = amax / 64.0f, dmq = bmax / 63.0f;", 0, "q4k"),
    "q4k: minimum added": ("    return t - bp;\n}", "    return t + bp;\n}", 0, "q4k"),
    "q4k: sub-blocks of 16": ("const int j = (int)((k % 256) / 32);", "const int j = (int)((k % 256) / 16) % 8;", 0, "q4k"),
    "q4k: sc read from the m word": ("sc[j] = (int)(((rec[1] >> (4 * j)) & 15)", "sc[j] = (int)(((rec[2] >> (4 * j)) & 15)",
                                     0, "q4k"),
    "q4k: range not widened to 0": ("        float lo = 0.0f, hi = 0.0f;\n        for (int i = 0; i < 32; ++i) {",
                                    "        float lo = w[32 * j], hi = w[32 * j];\n        for (int i = 0; i < 32; ++i) {",
                                    0, "q4k"),
    "q4k: codes truncated": ("q[32 * j + i] = (uint8_t)clamp_i64((int64_t)nearbyintf(t), 0, 15);",
                             "q[32 * j + i] = (uint8_t)clamp_i64((int64_t)t, 0, 15);", 0, "q4k"),
    "q4k: dmin not stored": ("rec[0] = (uint32_t)db | ((uint32_t)dmb << 16);", "rec[0] = (uint32_t)db;", 0, "q4k"),
}

_RUNNER = """
import os, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, os.path.join({root!r}, "tests"))
import oracle
oracle._build.build = lambda force=False: os.environ["ORACLE_MUTANT_SO"]
oracle._lib = None
import pytest
sys.exit(pytest.main(["-q", "-x", "-p", "no:cacheprovider", os.path.join({root!r}, "tests", "test_oracle.py"),
                      "-k", os.environ["ORACLE_MUTANT_PINS"]]))
"""


def _replace_nth(text, old, new, n):
    start = -1
    for _ in range(n + 1):
        start = text.index(old, start + 1)
    return text[:start] + new + text[start + len(old):]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name):
    old, new, occurrence, pins = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) > occurrence, f"mutation anchor not found: {old!r}"
    os.makedirs(WORK, exist_ok=True)
    tag = "".join(ch if ch.isalnum() else "_" for ch in name)
    c_path, so_path = os.path.join(WORK, tag + ".c"), os.path.join(WORK, tag + ".so")
    try:
        with open(c_path, "w") as f:
            f.write(_replace_nth(src, old, new, occurrence))
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fno-fast-math", "-ffp-contract=off", "-fopenmp", "-fPIC",
                               "-shared", c_path, "-o", so_path, "-lm"])
        env = dict(os.environ, ORACLE_MUTANT_SO=so_path, ORACLE_MUTANT_PINS=pins)
        r = subprocess.run([sys.executable, "-c", _RUNNER.format(root=ROOT)], env=env, capture_output=True,
                           text=True, cwd=ROOT, timeout=600)
        assert r.returncode == 1, f"no pin caught '{name}' (exit {r.returncode}):\n{r.stdout[-2000:]}"
    finally:
        for p in (c_path, so_path):
            if os.path.exists(p):
                os.remove(p)
