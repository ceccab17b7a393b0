"""The oracle's pins must catch plausible slips.  Each case plants one slip in
a copy of oracle.c (on the CPU, in a temporary directory), builds it, and runs
the pin suite against it in a child process; the suite must fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PINS = ["tests/test_oracle_formats.py", "tests/test_oracle_swizzle.py",
        "tests/test_oracle_method.py"]

# (name, text in oracle.c, replacement)
MUTATIONS = [
    ("drop_gemma_bias", "((double)weight_bias + wv)", "(wv)"),
    ("flip_weight_sign", "((double)weight_bias + wv)", "((double)weight_bias - wv)"),
    ("mean_over_h_minus_1", "ss / (double)H", "ss / (double)(H - 1)"),
    ("drop_eps", "ss / (double)H + (double)eps", "ss / (double)H"),
    ("residual_not_written", "residual[m * H + j] = h[j];", ";"),
    ("residual_not_used", "h[j] = or_round16((double)s, dtype);", ";"),
    ("partials_in_double", "float acc = (float)or_decode16", "double acc = or_decode16"),
    ("partials_skip_last", "for (int p = 1; p < k; ++p)", "for (int p = 1; p < k - 1; ++p)"),
    ("nibbles_swapped", "c[2 * i] | (c[2 * i + 1] << 4)", "c[2 * i + 1] | (c[2 * i] << 4)"),
    ("amax_over_4", "amax / 6.0f", "amax / 4.0f"),
    ("element_scale_inverted", "g / sfv", "sfv / g"),
    ("fp8_reciprocal", "yf[j] / s", "yf[j] * (1.0f / s)"),
    ("swizzle_group_stride", "((m % 128) / 32) * 4", "((m % 128) / 32) * 8"),
    ("swizzle_row_stride", "(m % 32) * 16", "(m % 32) * 4"),
    ("e4m3_ties_odd", "if (d < best_d || (d == best_d && (c & 1) == 0)) {\n            best = c;\n            best_d = d;\n        }\n    }\n    return (uint8_t)(sign | best);\n}\n\n/* ---",
     "if (d < best_d || (d == best_d && (c & 1) == 1)) {\n            best = c;\n            best_d = d;\n        }\n    }\n    return (uint8_t)(sign | best);\n}\n\n/* ---"),
    ("e2m1_no_saturation_sign", "uint8_t sign = signbit(v) ? 0x8 : 0x0;", "uint8_t sign = v < 0 ? 0x8 : 0x0;"),
    ("e2m1_no_explicit_saturation", "if (a >= 6.0) return sign | 0x7;", "if (isinf(a)) return sign | 0x7;"),
    ("bf16_truncates", "double n = rint(a / ulp);", "double n = floor(a / ulp);"),
    ("mx_scale_off_by_one", "code = (e2 - 1) - 8 + 127;", "code = e2 - 8 + 127;"),
    ("mx_infinite_block_code_zero", "} else if (isinf(amax)) {\n            code = 254;",
     "} else if (isinf(amax)) {\n            code = 0;"),
    ("mx_elements_unscaled", "or_e4m3_encode((double)yf[32 * b + j] / X)",
     "or_e4m3_encode((double)yf[32 * b + j])"),
    ("swizzle_tile_row_stride", "(m / 128) * (Kp / 4) + k / 4", "(m / 128) * Kp + k / 4"),
    ("swizzle_tile_col_stride", "(m / 128) * (Kp / 4) + k / 4", "(m / 128) * (Kp / 4) + k / 2"),
    ("no_square_root", "1.0 / sqrt(ss / (double)H + (double)eps)", "1.0 / (ss / (double)H + (double)eps)"),
]

# Slips the symmetry pins (tests/test_oracle_symmetries.py) must catch on
# their own, without the hand-worked examples.
SYMMETRY_MUTATIONS = [m for m in MUTATIONS
                      if m[0] in ("drop_eps", "residual_not_used", "e2m1_no_saturation_sign",
                                  "no_square_root")]


def _fails_with(tmp_path, name, old, new, pins):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mutated = tmp_path / "oracle.c"
    mutated.write_text(src.replace(old, new))
    (tmp_path / "oracle.h").write_text(open(os.path.join(ROOT, "oracle", "oracle.h")).read())
    lib = tmp_path / "liboracle_mut.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
                    str(mutated), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, GNQ_ORACLE_LIB=str(lib))
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                          *pins], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    # exit status 1: tests ran and one failed (not a collection or usage error)
    assert res.returncode == 1, (f"pins did not catch the planted slip {name} "
                                 f"(pytest status {res.returncode}):\n{res.stdout[-2000:]}")


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_slip(tmp_path, name, old, new):
    _fails_with(tmp_path, name, old, new, PINS)


@pytest.mark.parametrize("name,old,new", SYMMETRY_MUTATIONS, ids=[m[0] for m in SYMMETRY_MUTATIONS])
def test_symmetry_pins_alone_catch_planted_slip(tmp_path, name, old, new):
    _fails_with(tmp_path, name, old, new, ["tests/test_oracle_symmetries.py"])
