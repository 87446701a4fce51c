"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a private copy of ``oracle/oracle.c`` (a dropped
term, a wrong sign, a wrong index or stride, a wrong rounding rule), compiles
it into a temporary directory and runs the pin suite against it in a child
process; the suite must fail.  Nothing here touches a GPU, and the committed
oracle is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "q4_0_offset_7": ("w[j]      = d * (float)(lo - 8);", "w[j]      = d * (float)(lo - 7);"),
    "q4_0_nibbles_swapped": ("int lo = qs[j] & 0x0f;\n            int hi = qs[j] >> 4;\n            w[j]      = d * (float)(lo - 8);",
                             "int hi = qs[j] & 0x0f;\n            int lo = qs[j] >> 4;\n            w[j]      = d * (float)(lo - 8);"),
    "q4_1_min_dropped": ("w[j]      = plo + m;", "w[j]      = plo;"),
    "q4_1_min_sign": ("w[j + 16] = phi + m;", "w[j + 16] = phi - m;"),
    "q8_0_unsigned": ("int q = (int)(int8_t)qs[j];", "int q = (int)qs[j];"),
    "fp16_exponent_bias": ("v = ldexp((double)(1024 + frac), expo - 25);", "v = ldexp((double)(1024 + frac), expo - 24);"),
    "fp16_subnormal_scale": ("v = ldexp((double)frac, -24);", "v = ldexp((double)frac, -23);"),
    "rne_ties_up": ("(dropped == 0x1000u && (h & 1u))", "(dropped == 0x1000u)"),
    "gemv_x_stride": ("const float *xb = x + b * ncols;\n            double acc = 0.0, aacc = 0.0;\n            for (int64_t k = 0; k < ncols; ++k) {\n                double p = (double)w[k] * (double)xb[k];\n                acc += p;\n                aacc += fabs(p);\n            }\n            y[b * nrows + r] = (float)acc;",
                      "const float *xb = x + b * nrows;\n            double acc = 0.0, aacc = 0.0;\n            for (int64_t k = 0; k < ncols; ++k) {\n                double p = (double)w[k] * (double)xb[k];\n                acc += p;\n                aacc += fabs(p);\n            }\n            y[b * nrows + r] = (float)acc;"),
    "gemv_output_transposed": ("y[b * nrows + r] = (float)acc;", "y[r * batch + b] = (float)acc;"),
    "row_stride_blocks": ("const uint8_t *row = W + r * nb * bb;", "const uint8_t *row = W + r * nb * 18;"),
    "q8_1_ties_away_from_zero": ("if (frac > 0.5 || (frac == 0.5 && fmod(f, 2.0) != 0.0)) f += 1.0;",
                                 "if (frac >= 0.5) f += 1.0;"),
    "q8_1_scale_over_128": ("float dd = finite ? amax / 127.0f : NAN;", "float dd = finite ? amax / 128.0f : NAN;"),
    "q8_1_no_clamp": ("if (v > 127) v = 127;", "if (v > 128) v = 128;"),
    "q8_1_sum_of_magnitudes": ("sum += v;", "sum += v < 0 ? -v : v;"),
    "q8_1_scale_block_index": ("double xhat = (double)d[b * nb + k / 32] * (double)q[b * ncols + k];",
                               "double xhat = (double)d[b * nb + k % nb] * (double)q[b * ncols + k];"),
    "gemv_id_wrong_expert_stride": ("const uint8_t *We = W + ids[b] * ebytes;", "const uint8_t *We = W + ids[b] * (ebytes / 2);"),
    "gemv_id_first_expert_only": ("const uint8_t *We = W + ids[b] * ebytes;", "const uint8_t *We = W;"),
    "gemv_id_x_row_modulo": ("const float *xb = x + (b / x_group) * ncols;", "const float *xb = x + (b % x_group) * ncols;"),
    "gemm_reads_w_row_m": ("dequant_row(fmt, W, ncols, n, w);\n        for (int64_t m = 0; m < mrows; ++m) {\n            const uint16_t *xm = X + m * ncols;",
                           "dequant_row(fmt, W, ncols, n, w);\n        for (int64_t m = 0; m < mrows; ++m) {\n            const uint16_t *xm = X + n % mrows * ncols;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_fail_on_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, "mutation anchor not found: %s" % name
    mutated = src.replace(old, new, 1)
    cpath = tmp_path / "oracle_mutant.c"
    cpath.write_text(mutated)
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", str(cpath), "-o", str(lib), "-lm"], check=True, capture_output=True)
    env = dict(os.environ, QORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch mutant %s:\n%s" % (name, r.stdout[-2000:])
