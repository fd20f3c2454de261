"""The pins must be strong enough to catch a plausible mistake anywhere in the oracle.

Each case copies gq_oracle.c, plants one mistake (a wrong constant, sign, index, rounding
rule or a dropped term), compiles the copy on the CPU and runs the pin suite against it
in a child process: the suite has to fail. The oracle itself is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gq_oracle.c")

MUTANTS = {
    "scale_divisor": ("const float d = amax / 7.0f;", "const float d = amax / 8.0f;"),
    "code_offset": ("int c = (int)roundf(w[i] / d) + 8;", "int c = (int)roundf(w[i] / d) + 7;"),
    "nibble_order": ("(uint8_t)(code[j] | (code[j + 16] << 4))",
                     "(uint8_t)(code[j + 16] | (code[j] << 4))"),
    "ties_to_even": ("int c = (int)roundf(w[i] / d) + 8;", "int c = (int)rintf(w[i] / d) + 8;"),
    "q8_ties_to_even": ("c = (int)roundf(w[i] / d);", "c = (int)rintf(w[i] / d);"),
    "dequant_sign": ("w[j] = (float)(lo - 8) * d;", "w[j] = (float)(8 - lo) * d;"),
    "dequant_high_nibble": ("w[j + 16] = (float)(hi - 8) * d;", "w[j + 16] = (float)(hi - 7) * d;"),
    "dropped_term": ("for (int64_t k = 0; k < K; ++k)", "for (int64_t k = 0; k + 1 < K; ++k)"),
    "transposed_x": ("acc += (double)wrow[k] * (double)x[k];",
                     "acc += (double)wrow[k] * (double)X[k * N + n];"),
    "transposed_y": ("Y[n * M + m] = (float)acc;", "Y[m * N + n] = (float)acc;"),
    "fp32_accumulator": ("double acc = 0.0;", "float acc = 0.0f;"),
    "fp16_ties_away": ("if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;",
                       "if (rest >= 0x1000u) h += 1u;"),
    "fp16_flush_subnormal": ("if (drop > 24) return sign;", "if (drop > 13) return sign;"),
    "fp16_truncate": ("if (rest > 0x1000u || (rest == 0x1000u && (h & 1u))) h += 1u;", ""),
    "q8_scale_divisor": ("const float d = amax / 127.0f;", "const float d = amax / 128.0f;"),
    "q8x_code_offset": ("return (i < 16 ? (byte & 0x0F) : (byte >> 4)) - 8;",
                        "return (i < 16 ? (byte & 0x0F) : (byte >> 4)) - 7;"),
    "q8x_scale": ("acc += dw * dx * (double)sum;", "acc += dw * (double)sum;"),
    "q8x_x_block": ("const uint8_t* xb = xq + (n * nb + b) * 34;",
                    "const uint8_t* xb = xq + (n * nb + (nb - 1 - b)) * 34;"),
    "rmsnorm_sum_not_mean": ("const double rms = sqrt(ss / (double)K + eps);",
                             "const double rms = sqrt(ss + eps);"),
    "rmsnorm_eps_outside": ("const double rms = sqrt(ss / (double)K + eps);",
                            "const double rms = sqrt(ss / (double)K) + eps;"),
    "rmsnorm_no_gamma": ("xhat[k] = (double)x[k] / rms * (double)gamma[k];",
                         "xhat[k] = (double)x[k] / rms;"),
    "swiglu_exp_sign": ("H[n * M + m] = (float)(g / (1.0 + exp(-g)) * u);",
                        "H[n * M + m] = (float)(g / (1.0 + exp(g)) * u);"),
    "swiglu_no_up": ("H[n * M + m] = (float)(g / (1.0 + exp(-g)) * u);",
                     "H[n * M + m] = (float)(g / (1.0 + exp(-g)));"),
    "swiglu_roles_swapped": ("H[n * M + m] = (float)(g / (1.0 + exp(-g)) * u);",
                             "H[n * M + m] = (float)(u / (1.0 + exp(-u)) * g);"),
    # Q4_K super-blocks
    "q4k_nibble_order": ("(uint8_t)(code[64 * g + l] | (code[64 * g + 32 + l] << 4))",
                         "(uint8_t)(code[64 * g + 32 + l] | (code[64 * g + l] << 4))"),
    "q4k_min_added": ("w[32 * j + l] = D * (float)q - M;", "w[32 * j + l] = D * (float)q + M;"),
    "q4k_scale_high_bits": ("*sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);",
                            "*sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 3);"),
    "q4k_min_high_bits": ("*m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);",
                          "*m = (s[j + 4] >> 4) | ((s[j - 4] >> 6) << 4);"),
    "q4k_step_divisor": ("step[j] = (hi - lo) / 15.0f;", "step[j] = (hi - lo) / 16.0f;"),
    "q4k_no_zero_in_range": ("if (lo > 0.0f) lo = 0.0f;", ""),
    "q4k_scale_divisor": ("const float d = smax / 63.0f;", "const float d = smax / 64.0f;"),
    "q4k_codes_from_unrounded_scale": ("const float D = df * (float)sc[j];",
                                       "const float D = step[j];"),
}
PIN_FILES = ("test_oracle_pins.py", "test_oracle_q4k_pins.py")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    before, after = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(before) >= 1, f"mutation anchor for {name} not found"
    mutated = src.replace(before, after, 1)
    c_path = tmp_path / "mutant.c"
    so_path = tmp_path / "mutant.so"
    c_path.write_text(mutated)
    import oracle
    subprocess.check_call(["gcc", *oracle.CFLAGS, str(c_path), "-o", str(so_path), "-lm"])
    env = dict(os.environ, GQ_ORACLE_SO=str(so_path))
    r = subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
         *[os.path.join(ROOT, "tests", f) for f in PIN_FILES]],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"pins did not catch mutant {name}:\n{r.stdout[-2000:]}"
