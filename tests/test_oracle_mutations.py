"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake (a dropped term, a wrong sign, a wrong
index, a transposed operand, a wrong rounding rule) in a private copy of
oracle.c, builds it with gcc, and runs the oracle pin tests against that build
in a fresh process (ORACLE_LIB points the oracle loader at it).  The pins pass
on the real oracle, so each mutant must make at least one of them fail.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")
PIN_TESTS = ["tests/test_oracle_half.py", "tests/test_oracle_ssln.py",
             "tests/test_oracle_gated.py", "tests/test_oracle_sgn.py",
             "tests/test_oracle_bf16.py"]

MUTANTS = {
    "bias_sign": ("t = t + ld_f32(bias, dtype, bias_index);",
                  "t = t - ld_f32(bias, dtype, bias_index);"),
    "bias_index": ("t = t + ld_f32(bias, dtype, bias_index);",
                   "t = t + ld_f32(bias, dtype, 0);"),
    "sum_not_rounded_before_stats": ("        s = orc_f16_to_f64(h);\n",
                                     "        s = (double)t;\n"),
    "ssln_mean_count": ("double ms = ss / (double)hidden;",
                        "double ms = ss / (double)(hidden - 1);"),
    "ssln_eps_dropped": ("double inv = 1.0 / sqrt(ms + (double)epsilon);\n        for (int64_t j = 0; j < hidden;",
                         "double inv = 1.0 / sqrt(ms);\n        for (int64_t j = 0; j < hidden;"),
    "ssln_gamma_index": ("srow[j] * inv * (double)ld_f32(gamma, dtype, j)",
                         "srow[j] * inv * (double)ld_f32(gamma, dtype, hidden - 1 - j)"),
    "gated_scale_index": ("(double)ld_f32(scale, dtype, j)",
                          "(double)ld_f32(scale, dtype, r % C)"),
    "gated_eps_inside_sqrt": ("double inv = 1.0 / sqrt(ms + (double)epsilon);\n        for (int64_t j = 0; j < C;",
                              "double inv = 1.0 / (sqrt(ms) + (double)epsilon);\n        for (int64_t j = 0; j < C;"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "sgn_mean_sign": ("ga * (sv[k++] - mean) * rstd + be", "ga * (sv[k++] + mean) * rstd + be"),
    "sgn_sample_variance": ("double var = m2 / (double)cnt;",
                            "double var = m2 / (double)(cnt - 1);"),
    "sgn_beta_dropped": ("ga * (sv[k++] - mean) * rstd + be", "ga * (sv[k++] - mean) * rstd"),
    "sgn_nchw_nc_transposed": ("return ((n * C + c) * H + h) * W + w;",
                               "return ((c * N_ + n) * H + h) * W + w;"),
    "sgn_nhwc_as_nchw": ("if (channels_last) return ((n * H + h) * W + w) * C + c;",
                         "if (channels_last) return ((n * C + c) * H + h) * W + w;"),
    "sgn_bcast_ignores_batch": ("int64_t si = skip_bcast ? n * C + c : i;",
                                "int64_t si = skip_bcast ? c : i;"),
    "sgn_gamma_beta_swapped": ("double ga = (double)ld_f32(gamma, mdtype, c);",
                               "double ga = (double)ld_f32(beta, mdtype, c);"),
    "half_ties_away": ("if (frac > 0.5 || (frac == 0.5 && fmod(fl, 2.0) != 0.0)) r = fl + 1.0;",
                       "if (frac >= 0.5) r = fl + 1.0;"),
    "half_subnormal_quantum": ("if (unb < -14) q = -24;", "if (unb < -15) q = -24;"),
    "half_overflow_threshold": ("if (a >= 65520.0)", "if (a >= 65504.0)"),
    "bf16_ties_away": ("if (frac > 0.5 || (frac == 0.5 && odd)) r = fl + 1.0;",
                       "if (frac >= 0.5) r = fl + 1.0;"),
    "bf16_truncates": ("if (frac > 0.5 || (frac == 0.5 && odd)) r = fl + 1.0;",
                       "(void)odd;"),
    "bf16_subnormal_quantum": ("if (unb < -126) q = -133;", "if (unb < -127) q = -133;"),
    "bf16_overflow_threshold": ("ldexp(2.0 - ldexp(1.0, -8), 127)",
                                "ldexp(2.0 - ldexp(1.0, -7), 127)"),
    "bf16_decode_bias": ("v = ldexp((double)(128 + f), e - 134);",
                         "v = ldexp((double)(128 + f), e - 133);"),
    "bf16_sum_not_rounded_before_stats": ("        s = orc_bf16_to_f64(h);\n",
                                          "        s = (double)t;\n"),
    "bf16_read_as_half": ("if (dtype == ORC_BF16) return orc_bf16_to_f32(((const uint16_t*)p)[i]);",
                          "if (dtype == ORC_BF16) return orc_f16_to_f32(((const uint16_t*)p)[i]);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor for {name} no longer in oracle.c"
    mutated = src.replace(old, new, 1)
    if "N_" in new:  # the batch count is not an argument of the index helper
        mutated = mutated.replace("int64_t w, int64_t C, int64_t H, int64_t W) {",
                                  "int64_t w, int64_t C, int64_t H, int64_t W) {\n"
                                  "    const int64_t N_ = 2;", 1)
    c_path = tmp_path / "oracle_mutant.c"
    so_path = tmp_path / "liboracle_mutant.so"
    c_path.write_text(mutated)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", str(so_path), str(c_path), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        *PIN_TESTS], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
