"""Plant plausible mistakes in a copy of oracle.c and check that the pins in
test_oracle_pins.py catch every one of them (CPU only)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "flipped_kernel_rows": ("int ih = oh * c->sh - c->ph + kh;", "int ih = oh * c->sh - c->ph + (c->KH - 1 - kh);"),
    "kh_kw_transposed_weight": ("* c->KH + kh) * c->KW + kw]);", "* c->KW + kw) * c->KH + kh]);"),
    "wrong_pad_axis": ("int iw = ow * c->sw - c->pw + kw;", "int iw = ow * c->sw - c->ph + kw;"),
    "dropped_bn_bias": ("double v = acc * (double)c->scale[co] + (double)c->bias[co];", "double v = acc * (double)c->scale[co];"),
    "silu_sign": ("static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }",
                  "static double sigmoid(double v) { return 1.0 / (1.0 + exp(v)); }"),
    "gelu_sign": ("return 0.5 * s * erfc(-s / sqrt(2.0));", "return 0.5 * s * erfc(s / sqrt(2.0));"),
    "gelu_cancelling_form": ("return 0.5 * s * erfc(-s / sqrt(2.0));", "return 0.5 * s * (1.0 + erf(s / sqrt(2.0)));"),
    "bias_by_row": ("+ f16_value(c->bias[j]);", "+ f16_value(c->bias[r % c->cols]);"),
    "ln_unbiased_variance": ("double var = sq / (double)H;", "double var = sq / (double)(H - 1);"),
    "ln_eps_outside_sqrt": ("double inv = 1.0 / sqrt(var + c->eps);", "double inv = 1.0 / (sqrt(var) + c->eps);"),
    "ln_gamma_beta_swapped": ("nrm * (double)c->gamma[j] + (double)c->beta[j];", "nrm * (double)c->beta[j] + (double)c->gamma[j];"),
    "pack_kh_kw_swapped": ("w_ohwi[(((int64_t)co * KH + kh) * KW + kw) * C_in + ci] =",
                           "w_ohwi[(((int64_t)co * KW + kw) * KH + kh) * C_in + ci] ="),
    "f16_exponent_bias": ("v = ldexp((double)(f | 0x400), e - 25);", "v = ldexp((double)(f | 0x400), e - 24);"),
    "chain_skips_t1_rounding": ("double t1 = round_to_bf16(acc);", "double t1 = acc;"),
    "ln_mean_not_subtracted": ("sq += (s[j] - mean) * (s[j] - mean);", "sq += s[j] * s[j];"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    mutant = tmp_path / "oracle_mutant.c"
    mutant.write_text(src.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c99", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(lib), str(mutant), "-lm", "-lpthread"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
