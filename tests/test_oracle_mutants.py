"""The oracle's pins have teeth: plant one plausible mistake at a time in a
copy of oracle.c (CPU only), build it, and check that the pin suite
(tests/test_oracle.py) fails against it.  Every mutation keeps all memory
accesses in bounds."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "drop_beta_c_term": ("  if (p->use_c) dv += p->beta", "  if (0) dv += p->beta"),
    "x_term_wrong_sign": ("  if (p->use_x) dv += p->xf", "  if (p->use_x) dv -= p->xf"),
    "k_loop_skips_first": ("for (int64_t k = 0; k < p->K; ++k) {\n    double a = arow",
                           "for (int64_t k = 1; k < p->K; ++k) {\n    double a = arow"),
    "alpha_beta_swapped": ("double dv = p->alpha * acc;", "double dv = p->beta * acc;"),
    "y_is_d": ("  *y = acc;", "  *y = dv;"),
    "f16_bias_off_by_one": ("v = ldexp(1.0 + f / 1024.0, e - 15);",
                            "v = ldexp(1.0 + f / 1024.0, e - 14);"),
    "e4m3_subnormal_scale": ("v = ldexp((double)f, -9);", "v = ldexp((double)f, -10);"),
    "round_toward_zero": ("return nearbyint(x / q) * q;", "return trunc(x / q) * q;"),
    "cd_layout_swapped": ("return p->cd_m_major ? (l * p->N + n) * p->M + m : (l * p->M + m) * p->N + n;",
                          "return !p->cd_m_major ? (l * p->N + n) * p->M + m : (l * p->M + m) * p->N + n;"),
    "bf16_decoder_mantissa": ("v = ldexp(1.0 + f / 128.0, e - 127);",
                              "v = ldexp(1.0 + f / 256.0, e - 127);"),
    "e5m2_bias": ("v = ldexp(1.0 + f / 4.0, e - 15);", "v = ldexp(1.0 + f / 4.0, e - 16);"),
    "partial_boundary_shift": ("((k + 1) % p->acc_chunk == 0 || k + 1 == p->K)",
                               "(k % p->acc_chunk == 0 || k + 1 == p->K)"),
    "relu_after_x": ("  if (p->relu && dv < 0.0) dv = 0.0;\n  if (p->use_x) dv += p->xf",
                     "  if (p->use_x) dv += p->xf"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    src = tmp_path / "oracle_mutant.c"
    src.write_text(text.replace(old, new))
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-o", str(lib), str(src), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB_OVERRIDE=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle.py")],
                       capture_output=True, text=True, env=env, cwd=ROOT, timeout=600)
    assert r.returncode != 0, f"no pin caught mutant {name}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
