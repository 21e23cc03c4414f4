"""Plant plausible mistakes in copies of the oracle and check that the pins
in test_oracle.py catch every one (CPU only).

Each mutant is the oracle's C source with one small edit (a wrong unpack
order, a dropped term, a wrong sign or index, ...), compiled to a temporary
library and run under the full pin suite in a subprocess.  A mutant that
passes every pin would mean the pins cannot tell it from the real oracle.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qgemv_oracle.c")

MUTANTS = {
    "high_bits_first": ("int shift = bits * (k % per_word);",
                        "int shift = 32 - bits * (1 + k % per_word);"),
    "shifted_code_index": ("int shift = bits * (k % per_word);",
                           "int shift = bits * ((k + 1) % per_word);"),
    "group_of_32": ("scales[(int64_t)n * G + k / ORACLE_GROUP]",
                    "scales[(int64_t)n * G + (k / 32) % G]"),
    "bias_dropped": ("return (double)q * s + b;", "return (double)q * s;"),
    "bias_sign": ("return (double)q * s + b;", "return (double)q * s - b;"),
    "sum_sign": ("acc += w * x[k];", "acc -= w * x[k];"),
    "eps_outside_root": ("sqrt(ss / (double)K + eps)", "(sqrt(ss / (double)K) + eps)"),
    "gamma_dropped": ("xn[k] = oracle_half_to_double(x[k]) * r * oracle_half_to_double(gamma[k]);",
                      "xn[k] = oracle_half_to_double(x[k]) * r;"),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "residual_dropped": ("double v = acc[n] + r;", "double v = acc[n];"),
    "up_is_gate": ("gc + up_w, gs + up_g, gb + up_g", "gc, gs, gb"),
    "expert_weight_ignored": ("acc[n] += w * yd[n];", "acc[n] += yd[n];"),
    "half_truncates": ("double m = rint(ldexp(a, 10 - E));", "double m = floor(ldexp(a, 10 - E));"),
    "half_subnormal_scale": ("v = ldexp((double)mant, -24);", "v = ldexp((double)mant, -23);"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
    mutated = src.replace(old, new)
    csrc = tmp_path / "mutant.c"
    csrc.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o",
                    str(so), str(csrc), "-lm"], check=True)
    env = dict(os.environ, QGEMV_ORACLE_LIB=str(so), OMP_NUM_THREADS="2")
    res = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p",
                          "no:cacheprovider", os.path.join(ROOT, "tests", "test_oracle.py")],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert res.returncode != 0, f"mutant {name} passed every pin:\n{res.stdout[-2000:]}"
