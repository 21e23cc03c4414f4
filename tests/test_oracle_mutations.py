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
    "moe_tol_h_dropped": ("hb[j] = fabs(h[j]) + th[j] / 2e-3;", "hb[j] = fabs(h[j]);"),
    "moe_abs_matvec_signed": ("s += fabs(weight(codes, scales, biases, bits, K, n, k)) * v[k];",
                              "s += weight(codes, scales, biases, bits, K, n, k) * v[k];"),
    "moe_tol_signed_weight": ("mag[n] += fabs(w) * ab[n];", "mag[n] += w * ab[n];"),
    "moe_tol_without_residual": ("tol[n] = 2e-3 * (mag[n] + fabs(r)) + 1e-5;",
                                 "tol[n] = 2e-3 * mag[n] + 1e-5;"),
    "lut_one_table_per_row": ("lut + (int64_t)(n / rows_per_lut) * 16", "lut + (int64_t)n * 16"),
    "lut_table_stride": ("lut + (int64_t)(n / rows_per_lut) * 16",
                         "lut + (int64_t)(n / rows_per_lut) * 15"),
    "lut_reversed_index": ("table[oracle_code(row, 4, k)]", "table[15 - oracle_code(row, 4, k)]"),
    "lut_residual_dropped": ("            acc += r;\n", ""),
    "lut_bound_without_x": ("mag += fabs(w) * fabs(xv);", "mag += fabs(w);"),
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


# The routing oracle is Python: its mutants are copies of oracle/__init__.py
# with one edit in moe_route, run under the routing pins of test_oracle.py.
PY_SRC = os.path.join(ROOT, "oracle", "__init__.py")
ROUTE_MUTANTS = {
    "tie_to_higher_index": ("if best < 0 or lv[e] > lv[best]:", "if best < 0 or lv[e] >= lv[best]:"),
    "smallest_logits": ("if best < 0 or lv[e] > lv[best]:", "if best < 0 or lv[e] < lv[best]:"),
    "shared_dropped": ("chosen = [int(shared)] if shared >= 0 else []", "chosen = []"),
    "chosen_not_excluded": ("            if e in chosen:\n                continue\n", ""),
    "weights_unnormalised": ("[v / tot for v in ex]", "[v for v in ex]"),
    "hidden_temperature": ("float(np.exp(v - m))", "float(np.exp(2.0 * (v - m)))"),
}

_ROUTE_PINS = """
import importlib.util, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
spec = importlib.util.spec_from_file_location("oracle", {path!r},
                                              submodule_search_locations=[{pkg!r}])
mod = importlib.util.module_from_spec(spec); sys.modules["oracle"] = mod
spec.loader.exec_module(mod)
import test_oracle as t
t.oracle = mod
t.test_moe_route_hand_example()
t.test_moe_route_equal_logits_and_no_shared_expert()
for args in [(512, 4, 0), (64, 8, -1), (33, 1, 5), (16, 2, 15)]:
    t.test_moe_route_against_stable_sort(*args)
"""


@pytest.mark.parametrize("name", sorted(ROUTE_MUTANTS))
def test_route_pins_catch_mutant(name, tmp_path):
    old, new = ROUTE_MUTANTS[name]
    src = open(PY_SRC).read()
    assert src.count(old) == 1, f"mutation anchor missing: {old!r}"
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(src.replace(old, new))
    script = _ROUTE_PINS.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                                path=str(pkg / "__init__.py"), pkg=str(pkg))
    # the C library the copy would build is the real one (only moe_route differs)
    env = dict(os.environ, QGEMV_ORACLE_LIB=os.path.join(ROOT, "oracle", "_build", "liboracle.so"))
    res = subprocess.run([sys.executable, "-c", script], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode != 0, f"routing mutant {name} passed every pin:\n{res.stdout[-1000:]}"


def test_route_pins_pass_on_the_real_oracle(tmp_path):
    # the harness itself: the unmutated copy passes
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(open(PY_SRC).read())
    script = _ROUTE_PINS.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                                path=str(pkg / "__init__.py"), pkg=str(pkg))
    env = dict(os.environ, QGEMV_ORACLE_LIB=os.path.join(ROOT, "oracle", "_build", "liboracle.so"))
    res = subprocess.run([sys.executable, "-c", script], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr[-2000:]


# Planted mistakes in the top-k sampling oracle; the sampling pins must fail
# on each.
SAMPLE_MUTANTS = {
    "tie_to_higher_index": ('cand = np.argsort(-lv, kind="stable")[:top_k]',
                            'cand = (len(lv) - 1 - np.argsort(-lv[::-1], kind="stable"))[:top_k]'),
    "smallest_logits": ('cand = np.argsort(-lv, kind="stable")[:top_k]',
                        'cand = np.argsort(lv, kind="stable")[:top_k]'),
    "one_candidate_short": ('cand = np.argsort(-lv, kind="stable")[:top_k]',
                            'cand = np.argsort(-lv, kind="stable")[:max(top_k - 1, 1)]'),
    "temperature_multiplies": ("/ float(temperature))", "* float(temperature))"),
    "running_sum_unnormalised": ("cum = np.cumsum(p) / p.sum()", "cum = np.cumsum(p)"),
    "pick_at_equal_sum": ("j = int(np.argmax(cum > float(u))) if np.any(cum > float(u))",
                          "j = int(np.argmax(cum >= float(u))) if np.any(cum >= float(u))"),
    "fallback_to_first": ("else top_k - 1", "else 0"),
}

_SAMPLE_PINS = _ROUTE_PINS.split("import test_oracle as t")[0] + """import test_oracle as t
t.oracle = mod
t.test_lm_head_sample_hand_example()
t.test_lm_head_sample_top1_is_greedy_and_temperature()
t.test_lm_head_sample_frequencies_follow_the_softmax()
t.test_lm_head_sample_boundaries()
"""


def _run_pins(script_tmpl, src, tmp_path):
    pkg = tmp_path / "oracle"
    pkg.mkdir()
    (pkg / "__init__.py").write_text(src)
    script = script_tmpl.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                                path=str(pkg / "__init__.py"), pkg=str(pkg))
    env = dict(os.environ, QGEMV_ORACLE_LIB=os.path.join(ROOT, "oracle", "_build", "liboracle.so"))
    return subprocess.run([sys.executable, "-c", script], cwd=ROOT, env=env,
                          capture_output=True, text=True, timeout=300)


@pytest.mark.parametrize("name", sorted(SAMPLE_MUTANTS))
def test_sample_pins_catch_mutant(name, tmp_path):
    old, new = SAMPLE_MUTANTS[name]
    src = open(PY_SRC).read()
    assert src.count(old) == 1, f"mutation anchor missing: {old!r}"
    res = _run_pins(_SAMPLE_PINS, src.replace(old, new), tmp_path)
    assert res.returncode != 0, f"sampling mutant {name} passed every pin:\n{res.stdout[-1000:]}"


def test_sample_pins_pass_on_the_real_oracle(tmp_path):
    res = _run_pins(_SAMPLE_PINS, open(PY_SRC).read(), tmp_path)
    assert res.returncode == 0, res.stderr[-2000:]
