"""The pins must catch plausible mistakes: build copies of the oracle with one
planted mistake each (on the CPU, in the oracle only) and require that the pin
suite fails on every one of them."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "gdn_oracle.c")

# (name, exact source text, replacement)
MUTATIONS = [
    ("conv_taps_reversed", "acc += w[c * 4 + m] * conv_tap(t - 3 + m", "acc += w[c * 4 + (3 - m)] * conv_tap(t - 3 + m"),
    ("hist_oldest_last", "hist[c * 3 + (3 + s)]", "hist[c * 3 + (-1 - s)]"),
    ("l2_eps_outside_sqrt", "1.0 / sqrt(ss + eps)", "1.0 / (sqrt(ss) + eps)"),
    ("softplus_sign", "return m + log1p(exp(-fabs(x)));", "return m - log1p(exp(-fabs(x)));"),
    ("gate_no_exp", "double l = -exp(A_log[h]) *", "double l = -A_log[h] *"),
    ("decay_after_update", "for (int64_t i = 0; i < dk * dv; ++i) S[i] *= gt;            /* S <- g S      */",
     "/* decay moved */"),
    ("delta_sign", "u[j] = bt * (vt[j] - sk[j]);", "u[j] = bt * (vt[j] + sk[j]);"),
    ("no_q_scale", "const double qi = qt[i] * qscale;", "const double qi = qt[i];"),
    ("key_head_modulo", "const int64_t j = h / group;", "const int64_t j = h % hk;"),
    ("rms_sum_not_mean", "double inv = 1.0 / sqrt(ss / (double)dv + eps);", "double inv = 1.0 / sqrt(ss + eps);"),
    ("post_eps_outside_sqrt", "double inv = 1.0 / sqrt(ss / (double)dv + eps);",
     "double inv = 1.0 / (sqrt(ss / (double)dv) + eps);"),
    ("post_sigmoid_gate", "gamma[i] * gdn_oracle_silu_scalar(zrow[i]);", "gamma[i] * gdn_oracle_sigmoid(zrow[i]);"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation anchor for {name} no longer matches the oracle source"
    mutated = tmp_path / "gdn_oracle_mut.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-shared", "-fPIC", str(mutated), "-o",
                    str(lib), "-lm"], check=True)
    env = dict(os.environ, GDN_ORACLE_LIB=str(lib), OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode != 0, f"pins did not catch mutation {name}:\n{r.stdout[-2000:]}"
