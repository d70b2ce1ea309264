"""Mutation test of the oracle's pins (CPU only): each mutant is a copy of kda_oracle.c with one
plausible mistake planted (a dropped term, a wrong sign, a transposed index, a wrong constant);
the pin suite must fail for every one of them.  The mutants are compiled into a temporary
directory; nothing under oracle/ is modified."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "kda_oracle.c")

MUTANTS = {
    "softplus_threshold_flipped": ("if (x > threshold)", "if (x < threshold)"),
    "gate_sign": ("g[i] = -rate * kdao_softplus(", "g[i] = rate * kdao_softplus("),
    "safe_gate_drops_rate": ("g[i] = p->lower_bound * kdao_sigmoid(rate * x);", "g[i] = p->lower_bound * kdao_sigmoid(x);"),
    "sigmoid_sign": ("return 1.0 / (1.0 + exp(-x));", "return 1.0 / (1.0 + exp(x));"),
    "l2_eps_dropped": ("double r = scale / sqrt(ss + eps);", "double r = scale / sqrt(ss);"),
    "q_scale_wrong": ("1.0 / sqrt((double)p->dk)", "1.0 / (double)p->dk"),
    "error_sign": ("delta[j] = v[j] - vh;", "delta[j] = vh - v[j];"),
    "write_term_dropped": ("S[c * dv + j] += alpha_w * k[c] * v[j] + beta_w * k[c] * delta[j];",
                           "S[c * dv + j] += alpha_w * k[c] * v[j];"),
    "decay_dropped": ("            S[c * dv + j] *= gamma[c];\n    /* v_hat",
                            "            S[c * dv + j] *= 1.0;\n    /* v_hat"),
    "pool_not_transposed": ("S[c * dv + j] = src[(size_t)j * dk + c];", "S[c * dv + j] = src[(size_t)c * dv + j];"),
    "chunk_drops_P_Delta": ("acc += P[r * C + m] * Dl[m * dv + j];", "acc += 0.0 * P[r * C + m] * Dl[m * dv + j];"),
    "chunk_solve_sign": ("acc -= A[r * C + m] * U[m * dv + j];", "acc += A[r * C + m] * U[m * dv + j];"),
    "chunk_state_decay_index": ("acc += Kn[r * dk + c] * exp(GL - G[r * dk + c]) * Dl[r * dv + j];",
                                "acc += Kn[r * dk + c] * exp(G[r * dk + c] - G[0 * dk + c]) * Dl[r * dv + j];"),
}


def _build(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-I",
                    os.path.join(ROOT, "oracle"), "-o", str(so), str(path), "-lm"], check=True)
    return so


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    so = _build(tmp_path, name, old, new)
    env = dict(os.environ, KDA_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-x", "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"


def test_unmutated_oracle_passes_the_pins(tmp_path):
    so = _build(tmp_path, "identity", "#include <math.h>", "#include <math.h>")
    env = dict(os.environ, KDA_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"),
                        "-q", "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout[-2000:]
