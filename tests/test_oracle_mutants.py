"""Mutation test of the oracle's pins (CPU only): each mutant is a copy of kda_oracle.c with one
plausible mistake planted (a dropped term, a wrong sign, a transposed index, a wrong constant);
the pin suite must fail for every one of them.  The mutants are compiled into a temporary
directory; nothing under oracle/ is modified.  Mutants that cannot change any result are left
out: the diagonal of A, for instance, is never read by the forward substitution."""
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
    "pool_store_not_transposed": ("dst[(size_t)j * dk + c] = S[c * dv + j];", "dst[(size_t)c * dv + j] = S[c * dv + j];"),
    "gate_cumsum_exclusive": ("G[r * dk + c] = (r == 0 ? 0.0 : G[(r - 1) * dk + c]) + g[c];",
                              "G[r * dk + c] = (r == 0 ? 0.0 : G[(r - 1) * dk + c] + g[c]);"),
    "chunk_P_drops_diagonal": ("P[r * C + j] = (j <= r) ? pq : 0.0;", "P[r * C + j] = (j < r) ? pq : 0.0;"),
    "chunk_P_drops_decay": ("pq += Qn[r * dk + c] * Kn[j * dk + c] * d;", "pq += Qn[r * dk + c] * Kn[j * dk + c];"),
    "chunk_A_drops_beta": ("A[r * C + j] = (j < r) ? beta[r] * a : 0.0;", "A[r * C + j] = (j < r) ? a : 0.0;"),
    "chunk_A_beta_of_column": ("A[r * C + j] = (j < r) ? beta[r] * a : 0.0;", "A[r * C + j] = (j < r) ? beta[j] * a : 0.0;"),
    "chunk_U_drops_beta": ("double acc = beta[r] * vr[j];", "double acc = vr[j];"),
    "chunk_W_drops_decay": ("double acc = beta[r] * Kn[r * dk + c] * exp(G[r * dk + c]);",
                            "double acc = beta[r] * Kn[r * dk + c];"),
    "chunk_Delta_sign": ("acc -= W[r * dk + c] * S[c * dv + j];", "acc += W[r * dk + c] * S[c * dv + j];"),
    "chunk_O_inter_drops_decay": ("acc += Qn[r * dk + c] * exp(G[r * dk + c]) * S[c * dv + j];",
                                  "acc += Qn[r * dk + c] * S[c * dv + j];"),
    "chunk_state_drops_decay": ("double acc = exp(GL) * S[c * dv + j];", "double acc = S[c * dv + j];"),
    "beta_without_sigmoid": ("*beta = kdao_sigmoid(b_raw[(size_t)t * H + h]);", "*beta = b_raw[(size_t)t * H + h];"),
    "explicit_scale_ignored": ("return p->scale > 0.0 ? p->scale : 1.0 / sqrt((double)p->dk);",
                               "return 1.0 / sqrt((double)p->dk);"),
    "dt_bias_of_head_0": ("dt_bias ? dt_bias + (size_t)h * dk : NULL", "dt_bias ? dt_bias : NULL"),
    "gdn_dt_bias_of_head_0": ("dt_bias ? dt_bias + h : NULL", "dt_bias ? dt_bias : NULL"),
    "k_scaled_like_q": ("kdao_l2_normalize(dk, kt, p->l2_eps, 1.0, kn);",
                        "kdao_l2_normalize(dk, kt, p->l2_eps, q_scale(p), kn);"),
    "softplus_drops_log": ("return log1p(exp(x));", "return exp(x);"),
    "rate_not_exponentiated": ("double rate = exp(A_log_h);", "double rate = A_log_h;"),
    "prediction_reads_q": ("vh += k[c] * S[c * dv + j];", "vh += q[c] * S[c * dv + j];"),
    "write_weights_swapped": ("kdao_unified_step(dk, dv, S, gamma, 0.0, beta, kn,",
                              "kdao_unified_step(dk, dv, S, gamma, beta, 0.0, kn,"),
    "verify_states_at_local_index": ("pool_store(p, inter, (size_t)t, h, S);", "pool_store(p, inter, (size_t)(t - t0), h, S);"),
    "slot_bound_off_by_one": ("if (state_idx[i] >= num_slots)", "if (state_idx[i] > num_slots)"),
    "seqlen_order_unchecked": ("if (cu_seqlens[i + 1] < cu_seqlens[i])", "if (0)"),
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
