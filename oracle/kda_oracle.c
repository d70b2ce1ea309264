/*
 * kda_oracle.c -- plain fp64 CPU oracle of the KDA gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  The test-suite, the package smoke check and the benchmark's
 * CPU-baseline leg are the only users.  The CUDA library never links, loads or calls this
 * file, and the two share no code, header, table or helper.
 *
 * Everything is computed in double precision, token by token, in the order the pages state
 * it.  There is no blocking, fusion or reordering beyond that, so the code can be checked
 * against the pages by eye.
 *
 * Notation ("linear_attention", zdszero.github.io, section "递归形式"): row vectors,
 * q_t, k_t in R^{1 x d_k}, v_t in R^{1 x d_v}, state S in R^{d_k x d_v}.  Inside this file the
 * state is held as S[c][j] with c the key channel (row) and j the value column.  The state pool
 * the library uses is stored transposed, element (j, c) at [slot][h][j][c]; the oracle converts
 * at its boundary (pool_load / pool_store below).
 *
 * Pins: every function here is checked by tests that do not call this file's formulas again
 * (tests/test_oracle_pins.py): the overwrite property, orthonormal readback, the prefix-sum
 * special case, the gradient-step identity, the beta-interpolation identity, contraction with
 * v = 0, the GDN-inside-KDA special case, the printed safe-gate half-lives, the explicit q scale,
 * the argument checks and agreement of the chunk closed form with the token recurrence.  A
 * mutation test (tests/test_oracle_mutants.py) plants one-line mistakes in copies of this file
 * and checks that the pins catch each of them.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "kda_oracle.h"

/* ------------------------------------------------------------------------------------------ */
/* Gate activations                                                                           */
/* ------------------------------------------------------------------------------------------ */

/* softplus with the pages' overflow guard: log(1 + exp(x)) for x <= threshold, x above it.
 * "ReplaySSM -- buffered output-only decode" (yuyanqi.com), section 3.8 (the numerically stable
 * softplus of the GDN gate branch); "PR #26888 report", the target_verify call (softplus_beta
 * 1.0, softplus_threshold 20.0). */
double kdao_softplus(double x, double threshold)
{
    if (x > threshold)
        return x;
    return log1p(exp(x));
}

/* beta_t = sigmoid(b_t).  "linear_attention", section "Gated DeltaNet" (gate parameterisation). */
double kdao_sigmoid(double x)
{
    return 1.0 / (1.0 + exp(-x));
}

/* Log-space decay of one token of one head.
 *
 * Default gate ("linear_attention", sections "Gated DeltaNet" and "KDA：逐通道的遗忘门"):
 *     g = -exp(A_log[h]) * softplus(a + dt_bias)
 * Safe gate ("linear_attention", section "实例：Kimi K3", gate_lower_bound = -5):
 *     g = lower_bound * sigmoid(exp(A_log[h]) * (a + dt_bias))
 * n = d_k for the per-channel (KDA) gate, n = 1 for the per-head scalar (GDN) gate.
 * dt_bias may be NULL (read as zero). */
void kdao_gate(const kdao_params* p, int n, const double* a, const double* dt_bias,
               double A_log_h, double* g)
{
    double rate = exp(A_log_h);
    for (int i = 0; i < n; ++i) {
        double x = a[i] + (dt_bias ? dt_bias[i] : 0.0);
        if (p->use_lower_bound)
            g[i] = p->lower_bound * kdao_sigmoid(rate * x);
        else
            g[i] = -rate * kdao_softplus(x, p->softplus_threshold);
    }
}

/* out = x / sqrt(sum x^2 + eps) * scale.  The pages normalise q and k inside the kernel
 * ("ReplaySSM", section 3.10: the factor 1/sqrt(sum(x^2) + 1e-6)) and scale q by d_k^{-1/2}
 * after the normalisation ("linear_attention", the per-token reference gated_delta_rule_ref). */
void kdao_l2_normalize(int n, const double* x, double eps, double scale, double* out)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i)
        ss += x[i] * x[i];
    double r = scale / sqrt(ss + eps);
    for (int i = 0; i < n; ++i)
        out[i] = x[i] * r;
}

/* ------------------------------------------------------------------------------------------ */
/* The unified recurrence, one token                                                          */
/* ------------------------------------------------------------------------------------------ */

/* One step of the unified recurrence ("linear_attention", section "统一递归形式"):
 *     v_hat = k (gamma S_{t-1})              decay first, then read the old value
 *     Delta = v - v_hat                      prediction error
 *     S_t   = gamma S_{t-1} + alpha_w k^T v + beta_w k^T Delta
 *     o_t   = q S_t
 * gamma is a diagonal (one factor per key channel = per row of S); the page writes a scalar, the
 * KDA section generalises it to Diag(alpha_t) acting on the rows.  S is [dk][dv] and is updated
 * in place; o may be NULL. */
void kdao_unified_step(int dk, int dv, double* S, const double* gamma, double alpha_w,
                       double beta_w, const double* k, const double* v, const double* q,
                       double* o)
{
    /* gamma S_{t-1} */
    for (int c = 0; c < dk; ++c)
        for (int j = 0; j < dv; ++j)
            S[c * dv + j] *= gamma[c];
    /* v_hat = k (gamma S_{t-1});  Delta = v - v_hat */
    double* delta = (double*)malloc(sizeof(double) * (size_t)dv);
    for (int j = 0; j < dv; ++j) {
        double vh = 0.0;
        for (int c = 0; c < dk; ++c)
            vh += k[c] * S[c * dv + j];
        delta[j] = v[j] - vh;
    }
    /* S_t = gamma S_{t-1} + alpha_w k^T v + beta_w k^T Delta */
    for (int c = 0; c < dk; ++c)
        for (int j = 0; j < dv; ++j)
            S[c * dv + j] += alpha_w * k[c] * v[j] + beta_w * k[c] * delta[j];
    free(delta);
    /* o_t = q S_t */
    if (o) {
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c)
                acc += q[c] * S[c * dv + j];
            o[j] = acc;
        }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Helpers for the packed varlen layout                                                       */
/* ------------------------------------------------------------------------------------------ */

static void pool_load(const kdao_params* p, const double* pool, int64_t slot, int h, double* S)
{
    const int dk = p->dk, dv = p->dv;
    const double* src = pool + ((size_t)slot * p->num_heads + h) * (size_t)dk * dv;
    for (int j = 0; j < dv; ++j)
        for (int c = 0; c < dk; ++c)
            S[c * dv + j] = src[(size_t)j * dk + c];
}

static void pool_store(const kdao_params* p, double* dst_base, size_t index, int h, const double* S)
{
    const int dk = p->dk, dv = p->dv;
    double* dst = dst_base + (index * p->num_heads + h) * (size_t)dk * dv;
    for (int j = 0; j < dv; ++j)
        for (int c = 0; c < dk; ++c)
            dst[(size_t)j * dk + c] = S[c * dv + j];
}

static double q_scale(const kdao_params* p)
{
    return p->scale > 0.0 ? p->scale : 1.0 / sqrt((double)p->dk);
}

static int check_common(const kdao_params* p, const int32_t* cu_seqlens, int32_t num_seqs,
                        const int32_t* state_idx, int64_t num_slots, int32_t h_begin,
                        int32_t h_end)
{
    if (!p || p->dk <= 0 || p->dv <= 0 || p->num_heads <= 0)
        return KDAO_ERR_ARG;
    if (h_begin < 0 || h_end > p->num_heads || h_begin > h_end)
        return KDAO_ERR_ARG;
    if (num_seqs < 0 || (num_seqs > 0 && (!cu_seqlens || !state_idx)))
        return KDAO_ERR_ARG;
    for (int32_t i = 0; i < num_seqs; ++i) {
        if (cu_seqlens[i + 1] < cu_seqlens[i])
            return KDAO_ERR_ARG;
        if (state_idx[i] >= num_slots)
            return KDAO_ERR_ARG;
    }
    return KDAO_OK;
}

/* Per-token input preparation shared by both oracle forms: normalised q and k, the gate and
 * beta of token t of head h.  g has dk entries; the per-head gate is broadcast over them. */
static void prepare_token(const kdao_params* p, int64_t t, int h, const double* q,
                          const double* k, const double* g_raw, const double* b_raw,
                          const double* A_log, const double* dt_bias, double* qn, double* kn,
                          double* g, double* beta)
{
    const int H = p->num_heads, dk = p->dk;
    const double* qt = q + ((size_t)t * H + h) * dk;
    const double* kt = k + ((size_t)t * H + h) * dk;
    if (p->use_qk_l2norm) {
        kdao_l2_normalize(dk, qt, p->l2_eps, q_scale(p), qn);
        kdao_l2_normalize(dk, kt, p->l2_eps, 1.0, kn);
    } else {
        for (int c = 0; c < dk; ++c) {
            qn[c] = qt[c] * q_scale(p);
            kn[c] = kt[c];
        }
    }
    if (p->gate_kind == KDAO_GATE_PER_CHANNEL) {
        kdao_gate(p, dk, g_raw + ((size_t)t * H + h) * dk, dt_bias ? dt_bias + (size_t)h * dk : NULL,
                  A_log[h], g);
    } else {
        double g0;
        kdao_gate(p, 1, g_raw + (size_t)t * H + h, dt_bias ? dt_bias + h : NULL, A_log[h], &g0);
        for (int c = 0; c < dk; ++c)
            g[c] = g0;
    }
    *beta = kdao_sigmoid(b_raw[(size_t)t * H + h]);
}

/* ------------------------------------------------------------------------------------------ */
/* Token-by-token forward (the definition)                                                    */
/* ------------------------------------------------------------------------------------------ */

/* The KDA recurrence over packed varlen sequences, one token at a time
 * ("linear_attention", section "KDA：逐通道的遗忘门"):
 *     S_t = (I - beta_t k_t^T k_t) Diag(alpha_t) S_{t-1} + beta_t k_t^T v_t,  o_t = q_t S_t,
 * evaluated as the five steps of the page's per-token reference (decay, predict, error, write,
 * read), i.e. the unified step with gamma = Diag(exp g_t), alpha_w = 0, beta_w = beta_t.
 *
 * Sequence i holds tokens cu_seqlens[i] .. cu_seqlens[i+1]-1 and starts from the pool slot
 * state_idx[i] ("KDA inference components", section 4.5: per-request slots; slots are cleared
 * on allocation, so the caller zeroes a slot to start from S_0 = 0).  A negative state_idx marks
 * a padding row: its outputs are zero and nothing is read or written ("ReplaySSM", section
 * 3.6).  With inter == NULL the final state is written back to the same slot (prefill and
 * decode).  With inter != NULL the pool is left untouched and the state after every token t is
 * written to inter[t] (the verify mode of "PR #26888 report": disable_state_update with an
 * intermediate-state buffer).  Only heads h_begin .. h_end-1 are computed. */
int kdao_forward(const kdao_params* p, const double* q, const double* k, const double* v,
                 const double* g_raw, const double* b_raw, const double* A_log,
                 const double* dt_bias, const int32_t* cu_seqlens, int32_t num_seqs,
                 double* pool, int64_t num_slots, const int32_t* state_idx, double* out,
                 double* inter, int32_t h_begin, int32_t h_end)
{
    int rc = check_common(p, cu_seqlens, num_seqs, state_idx, num_slots, h_begin, h_end);
    if (rc != KDAO_OK)
        return rc;
    const int H = p->num_heads, dk = p->dk, dv = p->dv;
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
    double* qn = (double*)malloc(sizeof(double) * (size_t)dk);
    double* kn = (double*)malloc(sizeof(double) * (size_t)dk);
    double* g = (double*)malloc(sizeof(double) * (size_t)dk);
    double* gamma = (double*)malloc(sizeof(double) * (size_t)dk);
    double* o = (double*)malloc(sizeof(double) * (size_t)dv);

    for (int32_t i = 0; i < num_seqs; ++i) {
        const int64_t t0 = cu_seqlens[i], t1 = cu_seqlens[i + 1];
        for (int h = h_begin; h < h_end; ++h) {
            if (state_idx[i] < 0) {
                for (int64_t t = t0; t < t1; ++t)
                    memset(out + ((size_t)t * H + h) * dv, 0, sizeof(double) * (size_t)dv);
                continue;
            }
            pool_load(p, pool, state_idx[i], h, S);
            for (int64_t t = t0; t < t1; ++t) {
                double beta;
                prepare_token(p, t, h, q, k, g_raw, b_raw, A_log, dt_bias, qn, kn, g, &beta);
                for (int c = 0; c < dk; ++c)
                    gamma[c] = exp(g[c]);
                kdao_unified_step(dk, dv, S, gamma, 0.0, beta, kn, v + ((size_t)t * H + h) * dv,
                                  qn, o);
                memcpy(out + ((size_t)t * H + h) * dv, o, sizeof(double) * (size_t)dv);
                if (inter)
                    pool_store(p, inter, (size_t)t, h, S);
            }
            if (!inter)
                pool_store(p, pool, (size_t)state_idx[i], h, S);
        }
    }
    free(S); free(qn); free(kn); free(g); free(gamma); free(o);
    return KDAO_OK;
}

/* ------------------------------------------------------------------------------------------ */
/* Chunk closed form (self-check of the chunkwise algorithm)                                  */
/* ------------------------------------------------------------------------------------------ */

/* The chunkwise form of the same recurrence ("linear_attention", sections "矩阵（并行）形式"
 * and "两种计算形态"): each sequence is cut into chunks of C tokens (restarting at every sequence
 * start; the last chunk of a sequence may be shorter).  Within a chunk of L tokens entering
 * with state S0, with G_r = sum_{i<=r} g_i (per key channel, local index r):
 *     A[r][j] = beta_r sum_c k_r[c] k_j[c] exp(G_r[c] - G_j[c])   (j < r)
 *     P[r][j] =        sum_c q_r[c] k_j[c] exp(G_r[c] - G_j[c])   (j <= r)
 *     (I + A) U = diag(beta) V                  solved by forward substitution
 *     (I + A) W = diag(beta) (K o exp(G))
 *     Delta = U - W S0                          ("v_new = U - W S_i")
 *     O     = (Q o exp(G)) S0 + P Delta
 *     S_L   = Diag(exp(G_L)) S0 + (K o exp(G_L - G))^T Delta
 * The lower-triangular inverse (I + A)^{-1} is the closed form of the delta-rule chain that the
 * page describes; the page's own equation for it was lost, so the derivation is restated in the
 * project's design notes.  Every exponent above is <= 0, so nothing overflows.  Used only to
 * check the token recurrence and the chunk algorithm against each other. */
int kdao_chunk_forward(const kdao_params* p, int32_t chunk_size, const double* q,
                       const double* k, const double* v, const double* g_raw,
                       const double* b_raw, const double* A_log, const double* dt_bias,
                       const int32_t* cu_seqlens, int32_t num_seqs, double* pool,
                       int64_t num_slots, const int32_t* state_idx, double* out,
                       int32_t h_begin, int32_t h_end)
{
    int rc = check_common(p, cu_seqlens, num_seqs, state_idx, num_slots, h_begin, h_end);
    if (rc != KDAO_OK)
        return rc;
    if (chunk_size <= 0)
        return KDAO_ERR_ARG;
    const int H = p->num_heads, dk = p->dk, dv = p->dv, C = chunk_size;
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
    double* Qn = (double*)malloc(sizeof(double) * (size_t)C * dk);
    double* Kn = (double*)malloc(sizeof(double) * (size_t)C * dk);
    double* G = (double*)malloc(sizeof(double) * (size_t)C * dk);
    double* beta = (double*)malloc(sizeof(double) * (size_t)C);
    double* A = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* P = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* U = (double*)malloc(sizeof(double) * (size_t)C * dv);
    double* W = (double*)malloc(sizeof(double) * (size_t)C * dk);
    double* Dl = (double*)malloc(sizeof(double) * (size_t)C * dv);
    double* g = (double*)malloc(sizeof(double) * (size_t)dk);
    double* Snew = (double*)malloc(sizeof(double) * (size_t)dk * dv);

    for (int32_t i = 0; i < num_seqs; ++i) {
        const int64_t t0 = cu_seqlens[i], t1 = cu_seqlens[i + 1];
        for (int h = h_begin; h < h_end; ++h) {
            if (state_idx[i] < 0) {
                for (int64_t t = t0; t < t1; ++t)
                    memset(out + ((size_t)t * H + h) * dv, 0, sizeof(double) * (size_t)dv);
                continue;
            }
            pool_load(p, pool, state_idx[i], h, S);
            for (int64_t cs = t0; cs < t1; cs += C) {
                const int L = (int)((t1 - cs) < C ? (t1 - cs) : C);
                /* per-token preparation and the in-chunk cumulative log decay G */
                for (int r = 0; r < L; ++r) {
                    prepare_token(p, cs + r, h, q, k, g_raw, b_raw, A_log, dt_bias, Qn + r * dk,
                                  Kn + r * dk, g, &beta[r]);
                    for (int c = 0; c < dk; ++c)
                        G[r * dk + c] = (r == 0 ? 0.0 : G[(r - 1) * dk + c]) + g[c];
                }
                /* A (strictly lower) and P (lower, with diagonal) */
                for (int r = 0; r < L; ++r)
                    for (int j = 0; j < L; ++j) {
                        double a = 0.0, pq = 0.0;
                        if (j <= r) {
                            for (int c = 0; c < dk; ++c) {
                                double d = exp(G[r * dk + c] - G[j * dk + c]);
                                a += Kn[r * dk + c] * Kn[j * dk + c] * d;
                                pq += Qn[r * dk + c] * Kn[j * dk + c] * d;
                            }
                        }
                        A[r * C + j] = (j < r) ? beta[r] * a : 0.0;
                        P[r * C + j] = (j <= r) ? pq : 0.0;
                    }
                /* forward substitution: (I + A) U = diag(beta) V, (I + A) W = diag(beta)(K o e^G) */
                for (int r = 0; r < L; ++r) {
                    const double* vr = v + ((size_t)(cs + r) * H + h) * dv;
                    for (int j = 0; j < dv; ++j) {
                        double acc = beta[r] * vr[j];
                        for (int m = 0; m < r; ++m)
                            acc -= A[r * C + m] * U[m * dv + j];
                        U[r * dv + j] = acc;
                    }
                    for (int c = 0; c < dk; ++c) {
                        double acc = beta[r] * Kn[r * dk + c] * exp(G[r * dk + c]);
                        for (int m = 0; m < r; ++m)
                            acc -= A[r * C + m] * W[m * dk + c];
                        W[r * dk + c] = acc;
                    }
                }
                /* Delta = U - W S0 */
                for (int r = 0; r < L; ++r)
                    for (int j = 0; j < dv; ++j) {
                        double acc = U[r * dv + j];
                        for (int c = 0; c < dk; ++c)
                            acc -= W[r * dk + c] * S[c * dv + j];
                        Dl[r * dv + j] = acc;
                    }
                /* O = (Q o e^G) S0 + P Delta */
                for (int r = 0; r < L; ++r) {
                    double* orow = out + ((size_t)(cs + r) * H + h) * dv;
                    for (int j = 0; j < dv; ++j) {
                        double acc = 0.0;
                        for (int c = 0; c < dk; ++c)
                            acc += Qn[r * dk + c] * exp(G[r * dk + c]) * S[c * dv + j];
                        for (int m = 0; m <= r; ++m)
                            acc += P[r * C + m] * Dl[m * dv + j];
                        orow[j] = acc;
                    }
                }
                /* S_L = Diag(e^{G_L}) S0 + (K o e^{G_L - G})^T Delta */
                for (int c = 0; c < dk; ++c) {
                    const double GL = G[(L - 1) * dk + c];
                    for (int j = 0; j < dv; ++j) {
                        double acc = exp(GL) * S[c * dv + j];
                        for (int r = 0; r < L; ++r)
                            acc += Kn[r * dk + c] * exp(GL - G[r * dk + c]) * Dl[r * dv + j];
                        Snew[c * dv + j] = acc;
                    }
                }
                memcpy(S, Snew, sizeof(double) * (size_t)dk * dv);
            }
            pool_store(p, pool, (size_t)state_idx[i], h, S);
        }
    }
    free(S); free(Qn); free(Kn); free(G); free(beta); free(A); free(P); free(U); free(W);
    free(Dl); free(g); free(Snew);
    return KDAO_OK;
}
