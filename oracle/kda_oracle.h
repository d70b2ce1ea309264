/*
 * kda_oracle.h -- fp64 CPU oracle of the KDA gated delta-rule recurrence.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the package smoke check and the benchmark's
 * CPU-baseline leg.  Independent of the CUDA library (include/kda.h): no shared code or header.
 *
 * Layouts (all row-major, fp64):
 *   q, k      [T][H][dk]          v, out  [T][H][dv]
 *   g_raw     [T][H][dk] (per-channel gate) or [T][H] (per-head gate)
 *   b_raw     [T][H]              A_log   [H]
 *   dt_bias   [H][dk] or [H], may be NULL (zero)
 *   pool      [num_slots][H][dv][dk]   (element (j, c) = S[c][j], the transpose of the maths)
 *   inter     [T][H][dv][dk]           (state after every token; verify mode)
 *   cu_seqlens[num_seqs + 1] int32, state_idx[num_seqs] int32 (< 0: padding row)
 */
#ifndef KDA_ORACLE_H
#define KDA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { KDAO_OK = 0, KDAO_ERR_ARG = -1 };
enum { KDAO_GATE_PER_CHANNEL = 0, KDAO_GATE_PER_HEAD = 1 };

typedef struct kdao_params {
    int32_t num_heads;
    int32_t dk;
    int32_t dv;
    int32_t gate_kind;          /* KDAO_GATE_PER_CHANNEL (KDA) or KDAO_GATE_PER_HEAD (GDN) */
    int32_t use_lower_bound;    /* 1: safe gate lower_bound * sigmoid(exp(A_log) * x) */
    int32_t use_qk_l2norm;      /* 1: L2-normalise q and k per token and head */
    double lower_bound;
    double scale;               /* q scale; <= 0 selects dk^{-1/2} */
    double l2_eps;              /* 1e-6 on the pages */
    double softplus_threshold;  /* 20 on the pages */
} kdao_params;

double kdao_softplus(double x, double threshold);
double kdao_sigmoid(double x);
void kdao_gate(const kdao_params* p, int n, const double* a, const double* dt_bias,
               double A_log_h, double* g);
void kdao_l2_normalize(int n, const double* x, double eps, double scale, double* out);
void kdao_unified_step(int dk, int dv, double* S, const double* gamma, double alpha_w,
                       double beta_w, const double* k, const double* v, const double* q,
                       double* o);
int kdao_forward(const kdao_params* p, const double* q, const double* k, const double* v,
                 const double* g_raw, const double* b_raw, const double* A_log,
                 const double* dt_bias, const int32_t* cu_seqlens, int32_t num_seqs,
                 double* pool, int64_t num_slots, const int32_t* state_idx, double* out,
                 double* inter, int32_t h_begin, int32_t h_end);
int kdao_chunk_forward(const kdao_params* p, int32_t chunk_size, const double* q,
                       const double* k, const double* v, const double* g_raw,
                       const double* b_raw, const double* A_log, const double* dt_bias,
                       const int32_t* cu_seqlens, int32_t num_seqs, double* pool,
                       int64_t num_slots, const int32_t* state_idx, double* out,
                       int32_t h_begin, int32_t h_end);

#ifdef __cplusplus
}
#endif

#endif
