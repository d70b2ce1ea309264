// kda_prefill.cu -- chunkwise-parallel KDA prefill over packed varlen sequences.
//
// Algorithm ("linear_attention", zdszero.github.io, sections "矩阵（并行）形式" and
// "两种计算形态"): each sequence is cut into chunks of C tokens.  For a chunk of L tokens with
// per-channel cumulative log decay G_r = sum_{i<=r} g_i and entry state S0:
//   A[r][j] = beta_r sum_c k_r[c] k_j[c] e^{G_r[c]-G_j[c]}       (j <  r)
//   P[r][j] =        sum_c q_r[c] k_j[c] e^{G_r[c]-G_j[c]}       (j <= r)
//   U = (I + A)^{-1} diag(beta) V,   W = (I + A)^{-1} diag(beta) (K o e^{G})   (forward substitution)
//   Delta = U - W S0;   O = (Q o e^{G}) S0 + P Delta
//   S_L   = Diag(e^{G_L}) S0 + (K o e^{G_L - G})^T Delta
//
// Three kernels, all on the caller's stream, no host synchronisation:
//   chunk_table_kernel   builds the chunk list from the device cu_seqlens;
//   intra-chunk kernel   one CTA per (chunk, head): everything that does not depend on S0
//                        (W, U, Q o e^G, K o e^{G_L-G}, P, e^{G_L}) into the workspace;
//   state-pass kernel    the serial pass over a sequence's chunks, keeping S on chip.
// bf16 inputs at C = 64, D = 128 take the tensor-core pair (chunk_intra_tc_kernel, two CTAs per SM,
// and chunk_state_tc_kernel, one CTA per (sequence, head)), which exchange a per-(chunk, head)
// record laid out as the state pass's shared-memory operand images (TcRec).  Every other shape and
// fp32 inputs take the fp32 CUDA-core pair (chunk_intra_kernel; chunk_state_kernel with one CTA
// per (sequence, head, value tile)), which meets the 1e-5 bound of fp32 I/O.
//
// Overflow-free decay algebra.  With these gates g reaches tens per token, so e^{-G} overflows
// fp32 long before a chunk ends.  No decay factor here is ever formed from an exponent > 0:
//   * alpha = e^{g} <= 1 is computed once per (token, channel);
//   * every decay e^{G_r - G_j} (r >= j) is a product of alphas, split at 16-row sub-block
//     boundaries: r in block I, j in block J < I  ->  Rin_I(r) * M_IJ * Rout_J(j), with
//     Rin the in-block prefix product up to r, Rout the in-block suffix product after j and
//     M_IJ the product of the whole blocks strictly between them; inside a diagonal block the
//     running product is accumulated token by token.
// Products of factors in (0, 1] cannot overflow and lose at most one rounding per factor, so the
// fp32 path keeps the 1e-5 relative accuracy the fp32 configuration needs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

__device__ int32_t g_prefill_error = 0;
__device__ __forceinline__ void record_error(int32_t code) { atomicCAS(&g_prefill_error, 0, code); }

constexpr int kSub = 16;  // sub-block length of the decay split

// Record of one (chunk, head) for the tensor-core state pass (C = 64, D = 128), in bytes.  It is
// also the shared-memory image of that pass: operand images in the no-swizzle K-major layout of
// kda_tc.cuh, already rounded to tf32.
struct TcRec {
    static constexpr int C = 64, D = 128;
    static constexpr uint32_t W = 0;          // W:      rows r (64), K = c (128)  image
    static constexpr uint32_t KT = 32768;     // Ktil^T: rows c (128), K = r (64)  image
    static constexpr uint32_t U = 65536;      // U [r][v] fp32 (not rounded)
    static constexpr uint32_t GL = 98304;     // e^{G_L} [c] fp32, 128 values + padding
    static constexpr uint32_t QB = 98816;     // Qbar:   rows r (64), K = c (128)  image
    static constexpr uint32_t P = 131584;     // P:      rows r (64), K = j (64)   image
    static constexpr uint32_t BYTES = 147968;
};

// ---- workspace layout ----------------------------------------------------------------------
// [chunk table: 3 * max_chunks + (N + 1) + N int32, padded to 256 B]
// [per (chunk, head): W C*D | Qbar C*D | Ktil C*D | U C*D | P C*C | gL D  floats, padded to 64]
struct WsLayout {
    int64_t max_chunks;
    size_t table_bytes;
    size_t per_chunk_head;  // floats
    size_t total_bytes;
};

__host__ __device__ inline size_t round_up(size_t x, size_t m) { return (x + m - 1) / m * m; }

WsLayout ws_layout(int C, int D, int H, int32_t N, int64_t T)
{
    WsLayout w;
    w.max_chunks = (T + C - 1) / C + N;
    w.table_bytes = round_up(sizeof(int32_t) * (size_t)(3 * w.max_chunks + 2 * (int64_t)N + 1), 256);
    w.per_chunk_head = round_up((size_t)4 * C * D + (size_t)C * C + D, 64);
    w.total_bytes = w.table_bytes + sizeof(float) * w.per_chunk_head * (size_t)w.max_chunks * H;
    return w;
}

// ---- chunk table -----------------------------------------------------------------------------
// One CTA of 1024 threads.  chunk i of the packed batch covers tokens
// chunk_start[i] .. chunk_start[i] + chunk_len[i] - 1 of sequence chunk_seq[i]; the chunks of
// sequence s are seq_off[s] .. seq_off[s+1]-1 and seq_off[N] is the number of chunks.
// seq_order lists the sequences by decreasing chunk count (ties by index; identity when
// N > 4096), so that the state pass starts its longest serial chains first.
constexpr int32_t kMaxSortedSeqs = 4096;
// token range of sequence i, clamped into [0, T] (a malformed cu_seqlens is recorded, not trusted)
__device__ __forceinline__ void seq_range(const int32_t* __restrict__ cu, int32_t i, int32_t N, int64_t T,
                                          int64_t& s0, int64_t& s1, bool record)
{
    s0 = cu[i];
    s1 = cu[i + 1];
    const bool bad = s0 < 0 || s1 < s0 || s1 > T || (i == 0 && s0 != 0) || (i == N - 1 && s1 != T);
    if (bad) {
        if (record) record_error(kDevErrSeqlens);
        s0 = s0 < 0 ? 0 : (s0 > T ? T : s0);
        s1 = s1 < s0 ? s0 : (s1 > T ? T : s1);
    }
}

__global__ void __launch_bounds__(1024) chunk_table_kernel(const int32_t* __restrict__ cu, int32_t N, int64_t T,
                                                           int C, int64_t max_chunks,
                                                           int32_t* chunk_seq, int32_t* chunk_start,
                                                           int32_t* chunk_len, int32_t* seq_off,
                                                           int32_t* seq_order)
{
    __shared__ int32_t s_warp[32];
    __shared__ int32_t s_base;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) s_base = 0;
    __syncthreads();
    // 1. chunk counts and their exclusive prefix sum -> seq_off
    for (int32_t base = 0; base < N; base += blockDim.x) {
        const int32_t i = base + tid;
        int32_t n = 0;
        if (i < N) {
            int64_t s0, s1;
            seq_range(cu, i, N, T, s0, s1, true);
            n = (int32_t)((s1 - s0 + C - 1) / C);
        }
        // inclusive scan of n over the CTA
        int32_t x = n;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int32_t w = lane < (int)(blockDim.x >> 5) ? s_warp[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int32_t y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            s_warp[lane] = w;
        }
        __syncthreads();
        const int32_t incl = x + (warp > 0 ? s_warp[warp - 1] : 0);
        const int32_t off0 = s_base + incl - n;
        if (i < N) seq_off[i] = off0;
        __syncthreads();
        if (tid == blockDim.x - 1) s_base = off0 + n;
        __syncthreads();
    }
    if (tid == 0) {
        seq_off[N] = s_base;
        if (s_base > max_chunks) record_error(kDevErrSeqlens);
    }
    __syncthreads();
    // 2. one thread per chunk: its sequence by binary search over seq_off, then start and length
    const int64_t nch = s_base < max_chunks ? s_base : max_chunks;
    for (int64_t c = tid; c < nch; c += blockDim.x) {
        int32_t lo = 0, hi = N - 1;                  // last i with seq_off[i] <= c
        while (lo < hi) {
            const int32_t mid = (lo + hi + 1) >> 1;
            if (seq_off[mid] <= c) lo = mid;
            else hi = mid - 1;
        }
        int64_t s0, s1;
        seq_range(cu, lo, N, T, s0, s1, false);
        const int64_t st = s0 + (c - seq_off[lo]) * C;
        chunk_seq[c] = lo;
        chunk_start[c] = (int32_t)st;
        chunk_len[c] = (int32_t)((s1 - st) < C ? (s1 - st) : C);
    }
    // 3. sequences by decreasing chunk count
    for (int32_t i = tid; i < N; i += blockDim.x) {
        if (N > kMaxSortedSeqs) {
            seq_order[i] = i;
            continue;
        }
        const int32_t ni = seq_off[i + 1] - seq_off[i];
        int32_t rank = 0;
        for (int32_t j = 0; j < N; ++j) {
            const int32_t nj = seq_off[j + 1] - seq_off[j];
            rank += (nj > ni) || (nj == ni && j < i);
        }
        seq_order[rank] = i;
    }
}

// ---- intra-chunk kernel ----------------------------------------------------------------------
struct IntraArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g_raw;
    const float* b_raw;
    const float* A_log;
    const float* dt_bias;
    const int32_t* chunk_seq;
    const int32_t* chunk_start;
    const int32_t* chunk_len;
    const int32_t* seq_off;   // seq_off[N] = number of chunks
    const int32_t* state_idx;
    int64_t num_slots;
    int64_t max_chunks;
    int32_t N;
    int H;
    GateParams gp;
    float* ws;                // per-(chunk, head) records
    size_t ws_stride;         // floats per record
};

template <int C, int D>
struct IntraShape {
    static constexpr int THREADS = (2 * D > C ? 2 * D : C) < 64 ? 64 : (2 * D > C ? 2 * D : C);
    static constexpr int NB = C / kSub;           // sub-blocks per chunk
    static constexpr int NCG = THREADS / C;        // column groups per row j (diagonal blocks)
    static constexpr int CPT = D / NCG;            // columns per thread (diagonal blocks)
    static constexpr int PADC = C + 1;
    static_assert(C % kSub == 0, "chunk must be a multiple of 16");
    static_assert(NCG >= 1 && D % (4 * NCG) == 0, "column split");
    static_assert(THREADS >= 2 * D && THREADS >= C, "threads");
    // shared memory (floats)
    static constexpr size_t OFF_AL = 0;                       // alpha [C][D]
    static constexpr size_t OFF_K = OFF_AL + (size_t)C * D;   // k_hat -> k o Rin  [C][D]
    static constexpr size_t OFF_Q = OFF_K + (size_t)C * D;    // q_hat -> q o Rin  [C][D]
    static constexpr size_t OFF_KOT = OFF_Q + (size_t)C * D;  // (k o Rout)^T [D][C+1]
    static constexpr size_t OFF_A = OFF_KOT + (size_t)D * PADC;
    static constexpr size_t OFF_P = OFF_A + (size_t)C * PADC;
    static constexpr size_t OFF_BP = OFF_P + (size_t)C * PADC;  // block products [NB][D]
    static constexpr size_t OFF_BETA = OFF_BP + (size_t)NB * D;
    static constexpr size_t OFF_RED = OFF_BETA + C;            // row norms [2][C]
    static constexpr size_t FLOATS = OFF_RED + 2 * C;
    static constexpr size_t BYTES = FLOATS * sizeof(float);
};

// Record written per (chunk, head).  TCREC = false: plain fp32 arrays for the SIMT state pass.
// TCREC = true (C = 64, D = 128): the shared-memory image the tensor-core state pass copies in
// one piece (see TcRec): tf32-rounded K-major operand images plus plain U and e^{G_L}.
template <int C, int D, typename TIn, bool TCREC>
__global__ void __launch_bounds__(IntraShape<C, D>::THREADS, 1) chunk_intra_kernel(const IntraArgs a)
{
    using Sh = IntraShape<C, D>;
    constexpr int THREADS = Sh::THREADS, NB = Sh::NB, NCG = Sh::NCG, CPT = Sh::CPT, PADC = Sh::PADC;
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    float* s_al = sm + Sh::OFF_AL;
    float* s_k = sm + Sh::OFF_K;
    float* s_q = sm + Sh::OFF_Q;
    float* s_koT = sm + Sh::OFF_KOT;
    float* s_A = sm + Sh::OFF_A;
    float* s_P = sm + Sh::OFF_P;
    float* s_bp = sm + Sh::OFF_BP;
    float* s_beta = sm + Sh::OFF_BETA;
    float* s_rn = sm + Sh::OFF_RED;

    const int64_t ch = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t nch = a.seq_off[a.N];
    if (nch > a.max_chunks) nch = a.max_chunks;
    if (ch >= nch) return;
    const int32_t seq = a.chunk_seq[ch];
    const int64_t slot = a.state_idx[seq];
    if (slot < 0 || slot >= a.num_slots) return;  // padding row: the state pass writes zeros
    const int64_t t0 = a.chunk_start[ch];
    const int L = a.chunk_len[ch];
    const int H = a.H;
    const TIn* qp = reinterpret_cast<const TIn*>(a.q);
    const TIn* kp = reinterpret_cast<const TIn*>(a.k);
    const TIn* vp = reinterpret_cast<const TIn*>(a.v);
    const float rate = expf(a.A_log[h]);

    // 1. load k, q, alpha = e^{g}; rows past the chunk end are k = q = 0, alpha = 1, beta = 0
    for (int e = tid; e < C * D; e += THREADS) {
        const int r = e / D, c = e % D;
        float kv = 0.f, qv = 0.f, al = 1.f;
        if (r < L) {
            const size_t idx = ((size_t)(t0 + r) * H + h) * D + c;
            kv = to_f32(kp[idx]);
            qv = to_f32(qp[idx]);
            const float x = a.g_raw[idx] + (a.dt_bias ? a.dt_bias[(size_t)h * D + c] : 0.f);
            al = expf(gate_log_decay(x, rate, a.gp));
        }
        s_k[e] = kv;
        s_q[e] = qv;
        s_al[e] = al;
    }
    for (int r = tid; r < C; r += THREADS)
        s_beta[r] = r < L ? sigmoid_f32(a.b_raw[(size_t)(t0 + r) * H + h]) : 0.f;
    __syncthreads();

    // 2. L2-normalise the rows of k and q (one warp per row)
    for (int r = warp; r < C; r += THREADS / 32) {
        float kk = 0.f, qq = 0.f;
        for (int c = lane; c < D; c += 32) {
            kk += s_k[r * D + c] * s_k[r * D + c];
            qq += s_q[r * D + c] * s_q[r * D + c];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            qq += __shfl_xor_sync(0xffffffffu, qq, off);
        }
        if (lane == 0) {
            s_rn[r] = 1.0f / sqrtf(kk + a.gp.l2_eps);
            s_rn[C + r] = a.gp.scale / sqrtf(qq + a.gp.l2_eps);
        }
    }
    __syncthreads();
    for (int e = tid; e < C * D; e += THREADS) {
        const int r = e / D;
        s_k[e] *= s_rn[r];
        s_q[e] *= s_rn[C + r];
    }
    for (int e = tid; e < C * PADC; e += THREADS) {
        s_A[e] = 0.f;
        s_P[e] = 0.f;
    }
    __syncthreads();

    // 3. diagonal sub-blocks: running product of alphas, one (row j, column group) per thread
    {
        const int j = tid / NCG;       // 0 .. C-1
        const int cg = tid % NCG;
        const int blk0 = (j / kSub) * kSub;
        float kd[CPT];
#pragma unroll
        for (int m = 0; m < CPT / 4; ++m) {
            const float4 v4 = *reinterpret_cast<const float4*>(&s_k[j * D + 4 * cg + 4 * NCG * m]);
            kd[4 * m + 0] = v4.x; kd[4 * m + 1] = v4.y; kd[4 * m + 2] = v4.z; kd[4 * m + 3] = v4.w;
        }
#pragma unroll 1
        for (int rr = 0; rr < kSub; ++rr) {
            const int r = blk0 + rr;
            const bool act = r >= j;
            float pa = 0.f, pp = 0.f;
#pragma unroll
            for (int m = 0; m < CPT / 4; ++m) {
                const int c = 4 * cg + 4 * NCG * m;
                const float4 al4 = *reinterpret_cast<const float4*>(&s_al[r * D + c]);
                const float4 k4 = *reinterpret_cast<const float4*>(&s_k[r * D + c]);
                const float4 q4 = *reinterpret_cast<const float4*>(&s_q[r * D + c]);
                if (r > j) {
                    kd[4 * m + 0] *= al4.x; kd[4 * m + 1] *= al4.y;
                    kd[4 * m + 2] *= al4.z; kd[4 * m + 3] *= al4.w;
                }
                pa = fmaf(k4.x, kd[4 * m + 0], pa); pa = fmaf(k4.y, kd[4 * m + 1], pa);
                pa = fmaf(k4.z, kd[4 * m + 2], pa); pa = fmaf(k4.w, kd[4 * m + 3], pa);
                pp = fmaf(q4.x, kd[4 * m + 0], pp); pp = fmaf(q4.y, kd[4 * m + 1], pp);
                pp = fmaf(q4.z, kd[4 * m + 2], pp); pp = fmaf(q4.w, kd[4 * m + 3], pp);
            }
#pragma unroll
            for (int off = NCG / 2; off > 0; off >>= 1) {
                pa += __shfl_xor_sync(0xffffffffu, pa, off);
                pp += __shfl_xor_sync(0xffffffffu, pp, off);
            }
            if (act && cg == 0) {
                if (r > j) s_A[r * PADC + j] = s_beta[r] * pa;
                s_P[r * PADC + j] = pp;
            }
        }
    }
    __syncthreads();

    // 4. per-column sub-block products: k o Rin -> s_k, q o Rin -> s_q, (k o Rout)^T -> s_koT
    for (int c = tid; c < D; c += THREADS) {
        for (int blk = 0; blk < NB; ++blk) {
            float rout = 1.f;
            for (int rr = kSub - 1; rr >= 0; --rr) {
                const int r = blk * kSub + rr;
                s_koT[c * PADC + r] = s_k[r * D + c] * rout;
                rout *= s_al[r * D + c];
            }
            s_bp[blk * D + c] = rout;
            float rin = 1.f;
            for (int rr = 0; rr < kSub; ++rr) {
                const int r = blk * kSub + rr;
                rin *= s_al[r * D + c];
                s_k[r * D + c] *= rin;
                s_q[r * D + c] *= rin;
            }
        }
    }
    __syncthreads();

    // 5. off-diagonal sub-blocks: A[r][j] = beta_r sum_c kin[r][c] M_IJ[c] kout[j][c], same for P
    for (int e = tid; e < NB * (NB - 1) / 2 * kSub * kSub; e += THREADS) {
        int pair = e / (kSub * kSub);
        const int within = e % (kSub * kSub);
        int I = 1, J = 0;
        {   // enumerate (I, J) with J < I
            int cnt = pair;
            for (I = 1; I < NB; ++I) {
                if (cnt < I) { J = cnt; break; }
                cnt -= I;
            }
        }
        const int r = I * kSub + within / kSub;
        const int j = J * kSub + within % kSub;
        float pa = 0.f, pp = 0.f;
        for (int c = 0; c < D; ++c) {
            float m = 1.f;
            for (int bb = J + 1; bb < I; ++bb) m *= s_bp[bb * D + c];
            const float ko = s_koT[c * PADC + j] * m;
            pa = fmaf(s_k[r * D + c], ko, pa);
            pp = fmaf(s_q[r * D + c], ko, pp);
        }
        s_A[r * PADC + j] = s_beta[r] * pa;
        s_P[r * PADC + j] = pp;
    }
    __syncthreads();

    float* rec = a.ws + ((size_t)ch * H + h) * a.ws_stride;
    if constexpr (!TCREC) {
        float* wW = rec;
        float* wQ = rec + (size_t)C * D;
        float* wK = rec + (size_t)2 * C * D;
        float* wU = rec + (size_t)3 * C * D;
        float* wP = rec + (size_t)4 * C * D;
        float* wG = wP + (size_t)C * C;

        // 6. forward substitution, one column of [U | W] per thread: x_r = rhs_r - sum_{j<r} A[r][j] x_j
        if (tid < 2 * D) {
            const bool isU = tid < D;
            const int c = isU ? tid : tid - D;
            float x[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float rhs;
                if (isU) {
                    rhs = r < L ? s_beta[r] * to_f32(vp[((size_t)(t0 + r) * H + h) * D + c]) : 0.f;
                } else {
                    float eb = 1.f;  // e^{G} up to the start of r's sub-block
                    for (int bb = 0; bb < r / kSub; ++bb) eb *= s_bp[bb * D + c];
                    rhs = s_beta[r] * s_k[r * D + c] * eb;
                }
#pragma unroll
                for (int jj = 0; jj < r; ++jj) rhs = fmaf(-s_A[r * PADC + jj], x[jj], rhs);
                x[r] = rhs;
                (isU ? wU : wW)[(size_t)r * D + c] = rhs;
            }
        }
        // 7. Qbar = q o e^{G}, Ktil = k o e^{G_L - G}, P, e^{G_L}
        for (int e = tid; e < C * D; e += THREADS) {
            const int r = e / D, c = e % D;
            const int blk = r / kSub;
            float eb = 1.f, ea = 1.f;
            for (int bb = 0; bb < blk; ++bb) eb *= s_bp[bb * D + c];
            for (int bb = blk + 1; bb < NB; ++bb) ea *= s_bp[bb * D + c];
            wQ[e] = s_q[e] * eb;
            wK[e] = s_koT[c * PADC + r] * ea;
        }
        for (int e = tid; e < C * C; e += THREADS) wP[e] = s_P[(e / C) * PADC + (e % C)];
        for (int c = tid; c < D; c += THREADS) {
            float g = 1.f;
            for (int bb = 0; bb < NB; ++bb) g *= s_bp[bb * D + c];
            wG[c] = g;
        }
    } else {
        static_assert(C == TcRec::C && D == TcRec::D, "tensor-core record shape");
        float* wW = rec + TcRec::W / 4;
        float* wK = rec + TcRec::KT / 4;
        float* wU = rec + TcRec::U / 4;
        float* wG = rec + TcRec::GL / 4;
        float* wQ = rec + TcRec::QB / 4;
        float* wP = rec + TcRec::P / 4;
        // 6. forward substitution as above; U plain [r][v], W as a tf32 image (rows r, K = c)
        if (tid < 2 * D) {
            const bool isU = tid < D;
            const int c = isU ? tid : tid - D;
            float x[C];
#pragma unroll
            for (int r = 0; r < C; ++r) {
                float rhs;
                if (isU) {
                    rhs = r < L ? s_beta[r] * to_f32(vp[((size_t)(t0 + r) * H + h) * D + c]) : 0.f;
                } else {
                    float eb = 1.f;
                    for (int bb = 0; bb < r / kSub; ++bb) eb *= s_bp[bb * D + c];
                    rhs = s_beta[r] * s_k[r * D + c] * eb;
                }
#pragma unroll
                for (int jj = 0; jj < r; ++jj) rhs = fmaf(-s_A[r * PADC + jj], x[jj], rhs);
                x[r] = rhs;
                if (isU)
                    wU[(size_t)r * D + c] = rhs;
                else
                    wW[tc::img_index(r, c, D)] = tc::round_tf32(rhs);
            }
        }
        // 7. Qbar image (rows r, K = c), Ktil^T image (rows c, K = r), P image (rows r, K = j), e^{G_L}
        for (int e = tid; e < C * D; e += THREADS) {
            const int r = e / D, c = e % D;
            const int blk = r / kSub;
            float eb = 1.f, ea = 1.f;
            for (int bb = 0; bb < blk; ++bb) eb *= s_bp[bb * D + c];
            for (int bb = blk + 1; bb < NB; ++bb) ea *= s_bp[bb * D + c];
            wQ[tc::img_index(r, c, D)] = tc::round_tf32(s_q[e] * eb);
            wK[tc::img_index(c, r, C)] = tc::round_tf32(s_koT[c * PADC + r] * ea);
        }
        for (int e = tid; e < C * C; e += THREADS) {
            const int r = e / C, j = e % C;
            wP[tc::img_index(r, j, C)] = tc::round_tf32(s_P[r * PADC + j]);
        }
        for (int c = tid; c < D; c += THREADS) {
            float g = 1.f;
            for (int bb = 0; bb < NB; ++bb) g *= s_bp[bb * D + c];
            wG[c] = g;
        }
    }
}

// ---- inter-chunk state pass ----------------------------------------------------------------------
struct StateArgs {
    const int32_t* seq_order;   // sequences by decreasing chunk count (tensor-core pass)
    const int32_t* chunk_start;
    const int32_t* chunk_len;
    const int32_t* seq_off;
    const int32_t* cu;
    const int32_t* state_idx;
    float* pool;
    int64_t num_slots;
    int64_t max_chunks;
    int64_t T;
    int32_t N;
    int H;
    const float* ws;
    size_t ws_stride;
    void* out;
    float* snap;           // optional chunk-boundary states [chunks][H][D][D]
    int64_t snap_cap;      // entries in snap
};

template <int C, int D, int NV>
struct StateShape {
    static constexpr int THREADS = 256;
    static constexpr int TR = THREADS / NV;    // threads along r (or c)
    static constexpr int RPT = C / TR;         // rows per thread (Delta, O)
    static constexpr int CPT = D / TR;         // key channels per thread (S update)
    static_assert(THREADS % NV == 0 && C % TR == 0 && D % TR == 0, "tiling");
    static constexpr size_t OFF_S = 0;                          // S [D][NV]
    static constexpr size_t OFF_W = OFF_S + (size_t)D * NV;     // W [C][D]
    static constexpr size_t OFF_Q = OFF_W + (size_t)C * D;      // Qbar [C][D]
    static constexpr size_t OFF_K = OFF_Q + (size_t)C * D;      // Ktil [C][D]
    static constexpr size_t OFF_P = OFF_K + (size_t)C * D;      // P [C][C]
    static constexpr size_t OFF_U = OFF_P + (size_t)C * C;      // U -> Delta [C][NV]
    static constexpr size_t OFF_G = OFF_U + (size_t)C * NV;     // e^{G_L} [D]
    static constexpr size_t FLOATS = OFF_G + D;
    static constexpr size_t BYTES = FLOATS * sizeof(float);
};

template <int C, int D, int NV, typename TOut>
__global__ void __launch_bounds__(256, 1) chunk_state_kernel(const StateArgs a)
{
    using Sh = StateShape<C, D, NV>;
    constexpr int THREADS = Sh::THREADS, TR = Sh::TR, RPT = Sh::RPT, CPT = Sh::CPT;
    extern __shared__ float4 smem4[];
    float* sm = reinterpret_cast<float*>(smem4);
    float* s_S = sm + Sh::OFF_S;
    float* s_W = sm + Sh::OFF_W;
    float* s_Q = sm + Sh::OFF_Q;
    float* s_K = sm + Sh::OFF_K;
    float* s_P = sm + Sh::OFF_P;
    float* s_U = sm + Sh::OFF_U;
    float* s_G = sm + Sh::OFF_G;

    const int seq = blockIdx.x;
    const int h = blockIdx.y;
    const int v0 = blockIdx.z * NV;
    const int tid = threadIdx.x;
    const int tv = tid % NV, tr = tid / NV;
    const int H = a.H;
    TOut* out = reinterpret_cast<TOut*>(a.out);

    int64_t slot = a.state_idx[seq];
    if (slot >= a.num_slots) {
        if (tid == 0 && blockIdx.y == 0 && blockIdx.z == 0) record_error(kDevErrStateIndex);
        slot = -1;
    }
    int64_t c_begin = a.seq_off[seq], c_end = a.seq_off[seq + 1];
    if (c_end > a.max_chunks) c_end = a.max_chunks;
    if (slot < 0) {  // padding row: zero outputs over the sequence's tokens
        int64_t s0 = a.cu[seq], s1 = a.cu[seq + 1];
        s0 = s0 < 0 ? 0 : (s0 > a.T ? a.T : s0);
        s1 = s1 < s0 ? s0 : (s1 > a.T ? a.T : s1);
        for (int64_t e = tid; e < (s1 - s0) * NV; e += THREADS) {
            const int64_t t = s0 + e / NV;
            out[((size_t)t * H + h) * D + v0 + e % NV] = from_f32<TOut>(0.f);
        }
        return;
    }
    float* Sg = a.pool + ((size_t)slot * H + h) * (size_t)D * D;
    for (int e = tid; e < D * NV; e += THREADS) {   // S[c][v] = pool[v0 + v][c]
        const int v = e / D, c = e % D;
        s_S[c * NV + v] = Sg[(size_t)(v0 + v) * D + c];
    }

    for (int64_t ch = c_begin; ch < c_end; ++ch) {
        const float* rec = a.ws + ((size_t)ch * H + h) * a.ws_stride;
        const int64_t t0 = a.chunk_start[ch];
        const int L = a.chunk_len[ch];
        __syncthreads();  // previous chunk done with the staging buffers
        {
            const float4* src = reinterpret_cast<const float4*>(rec);
            float4* dW = reinterpret_cast<float4*>(s_W);
            for (int e = tid; e < 3 * C * D / 4; e += THREADS) dW[e] = src[e];  // W, Qbar, Ktil contiguous
            const float4* srcP = reinterpret_cast<const float4*>(rec + (size_t)4 * C * D);
            float4* dP = reinterpret_cast<float4*>(s_P);
            for (int e = tid; e < C * C / 4; e += THREADS) dP[e] = srcP[e];
            for (int e = tid; e < C * NV; e += THREADS) {
                const int r = e / NV, v = e % NV;
                s_U[e] = rec[(size_t)3 * C * D + (size_t)r * D + v0 + v];
            }
            for (int e = tid; e < D; e += THREADS) s_G[e] = rec[(size_t)4 * C * D + (size_t)C * C + e];
        }
        __syncthreads();
        // Delta = U - W S
        {
            float acc[RPT];
#pragma unroll
            for (int i = 0; i < RPT; ++i) acc[i] = s_U[(tr + TR * i) * NV + tv];
            for (int c = 0; c < D; c += 4) {
                const float s0 = s_S[(c + 0) * NV + tv], s1 = s_S[(c + 1) * NV + tv];
                const float s2 = s_S[(c + 2) * NV + tv], s3 = s_S[(c + 3) * NV + tv];
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const float4 w = *reinterpret_cast<const float4*>(&s_W[(tr + TR * i) * D + c]);
                    acc[i] = fmaf(-w.x, s0, acc[i]); acc[i] = fmaf(-w.y, s1, acc[i]);
                    acc[i] = fmaf(-w.z, s2, acc[i]); acc[i] = fmaf(-w.w, s3, acc[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < RPT; ++i) s_U[(tr + TR * i) * NV + tv] = acc[i];
        }
        __syncthreads();
        // O = Qbar S + P Delta (rows past the chunk end are not stored)
        {
            float acc[RPT];
#pragma unroll
            for (int i = 0; i < RPT; ++i) acc[i] = 0.f;
            for (int c = 0; c < D; c += 4) {
                const float s0 = s_S[(c + 0) * NV + tv], s1 = s_S[(c + 1) * NV + tv];
                const float s2 = s_S[(c + 2) * NV + tv], s3 = s_S[(c + 3) * NV + tv];
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const float4 qv = *reinterpret_cast<const float4*>(&s_Q[(tr + TR * i) * D + c]);
                    acc[i] = fmaf(qv.x, s0, acc[i]); acc[i] = fmaf(qv.y, s1, acc[i]);
                    acc[i] = fmaf(qv.z, s2, acc[i]); acc[i] = fmaf(qv.w, s3, acc[i]);
                }
            }
            for (int j = 0; j < C; ++j) {
                const float dj = s_U[j * NV + tv];
#pragma unroll
                for (int i = 0; i < RPT; ++i) {
                    const int r = tr + TR * i;
                    if (j <= r) acc[i] = fmaf(s_P[r * C + j], dj, acc[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < RPT; ++i) {
                const int r = tr + TR * i;
                if (r < L) out[((size_t)(t0 + r) * H + h) * D + v0 + tv] = from_f32<TOut>(acc[i]);
            }
        }
        // S <- Diag(e^{G_L}) S + Ktil^T Delta
        {
            float acc[CPT];
#pragma unroll
            for (int i = 0; i < CPT; ++i) {
                const int c = tr + TR * i;
                acc[i] = s_G[c] * s_S[c * NV + tv];
            }
            for (int r = 0; r < C; ++r) {
                const float dr = s_U[r * NV + tv];
#pragma unroll
                for (int i = 0; i < CPT; ++i) acc[i] = fmaf(s_K[r * D + tr + TR * i], dr, acc[i]);
            }
            __syncthreads();  // every thread has finished reading the old S
#pragma unroll
            for (int i = 0; i < CPT; ++i) s_S[(tr + TR * i) * NV + tv] = acc[i];
        }
        if (a.snap) {                                // state after this chunk
            __syncthreads();
            if (ch < a.snap_cap) {
                for (int e = tid; e < D * NV; e += THREADS) {
                    const int v = e / D, c = e % D;
                    a.snap[(((size_t)ch * H + h) * D + v0 + v) * D + c] = s_S[c * NV + v];
                }
            } else if (tid == 0) {
                record_error(kDevErrSeqlens);
            }
        }
    }
    __syncthreads();
    for (int e = tid; e < D * NV; e += THREADS) {
        const int v = e / D, c = e % D;
        Sg[(size_t)(v0 + v) * D + c] = s_S[c * NV + v];
    }
}

// ---- inter-chunk state pass on the tensor cores (C = 64, D = 128) --------------------------------
// One CTA of 384 threads per (sequence, head), in the transposed ("value-major") form so that every
// MMA has M = 128 rows = the 128 value rows (TMEM lane v).  Per chunk:
//   (a)  Dd   = S^T W^T                  A = tf32 copy of S^T in TMEM, B = W image       (N = 64)
//   Delta^T = U^T - Dd, rounded to tf32, written over Dd
//   (c)  Dc   = Delta^T Ktil             A = Delta^T in TMEM,          B = Ktil^T image  (N = 128)
//   S^T <- S^T Diag(e^{G_L}) + Dc (fp32 in registers), its tf32 copy into the other TMEM buffer
//   (b2) Do   = Delta^T P^T              A = Delta^T,                  B = P image       (N = 64)
//   (b)  Do  += S^T Qbar^T               A = S^T (this chunk's copy),  B = Qbar image    (N = 64)
//   O^T = Do -> out
// Warps 0..7 share the chain: thread v of warp group g (0: warps 0..3, 1: warps 4..7) is TMEM
// lane v and owns columns 64 g .. 64 g + 63 of row v of S^T in registers; each group computes half
// of Delta (rows r = 32 g ..) and half of the S update.  Thread 0 issues (a) and (c) and loads W,
// U/gL and Ktil^T.  Warps 8..11 produce the output: thread 256 issues (b2) and (b) once Delta is
// ready and P / Qbar have landed, and loads P and Qbar; the four warps copy Do to the output.
// Neither the output MMAs, their operands nor the output stores sit on the chain.  The S^T copy is
// double-buffered (chunk i reads buffer i & 1), so the S update of chunk i only waits for (b) of
// chunk i - 1.  Hand-offs are mbarriers (delta_ready: an arrival of thread 0; b2_done,
// out_ready[2]: tensor-core commits of thread 256).  Operand images arrive by bulk async copy from
// the record: W and U/gL double-buffered (two chunks ahead), Ktil^T, P and Qbar one chunk ahead.
// All waits are bounded and give up early once any thread has recorded a failure; loop exits are
// made uniform with barrier reductions.
constexpr uint32_t kWaitPolls = 1u << 24;

// shared memory: the record image (one buffer set) followed by the second W and U/gL buffers
constexpr uint32_t kSmW1 = TcRec::BYTES;
constexpr uint32_t kSmUG1 = kSmW1 + 32768;
constexpr uint32_t kUGBytes = 32768 + 512;
constexpr uint32_t kSmBars = kSmUG1 + kUGBytes;
struct TcBars {
    uint64_t w[2], ug[2], kt, qb, p;  // operand buffers filled (tx bytes); these seven come first
    uint64_t mma_a;                   // (a) complete                    (thread 0 commit)
    uint64_t mma_c;                   // (c) complete                    (thread 0 commit)
    uint64_t delta_ready;             // Delta^T of the chunk is in TMEM (thread 0 arrives)
    uint64_t b2_done;                 // (b2) complete: Delta^T may be overwritten (issuer commit)
    uint64_t out_ready[2];            // (b) of chunk i complete, Do ready; index i & 1 (issuer commit)
    uint64_t drain[2];                // used once each, to drain the tensor core after a failed wait
};
constexpr size_t kTcSmemBytes = kSmBars + 1024;
static_assert(sizeof(TcBars) + 32 + 512 <= 1024, "barriers, TMEM base, abort flag and e^{G_L}");
static_assert(kTcSmemBytes <= 232448, "state-pass shared memory");
constexpr int kStateThreads = 384;

// TMEM column map (512 columns allocated; each accumulator starts at a multiple of its width)
constexpr uint32_t kT_SOP = 0;     // tf32 S^T, two buffers   (2 x 128 cols, A operand)
constexpr uint32_t kT_SC = 256;    // Delta^T Ktil            (128, accumulator)
constexpr uint32_t kT_DD = 384;    // S^T W^T, then Delta^T   (64, accumulator, then A operand)
constexpr uint32_t kT_OUT = 448;   // O^T                     (64, accumulator)

__device__ __forceinline__ void chain_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// Named barrier that also returns, to every participating thread, whether any of them passed a
// true flag: a loop exit after a failure is uniform even though the failure flag is written
// asynchronously by other warps.  Barrier 1: the 256 chain threads; barrier 2: the 128 output threads.
template <int ID, int COUNT>
__device__ __forceinline__ bool sync_any(bool flag)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\t"
        "setp.ne.u32 pi, %1, 0;\n\t"
        "bar.red.or.pred po, %2, %3, pi;\n\t"
        "selp.u32 %0, 1, 0, po;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)flag), "n"(ID), "n"(COUNT)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ bool chain_sync_any(bool flag) { return sync_any<1, 256>(flag); }
__device__ __forceinline__ bool output_sync_any(bool flag) { return sync_any<2, 128>(flag); }

template <typename TOut>
__global__ void __launch_bounds__(kStateThreads, 1) chunk_state_tc_kernel(const StateArgs a)
{
    constexpr int C = TcRec::C, D = TcRec::D, DH = D / 2;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw;
    TcBars* bars = reinterpret_cast<TcBars*>(sm + kSmBars);
    uint32_t* s_taddr = reinterpret_cast<uint32_t*>(sm + kSmBars + sizeof(TcBars));
    volatile int* s_abort = reinterpret_cast<volatile int*>(sm + kSmBars + sizeof(TcBars) + 16);
    float* s_gl = reinterpret_cast<float*>(sm + kSmBars + sizeof(TcBars) + 32);  // e^{G_L} of the chunk

    // longest sequences first: CTA x -> (rank, head), rank -> sequence through seq_order
    const int H = a.H;
    const int rank = blockIdx.x / H;
    const int h = blockIdx.x - rank * H;
    const int seq = a.seq_order[rank];
    const int tid = threadIdx.x, warp = tid >> 5;
    TOut* out = reinterpret_cast<TOut*>(a.out);

    int64_t slot = a.state_idx[seq];
    if (slot >= a.num_slots) {
        if (tid == 0 && h == 0) record_error(kDevErrStateIndex);
        slot = -1;
    }
    int64_t c_begin = a.seq_off[seq], c_end = a.seq_off[seq + 1];
    if (c_end > a.max_chunks) c_end = a.max_chunks;
    if (slot < 0) {
        int64_t s0 = a.cu[seq], s1 = a.cu[seq + 1];
        s0 = s0 < 0 ? 0 : (s0 > a.T ? a.T : s0);
        s1 = s1 < s0 ? s0 : (s1 > a.T ? a.T : s1);
        if (tid < D)
            for (int64_t t = s0; t < s1; ++t) out[((size_t)t * H + h) * D + tid] = from_f32<TOut>(0.f);
        return;
    }
    if (c_begin >= c_end) return;  // empty sequence: the slot keeps its state

    if (warp == 0) {
        tc::tmem_alloc(s_taddr, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        uint64_t* b = reinterpret_cast<uint64_t*>(bars);
        for (int i = 0; i < (int)(sizeof(TcBars) / 8); ++i) tc::mbar_init(b + i, 1);
        *s_abort = 0;
        tc::fence_mbar_init();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *s_taddr;
    const uint32_t lane = (uint32_t)((warp & 3) * 32) << 16;

    // bounded wait that also gives up once any thread has recorded a failure
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        for (uint32_t it = 0; it < kWaitPolls; ++it) {
            if (tc::mbar_try_wait(bar, parity)) return true;
            if ((it & 63u) == 63u && *s_abort) return false;
        }
        *s_abort = 1;
        return false;
    };
    auto rec_of = [&](int64_t ch) -> const unsigned char* {
        return reinterpret_cast<const unsigned char*>(a.ws + ((size_t)ch * H + h) * a.ws_stride);
    };
    // copies in flight per load barrier (bookkeeping of the issuing thread, for the drain)
    uint64_t* const bar0 = &bars->w[0];
    uint32_t pend_mask = 0, pend_par = 0, uses[7] = {0, 0, 0, 0, 0, 0, 0};
    auto load = [&](uint64_t* bar, uint32_t dst_off, uint32_t src_off, uint32_t bytes, int64_t ch) {
        const uint32_t bi = (uint32_t)(bar - bar0), bit = 1u << bi;
        pend_mask |= bit;
        pend_par = (pend_par & ~bit) | ((uses[bi] & 1u) ? bit : 0u);
        ++uses[bi];
        tc::mbar_arrive_expect_tx(bar, bytes);
        tc::bulk_g2s(sm + dst_off, rec_of(ch) + src_off, bytes, bar);
    };
    auto landed = [&](uint64_t* bar) { pend_mask &= ~(1u << (uint32_t)(bar - bar0)); };
    auto drain = [&](uint64_t* dbar) {          // after a failure: own MMAs and copies land, bounded
        tc::mma_commit(dbar);
        tc::mbar_wait(dbar, 0, kWaitPolls);
        for (uint32_t bi = 0; bi < 7; ++bi)
            if (pend_mask & (1u << bi)) tc::mbar_wait(bar0 + bi, (pend_par >> bi) & 1u, kWaitPolls);
    };
    constexpr uint32_t kId64 = tc::idesc_tf32(128, 64), kId128 = tc::idesc_tf32(128, 128);

    if (warp >= 8) {
        // ---- output side: thread 256 issues (b2) and (b); warps 8..11 copy Do to the output
        const int v = tid - 256;
        const bool issuer = (v == 0);
        const uint32_t sQB = tc::smem_u32(sm + TcRec::QB), sP = tc::smem_u32(sm + TcRec::P);
        if (issuer) {
            load(&bars->p, TcRec::P, TcRec::P, 16384, c_begin);
            load(&bars->qb, TcRec::QB, TcRec::QB, 32768, c_begin);
        }
        bool ok = true;
        for (int64_t ch = c_begin; ch < c_end; ++ch) {
            const uint32_t i = (uint32_t)(ch - c_begin), ph = i & 1u;
            if (issuer) {
                ok = wait(&bars->delta_ready, ph) && wait(&bars->p, ph);
                if (ok) {
                    landed(&bars->p);
                    tc::tc_fence_after();
#pragma unroll
                    for (int s = 0; s < C / 8; ++s)
                        tc::mma_tf32_ts(tmem + kT_OUT, tmem + kT_DD + 8 * s, tc::smem_desc(sP + 256 * s, 128, 2048), kId64, s > 0);
                    tc::mma_commit(&bars->b2_done);
                    ok = wait(&bars->qb, ph);
                }
                if (ok) {
                    landed(&bars->qb);
#pragma unroll
                    for (int s = 0; s < D / 8; ++s)
                        tc::mma_tf32_ts(tmem + kT_OUT, tmem + kT_SOP + 128 * (i & 1u) + 8 * s,
                                        tc::smem_desc(sQB + 256 * s, 128, 4096), kId64, 1);
                    tc::mma_commit(&bars->out_ready[i & 1u]);
                }
            }
            const bool okr = ok && wait(&bars->out_ready[i & 1u], (i >> 1) & 1u);   // every output thread
            if (okr) {
                tc::tc_fence_after();
                if (issuer && ch + 1 < c_end) {          // (b2) and (b) are done with P and Qbar
                    load(&bars->p, TcRec::P, TcRec::P, 16384, ch + 1);
                    load(&bars->qb, TcRec::QB, TcRec::QB, 32768, ch + 1);
                }
                const int64_t t0 = a.chunk_start[ch];
                const int L = a.chunk_len[ch];
#pragma unroll
                for (int r0 = 0; r0 < C; r0 += 16) {
                    float o[16];
                    tc::tmem_ld16(tmem + lane + kT_OUT + r0, o);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (r0 + j < L) out[((size_t)(t0 + r0 + j) * H + h) * D + v] = from_f32<TOut>(o[j]);
                }
            }
            tc::tc_fence_before();
            if (output_sync_any(!okr || *s_abort != 0)) break;   // Do is free for the next (b2)
        }
        if (issuer && *s_abort) drain(&bars->drain[1]);
        __syncwarp();
    } else {
        // ---- the chain: warp group g = warp >> 2 owns S^T columns 64 g .. 64 g + 63 of row v
        const int g = warp >> 2, v = tid & (D - 1);
        auto w_off = [](uint32_t b) { return b ? kSmW1 : TcRec::W; };
        auto ug_off = [](uint32_t b) { return b ? kSmUG1 : TcRec::U; };
        if (tid == 0) {
            load(&bars->w[0], TcRec::W, TcRec::W, 32768, c_begin);
            load(&bars->ug[0], TcRec::U, TcRec::U, kUGBytes, c_begin);
            load(&bars->kt, TcRec::KT, TcRec::KT, 32768, c_begin);
            if (c_begin + 1 < c_end) {
                load(&bars->w[1], kSmW1, TcRec::W, 32768, c_begin + 1);
                load(&bars->ug[1], kSmUG1, TcRec::U, kUGBytes, c_begin + 1);
            }
        }

        // entry state: columns 64 g .. of row v of S^T = pool[slot][h][v][:]; tf32 copy -> buffer 0
        float S[DH];
        const float* Sg = a.pool + ((size_t)slot * H + h) * (size_t)D * D + (size_t)v * D + DH * g;
#pragma unroll
        for (int c = 0; c < DH; c += 4) {
            const float4 x = *reinterpret_cast<const float4*>(Sg + c);
            S[c] = x.x; S[c + 1] = x.y; S[c + 2] = x.z; S[c + 3] = x.w;
        }
#pragma unroll
        for (int c = 0; c < DH; c += 16) {
            float t[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) t[j] = tc::round_tf32(S[c + j]);
            tc::tmem_st16_nowait(tmem + lane + kT_SOP + DH * g + c, t);
        }
        tc::tmem_wait_st();
        tc::tc_fence_before();
        chain_sync();

        const uint32_t sKT = tc::smem_u32(sm + TcRec::KT);
        bool ok = true;
        for (int64_t ch = c_begin; ch < c_end; ++ch) {
            const uint32_t i = (uint32_t)(ch - c_begin);
            const uint32_t ph = i & 1u, b = i & 1u, phb = (i >> 1) & 1u;
            const float* sU = reinterpret_cast<const float*>(sm + ug_off(b));
            const float* sG = sU + 32768 / 4;

            // (a): Dd is the previous chunk's Delta^T, free once its (b2) is done
            if (tid == 0) {
                tc::tc_fence_after();
                ok = wait(&bars->w[b], phb) && (i == 0 || wait(&bars->b2_done, (i - 1) & 1u)) && ok;
                if (ok) {
                    landed(&bars->w[b]);
                    tc::tc_fence_after();
                    const uint32_t sW = tc::smem_u32(sm + w_off(b));
#pragma unroll
                    for (int s = 0; s < D / 8; ++s)
                        tc::mma_tf32_ts(tmem + kT_DD, tmem + kT_SOP + 128 * b + 8 * s, tc::smem_desc(sW + 256 * s, 128, 4096),
                                        kId64, s > 0);
                    tc::mma_commit(&bars->mma_a);
                }
            }
            // Delta^T = U^T - S^T W^T (rows r = 32 g .. 32 g + 31), rounded, over Dd
            {
                const bool okw = wait(&bars->ug[b], phb) && wait(&bars->mma_a, ph);
                if (okw && tid == 0) landed(&bars->ug[b]);
                tc::tc_fence_after();
                if (okw) {
#pragma unroll
                    for (int r0 = 32 * g; r0 < 32 * g + 32; r0 += 16) {
                        float d[16];
                        tc::tmem_ld16(tmem + lane + kT_DD + r0, d);
#pragma unroll
                        for (int j = 0; j < 16; ++j) d[j] = tc::round_tf32(sU[(r0 + j) * D + v] - d[j]);
                        tc::tmem_st16_nowait(tmem + lane + kT_DD + r0, d);
                    }
                    if (g == 0) s_gl[v] = sG[v];         // the buffer is refilled before (c) retires
                    tc::tmem_wait_st();
                }
            }
            tc::tc_fence_before();
            if (chain_sync_any(*s_abort != 0)) break;
            if (tid == 0) {                              // Delta ready; refill W, U/gL(b); (c)
                tc::tc_fence_after();
                tc::mbar_arrive(&bars->delta_ready);
                if (ch + 2 < c_end) {
                    load(&bars->w[b], w_off(b), TcRec::W, 32768, ch + 2);
                    load(&bars->ug[b], ug_off(b), TcRec::U, kUGBytes, ch + 2);
                }
                ok = wait(&bars->kt, ph) && ok;
                if (ok) {
                    landed(&bars->kt);
                    tc::tc_fence_after();
#pragma unroll
                    for (int s = 0; s < C / 8; ++s)
                        tc::mma_tf32_ts(tmem + kT_SC, tmem + kT_DD + 8 * s, tc::smem_desc(sKT + 256 * s, 128, 2048), kId128, s > 0);
                    tc::mma_commit(&bars->mma_c);
                }
            }
            // S^T <- S^T Diag(e^{G_L}) + Delta^T Ktil on this group's columns; tf32 copy -> buffer
            // (i + 1) & 1, which (b) of chunk i - 1 reads
            {
                bool okc = wait(&bars->mma_c, ph);
                if (okc && i >= 1) okc = wait(&bars->out_ready[(i - 1) & 1u], ((i - 1) >> 1) & 1u);
                tc::tc_fence_after();
                if (okc && tid == 0 && ch + 1 < c_end) load(&bars->kt, TcRec::KT, TcRec::KT, 32768, ch + 1);
                if (okc) {
                    const uint32_t sop = kT_SOP + 128 * (b ^ 1u) + DH * g;
#pragma unroll
                    for (int c = 0; c < DH; c += 16) {
                        float d[16];
                        tc::tmem_ld16(tmem + lane + kT_SC + DH * g + c, d);
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            S[c + j] = fmaf(S[c + j], s_gl[DH * g + c + j], d[j]);
                            d[j] = tc::round_tf32(S[c + j]);
                        }
                        tc::tmem_st16_nowait(tmem + lane + sop + c, d);
                    }
                    tc::tmem_wait_st();
                    if (a.snap) {                        // state after this chunk
                        if (ch < a.snap_cap) {
                            float* Sd = a.snap + (((size_t)ch * H + h) * D + v) * (size_t)D + DH * g;
#pragma unroll
                            for (int c = 0; c < DH; c += 4)
                                *reinterpret_cast<float4*>(Sd + c) = make_float4(S[c], S[c + 1], S[c + 2], S[c + 3]);
                        } else if (tid == 0) {
                            record_error(kDevErrSeqlens);
                        }
                    }
                }
            }
            tc::tc_fence_before();
            if (chain_sync_any(*s_abort != 0)) break;
        }
        const bool aborted = chain_sync_any(*s_abort != 0);
        if (aborted) {
            // A wait gave up: record it, let this side's MMAs and copies land.  The slot is left as it was.
            if (tid == 0) {
                record_error(kDevErrTimeout);
                drain(&bars->drain[0]);
            }
        } else {
            float* Sd = a.pool + ((size_t)slot * H + h) * (size_t)D * D + (size_t)v * D + DH * g;
#pragma unroll
            for (int c = 0; c < DH; c += 4) *reinterpret_cast<float4*>(Sd + c) = make_float4(S[c], S[c + 1], S[c + 2], S[c + 3]);
        }
        __syncwarp();
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ---- helpers of the bf16 intra-chunk kernel (C = 64, D = 128) -----------------------------------
namespace itc {
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 mul4(float4 a, float4 b) { return make_float4(a.x * b.x, a.y * b.y, a.z * b.z, a.w * b.w); }
__device__ __forceinline__ float4 rnd4(float4 a)
{
    return make_float4(tc::round_tf32(a.x), tc::round_tf32(a.y), tc::round_tf32(a.z), tc::round_tf32(a.w));
}
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// alpha = e^{g} from the identities e^{-r softplus(x)} = 2^{-r log2(1 + 2^{x log2 e})} and
// e^{lb sigmoid(r x)} = 2^{lb log2 e / (1 + 2^{-r x log2 e})}, on the special-function unit.
__device__ __forceinline__ float alpha_mufu(float x, float rate, const GateParams& gp)
{
    constexpr float kLog2e = 1.4426950408889634f;
    if (gp.use_lower_bound) {
        const float sig = __fdividef(1.0f, 1.0f + ex2_approx(-rate * x * kLog2e));
        return ex2_approx(gp.lower_bound * kLog2e * sig);
    }
    const float sp2 = x > gp.softplus_threshold ? x * kLog2e : lg2_approx(1.0f + ex2_approx(x * kLog2e));
    return ex2_approx(-rate * sp2);
}
// Packed fp32 pairs (one 64-bit register pair) and the sm_100+ paired FP32 instructions; each lane
// of a pair is an ordinary IEEE fp32 multiply / fused multiply-add.
__device__ __forceinline__ float f2sum(uint64_t r)
{
    float x, y;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
    return x + y;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
// 16 bytes of shared memory as two packed pairs
__device__ __forceinline__ void ld2x2(const float* p, uint64_t& lo, uint64_t& hi)
{
    const ulonglong2 v = *reinterpret_cast<const ulonglong2*>(p);
    lo = v.x;
    hi = v.y;
}
// Gram row m (0..95) -> row block I and key row j
__device__ __forceinline__ void gram_row(int m, int& I, int& j)
{
    I = m < 16 ? 1 : (m < 48 ? 2 : 3);
    j = m - (I == 1 ? 0 : (I == 2 ? 16 : 48));
}
}  // namespace itc

// ---- intra-chunk kernel for bf16 inputs at C = 64, D = 128: two CTAs per SM -----------------------
// One CTA of 256 threads per (chunk, head) with 105 KB of shared memory and 256 TMEM columns, so
// that two CTAs share an SM and each one's loads, barriers and single-thread MMA issue overlap the
// other's arithmetic.  Three [C][LD] fp32 tiles hold k_hat, q_hat and alpha; each is reused in
// place as the pass over it ends.  It writes the tensor-core record (TcRec) that the state pass reads:
//   1. loads; alpha = e^{g} (MUFU form of the gate); L2 norms fused into the loads
//   2. diagonal 16 x 16 sub-blocks of A and P by running products of alphas (CUDA cores); each
//      thread takes key rows j and 15 - j so that all warps do the same number of rows; P goes
//      straight to the record image, A to a small buffer
//   3. per (column, sub-block): k o Rout -> Ktil^T record, k o Rin, q o Rin (in place),
//      (beta Kbar)^T -> TMEM (the thread's TMEM lane is its column)
//   4. Gram operands in fp16 (kind::f16; same 11-bit significand as tf32, every operand <= 1 in
//      magnitude): B image = rows of k o Rin and q o Rin of blocks 1..3 (over the q tile), A = key
//      j decayed to the start of row block I in TMEM (lane m <-> (I, j)); Qbar record
//   5. while the MMA runs: value loads for (beta V)^T; Gram result -> off-diagonal A and P
//   6. T = (I + A)^{-1} by blocks (over the alpha tile), then U^T = (beta V)^T T^T and
//      W^T = (beta Kbar)^T T^T with both A operands in TMEM (kind::tf32)
namespace itc {
constexpr int C = 64, D = 128, NB = 4, THREADS = 256;
constexpr int LD = 132;   // padded row stride (floats) of the [C][D] tiles
constexpr int LDA = 68;   // padded row stride of the [C][C] tiles
constexpr uint32_t TILE = C * LD * 4;
constexpr uint32_t OFF_K = 0;                        // k_hat -> k o Rin; then A and X
constexpr uint32_t OFF_Q = TILE;                     // q_hat -> q o Rin; then the Gram B image
constexpr uint32_t OFF_AL = 2 * TILE;                // alpha -> k o Rout; then T and its image
constexpr uint32_t OFF_AD = 3 * TILE;                // diagonal blocks of A   [NB][16][16]
constexpr uint32_t OFF_BP = OFF_AD + NB * 256 * 4;   // block products bp      [NB][D]
constexpr uint32_t OFF_EB = OFF_BP + NB * D * 4;     // e^{G} before block b: prod_{b' < b} bp  [NB][D]
constexpr uint32_t OFF_B12 = OFF_EB + NB * D * 4;    // bp[1] * bp[2]          [D]
constexpr uint32_t OFF_BETA = OFF_B12 + D * 4;       // beta                   [C]
constexpr uint32_t OFF_BAR = OFF_BETA + C * 4;       // 3 mbarriers: Gram done, U/W done, drain
constexpr uint32_t OFF_TM = OFF_BAR + 24;            // TMEM base
constexpr uint32_t BYTES = OFF_TM + 16;
constexpr uint32_t OFF_A = OFF_K;                    // A = sum of diagonal and Gram blocks [C][LDA]
constexpr uint32_t OFF_X = OFF_K + C * LDA * 4;      // 3 scratch 16 x 16 blocks
constexpr uint32_t OFF_IB = OFF_Q;                   // Gram B image: 96 rows x 128 fp16
constexpr uint32_t OFF_T = OFF_AL;                   // T [C][LDA]
constexpr uint32_t OFF_IT = OFF_AL + C * LDA * 4;    // T image (rows r, K = j), tf32
static_assert(OFF_X + 3 * 256 * 4 <= OFF_Q, "A and X fit in the k tile");
static_assert(96 * D * 2 <= TILE, "the fp16 B image fits in the q tile");
static_assert(OFF_IT + C * C * 4 <= OFF_AD, "T and its image fit in the alpha tile");
static_assert(2 * (BYTES + 1024) <= 233472, "two CTAs per SM");
// TMEM columns (256 allocated)
constexpr uint32_t T_KD = 0;      // decayed keys, fp16 pairs (64 cols); then (beta V)^T (64)
constexpr uint32_t T_KB = 64;     // (beta Kbar)^T (64)
constexpr uint32_t T_G = 128;     // Gram result (96); then U^T (64) and W^T (64)
}  // namespace itc

__global__ void __launch_bounds__(itc::THREADS, 2) chunk_intra_tc_kernel(const IntraArgs a)
{
    using namespace itc;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* sm = smem_raw;
    float* sK = reinterpret_cast<float*>(sm + OFF_K);
    float* sQ = reinterpret_cast<float*>(sm + OFF_Q);
    float* sAl = reinterpret_cast<float*>(sm + OFF_AL);
    float* sAD = reinterpret_cast<float*>(sm + OFF_AD);
    float* sBp = reinterpret_cast<float*>(sm + OFF_BP);
    float* sEb = reinterpret_cast<float*>(sm + OFF_EB);
    float* sB12 = reinterpret_cast<float*>(sm + OFF_B12);
    float* sBeta = reinterpret_cast<float*>(sm + OFF_BETA);
    float* sA = reinterpret_cast<float*>(sm + OFF_A);
    float* sX = reinterpret_cast<float*>(sm + OFF_X);
    float* sT = reinterpret_cast<float*>(sm + OFF_T);
    float* sIT = reinterpret_cast<float*>(sm + OFF_IT);
    unsigned char* sIB = sm + OFF_IB;
    uint64_t* bar_g = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
    uint64_t* bar_uw = bar_g + 1;
    uint64_t* bar_drain = bar_g + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + OFF_TM);

    const int64_t ch = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int64_t nch = a.seq_off[a.N];
    if (nch > a.max_chunks) nch = a.max_chunks;
    if (ch >= nch) return;
    const int32_t seq = a.chunk_seq[ch];
    const int64_t slot = a.state_idx[seq];
    if (slot < 0 || slot >= a.num_slots) return;
    const int64_t t0 = a.chunk_start[ch];
    const int L = a.chunk_len[ch];
    const int H = a.H;
    const float rate = expf(a.A_log[h]);
    bool tc_ok = true;                                       // thread 0: every tcgen05 wait completed
    const __nv_bfloat16* kp = reinterpret_cast<const __nv_bfloat16*>(a.k);
    const __nv_bfloat16* qp = reinterpret_cast<const __nv_bfloat16*>(a.q);
    const __nv_bfloat16* vp = reinterpret_cast<const __nv_bfloat16*>(a.v);

    // record fields, addressed from one base pointer where they are written
    unsigned char* const rec = reinterpret_cast<unsigned char*>(a.ws + ((size_t)ch * H + h) * a.ws_stride);
#define KDA_REC(field) reinterpret_cast<float*>(rec + TcRec::field)

    if (warp == 0) {
        tc::tmem_alloc(s_tmem, 256);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(bar_g, 1);
        tc::mbar_init(bar_uw, 1);
        tc::mbar_init(bar_drain, 1);
        tc::fence_mbar_init();
    }
    if (warp == 1) {               // the value rows are read after the Gram: start them towards L2 now
        for (int r = lane; r < L; r += 32)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], 256;" ::"l"(vp + ((size_t)(t0 + r) * H + h) * D)
                         : "memory");
    }
    // 1. loads, all issued before any is used (rows past the chunk end: k = q = 0, alpha = 1,
    //    beta = 0).  k, q: 8 elements in rows 2 warp + (lane bit 2) + 16 i, columns 32 (lane >> 3) +
    //    8 (lane & 3): the two 8-lane halves of a quarter-warp hold adjacent rows, so that with the
    //    132-float row stride each 16-byte shared store of a quarter-warp covers all 32 banks once.
    //    g: 4 elements in rows (tid >> 5) + 8 i
    {
        uint4 kv[4], qv[4];
        float4 gv[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 2 * warp + ((lane >> 2) & 1) + 16 * i, c8 = 32 * (lane >> 3) + 8 * (lane & 3);
            kv[i] = qv[i] = make_uint4(0, 0, 0, 0);
            if (r < L) {
                const size_t idx = ((size_t)(t0 + r) * H + h) * D + c8;
                kv[i] = *reinterpret_cast<const uint4*>(kp + idx);
                qv[i] = *reinterpret_cast<const uint4*>(qp + idx);
            }
        }
        const int c4 = (tid & 31) * 4;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = (tid >> 5) + 8 * i;
            gv[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < L) gv[i] = *reinterpret_cast<const float4*>(a.g_raw + ((size_t)(t0 + r) * H + h) * D + c4);
        }
        float bt = 0.f;
        if (tid < L) bt = a.b_raw[(size_t)(t0 + tid) * H + h];
        float4 db = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.dt_bias) db = *reinterpret_cast<const float4*>(a.dt_bias + (size_t)h * D + c4);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            // the 16 lanes that hold row r (lane bit 2 fixed) reduce its squared norms with shuffles
            const int r = 2 * warp + ((lane >> 2) & 1) + 16 * i, c8 = 32 * (lane >> 3) + 8 * (lane & 3);
            const __nv_bfloat16* kb = reinterpret_cast<const __nv_bfloat16*>(&kv[i]);
            const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(&qv[i]);
            float kf[8], qf[8], kk = 0.f, qq = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                kf[t] = __bfloat162float(kb[t]);
                qf[t] = __bfloat162float(qb[t]);
                kk = fmaf(kf[t], kf[t], kk);
                qq = fmaf(qf[t], qf[t], qq);
            }
#pragma unroll
            for (int off = 1; off <= 16; off <<= 1) {
                if (off == 4) continue;
                kk += __shfl_xor_sync(0xffffffffu, kk, off);
                qq += __shfl_xor_sync(0xffffffffu, qq, off);
            }
            const float rk = 1.0f / sqrtf(kk + a.gp.l2_eps), rq = a.gp.scale / sqrtf(qq + a.gp.l2_eps);
#pragma unroll
            for (int t = 0; t < 8; ++t) { kf[t] *= rk; qf[t] *= rq; }
            st4(sK + r * LD + c8, make_float4(kf[0], kf[1], kf[2], kf[3]));
            st4(sK + r * LD + c8 + 4, make_float4(kf[4], kf[5], kf[6], kf[7]));
            st4(sQ + r * LD + c8, make_float4(qf[0], qf[1], qf[2], qf[3]));
            st4(sQ + r * LD + c8 + 4, make_float4(qf[4], qf[5], qf[6], qf[7]));
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int r = (tid >> 5) + 8 * i;
            float4 al = make_float4(1.f, 1.f, 1.f, 1.f);
            if (r < L) {
                al.x = alpha_mufu(gv[i].x + db.x, rate, a.gp);
                al.y = alpha_mufu(gv[i].y + db.y, rate, a.gp);
                al.z = alpha_mufu(gv[i].z + db.z, rate, a.gp);
                al.w = alpha_mufu(gv[i].w + db.w, rate, a.gp);
            }
            st4(sAl + r * LD + c4, al);
        }
        if (tid < C) sBeta[tid] = tid < L ? sigmoid_f32(bt) : 0.f;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;

    // 2. diagonal sub-blocks.  Warp w: block w >> 1; lane = (jq, cg), 8 channel groups of 16
    //    columns (4 cg + 32 m); the thread runs key row j = 4 (w & 1) + jq, then 15 - that, from the
    //    first row its warp needs (rows below a thread's own j are computed and dropped).  The 32
    //    partial sums of a row j (16 of A, 16 of P) are reduced over the 8 cg lanes at the end with
    //    one transposed reduction (each lane ends with 4 of the totals).
    {
        const int blk = warp >> 1, cg = lane & 7, jq = lane >> 3;
        const int blk0 = 16 * blk;
#pragma unroll 1
        for (int ps = 0; ps < 2; ++ps) {
            const int jp = 4 * (warp & 1) + jq;
            const int j = blk0 + (ps == 0 ? jp : 15 - jp);
            const int rs = ps == 0 ? 4 * (warp & 1) : 12 - 4 * (warp & 1);   // warp-uniform
            uint64_t kd[8];                       // key j decayed to row r, as packed pairs
#pragma unroll
            for (int m = 0; m < 4; ++m) ld2x2(sK + j * LD + 4 * cg + 32 * m, kd[2 * m], kd[2 * m + 1]);
            float red[32];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                red[rr] = 0.f;
                red[16 + rr] = 0.f;
                if (rr < rs) continue;
                const int r = blk0 + rr;
                uint64_t pa0 = 0, pa1 = 0, pp0 = 0, pp1 = 0;
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const int c = 4 * cg + 32 * m;
                    uint64_t x0, x1;
                    if (r > j) {
                        ld2x2(sAl + r * LD + c, x0, x1);
                        kd[2 * m] = mul2(kd[2 * m], x0);
                        kd[2 * m + 1] = mul2(kd[2 * m + 1], x1);
                    }
                    ld2x2(sK + r * LD + c, x0, x1);
                    pa0 = fma2(x0, kd[2 * m], pa0);
                    pa1 = fma2(x1, kd[2 * m + 1], pa1);
                    ld2x2(sQ + r * LD + c, x0, x1);
                    pp0 = fma2(x0, kd[2 * m], pp0);
                    pp1 = fma2(x1, kd[2 * m + 1], pp1);
                }
                red[rr] = f2sum(pa0) + f2sum(pa1);
                red[16 + rr] = f2sum(pp0) + f2sum(pp1);
            }
#pragma unroll
            for (int lvl = 0; lvl < 3; ++lvl) {
                const int half = 16 >> lvl, off = 4 >> lvl;
                const bool upper = (cg & off) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float keep = upper ? red[half + i] : red[i];
                    const float give = upper ? red[i] : red[half + i];
                    red[i] = keep + __shfl_xor_sync(0xffffffffu, give, off);
                }
            }
            // lane cg holds the totals of sums 4 cg .. 4 cg + 3 (0..15: A rows, 16..31: P rows)
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int idx = 4 * cg + t, rr = idx & 15, r = blk0 + rr;
                if (idx < 16) sAD[r * 16 + (j & 15)] = r > j ? sBeta[r] * red[t] : 0.f;
                else KDA_REC(P)[tc::img_index(r, j, C)] = r >= j ? tc::round_tf32(red[t]) : 0.f;
            }
        }
        // zero upper off-diagonal blocks of the P image: (I, J) = (0,1) (0,2) (0,3) (1,2) (1,3) (2,3)
        for (int e = tid; e < 6 * 64; e += THREADS) {
            const int b = e >> 6, i = (e >> 2) & 15, q4 = e & 3;
            const int I = b < 3 ? 0 : (b < 5 ? 1 : 2);
            const int J = b < 3 ? b + 1 : (b < 5 ? b - 1 : 3);
            st4(KDA_REC(P) + tc::img_index(16 * I + i, 16 * J + 4 * q4, C), make_float4(0.f, 0.f, 0.f, 0.f));
        }
    }
    __syncthreads();

    // 3. per (column c, sub-block): block products (every thread forms all four, in one order),
    //    k o Rout -> alpha tile and Ktil^T record, k o Rin and q o Rin in place, (beta Kbar)^T -> TMEM
    {
        const int c = tid & (D - 1), hf = tid >> 7;
        float bp[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            float p = 1.f;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) p *= sAl[(16 * b + rr) * LD + c];
            bp[b] = p;
        }
        sBp[(2 * hf) * D + c] = hf ? bp[2] : bp[0];
        sBp[(2 * hf + 1) * D + c] = hf ? bp[3] : bp[1];
        if (hf == 0) {
            KDA_REC(GL)[c] = ((bp[0] * bp[1]) * bp[2]) * bp[3];
            sB12[c] = bp[1] * bp[2];
        }
#pragma unroll
        for (int bi = 0; bi < 2; ++bi) {
            const int blk = 2 * hf + bi;
            float eb = 1.f, ea = 1.f;
#pragma unroll
            for (int b = 0; b < NB; ++b) {
                if (b < blk) eb *= bp[b];
                if (b > blk) ea *= bp[b];
            }
            sEb[blk * D + c] = eb;
            float al[16], kk[16], qq[16];
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const int r = 16 * blk + rr;
                al[rr] = sAl[r * LD + c];
                kk[rr] = sK[r * LD + c];
                qq[rr] = sQ[r * LD + c];
            }
            float kt[16];
            float rout = 1.f;
#pragma unroll
            for (int rr = 15; rr >= 0; --rr) {
                const float ko = kk[rr] * rout;
                sAl[(16 * blk + rr) * LD + c] = ko;
                kt[rr] = tc::round_tf32(ko * ea);
                rout *= al[rr];
            }
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
                st4(KDA_REC(KT) + tc::img_index(c, 16 * blk + 4 * q4, C),
                    make_float4(kt[4 * q4], kt[4 * q4 + 1], kt[4 * q4 + 2], kt[4 * q4 + 3]));
            float kb[16];
            float rin = 1.f;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const int r = 16 * blk + rr;
                rin *= al[rr];
                const float ki = kk[rr] * rin;
                sK[r * LD + c] = ki;
                sQ[r * LD + c] = qq[rr] * rin;
                kb[rr] = tc::round_tf32(sBeta[r] * ki * eb);
            }
            tc::tmem_st16_nowait(tmem + lane_base + T_KB + 16 * blk, kb);
        }
        tc::tmem_wait_st();
    }
    __syncthreads();

    // value loads for (beta V)^T (lane v, columns j = 32 jh ..), issued here so that their latency
    // overlaps the Gram operands; consumed after the Gram completes.  They stay raw bf16 bits until
    // then: converting at the load would make the thread wait for the data here.
    const int vv_ = tid & (D - 1), jh = tid >> 7;
    unsigned short vr[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const int j = 32 * jh + i;
        vr[i] = j < L ? __bfloat16_as_ushort(vp[((size_t)(t0 + j) * H + h) * D + vv_]) : (unsigned short)0;
    }

    // 4. Gram operands and the Qbar record.  B image chunk f (16 bytes = 8 fp16 of one row) sits at
    //    byte 16 f: core (n >> 3, c >> 3) = f >> 3, row n & 7 = f & 7; rows n = 32 (I - 1) + {0..15:
    //    k o Rin, 16..31: q o Rin} of row block I.  Read now, written over the q tile after a barrier.
    uint32_t bimg[6][4];
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        const int f = tid + THREADS * i, core = f >> 3;
        const int n = (core >> 4) * 8 + (f & 7), c = (core & 15) * 8;
        const int I = (n >> 5) + 1, w = n & 31;
        const float* src = (w < 16 ? sK : sQ) + (16 * I + (w & 15)) * LD + c;
        const float4 x0 = ld4(src), x1 = ld4(src + 4);
        bimg[i][0] = tc::pack_f16x2(x0.x, x0.y);
        bimg[i][1] = tc::pack_f16x2(x0.z, x0.w);
        bimg[i][2] = tc::pack_f16x2(x1.x, x1.y);
        bimg[i][3] = tc::pack_f16x2(x1.z, x1.w);
    }
    for (int f = tid; f < C * D / 4; f += THREADS) {          // Qbar: rows r, K = c
        const int core = f >> 3, rr = (core >> 5) * 8 + (f & 7), c = (core & 31) * 4;
        st4(KDA_REC(QB) + 4 * f, rnd4(mul4(ld4(sQ + rr * LD + c), ld4(sEb + (rr >> 4) * D + c))));
    }
    if ((warp & 3) < 3) {          // lanes 0..95: key j decayed to the start of row block I, fp16 pairs
        const int m = (warp & 3) * 32 + lane;
        int I, j;
        gram_row(m, I, j);
        const int J = j >> 4;
        const int c0 = (warp >> 2) * 64;
        // decay over the whole blocks between J and I: none, bp[1], bp[2] or bp[1] bp[2]
        const float* mid = I - J < 2 ? nullptr : (I - J == 3 ? sB12 : sBp + (J + 1) * D);
        uint32_t w32[32];
#pragma unroll
        for (int q4 = 0; q4 < 16; ++q4) {
            const int c = c0 + 4 * q4;
            float4 v = ld4(sAl + j * LD + c);
            if (mid) v = mul4(v, ld4(mid + c));
            w32[2 * q4] = tc::pack_f16x2(v.x, v.y);
            w32[2 * q4 + 1] = tc::pack_f16x2(v.z, v.w);
        }
        tc::tmem_st16u_nowait(tmem + lane_base + T_KD + c0 / 2, w32);
        tc::tmem_st16u_nowait(tmem + lane_base + T_KD + c0 / 2 + 16, w32 + 16);
        tc::tmem_wait_st();
    }
    __syncthreads();               // k and q tiles are read; the alpha tile (k o Rout) is read
#pragma unroll
    for (int i = 0; i < 6; ++i)
        *reinterpret_cast<uint4*>(sIB + 16 * (tid + THREADS * i)) = make_uint4(bimg[i][0], bimg[i][1], bimg[i][2], bimg[i][3]);
    {                                                         // A <- diagonal blocks; T <- 0
        const int r = tid >> 2, q = tid & 3;                  // row r, float4 groups q, q + 4, ..
        const int b4 = (r >> 4) * 4;                          // the row's diagonal block: groups b4 .. b4 + 3
        for (int f = q; f < LDA / 4; f += 4) {
            float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
            if (f >= b4 && f < b4 + 4) x = ld4(sAD + r * 16 + 4 * (f - b4));
            st4(sA + r * LDA + 4 * f, x);
            st4(sT + r * LDA + 4 * f, make_float4(0.f, 0.f, 0.f, 0.f));
        }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        tc::tc_fence_after();
        const uint32_t bB = tc::smem_u32(sIB);
        constexpr uint32_t idesc = tc::idesc_f16(128, 96);
#pragma unroll
        for (int s = 0; s < D / 16; ++s)
            tc::mma_f16_ts(tmem + T_G, tmem + T_KD + 8 * s, tc::smem_desc(bB + 256 * s, 128, 2048), idesc, s > 0);
        tc::mma_commit(bar_g);
    }

    // 5. the Gram result; (beta V)^T from the values loaded before the Gram operands
    {
        const bool done = tc::mbar_wait(bar_g, 0, kWaitPolls);
        tc::tc_fence_after();
        if (!done && tid == 0) record_error(kDevErrTimeout);
        if (tid == 0) tc_ok = tc_ok && done;
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        float x[16];
#pragma unroll
        for (int i4 = 0; i4 < 4; ++i4) {
            const float4 b4 = ld4(sBeta + 32 * jh + 16 * hh + 4 * i4);
#define KDA_VF(i) __bfloat162float(__ushort_as_bfloat16(vr[i]))
            x[4 * i4 + 0] = tc::round_tf32(b4.x * KDA_VF(16 * hh + 4 * i4 + 0));
            x[4 * i4 + 1] = tc::round_tf32(b4.y * KDA_VF(16 * hh + 4 * i4 + 1));
            x[4 * i4 + 2] = tc::round_tf32(b4.z * KDA_VF(16 * hh + 4 * i4 + 2));
            x[4 * i4 + 3] = tc::round_tf32(b4.w * KDA_VF(16 * hh + 4 * i4 + 3));
#undef KDA_VF
        }
        tc::tmem_st16_nowait(tmem + lane_base + T_KD + 32 * jh + 16 * hh, x);
    }
    if ((warp & 3) < 3) {          // Gram rows m = (I, j): warp half 0 -> A (k rows), half 1 -> P (q rows)
        const int q = warp & 3, hf = warp >> 2;
        const int m = 32 * q + lane;
        int I, j;
        gram_row(m, I, j);
        const int Ia = q + 1, Ib = q < 2 ? q + 2 : 3;
        float ga[16], gb[16];
        tc::tmem_ld16(tmem + lane_base + T_G + 32 * (Ia - 1) + 16 * hf, ga);
        tc::tmem_ld16(tmem + lane_base + T_G + 32 * (Ib - 1) + 16 * hf, gb);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int r = 16 * I + i;
            const float g = I == Ia ? ga[i] : gb[i];
            if (hf == 0) sA[r * LDA + j] = sBeta[r] * g;
            else KDA_REC(P)[tc::img_index(r, j, C)] = tc::round_tf32(g);
        }
    }
    tc::tmem_wait_st();
    tc::tc_fence_before();
    __syncthreads();

    // 6. T = (I + A)^{-1}: 16 x 16 diagonal blocks by forward substitution, then by block distance
    if (tid < C) {
        const int I = tid >> 4, jj = tid & 15, j = tid;
        float col[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) col[i] = (i == jj) ? 1.f : 0.f;
#pragma unroll
        for (int i = 1; i < 16; ++i) {
            float acc = col[i];
#pragma unroll
            for (int k = 0; k < i; ++k) acc = fmaf(-sA[(16 * I + i) * LDA + 16 * I + k], col[k], acc);
            col[i] = (i > jj) ? acc : col[i];
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) sT[(16 * I + i) * LDA + j] = col[i];
    }
    __syncthreads();
    auto tblocks = [&](auto dc) {
        constexpr int d = decltype(dc)::value;
        constexpr int nb = NB - d;
        for (int e = tid; e < nb * 256; e += THREADS) {      // X_IJ = sum_{J<=K<I} A_IK T_KJ
            const int J = e >> 8, I = J + d, i = (e >> 4) & 15, jj = e & 15;
            const float* ar = sA + (16 * I + i) * LDA + 16 * J;
            const float* tc0 = sT + 16 * J * LDA + 16 * J + jj;
            float acc = 0.f;
#pragma unroll
            for (int kk = 0; kk < 16 * d; kk += 4) {                // a row of A as float4s
                const float4 av = ld4(ar + kk);
                acc = fmaf(av.x, tc0[kk * LDA], acc);
                acc = fmaf(av.y, tc0[(kk + 1) * LDA], acc);
                acc = fmaf(av.z, tc0[(kk + 2) * LDA], acc);
                acc = fmaf(av.w, tc0[(kk + 3) * LDA], acc);
            }
            sX[e] = acc;
        }
        __syncthreads();
        for (int e = tid; e < nb * 256; e += THREADS) {      // T_IJ = -T_II X_IJ
            const int J = e >> 8, I = J + d, i = (e >> 4) & 15, jj = e & 15;
            const float* tr = sT + (16 * I + i) * LDA + 16 * I;
            const float* xc = sX + (J << 8) + jj;
            float acc = 0.f;
#pragma unroll
            for (int kk = 0; kk < 16; kk += 4) {                    // T_II is lower triangular
                const float4 tv = ld4(tr + kk);
                acc = kk + 0 <= i ? fmaf(tv.x, xc[kk * 16], acc) : acc;
                acc = kk + 1 <= i ? fmaf(tv.y, xc[(kk + 1) * 16], acc) : acc;
                acc = kk + 2 <= i ? fmaf(tv.z, xc[(kk + 2) * 16], acc) : acc;
                acc = kk + 3 <= i ? fmaf(tv.w, xc[(kk + 3) * 16], acc) : acc;
            }
            sT[(16 * I + i) * LDA + 16 * J + jj] = -acc;
        }
        __syncthreads();
    };
    tblocks(std::integral_constant<int, 1>{});
    tblocks(std::integral_constant<int, 2>{});
    tblocks(std::integral_constant<int, 3>{});

    // T image (rows r, K = j); U^T = (beta V)^T T^T, W^T = (beta Kbar)^T T^T
    for (int f = tid; f < C * C / 4; f += THREADS) {
        const int core = f >> 3, rr = (core >> 4) * 8 + (f & 7), j0 = (core & 15) * 4;
        st4(sIT + 4 * f, rnd4(ld4(sT + rr * LDA + j0)));
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc::tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        tc::tc_fence_after();
        constexpr uint32_t idesc = tc::idesc_tf32(128, 64);
        const uint32_t bT = tc::smem_u32(sIT);
#pragma unroll
        for (int s = 0; s < C / 8; ++s)
            tc::mma_tf32_ts(tmem + T_G, tmem + T_KD + 8 * s, tc::smem_desc(bT + 256 * s, 128, 2048), idesc, s > 0);
#pragma unroll
        for (int s = 0; s < C / 8; ++s)
            tc::mma_tf32_ts(tmem + T_G + 64, tmem + T_KB + 8 * s, tc::smem_desc(bT + 256 * s, 128, 2048), idesc, s > 0);
        tc::mma_commit(bar_uw);
    }
    {
        const bool done = tc::mbar_wait(bar_uw, 0, kWaitPolls);
        tc::tc_fence_after();
        if (tid == 0) tc_ok = tc_ok && done;
        if (!done) {
            if (lane == 0) record_error(kDevErrTimeout);
        } else {
            const int row = (warp & 3) * 32 + lane, hf = warp >> 2;
            const uint32_t taddr = tmem + lane_base + T_G + 64 * hf;
#pragma unroll
            for (int r0 = 0; r0 < C; r0 += 16) {
                float x[16];
                tc::tmem_ld16(taddr + r0, x);
                if (hf == 0) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) KDA_REC(U)[(r0 + j) * D + row] = x[j];
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j) KDA_REC(W)[tc::img_index(r0 + j, row, D)] = tc::round_tf32(x[j]);
                }
            }
        }
    }
    if (tid == 0 && !tc_ok) {      // a wait gave up: let this CTA's MMAs land (bounded) before freeing TMEM
        tc::mma_commit(bar_drain);
        tc::mbar_wait(bar_drain, 0, kWaitPolls);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 256);
    }
#undef KDA_REC
}

// ---- host-side dispatch --------------------------------------------------------------------------
template <int C, int D, typename TIn, typename TOut>
cudaError_t run_prefill(const kda_params& p, const GateParams& gp, const void* q, const void* k,
                        const void* v, const float* g_raw, const float* b_raw, const float* A_log,
                        const float* dt_bias, const int32_t* cu, int32_t N, int64_t T, float* pool,
                        int64_t num_slots, const int32_t* state_idx, void* out, void* workspace,
                        cudaStream_t stream, const cudaEvent_t* ev, float* snap, int64_t snap_cap)
{
    const int H = p.num_heads;
    const WsLayout w = ws_layout(C, D, H, N, T);
    int32_t* tab = reinterpret_cast<int32_t*>(workspace);
    int32_t* chunk_seq = tab;
    int32_t* chunk_start = tab + w.max_chunks;
    int32_t* chunk_len = tab + 2 * w.max_chunks;
    int32_t* seq_off = tab + 3 * w.max_chunks;
    int32_t* seq_order = seq_off + N + 1;
    float* ws = reinterpret_cast<float*>(reinterpret_cast<char*>(workspace) + w.table_bytes);

    cudaError_t e;
    if (ev && (e = cudaEventRecord(ev[0], stream)) != cudaSuccess) return e;
    chunk_table_kernel<<<1, 1024, 0, stream>>>(cu, N, T, C, w.max_chunks, chunk_seq, chunk_start, chunk_len, seq_off,
                                               seq_order);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[1], stream)) != cudaSuccess) return e;

    IntraArgs ia;
    ia.q = q; ia.k = k; ia.v = v; ia.g_raw = g_raw; ia.b_raw = b_raw; ia.A_log = A_log; ia.dt_bias = dt_bias;
    ia.chunk_seq = chunk_seq; ia.chunk_start = chunk_start; ia.chunk_len = chunk_len; ia.seq_off = seq_off;
    ia.state_idx = state_idx; ia.num_slots = num_slots; ia.max_chunks = w.max_chunks; ia.N = N; ia.H = H;
    ia.gp = gp; ia.ws = ws; ia.ws_stride = w.per_chunk_head;
    // bf16 inputs at the 64 x 128 shape take the tensor-core (tf32) state pass.  fp32 inputs keep
    // the fp32 SIMT pass: tf32 operands (unit roundoff 2^-11) cannot meet the 1e-5 relative bound
    // that fp32 I/O carries, while they sit well inside the 2e-3 bound of bf16 I/O.
    constexpr bool kTensorCore = (C == TcRec::C && D == TcRec::D && std::is_same<TIn, __nv_bfloat16>::value);
    dim3 gi((unsigned)w.max_chunks, (unsigned)H);
    if constexpr (kTensorCore) {
        e = cudaFuncSetAttribute(chunk_intra_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)itc::BYTES);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(chunk_intra_tc_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
        if (e != cudaSuccess) return e;
        chunk_intra_tc_kernel<<<gi, itc::THREADS, itc::BYTES, stream>>>(ia);
    } else {
        using IS = IntraShape<C, D>;
        auto intra = chunk_intra_kernel<C, D, TIn, false>;
        e = cudaFuncSetAttribute(intra, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)IS::BYTES);
        if (e != cudaSuccess) return e;
        intra<<<gi, IS::THREADS, IS::BYTES, stream>>>(ia);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[2], stream)) != cudaSuccess) return e;

    StateArgs sa;
    sa.seq_order = seq_order;
    sa.chunk_start = chunk_start; sa.chunk_len = chunk_len; sa.seq_off = seq_off; sa.cu = cu;
    sa.state_idx = state_idx; sa.pool = pool; sa.num_slots = num_slots; sa.max_chunks = w.max_chunks;
    sa.T = T; sa.N = N; sa.H = H; sa.ws = ws; sa.ws_stride = w.per_chunk_head; sa.out = out;
    sa.snap = snap; sa.snap_cap = snap_cap;
    if constexpr (kTensorCore) {
        auto state = chunk_state_tc_kernel<TOut>;
        e = cudaFuncSetAttribute(state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmemBytes);
        if (e != cudaSuccess) return e;
        state<<<(unsigned)((int64_t)N * H), kStateThreads, kTcSmemBytes, stream>>>(sa);
    } else {
        constexpr int NV = D < 32 ? D : 32;
        using SS = StateShape<C, D, NV>;
        auto state = chunk_state_kernel<C, D, NV, TOut>;
        e = cudaFuncSetAttribute(state, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SS::BYTES);
        if (e != cudaSuccess) return e;
        dim3 gs((unsigned)N, (unsigned)H, (unsigned)(D / NV));
        state<<<gs, SS::THREADS, SS::BYTES, stream>>>(sa);
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (ev && (e = cudaEventRecord(ev[3], stream)) != cudaSuccess) return e;
    return cudaSuccess;
}

template <int C, int D>
cudaError_t dispatch_dtypes(const kda_params& p, const GateParams& gp, const void* q, const void* k,
                            const void* v, const float* g_raw, const float* b_raw, const float* A_log,
                            const float* dt_bias, const int32_t* cu, int32_t N, int64_t T, float* pool,
                            int64_t num_slots, const int32_t* state_idx, void* out, void* ws,
                            cudaStream_t s, const cudaEvent_t* ev, float* snap, int64_t snap_cap)
{
#define KDA_RUN(TI, TO) run_prefill<C, D, TI, TO>(p, gp, q, k, v, g_raw, b_raw, A_log, dt_bias, cu, N, T, pool, num_slots, state_idx, out, ws, s, ev, snap, snap_cap)
    if (p.io_dtype == KDA_BF16) {
        if (p.out_dtype == KDA_BF16) return KDA_RUN(__nv_bfloat16, __nv_bfloat16);
        return KDA_RUN(__nv_bfloat16, float);
    }
    if (p.out_dtype == KDA_BF16) return KDA_RUN(float, __nv_bfloat16);
    return KDA_RUN(float, float);
#undef KDA_RUN
}

}  // namespace

bool prefill_supported(const kda_params& p)
{
    const bool dim = p.head_dim == 16 || p.head_dim == 32 || p.head_dim == 64 || p.head_dim == 128;
    const bool chunk = p.chunk_size == 16 || p.chunk_size == 32 || p.chunk_size == 64;
    const bool dt = (p.io_dtype == KDA_F32 || p.io_dtype == KDA_BF16) &&
                    (p.out_dtype == KDA_F32 || p.out_dtype == KDA_BF16);
    return dim && chunk && dt && p.gate_kind == KDA_GATE_PER_CHANNEL;
}

size_t prefill_workspace_bytes(const kda_params& p, int32_t num_seqs, int64_t total_tokens)
{
    return ws_layout(p.chunk_size, p.head_dim, p.num_heads, num_seqs, total_tokens).total_bytes;
}

cudaError_t launch_prefill(const kda_params& p, const GateParams& gp, const void* q,
                           const void* k, const void* v, const float* g_raw, const float* b_raw,
                           const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
                           int32_t num_seqs, int64_t total_tokens, float* pool,
                           int64_t num_slots, const int32_t* state_idx, void* out,
                           void* workspace, cudaStream_t stream, const cudaEvent_t* events,
                           float* chunk_states, int64_t chunk_states_capacity)
{
#define KDA_DIM(CC, DD)                                                                            \
    if (p.chunk_size == CC && p.head_dim == DD)                                                    \
        return dispatch_dtypes<CC, DD>(p, gp, q, k, v, g_raw, b_raw, A_log, dt_bias, cu_seqlens,  \
                                       num_seqs, total_tokens, pool, num_slots, state_idx, out,    \
                                       workspace, stream, events, chunk_states,                    \
                                       chunk_states_capacity);
    KDA_DIM(16, 16) KDA_DIM(16, 32) KDA_DIM(16, 64) KDA_DIM(16, 128)
    KDA_DIM(32, 16) KDA_DIM(32, 32) KDA_DIM(32, 64) KDA_DIM(32, 128)
    KDA_DIM(64, 16) KDA_DIM(64, 32) KDA_DIM(64, 64) KDA_DIM(64, 128)
#undef KDA_DIM
    return cudaErrorInvalidValue;
}

cudaError_t prefill_read_and_clear_error(int32_t* code)
{
    int32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_prefill_error, sizeof(int32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_prefill_error, &zero, sizeof(int32_t));
}

}  // namespace kda
