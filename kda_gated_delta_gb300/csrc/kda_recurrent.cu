// kda_recurrent.cu -- single-token decode and multi-token verify of the KDA / GDN recurrence.
//
// One CTA owns one (request, head) state tile S^T [D][D] fp32 (value row j, key channel c
// contiguous, the pool's layout).  The tile is streamed from HBM once with 16-byte loads,
// kept in registers across the request's tokens, and written once (decode: back into the pool
// slot; verify: once per draft token into the intermediate-state buffer).
//
// Per token, following the five steps of "linear_attention" (zdszero.github.io), section
// "Gated DeltaNet", with the per-channel decay of section "KDA：逐通道的遗忘门":
//   S' = S Diag(alpha) (transposed storage: column c of S^T scaled by alpha_c)   decay
//   v_hat_j = sum_c S'[j][c] k_c                                                 predict
//   delta_j = beta (v_j - v_hat_j)                                                error
//   S[j][c] = S'[j][c] + delta_j k_c                                             write
//   o_j     = sum_c S'[j][c] q_c + delta_j (q . k)  ( = q S_t )                  read
// The readout uses the decomposition of "ReplaySSM -- buffered output-only decode", section
// 3.12, so both row reductions (k . S'_j and q . S'_j) are taken in one pass.
//
// Thread mapping: a warp handles 16 rows; a row is split over LPR lanes, each lane holding CPL
// consecutive-in-pattern columns (float4 groups 4*li + 4*LPR*j), so every load instruction of a
// warp reads whole 128-byte row segments.  Row sums are reduced with log2(LPR) xor-shuffles.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "kda_internal.cuh"
#include "kda_tc.cuh"

namespace kda {
namespace {

__device__ int32_t g_recurrent_error = 0;

__device__ __forceinline__ void record_error(int32_t code) { atomicCAS(&g_recurrent_error, 0, code); }

struct RecArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* g_raw;
    const float* b_raw;
    const float* A_log;
    const float* dt_bias;
    const float* pool_in;
    float* pool_out;    // decode: == pool_in (in place); verify: unused
    float* inter;       // verify: [batch][t_draft][H][D][D]; decode: unused
    const int32_t* state_idx;
    void* out;
    int64_t num_slots;
    int H;
    int t_draft;
    GateParams gp;
    // replay mode: per-slot rings of the last steps since the checkpoint (see kda_replay_decode)
    float* ring_d;            // [slots][H][L][D] corrected deltas
    float* ring_k;            // [slots][H][L][D] normalised keys
    float* ring_a;            // [slots][H][L][D] (per-channel) or [slots][H][L] (per-head) decays
    int ring_len;             // L
    const int32_t* write_pos; // [batch] entries committed in the ring (0 .. L-1)
    const int32_t* force_flush;  // [batch] or null
    int64_t prefetch_ahead;   // CTAs between this one and the one whose state it prefetches into L2; 0 off
};

enum { kModeDecode = 0, kModeVerify = 1, kModeReplay = 2 };

// 16-byte asynchronous copy global -> shared (both addresses 16-byte aligned), bypassing L1
__device__ __forceinline__ void cp_async16(void* dst, const void* src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}

// SPLIT CTAs share one (request, head), each owning D / SPLIT consecutive value rows of the state.
template <int D, int SPLIT = 1>
struct RecShape {
    static constexpr int ROWS = D / SPLIT;          // state rows of one CTA
    static constexpr int NWARPS = D >= 32 ? D / 16 / SPLIT : 1;
    static constexpr int THREADS = NWARPS * 32;
    static constexpr int CPL = D >= 32 ? 16 : 8;   // columns per lane
    static constexpr int LPR = D / CPL;             // lanes per row
    static constexpr int RPS = 32 / LPR;            // rows per warp step
    static constexpr int ROWS_PER_WARP = ROWS / NWARPS;
    static constexpr int STEPS = ROWS_PER_WARP / RPS;
    static constexpr int NV4 = CPL / 4;             // float4 groups per lane and row
    static_assert(ROWS_PER_WARP % RPS == 0, "row split");
    static_assert(NWARPS * ROWS_PER_WARP == ROWS, "rows");
    static_assert(THREADS >= D || SPLIT == 1, "one thread per channel in the prologue");
};

// The buffered decode at d = 128 runs two CTAs of 128 threads per (request, head), 64 state rows
// each: a CTA streams its 32 KB of the checkpoint, and four CTAs fit on an SM instead of two, so
// that more of the checkpoint is in flight while other CTAs work through the ring.  Both halves
// form the per-channel prologue (norms, gate, ring products); rows are independent after it.
template <int D, int MODE>
__host__ __device__ constexpr int rec_split() { return MODE == kModeReplay && D == 128 ? 2 : 1; }

// GATE: KDA_GATE_PER_CHANNEL or KDA_GATE_PER_HEAD.  MODE: kModeDecode updates the pool slot in
// place; kModeVerify writes every intermediate state to `inter` and leaves the pool untouched;
// kModeReplay either appends this step to the ring, computing the outputs from the checkpoint and
// the committed entries without materializing the state (readout decomposition), or (flush)
// rebuilds the state from the checkpoint and ring and writes the new state to the checkpoint.
template <int D, int GATE, int MODE, typename TIn, typename TOut>
__global__ void __launch_bounds__(RecShape<D, rec_split<D, MODE>()>::THREADS, (D >= 128 ? 2 * rec_split<D, MODE>() : 4))
recurrent_kernel(const RecArgs a)
{
    constexpr int SPLIT = rec_split<D, MODE>();
    using Sh = RecShape<D, SPLIT>;
    constexpr int NWARPS = Sh::NWARPS, CPL = Sh::CPL, LPR = Sh::LPR, RPS = Sh::RPS;
    constexpr int STEPS = Sh::STEPS, NV4 = Sh::NV4;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int H = a.H;
    const int64_t bh = blockIdx.x / SPLIT;
    const int half = SPLIT == 1 ? 0 : (int)(blockIdx.x % SPLIT);
    const int row0 = half * Sh::ROWS;                // this CTA's first state row
    const int64_t b = bh / H;
    const int h = (int)(bh - b * H);
    constexpr bool VERIFY = MODE == kModeVerify;
    const int T = VERIFY ? a.t_draft : 1;

    int64_t slot = a.state_idx[b];
    if (slot >= a.num_slots) {
        if (tid == 0) record_error(kDevErrStateIndex);
        slot = -1;
    }
    int wp = 0;
    bool flush = false;
    if (MODE == kModeReplay && slot >= 0) {
        wp = a.write_pos[b];
        if (wp < 0 || wp >= a.ring_len) {
            if (tid == 0) record_error(kDevErrWritePos);
            slot = -1;
        }
        flush = wp == a.ring_len - 1 || (a.force_flush && a.force_flush[b] != 0);
    }
    TOut* out = reinterpret_cast<TOut*>(a.out);
    if (slot < 0) {  // padding row: zero outputs, no state traffic
        for (int t = 0; t < T; ++t) {
            const int64_t tok = b * T + t;
            for (int j = row0 + tid; j < row0 + Sh::ROWS; j += Sh::THREADS) out[(tok * H + h) * D + j] = from_f32<TOut>(0.f);
        }
        return;
    }

    const int row_in_step = lane / LPR;
    const int li = lane % LPR;
    const size_t tile = ((size_t)slot * H + h) * (size_t)D * D;

    // ---- prologue for all T tokens at once: inputs to shared memory, then norms, q.k, beta, alpha
    extern __shared__ float4 rec_smem4[];
    float* s_k = reinterpret_cast<float*>(rec_smem4);    // [T][D] k -> k_hat
    float* s_q = s_k + T * D;                            // [T][D] q -> q_hat * scale
    float* s_al = s_q + T * D;                           // [T][D] alpha (per-channel gate)
    float* s_v = s_al + T * D;                           // [T][D] v
    float* s_sc = s_v + T * D;                           // [T][8]: beta, q.k, alpha (per head), 1/|k|, scale/|q|
    if (MODE == kModeReplay && wp > 0) {
        // the committed ring entries travel to shared memory (asynchronous 16-byte copies), issued
        // ahead of the state loads so that they land first
        float* s_rk = s_sc + 8 * T;
        float* s_rd = s_rk + a.ring_len * D;
        float* s_ra = s_rd + a.ring_len * D;
        const size_t rb = ((size_t)slot * H + h) * (size_t)a.ring_len;
        const float4* gk = reinterpret_cast<const float4*>(a.ring_k + rb * D);
        const float4* gd = reinterpret_cast<const float4*>(a.ring_d + rb * D);
        const float4* ga = reinterpret_cast<const float4*>(a.ring_a + rb * D);
        for (int e = tid; e < wp * D / 4; e += Sh::THREADS) {
            cp_async16(reinterpret_cast<float4*>(s_rk) + e, gk + e);
            cp_async16(reinterpret_cast<float4*>(s_rd) + e, gd + e);
            if (GATE == KDA_GATE_PER_CHANNEL) cp_async16(reinterpret_cast<float4*>(s_ra) + e, ga + e);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    }
    const TIn* qp = reinterpret_cast<const TIn*>(a.q);
    const TIn* kp = reinterpret_cast<const TIn*>(a.k);
    const TIn* vp = reinterpret_cast<const TIn*>(a.v);
    // One token (decode, replay): its inputs are loaded raw before the state, so that they arrive
    // first and the prologue's arithmetic overlaps the state's latency instead of following it.
    TIn k_raw{}, q_raw{}, v_raw{};
    float g_r = 0.f, dt_r = 0.f, b_r = 0.f;
    if (!VERIFY) {
        if (tid < D) {
            const size_t idx = ((size_t)b * H + h) * D + tid;
            k_raw = kp[idx];
            q_raw = qp[idx];
            v_raw = vp[idx];
            if (GATE == KDA_GATE_PER_CHANNEL) {
                g_r = a.g_raw[idx];
                if (a.dt_bias) dt_r = a.dt_bias[(size_t)h * D + tid];
            }
        }
        if (tid == 0) {
            b_r = a.b_raw[(size_t)b * H + h];
            if (GATE == KDA_GATE_PER_HEAD) {
                g_r = a.g_raw[(size_t)b * H + h];
                if (a.dt_bias) dt_r = a.dt_bias[h];
            }
        }
    }
    const float a_log = a.A_log[h];
    // Then every state load of this thread; the token prologue overlaps their latency.
    float4 st[STEPS][NV4];
#pragma unroll
    for (int s = 0; s < STEPS; ++s) {
        const int row = row0 + warp * Sh::ROWS_PER_WARP + s * RPS + row_in_step;
        const float4* src = reinterpret_cast<const float4*>(a.pool_in + tile + (size_t)row * D);
#pragma unroll
        for (int j = 0; j < NV4; ++j) st[s][j] = __ldcs(src + li + LPR * j);
    }
    // L2 prefetch of the state rows of the CTA prefetch_ahead places later in the grid: CTAs start in
    // index order, so that one starts about one CTA lifetime from now and finds its state in L2.
    // Registers cap the state bytes the resident CTAs hold in flight; an L2 prefetch takes none.
    if (tid == 0 && a.prefetch_ahead > 0) {
        const int64_t nb = (int64_t)blockIdx.x + a.prefetch_ahead;
        if (nb < (int64_t)gridDim.x) {
            const int64_t bh2 = nb / SPLIT, b2 = bh2 / H;
            const int h2 = (int)(bh2 - b2 * H);
            const int64_t slot2 = a.state_idx[b2];
            if (slot2 >= 0 && slot2 < a.num_slots)
                tc::bulk_prefetch_l2(a.pool_in + ((size_t)slot2 * H + h2) * (size_t)D * D + (size_t)(nb % SPLIT) * Sh::ROWS * D,
                                     (uint32_t)(Sh::ROWS * D * sizeof(float)));
        }
    }

    const float rate = expf(a_log);
    if (VERIFY) {
        for (int e = tid; e < T * D; e += Sh::THREADS) {
            const int t = e / D, c = e - t * D;
            const size_t idx = ((size_t)(b * T + t) * H + h) * D + c;
            s_k[e] = to_f32(kp[idx]);
            s_q[e] = to_f32(qp[idx]);
            s_v[e] = to_f32(vp[idx]);
            if (GATE == KDA_GATE_PER_CHANNEL) {
                const float x = a.g_raw[idx] + (a.dt_bias ? a.dt_bias[(size_t)h * D + c] : 0.f);
                s_al[e] = expf(gate_log_decay(x, rate, a.gp));
            }
        }
        for (int t = tid; t < T; t += Sh::THREADS) {
            const size_t th = (size_t)(b * T + t) * H + h;
            s_sc[8 * t + 0] = sigmoid_f32(a.b_raw[th]);
            float alpha_h = 1.f;
            if (GATE == KDA_GATE_PER_HEAD) alpha_h = expf(gate_log_decay(a.g_raw[th] + (a.dt_bias ? a.dt_bias[h] : 0.f), rate, a.gp));
            s_sc[8 * t + 2] = alpha_h;
        }
    } else {
        if (tid < D) {
            s_k[tid] = to_f32(k_raw);
            s_q[tid] = to_f32(q_raw);
            s_v[tid] = to_f32(v_raw);
            if (GATE == KDA_GATE_PER_CHANNEL) s_al[tid] = expf(gate_log_decay(g_r + dt_r, rate, a.gp));
        }
        if (tid == 0) {
            s_sc[0] = sigmoid_f32(b_r);
            s_sc[2] = GATE == KDA_GATE_PER_HEAD ? expf(gate_log_decay(g_r + dt_r, rate, a.gp)) : 1.f;
        }
    }
    __syncthreads();
    // Norms and q.k.  Verify (T tokens): one warp per token, scaled k_hat and q_hat back to shared
    // memory.  Decode and replay (one token): every warp reduces the token's norms itself and keeps
    // 1/|k|, scale/|q| and q_hat.k_hat in registers, which saves two barriers.
    float rk1 = 1.f, rq1 = 1.f, qk1 = 0.f;
    if (MODE != kModeVerify) {
        float kk = 0.f, qq = 0.f, kq = 0.f;
        for (int c = lane; c < D; c += 32) {
            const float kc = s_k[c], qc = s_q[c];
            kk = fmaf(kc, kc, kk);
            qq = fmaf(qc, qc, qq);
            kq = fmaf(kc, qc, kq);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            kk += __shfl_xor_sync(0xffffffffu, kk, off);
            qq += __shfl_xor_sync(0xffffffffu, qq, off);
            kq += __shfl_xor_sync(0xffffffffu, kq, off);
        }
        rk1 = 1.0f / sqrtf(kk + a.gp.l2_eps);
        rq1 = a.gp.scale / sqrtf(qq + a.gp.l2_eps);
        qk1 = kq * rk1 * rq1;
    } else {
        for (int t = warp; t < T; t += NWARPS) {         // one warp per token
            float kk = 0.f, qq = 0.f, kq = 0.f;
            for (int c = lane; c < D; c += 32) {
                const float kc = s_k[t * D + c], qc = s_q[t * D + c];
                kk = fmaf(kc, kc, kk);
                qq = fmaf(qc, qc, qq);
                kq = fmaf(kc, qc, kq);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                kk += __shfl_xor_sync(0xffffffffu, kk, off);
                qq += __shfl_xor_sync(0xffffffffu, qq, off);
                kq += __shfl_xor_sync(0xffffffffu, kq, off);
            }
            if (lane == 0) {
                const float rk = 1.0f / sqrtf(kk + a.gp.l2_eps);
                const float rq = a.gp.scale / sqrtf(qq + a.gp.l2_eps);
                s_sc[8 * t + 1] = kq * rk * rq;
                s_sc[8 * t + 3] = rk;
                s_sc[8 * t + 4] = rq;
            }
        }
        __syncthreads();
        for (int e = tid; e < T * D; e += Sh::THREADS) {
            const int t = e / D;
            s_k[e] *= s_sc[8 * t + 3];
            s_q[e] *= s_sc[8 * t + 4];
        }
    }
    if (MODE == kModeReplay && wp > 0) {
        // S = Diag(prod_j a_j) S0 + sum_j d_j^T (k_j o prod_{i>j} a_i) over the wp committed steps
        // (ReplaySSM, section 3.11): stage the ring, turn k_j into k_j o prod_{i>j} a_i in place
        float* s_rk = s_sc + 8 * T;               // [L][D]
        float* s_rd = s_rk + a.ring_len * D;      // [L][D]
        float* s_ra = s_rd + a.ring_len * D;      // [L][D] (per-channel) or [L]
        float* s_tot = s_ra + a.ring_len * D;     // [D]
        float* s_ck = s_tot + D;                  // [L] k~_j . (a o k_hat)
        float* s_cq = s_ck + a.ring_len;          // [L] k~_j . (a o q_hat)
        const size_t rb = ((size_t)slot * H + h) * (size_t)a.ring_len;
        if (GATE == KDA_GATE_PER_HEAD)
            for (int j = tid; j < wp; j += Sh::THREADS) s_ra[j] = a.ring_a[rb + j];
        asm volatile("cp.async.wait_group 0;" ::: "memory");   // this thread's ring copies
        __syncthreads();
        for (int c = tid; c < D; c += Sh::THREADS) {
            float pr = 1.f;
            for (int j = wp - 1; j >= 0; --j) {
                s_rk[j * D + c] *= pr;
                pr *= (GATE == KDA_GATE_PER_CHANNEL) ? s_ra[j * D + c] : s_ra[j];
            }
            s_tot[c] = pr;
        }
        __syncthreads();
        if (!flush) {
            // Readout decomposition (ReplaySSM): with S' = Diag(P) S0 + sum_j k~_j^T d_j, a row of
            // (a o z) S' is sum_c S0[c] (P o a o z)[c] + sum_j (k~_j . (a o z)) d_j, so a step that
            // does not flush needs only these dot products and never materializes S'.
            for (int j = warp; j < wp; j += NWARPS) {
                float ck = 0.f, cq = 0.f;
                for (int c = lane; c < D; c += 32) {
                    const float za = (GATE == KDA_GATE_PER_CHANNEL) ? s_al[c] : s_sc[2];
                    const float r = s_rk[j * D + c] * za;
                    ck = fmaf(r, s_k[c], ck);
                    cq = fmaf(r, s_q[c], cq);
                }
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) {
                    ck += __shfl_xor_sync(0xffffffffu, ck, off);
                    cq += __shfl_xor_sync(0xffffffffu, cq, off);
                }
                if (lane == 0) {                     // raw k, q in shared memory: apply the norms
                    s_ck[j] = ck * rk1;
                    s_cq[j] = cq * rq1;
                }
            }
        } else {
#pragma unroll
        for (int s = 0; s < STEPS; ++s)
#pragma unroll
            for (int j4 = 0; j4 < NV4; ++j4) {
                const float4 tt = *reinterpret_cast<const float4*>(&s_tot[4 * (li + LPR * j4)]);
                st[s][j4] = make_float4(st[s][j4].x * tt.x, st[s][j4].y * tt.y, st[s][j4].z * tt.z, st[s][j4].w * tt.w);
            }
        for (int j = 0; j < wp; ++j) {                 // one ring entry: CPL keys x STEPS deltas per lane
            float4 kw[NV4];
            float dj[STEPS];
#pragma unroll
            for (int j4 = 0; j4 < NV4; ++j4) kw[j4] = *reinterpret_cast<const float4*>(&s_rk[j * D + 4 * (li + LPR * j4)]);
#pragma unroll
            for (int s = 0; s < STEPS; ++s) dj[s] = s_rd[j * D + row0 + warp * Sh::ROWS_PER_WARP + s * RPS + row_in_step];
#pragma unroll
            for (int s = 0; s < STEPS; ++s)
#pragma unroll
                for (int j4 = 0; j4 < NV4; ++j4) {
                    float4& e = st[s][j4];
                    e.x = fmaf(dj[s], kw[j4].x, e.x); e.y = fmaf(dj[s], kw[j4].y, e.y);
                    e.z = fmaf(dj[s], kw[j4].z, e.z); e.w = fmaf(dj[s], kw[j4].w, e.w);
                }
        }
        }
        __syncthreads();
    }
    if (MODE == kModeVerify) __syncthreads();

    for (int t = 0; t < T; ++t) {
        const int64_t tok = b * T + t;
        const size_t rowbase = ((size_t)tok * H + h) * D;
        const float beta = s_sc[8 * t + 0];
        const float qk = MODE == kModeVerify ? s_sc[8 * t + 1] : qk1;
        const float alpha_h = s_sc[8 * t + 2];
        const float sk = MODE == kModeVerify ? 1.f : rk1;   // k_hat = k * sk, q_hat = q * sq
        const float sq = MODE == kModeVerify ? 1.f : rq1;

        // ---- per-lane column constants --------------------------------------------------------
        float kh[CPL], qh[CPL], al[CPL];
#pragma unroll
        for (int j = 0; j < NV4; ++j) {
            const int c = t * D + 4 * (li + LPR * j);
            const float4 k4 = *reinterpret_cast<const float4*>(&s_k[c]);
            const float4 q4 = *reinterpret_cast<const float4*>(&s_q[c]);
            if (MODE == kModeVerify) {
                kh[4 * j + 0] = k4.x; kh[4 * j + 1] = k4.y; kh[4 * j + 2] = k4.z; kh[4 * j + 3] = k4.w;
                qh[4 * j + 0] = q4.x; qh[4 * j + 1] = q4.y; qh[4 * j + 2] = q4.z; qh[4 * j + 3] = q4.w;
            } else {
                kh[4 * j + 0] = k4.x * sk; kh[4 * j + 1] = k4.y * sk; kh[4 * j + 2] = k4.z * sk; kh[4 * j + 3] = k4.w * sk;
                qh[4 * j + 0] = q4.x * sq; qh[4 * j + 1] = q4.y * sq; qh[4 * j + 2] = q4.z * sq; qh[4 * j + 3] = q4.w * sq;
            }
            if (GATE == KDA_GATE_PER_CHANNEL) {
                const float4 a4 = *reinterpret_cast<const float4*>(&s_al[c]);
                al[4 * j + 0] = a4.x; al[4 * j + 1] = a4.y; al[4 * j + 2] = a4.z; al[4 * j + 3] = a4.w;
            } else {
                al[4 * j + 0] = al[4 * j + 1] = al[4 * j + 2] = al[4 * j + 3] = alpha_h;
            }
        }

        // replay step that does not flush, with committed entries: the readout decomposition
        const bool decomp = MODE == kModeReplay && !flush && wp > 0;
        if (decomp) {                                   // fold P o a into the column constants
            const float* s_tot = s_sc + 8 * T + (size_t)3 * a.ring_len * D;
#pragma unroll
            for (int j = 0; j < NV4; ++j) {
                const float4 tt = *reinterpret_cast<const float4*>(&s_tot[4 * (li + LPR * j)]);
                const float pa[4] = {tt.x * al[4 * j + 0], tt.y * al[4 * j + 1], tt.z * al[4 * j + 2], tt.w * al[4 * j + 3]};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    kh[4 * j + u] *= pa[u];
                    qh[4 * j + u] *= pa[u];
                }
            }
        }

        // ---- rows: decay, predict, error, write, read -----------------------------------------
#pragma unroll
        for (int s = 0; s < STEPS; ++s) {
            const int row = row0 + warp * Sh::ROWS_PER_WARP + s * RPS + row_in_step;
            const float vj = s_v[t * D + row];
            float pk = 0.f, pq = 0.f;
#pragma unroll
            for (int j = 0; j < NV4; ++j) {
                float4& e = st[s][j];
                if (!decomp) {
                    e.x *= al[4 * j + 0]; e.y *= al[4 * j + 1]; e.z *= al[4 * j + 2]; e.w *= al[4 * j + 3];
                }
                pk = fmaf(e.x, kh[4 * j + 0], pk); pk = fmaf(e.y, kh[4 * j + 1], pk);
                pk = fmaf(e.z, kh[4 * j + 2], pk); pk = fmaf(e.w, kh[4 * j + 3], pk);
                pq = fmaf(e.x, qh[4 * j + 0], pq); pq = fmaf(e.y, qh[4 * j + 1], pq);
                pq = fmaf(e.z, qh[4 * j + 2], pq); pq = fmaf(e.w, qh[4 * j + 3], pq);
            }
            if (decomp) {          // + sum_j (k~_j . (a o z)) d_j[row], the entries split over the row's lanes
                const float* s_rd = s_sc + 8 * T + (size_t)a.ring_len * D;
                const float* s_ck = s_sc + 8 * T + (size_t)3 * a.ring_len * D + D;
                for (int j = li; j < wp; j += LPR) {
                    const float dj = s_rd[j * D + row];
                    pk = fmaf(s_ck[j], dj, pk);
                    pq = fmaf(s_ck[a.ring_len + j], dj, pq);
                }
            }
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) {
                pk += __shfl_xor_sync(0xffffffffu, pk, off);
                pq += __shfl_xor_sync(0xffffffffu, pq, off);
            }
            const float delta = beta * (vj - pk);
            const float o = fmaf(delta, qk, pq);
            if (!(MODE == kModeReplay && !flush)) {     // a replay step that does not flush keeps S0
#pragma unroll
                for (int j = 0; j < NV4; ++j) {
                    float4& e = st[s][j];
                    e.x = fmaf(delta, kh[4 * j + 0], e.x); e.y = fmaf(delta, kh[4 * j + 1], e.y);
                    e.z = fmaf(delta, kh[4 * j + 2], e.z); e.w = fmaf(delta, kh[4 * j + 3], e.w);
                }
            }
            if (li == 0) out[rowbase + row] = from_f32<TOut>(o);
            if (MODE == kModeReplay && !flush) {      // append d to the ring; the state stays put
                if (li == 0) a.ring_d[(((size_t)slot * H + h) * a.ring_len + wp) * D + row] = delta;
                continue;
            }
            float* dst;
            if (VERIFY) {
                dst = a.inter + ((((size_t)b * T + t) * H + h) * (size_t)D + row) * D;
            } else {
                dst = a.pool_out + tile + (size_t)row * D;
            }
            float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
            for (int j = 0; j < NV4; ++j) __stcs(d4 + li + LPR * j, st[s][j]);
        }
        if (MODE == kModeReplay && !flush && half == 0) {   // append k_hat and the decay of this step
            const size_t re = ((size_t)slot * H + h) * a.ring_len + wp;
            for (int c = tid; c < D; c += Sh::THREADS) {
                a.ring_k[re * D + c] = s_k[c] * rk1;
                if (GATE == KDA_GATE_PER_CHANNEL) a.ring_a[re * D + c] = s_al[c];
            }
            if (GATE == KDA_GATE_PER_HEAD && tid == 0) a.ring_a[re] = alpha_h;
        }
    }
}

// Dynamic shared memory of one recurrent CTA: four [T][D] tiles and 8 scalars per token, plus in
// replay mode three [L][D] ring tiles, one [D] vector and two [L] vectors.
inline size_t recurrent_smem_bytes(int D, int T, int L)
{
    return sizeof(float) * ((size_t)4 * T * D + 8 * (size_t)T + (size_t)3 * L * D + D + (size_t)2 * L);
}

template <int D, int GATE, int MODE, typename TIn, typename TOut>
cudaError_t launch_t(const RecArgs& a, int64_t batch, cudaStream_t stream)
{
    constexpr int SPLIT = rec_split<D, MODE>();
    const int64_t blocks = batch * a.H * SPLIT;
    if (blocks <= 0) return cudaSuccess;
    const size_t smem = recurrent_smem_bytes(D, MODE == kModeVerify ? a.t_draft : 1, MODE == kModeReplay ? a.ring_len : 0);
    if (smem > 48 * 1024) {
        const cudaError_t e = cudaFuncSetAttribute(recurrent_kernel<D, GATE, MODE, TIn, TOut>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    // resident CTAs on the device (computed once per device and shared memory size class): the
    // prefetch distance; no prefetch if the occupancy query fails
    static std::atomic<int> resident[64][2];
    const int cls = smem > 48 * 1024 ? 1 : 0;
    int dev = 0;
    RecArgs la = a;
    la.prefetch_ahead = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64) {
        int r = resident[dev][cls].load(std::memory_order_relaxed);
        if (r == 0) {
            int per_sm = 0, sms = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, recurrent_kernel<D, GATE, MODE, TIn, TOut>,
                                                              RecShape<D, SPLIT>::THREADS, smem) == cudaSuccess &&
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && per_sm * sms > 0) {
                r = per_sm * sms;
            } else {
                cudaGetLastError();
                r = -1;
            }
            resident[dev][cls].store(r, std::memory_order_relaxed);
        }
        if (r > 0) la.prefetch_ahead = r;
    }
    recurrent_kernel<D, GATE, MODE, TIn, TOut><<<(unsigned)blocks, RecShape<D, SPLIT>::THREADS, smem, stream>>>(la);
    return cudaGetLastError();
}

template <int D, int GATE, int MODE>
cudaError_t dispatch_dtypes(const kda_params& p, const RecArgs& a, int64_t batch, cudaStream_t s)
{
    if (p.io_dtype == KDA_BF16) {
        if (p.out_dtype == KDA_BF16) return launch_t<D, GATE, MODE, __nv_bfloat16, __nv_bfloat16>(a, batch, s);
        return launch_t<D, GATE, MODE, __nv_bfloat16, float>(a, batch, s);
    }
    if (p.out_dtype == KDA_BF16) return launch_t<D, GATE, MODE, float, __nv_bfloat16>(a, batch, s);
    return launch_t<D, GATE, MODE, float, float>(a, batch, s);
}

template <int D, int MODE>
cudaError_t dispatch_gate(const kda_params& p, const RecArgs& a, int64_t batch, cudaStream_t s)
{
    if (p.gate_kind == KDA_GATE_PER_HEAD) return dispatch_dtypes<D, KDA_GATE_PER_HEAD, MODE>(p, a, batch, s);
    return dispatch_dtypes<D, KDA_GATE_PER_CHANNEL, MODE>(p, a, batch, s);
}

template <int MODE>
cudaError_t dispatch_dim(const kda_params& p, const RecArgs& a, int64_t batch, cudaStream_t s)
{
    switch (p.head_dim) {
    case 16: return dispatch_gate<16, MODE>(p, a, batch, s);
    case 32: return dispatch_gate<32, MODE>(p, a, batch, s);
    case 64: return dispatch_gate<64, MODE>(p, a, batch, s);
    case 128: return dispatch_gate<128, MODE>(p, a, batch, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool recurrent_supported(const kda_params& p)
{
    const bool dim = p.head_dim == 16 || p.head_dim == 32 || p.head_dim == 64 || p.head_dim == 128;
    const bool dt = (p.io_dtype == KDA_F32 || p.io_dtype == KDA_BF16) &&
                    (p.out_dtype == KDA_F32 || p.out_dtype == KDA_BF16);
    const bool gate = p.gate_kind == KDA_GATE_PER_CHANNEL || p.gate_kind == KDA_GATE_PER_HEAD;
    return dim && dt && gate;
}

cudaError_t launch_recurrent(const kda_params& p, const GateParams& gp, const void* q,
                             const void* k, const void* v, const float* g_raw,
                             const float* b_raw, const float* A_log, const float* dt_bias,
                             int32_t batch, int32_t t_draft, const float* pool_in,
                             float* pool_out, float* inter, int64_t num_slots,
                             const int32_t* state_idx, void* out, cudaStream_t stream)
{
    RecArgs a;
    a.q = q; a.k = k; a.v = v; a.g_raw = g_raw; a.b_raw = b_raw; a.A_log = A_log; a.dt_bias = dt_bias;
    a.pool_in = pool_in; a.pool_out = pool_out; a.inter = inter; a.state_idx = state_idx; a.out = out;
    a.num_slots = num_slots; a.H = p.num_heads; a.t_draft = t_draft; a.gp = gp;
    a.ring_d = a.ring_k = a.ring_a = nullptr; a.ring_len = 0; a.write_pos = nullptr; a.force_flush = nullptr;
    if (inter != nullptr) return dispatch_dim<kModeVerify>(p, a, batch, stream);
    return dispatch_dim<kModeDecode>(p, a, batch, stream);
}

cudaError_t launch_replay(const kda_params& p, const GateParams& gp, const void* q, const void* k,
                          const void* v, const float* g_raw, const float* b_raw, const float* A_log,
                          const float* dt_bias, int32_t batch, float* pool, int64_t num_slots,
                          const int32_t* state_idx, float* ring_d, float* ring_k, float* ring_a,
                          int32_t ring_len, const int32_t* write_pos, const int32_t* force_flush,
                          void* out, cudaStream_t stream)
{
    RecArgs a;
    a.q = q; a.k = k; a.v = v; a.g_raw = g_raw; a.b_raw = b_raw; a.A_log = A_log; a.dt_bias = dt_bias;
    a.pool_in = pool; a.pool_out = pool; a.inter = nullptr; a.state_idx = state_idx; a.out = out;
    a.num_slots = num_slots; a.H = p.num_heads; a.t_draft = 1; a.gp = gp;
    a.ring_d = ring_d; a.ring_k = ring_k; a.ring_a = ring_a; a.ring_len = ring_len;
    a.write_pos = write_pos; a.force_flush = force_flush;
    return dispatch_dim<kModeReplay>(p, a, batch, stream);
}

namespace {
// One CTA of 256 threads per (request, head): copy the accepted draft's state into the pool slot.
__global__ void __launch_bounds__(256) commit_kernel(const float* __restrict__ inter, int32_t t_draft,
                                                     const int32_t* __restrict__ accept_len, float* pool,
                                                     int64_t num_slots, const int32_t* __restrict__ state_idx,
                                                     int H, int D)
{
    const int64_t bh = blockIdx.x;
    const int64_t b = bh / H;
    const int h = (int)(bh - b * H);
    const int64_t slot = state_idx[b];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (threadIdx.x == 0 && h == 0) record_error(kDevErrStateIndex);
        return;
    }
    const int acc = accept_len[b];
    if (acc < 0 || acc > t_draft) {
        if (threadIdx.x == 0 && h == 0) record_error(kDevErrAcceptLen);
        return;
    }
    if (acc == 0) return;
    const size_t n4 = (size_t)D * D / 4;
    const float4* src = reinterpret_cast<const float4*>(inter + (((size_t)b * t_draft + acc - 1) * H + h) * (size_t)D * D);
    float4* dst = reinterpret_cast<float4*>(pool + ((size_t)slot * H + h) * (size_t)D * D);
    for (size_t i = threadIdx.x; i < n4; i += blockDim.x) __stcs(dst + i, __ldcs(src + i));
}
}  // namespace

cudaError_t launch_commit(int H, int D, const float* inter, int32_t batch, int32_t t_draft,
                          const int32_t* accept_len, float* pool, int64_t num_slots,
                          const int32_t* state_idx, cudaStream_t stream)
{
    const int64_t blocks = (int64_t)batch * H;
    if (blocks <= 0) return cudaSuccess;
    commit_kernel<<<(unsigned)blocks, 256, 0, stream>>>(inter, t_draft, accept_len, pool, num_slots, state_idx, H, D);
    return cudaGetLastError();
}

cudaError_t recurrent_read_and_clear_error(int32_t* code)
{
    int32_t zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(code, g_recurrent_error, sizeof(int32_t));
    if (e != cudaSuccess) return e;
    return cudaMemcpyToSymbol(g_recurrent_error, &zero, sizeof(int32_t));
}

}  // namespace kda
