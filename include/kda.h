/*
 * kda.h -- C ABI of libkda: the KDA (Kimi Delta Attention) gated delta-rule recurrence on
 * NVIDIA GB300 (sm_103a).
 *
 * The recurrence ("linear_attention", zdszero.github.io, section "KDA：逐通道的遗忘门"), per
 * head, with row vectors q_t, k_t in R^{1 x d_k}, v_t in R^{1 x d_v} and state S in R^{d_k x d_v}:
 *
 *     g_t     = -exp(A_log[h]) * softplus(g_raw_t + dt_bias[h])      (one value per key channel)
 *     alpha_t = exp(g_t),  beta_t = sigmoid(b_raw_t)
 *     k_t <- k_t / sqrt(|k_t|^2 + eps),   q_t <- q_t / sqrt(|q_t|^2 + eps) * scale
 *     S_t     = (I - beta_t k_t^T k_t) Diag(alpha_t) S_{t-1} + beta_t k_t^T v_t
 *     o_t     = q_t S_t
 *
 * Conventions shared by every entry point:
 *   - Every tensor pointer is caller-owned DEVICE memory (except `p`, a host struct).  The
 *     library never allocates, frees or keeps a pointer after a call returns.
 *   - Layouts are row-major with no padding:
 *       q, k      [T][H][D]    (io_dtype)        v    [T][H][D]  (io_dtype)
 *       out       [T][H][D]    (out_dtype)
 *       g_raw     [T][H][D] fp32 for the per-channel (KDA) gate, [T][H] fp32 for the per-head
 *                 (GDN) gate;  b_raw [T][H] fp32;  A_log [H] fp32;
 *       dt_bias   [H][D] fp32 (per-channel) or [H] fp32 (per-head); NULL means zero.
 *       state_pool[num_slots][H][D][D] fp32.  Element [s][h][j][c] holds S[c][j] of slot s: the
 *                 state is stored transposed (value row j, key channel c contiguous), as in the
 *                 SGLang pool the pages describe ("linear_attention", section "状态存在哪里").
 *       state_idx [num_seqs] int32: the slot of each sequence/request.  A negative entry marks a
 *                 padding row: its outputs are written as zeros and no state is read or written
 *                 ("ReplaySSM -- buffered output-only decode", yuyanqi.com, section 3.6).  The
 *                 non-negative entries must be distinct.  An entry >= num_slots is treated as
 *                 padding and recorded as a device error (kda_check_device_errors).
 *   - D = d_k = d_v = head_dim.
 *   - q, k, v, g_raw, dt_bias (when given), state_pool, out and the intermediate-state, snapshot
 *     and ring buffers must be 16-byte aligned (KDA_ERR_MISALIGNED otherwise); b_raw, A_log,
 *     cu_seqlens, state_idx and the other int32 tables need only their element alignment.
 *   - All host-side checks (NULL pointers, sizes, alignment, supported shapes) run before any
 *     work is enqueued and return a status without touching memory.  Work is then enqueued on
 *     `stream` and the call returns without synchronising; a launch failure is reported as
 *     KDA_ERR_CUDA.  No call aborts, throws or prints.
 *   - The entry points keep no state between calls beyond device properties looked up once per
 *     process (the driver's tensor-map encoder; the number of CTAs of each recurrent kernel that
 *     fit on a device at once), and may be called from several host threads on different
 *     streams.  Calls on the same state slots must be ordered by the caller.
 */
#ifndef KDA_H
#define KDA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Identical to cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st* kda_stream_t;
/* Identical to cudaEvent_t. */
typedef struct CUevent_st* kda_event_t;

typedef enum kda_status {
    KDA_OK = 0,
    KDA_ERR_INVALID_ARG = -1,  /* NULL pointer, negative size, inconsistent sizes */
    KDA_ERR_UNSUPPORTED = -2,  /* head_dim, chunk_size, dtype or gate combination not built */
    KDA_ERR_MISALIGNED = -3,   /* a tensor pointer is not 16-byte aligned */
    KDA_ERR_WORKSPACE = -4,    /* workspace NULL, too small or not 256-byte aligned */
    KDA_ERR_CUDA = -5,         /* a CUDA runtime call or kernel launch failed */
    KDA_ERR_DEVICE_CHECK = -6, /* kda_check_device_errors found an error a kernel recorded */
    KDA_ERR_SCRATCH_LIMIT = -7 /* the problem needs more scratch than KDA_STATIC_SCRATCH_BYTES */
} kda_status;

typedef enum kda_dtype { KDA_F32 = 0, KDA_BF16 = 1 } kda_dtype;

typedef enum kda_gate_kind {
    KDA_GATE_PER_CHANNEL = 0,  /* KDA: one decay per key channel */
    KDA_GATE_PER_HEAD = 1      /* GDN: one scalar decay per head ("linear_attention", "Gated DeltaNet") */
} kda_gate_kind;

typedef struct kda_params {
    int32_t num_heads;          /* H >= 1 */
    int32_t head_dim;           /* D = d_k = d_v: 16, 32, 64 or 128 */
    int32_t io_dtype;           /* kda_dtype of q, k, v */
    int32_t out_dtype;          /* kda_dtype of out */
    int32_t gate_kind;          /* kda_gate_kind */
    int32_t chunk_size;         /* prefill chunk length: 16, 32 or 64 (<= 64, multiple of 16) */
    int32_t use_lower_bound;    /* 0: g = -exp(A_log) * softplus(x)
                                   1: safe gate g = lower_bound * sigmoid(exp(A_log) * x)
                                   ("linear_attention", section "实例：Kimi K3") */
    float lower_bound;          /* e.g. -5; used when use_lower_bound = 1 */
    float scale;                /* q scale after normalisation; <= 0 selects head_dim^{-1/2} */
    float l2_eps;               /* 1e-6 ("ReplaySSM", section 3.10) */
    float softplus_threshold;   /* 20: softplus(x) = x above it ("PR #26888 report") */
} kda_params;

/* Fill `p` with the pages' defaults: bf16 inputs and output, per-channel gate, chunk 64,
 * no lower bound, scale = head_dim^{-1/2}, eps = 1e-6, softplus threshold 20. */
void kda_params_init(kda_params* p, int32_t num_heads, int32_t head_dim);

/* Static description of a status code (never NULL). */
const char* kda_status_string(int32_t status);

/*
 * Chunkwise-parallel prefill over packed varlen sequences ("linear_attention", sections
 * "矩阵（并行）形式" and "两种计算形态"; the interface mirrors chunk_kda of "KDA inference
 * components", section 4.1, with the gate activation and the q/k L2 norm always fused).
 *
 * Sequence i holds tokens cu_seqlens[i] .. cu_seqlens[i+1]-1 of the packed [T][H][..] inputs
 * and starts from state_pool[state_idx[i]]; the final state is written back to the same slot.
 * Each sequence is cut into chunks of p->chunk_size tokens starting at its first token.
 *   cu_seqlens    device int32 [num_seqs + 1], non-decreasing, cu_seqlens[0] = 0,
 *                 cu_seqlens[num_seqs] = total_tokens.  Never read back to the host; a malformed
 *                 table is clamped and recorded as a device error.
 *   total_tokens  0 <= T < 2^31 - 64 (the number of rows of q, k, v, g_raw, b_raw, out); a
 *                 larger T returns KDA_ERR_UNSUPPORTED.
 *   workspace     device scratch of at least kda_chunk_prefill_workspace_size(...) bytes,
 *                 256-byte aligned, owned by the caller; its contents need not be initialised
 *                 and are garbage afterwards.  It must not be shared with a call that overlaps
 *                 in time.
 * T = 0 or num_seqs = 0 is a no-op.
 */
size_t kda_chunk_prefill_workspace_size(const kda_params* p, int32_t num_seqs, int64_t total_tokens);

int32_t kda_chunk_prefill(const kda_params* p,
                          const void* q, const void* k, const void* v,
                          const float* g_raw, const float* b_raw,
                          const float* A_log, const float* dt_bias,
                          const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                          float* state_pool, int64_t num_slots, const int32_t* state_idx,
                          void* out,
                          void* workspace, size_t workspace_bytes,
                          kda_stream_t stream);

/*
 * kda_chunk_prefill with per-phase timing: the same work, plus caller-created CUDA events
 * recorded on `stream` around its kernels: events[0] before the chunk-table kernel, events[1]
 * after it, events[2] after the intra-chunk kernel, events[3] after the inter-chunk state pass.
 * `events` must hold KDA_PREFILL_PHASE_EVENTS valid event handles (owned by the caller).
 */
#define KDA_PREFILL_PHASE_EVENTS 4
int32_t kda_chunk_prefill_timed(const kda_params* p,
                                const void* q, const void* k, const void* v,
                                const float* g_raw, const float* b_raw,
                                const float* A_log, const float* dt_bias,
                                const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                float* state_pool, int64_t num_slots, const int32_t* state_idx,
                                void* out,
                                void* workspace, size_t workspace_bytes,
                                kda_stream_t stream, kda_event_t const* events);

/*
 * Single-token recurrent decode against the pooled state, updated in place ("linear_attention",
 * section "两种计算形态", the fused recurrent kernel; per-token steps of section "Gated DeltaNet":
 * decay, predict, error, write, read).  Request b is token b of the [batch][H][..] inputs.
 */
int32_t kda_recurrent_decode(const kda_params* p,
                             const void* q, const void* k, const void* v,
                             const float* g_raw, const float* b_raw,
                             const float* A_log, const float* dt_bias,
                             int32_t batch,
                             float* state_pool, int64_t num_slots, const int32_t* state_idx,
                             void* out,
                             kda_stream_t stream);

/*
 * Buffered single-token decode ("ReplaySSM -- buffered output-only decode", sections 2, 3 and 5):
 * the slot's state is kept as a checkpoint in state_pool plus a ring of the steps taken since,
 * and the state before the current token is rebuilt as
 *     S = Diag(prod_j a_j) S_checkpoint + sum_j (k_j o prod_{i>j} a_i)^T d_j   (j < write_pos[b])
 * The token then takes the same decode step as kda_recurrent_decode (its output is that of the
 * plain recurrence).  A non-flush step appends (d, k_hat, a) of this token at ring position
 * write_pos[b] and leaves the checkpoint untouched; a flush step (write_pos[b] == ring_len - 1,
 * or force_flush[b] != 0) writes the new state into the checkpoint instead.  The caller then
 * advances the cursor of the slot: 0 after a flush, write_pos + 1 otherwise; a new or copied slot
 * starts at 0 (an empty ring).
 *   ring_d   device fp32 [num_slots][H][ring_len][D]   corrected deltas d = beta (v - v_hat)
 *   ring_k   device fp32 [num_slots][H][ring_len][D]   normalised keys
 *   ring_a   device fp32 [num_slots][H][ring_len][D] (per-channel gate) or
 *            [num_slots][H][ring_len] (per-head gate)    decays a = e^{g} (not g: products of
 *            factors <= 1 keep the rebuild exact to fp32 rounding)
 *   write_pos  device int32 [batch] in [0, ring_len); outside it the row is treated as padding
 *            and recorded as device error 5.  force_flush: device int32 [batch] or NULL.
 *   1 <= ring_len <= 32.  With ring_len = 1 every step flushes and the call computes exactly
 *   what kda_recurrent_decode computes.
 */
int32_t kda_replay_decode(const kda_params* p,
                          const void* q, const void* k, const void* v,
                          const float* g_raw, const float* b_raw,
                          const float* A_log, const float* dt_bias,
                          int32_t batch,
                          float* state_pool, int64_t num_slots, const int32_t* state_idx,
                          float* ring_d, float* ring_k, float* ring_a, int32_t ring_len,
                          const int32_t* write_pos, const int32_t* force_flush,
                          void* out,
                          kda_stream_t stream);

/*
 * Multi-token verify ("PR #26888 report": target_verify with disable_state_update and an
 * intermediate-state buffer; "linear_attention", section "prefix cache 与投机解码").
 * Request b owns tokens b*t_draft .. b*t_draft + t_draft - 1 of the inputs (request-major).
 * The pool is only read.  The state after draft token t of request b is written to
 *   inter_states [batch][t_draft][H][D][D] fp32 (same transposed layout as the pool),
 * and out is [batch * t_draft][H][D].  Padding rows (state_idx < 0) write zero outputs and
 * leave their inter_states untouched.  1 <= t_draft <= 16.
 */
int32_t kda_recurrent_verify(const kda_params* p,
                             const void* q, const void* k, const void* v,
                             const float* g_raw, const float* b_raw,
                             const float* A_log, const float* dt_bias,
                             int32_t batch, int32_t t_draft,
                             const float* state_pool, int64_t num_slots, const int32_t* state_idx,
                             float* inter_states, void* out,
                             kda_stream_t stream);

/*
 * kda_chunk_prefill that also keeps the state at every chunk boundary, the snapshots a prefix
 * cache stores ("linear_attention", section "两种计算形态": the state h at each chunk boundary is
 * materialised; section "prefix cache 与投机解码").
 *   chunk_states   device fp32 [num_chunks][H][D][D] (transposed like the pool), where chunk
 *                  c = seq_chunk_offset(i) + m is chunk m of sequence i, seq_chunk_offset(i) =
 *                  sum_{j<i} ceil(len_j / chunk_size), num_chunks = seq_chunk_offset(num_seqs).
 *                  Entry c holds the state after chunk c (prefix length (m + 1) * chunk_size,
 *                  or the whole sequence for its last chunk).  Padding rows write nothing.
 *   chunk_states_capacity  number of [H][D][D] entries the buffer holds; a table that needs more
 *                  entries is recorded as device error 2 and the extra snapshots are dropped.
 * Everything else is as kda_chunk_prefill.
 */
int32_t kda_chunk_prefill_snapshots(const kda_params* p,
                                    const void* q, const void* k, const void* v,
                                    const float* g_raw, const float* b_raw,
                                    const float* A_log, const float* dt_bias,
                                    const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens,
                                    float* state_pool, int64_t num_slots, const int32_t* state_idx,
                                    void* out,
                                    void* workspace, size_t workspace_bytes,
                                    float* chunk_states, int64_t chunk_states_capacity,
                                    kda_stream_t stream);

/*
 * Commit accepted drafts after kda_recurrent_verify ("linear_attention", section "prefix cache 与
 * 投机解码": after acceptance the intermediate state of the accepted length is scattered back to
 * the pool).  For request b with a = accept_len[b] (device int32 [batch]): 1 <= a <= t_draft copies
 * inter_states[b][a - 1] into state_pool[state_idx[b]]; a = 0 leaves the slot unchanged; a padding
 * row (state_idx < 0) is skipped.  An accept_len outside [0, t_draft] or a slot >= num_slots is
 * skipped and recorded as device error 4 or 1.  The buffers may not overlap.
 */
int32_t kda_commit_verified_states(const kda_params* p,
                                   const float* inter_states, int32_t batch, int32_t t_draft,
                                   const int32_t* accept_len,
                                   float* state_pool, int64_t num_slots, const int32_t* state_idx,
                                   kda_stream_t stream);

/*
 * kda_chunk_prefill for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point; it exists for the library's users.
 *
 * Who needs it: code that may not call cudaMalloc or any allocator, for example a plugin inside
 * a serving process that has already handed all device memory to its own pools, a runtime with
 * no binding to a CUDA allocator, or a latency-critical loop that must not risk the device-wide
 * synchronisation a cudaMalloc can cause.  Such a caller cannot provide the workspace that
 * kda_chunk_prefill asks for.
 *
 * What it does: exactly the work of kda_chunk_prefill, with the same arguments minus the
 * workspace, and the same host-side checks.  Its scratch is a fixed array of
 * KDA_STATIC_SCRATCH_BYTES compiled into the library.  A device holds that much memory for it
 * until its context is destroyed (normally at process exit): under CUDA's default lazy module
 * loading from the first call of this entry point on that device, under eager loading
 * (CUDA_MODULE_LOADING=EAGER) from the creation of the context.  The call allocates nothing.
 * A problem whose kda_chunk_prefill_workspace_size(...) exceeds KDA_STATIC_SCRATCH_BYTES is
 * rejected with KDA_ERR_SCRATCH_LIMIT before any work is enqueued
 * (with bf16 inputs, H = 32, head_dim = 128, chunk 64 the array covers ceil(T / 64) + num_seqs
 * <= 112 chunks, about 7,000 tokens per call).
 *
 * Every call looks up the device address of the array in the current context (nothing is
 * cached, so a context that was reset and created again is handled); under lazy loading the
 * first call on a device also loads the library's device code there, so make that first call
 * outside any stream capture.  All calls share the one array and it keeps whatever the last
 * call left in it (nothing in it needs to start at zero).  Calls whose kernels overlap on the
 * GPU, on different streams or from different host threads, race on the array and produce
 * garbage: order them.
 */
#define KDA_STATIC_SCRATCH_BYTES ((size_t)256 << 20)
int32_t kda_chunk_prefill_static_scratch(const kda_params* p,
                                         const void* q, const void* k, const void* v,
                                         const float* g_raw, const float* b_raw,
                                         const float* A_log, const float* dt_bias,
                                         const int32_t* cu_seqlens, int32_t num_seqs,
                                         int64_t total_tokens,
                                         float* state_pool, int64_t num_slots,
                                         const int32_t* state_idx,
                                         void* out,
                                         kda_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the device error word that the kernels set when
 * they meet an out-of-range state_idx (code 1), a malformed cu_seqlens or a snapshot table too
 * small for it (code 2), a bounded wait inside a kernel that gave up (code 3; that call's
 * results are invalid), an accept_len outside [0, t_draft] (code 4) or a replay write_pos
 * outside [0, ring_len) (code 5).  *code receives
 * the first recorded code (0 when none) for the current device.  Returns KDA_OK when no error was
 * recorded, KDA_ERR_DEVICE_CHECK when one was, KDA_ERR_CUDA when the synchronisation failed.
 */
int32_t kda_check_device_errors(kda_stream_t stream, int32_t* code);

/*
 * Failure-detection self-test of the bounded waits in the tensor-core kernels.  Enqueues one
 * warp on `stream` that allocates 32 TMEM columns, waits with a limit of `polls` polls on an
 * mbarrier that nothing arrives on, records device error 3 (timeout) when the wait gives up,
 * then takes the same exit path as the prefill kernels after a timeout: commit to a second
 * mbarrier and wait for it (again at most `polls` polls), free TMEM, return.  No fault, trap or
 * unbounded loop is involved, and the context stays usable.
 *   polls   in [1, 1 << 24]; one poll is one mbarrier try_wait.
 *   result  NULL, or caller-owned device int32[2]: result[0] = 1 if the first wait completed
 *           (it never should), result[1] = 1 if the drain completed.  Written by the kernel.
 * Returns KDA_OK when the kernel was enqueued, KDA_ERR_INVALID_ARG for polls outside the range,
 * KDA_ERR_MISALIGNED when result is not 4-byte aligned, KDA_ERR_CUDA when the launch failed.
 * kda_check_device_errors then reports code 3.
 */
int32_t kda_selftest_wait_timeout(uint32_t polls, int32_t* result, kda_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_H */
