// kda_api.cu -- the extern "C" entry points of libkda (declared in include/kda.h): host-side
// argument validation, then dispatch to the kernels of kda_recurrent.cu and kda_prefill.cu.
// Nothing here allocates memory, synchronises (except kda_check_device_errors) or keeps state.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kda.h"
#include "kda_internal.cuh"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by all entry points; `tokens` is the number of input rows.
int32_t check_common(const kda_params* p, const void* q, const void* k, const void* v,
                     const float* g_raw, const float* b_raw, const float* A_log,
                     const float* dt_bias, int64_t tokens, const void* pool, int64_t num_slots,
                     const int32_t* state_idx, const void* out)
{
    if (!p) return KDA_ERR_INVALID_ARG;
    if (p->num_heads <= 0 || p->head_dim <= 0 || tokens < 0 || num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (!(p->l2_eps >= 0.f) || !(p->softplus_threshold == p->softplus_threshold)) return KDA_ERR_INVALID_ARG;
    if (tokens == 0) return KDA_OK;
    if (!q || !k || !v || !g_raw || !b_raw || !A_log || !pool || !state_idx || !out) return KDA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g_raw) || !aligned16(pool) ||
        !aligned16(out) || (dt_bias && !aligned16(dt_bias)))
        return KDA_ERR_MISALIGNED;
    (void)b_raw;
    return KDA_OK;
}

int32_t from_cuda(cudaError_t e) { return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA; }

using kda::gate_params;

}  // namespace

namespace kda {

GateParams gate_params(const kda_params& p)
{
    GateParams g;
    g.scale = p.scale > 0.f ? p.scale : 1.0f / sqrtf((float)p.head_dim);
    g.l2_eps = p.l2_eps;
    g.softplus_threshold = p.softplus_threshold;
    g.lower_bound = p.lower_bound;
    g.use_lower_bound = p.use_lower_bound ? 1 : 0;
    return g;
}

int32_t check_prefill(const kda_params* p, const void* q, const void* k, const void* v, const float* g_raw,
                      const float* b_raw, const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
                      int32_t num_seqs, int64_t total_tokens, const void* state_pool, int64_t num_slots,
                      const int32_t* state_idx, const void* out, bool* noop)
{
    *noop = false;
    if (num_seqs < 0) return KDA_ERR_INVALID_ARG;
    const int32_t rc = check_common(p, q, k, v, g_raw, b_raw, A_log, dt_bias, total_tokens, state_pool,
                                    num_slots, state_idx, out);
    if (rc != KDA_OK) return rc;
    if (!prefill_supported(*p)) return KDA_ERR_UNSUPPORTED;
    if (total_tokens == 0 || num_seqs == 0) {
        *noop = true;
        return KDA_OK;
    }
    if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (total_tokens >= ((int64_t)1 << 31) - 64) return KDA_ERR_UNSUPPORTED;
    return KDA_OK;
}

}  // namespace kda

extern "C" {

void kda_params_init(kda_params* p, int32_t num_heads, int32_t head_dim)
{
    if (!p) return;
    p->num_heads = num_heads;
    p->head_dim = head_dim;
    p->io_dtype = KDA_BF16;
    p->out_dtype = KDA_BF16;
    p->gate_kind = KDA_GATE_PER_CHANNEL;
    p->chunk_size = 64;
    p->use_lower_bound = 0;
    p->lower_bound = -5.0f;
    p->scale = 0.0f;
    p->l2_eps = 1e-6f;
    p->softplus_threshold = 20.0f;
}

const char* kda_status_string(int32_t status)
{
    switch (status) {
    case KDA_OK: return "ok";
    case KDA_ERR_INVALID_ARG: return "invalid argument";
    case KDA_ERR_UNSUPPORTED: return "unsupported head_dim, chunk_size, dtype or gate combination";
    case KDA_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
    case KDA_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case KDA_ERR_CUDA: return "CUDA runtime error";
    case KDA_ERR_DEVICE_CHECK: return "a kernel recorded an error (bad state_idx, cu_seqlens, accept_len or write_pos, or a bounded wait that gave up)";
    case KDA_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the library's fixed scratch array holds";
    default: return "unknown status";
    }
}

size_t kda_chunk_prefill_workspace_size(const kda_params* p, int32_t num_seqs, int64_t total_tokens)
{
    if (!p || num_seqs < 0 || total_tokens < 0 || !kda::prefill_supported(*p) || p->num_heads <= 0) return 0;
    return kda::prefill_workspace_bytes(*p, num_seqs, total_tokens);
}

namespace {
int32_t prefill_impl(const kda_params* p, const void* q, const void* k, const void* v,
                     const float* g_raw, const float* b_raw, const float* A_log,
                     const float* dt_bias, const int32_t* cu_seqlens, int32_t num_seqs,
                     int64_t total_tokens, float* state_pool, int64_t num_slots,
                     const int32_t* state_idx, void* out, void* workspace,
                     size_t workspace_bytes, kda_stream_t stream, const cudaEvent_t* events,
                     float* chunk_states = nullptr, int64_t chunk_states_capacity = 0)
{
    bool noop = false;
    const int32_t rc = kda::check_prefill(p, q, k, v, g_raw, b_raw, A_log, dt_bias, cu_seqlens, num_seqs,
                                          total_tokens, state_pool, num_slots, state_idx, out, &noop);
    if (rc != KDA_OK || noop) return rc;
    const size_t need = kda::prefill_workspace_bytes(*p, num_seqs, total_tokens);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return KDA_ERR_WORKSPACE;
    return from_cuda(kda::launch_prefill(*p, gate_params(*p), q, k, v, g_raw, b_raw, A_log, dt_bias,
                                         cu_seqlens, num_seqs, total_tokens, state_pool, num_slots,
                                         state_idx, out, workspace, (cudaStream_t)stream, events,
                                         chunk_states, chunk_states_capacity));
}
}  // namespace

int32_t kda_chunk_prefill(const kda_params* p, const void* q, const void* k, const void* v,
                          const float* g_raw, const float* b_raw, const float* A_log,
                          const float* dt_bias, const int32_t* cu_seqlens, int32_t num_seqs,
                          int64_t total_tokens, float* state_pool, int64_t num_slots,
                          const int32_t* state_idx, void* out, void* workspace,
                          size_t workspace_bytes, kda_stream_t stream)
{
    return prefill_impl(p, q, k, v, g_raw, b_raw, A_log, dt_bias, cu_seqlens, num_seqs, total_tokens,
                        state_pool, num_slots, state_idx, out, workspace, workspace_bytes, stream, nullptr);
}

int32_t kda_chunk_prefill_timed(const kda_params* p, const void* q, const void* k, const void* v,
                                const float* g_raw, const float* b_raw, const float* A_log,
                                const float* dt_bias, const int32_t* cu_seqlens, int32_t num_seqs,
                                int64_t total_tokens, float* state_pool, int64_t num_slots,
                                const int32_t* state_idx, void* out, void* workspace,
                                size_t workspace_bytes, kda_stream_t stream, kda_event_t const* events)
{
    if (!events) return KDA_ERR_INVALID_ARG;
    for (int i = 0; i < KDA_PREFILL_PHASE_EVENTS; ++i)
        if (!events[i]) return KDA_ERR_INVALID_ARG;
    return prefill_impl(p, q, k, v, g_raw, b_raw, A_log, dt_bias, cu_seqlens, num_seqs, total_tokens,
                        state_pool, num_slots, state_idx, out, workspace, workspace_bytes, stream,
                        reinterpret_cast<const cudaEvent_t*>(events));
}

int32_t kda_chunk_prefill_snapshots(const kda_params* p, const void* q, const void* k, const void* v,
                                    const float* g_raw, const float* b_raw, const float* A_log,
                                    const float* dt_bias, const int32_t* cu_seqlens, int32_t num_seqs,
                                    int64_t total_tokens, float* state_pool, int64_t num_slots,
                                    const int32_t* state_idx, void* out, void* workspace,
                                    size_t workspace_bytes, float* chunk_states,
                                    int64_t chunk_states_capacity, kda_stream_t stream)
{
    if (!chunk_states || chunk_states_capacity < 0) return KDA_ERR_INVALID_ARG;
    if (!aligned16(chunk_states)) return KDA_ERR_MISALIGNED;
    return prefill_impl(p, q, k, v, g_raw, b_raw, A_log, dt_bias, cu_seqlens, num_seqs, total_tokens,
                        state_pool, num_slots, state_idx, out, workspace, workspace_bytes, stream, nullptr,
                        chunk_states, chunk_states_capacity);
}

int32_t kda_commit_verified_states(const kda_params* p, const float* inter_states, int32_t batch,
                                   int32_t t_draft, const int32_t* accept_len, float* state_pool,
                                   int64_t num_slots, const int32_t* state_idx, kda_stream_t stream)
{
    if (!p || batch < 0 || t_draft < 1 || t_draft > 16 || num_slots < 0 || p->num_heads <= 0)
        return KDA_ERR_INVALID_ARG;
    if (!kda::recurrent_supported(*p)) return KDA_ERR_UNSUPPORTED;
    if (batch == 0) return KDA_OK;
    if (!inter_states || !accept_len || !state_pool || !state_idx) return KDA_ERR_INVALID_ARG;
    if (!aligned16(inter_states) || !aligned16(state_pool)) return KDA_ERR_MISALIGNED;
    return from_cuda(kda::launch_commit(p->num_heads, p->head_dim, inter_states, batch, t_draft, accept_len,
                                        state_pool, num_slots, state_idx, (cudaStream_t)stream));
}

int32_t kda_recurrent_decode(const kda_params* p, const void* q, const void* k, const void* v,
                             const float* g_raw, const float* b_raw, const float* A_log,
                             const float* dt_bias, int32_t batch, float* state_pool,
                             int64_t num_slots, const int32_t* state_idx, void* out,
                             kda_stream_t stream)
{
    if (batch < 0) return KDA_ERR_INVALID_ARG;
    int32_t rc = check_common(p, q, k, v, g_raw, b_raw, A_log, dt_bias, batch, state_pool,
                              num_slots, state_idx, out);
    if (rc != KDA_OK) return rc;
    if (!kda::recurrent_supported(*p)) return KDA_ERR_UNSUPPORTED;
    if (batch == 0) return KDA_OK;
    return from_cuda(kda::launch_recurrent(*p, gate_params(*p), q, k, v, g_raw, b_raw, A_log, dt_bias,
                                           batch, 1, state_pool, state_pool, nullptr, num_slots,
                                           state_idx, out, (cudaStream_t)stream));
}

int32_t kda_replay_decode(const kda_params* p, const void* q, const void* k, const void* v,
                          const float* g_raw, const float* b_raw, const float* A_log,
                          const float* dt_bias, int32_t batch, float* state_pool, int64_t num_slots,
                          const int32_t* state_idx, float* ring_d, float* ring_k, float* ring_a,
                          int32_t ring_len, const int32_t* write_pos, const int32_t* force_flush,
                          void* out, kda_stream_t stream)
{
    if (batch < 0 || ring_len < 1 || ring_len > 32) return KDA_ERR_INVALID_ARG;
    int32_t rc = check_common(p, q, k, v, g_raw, b_raw, A_log, dt_bias, batch, state_pool,
                              num_slots, state_idx, out);
    if (rc != KDA_OK) return rc;
    if (!kda::recurrent_supported(*p)) return KDA_ERR_UNSUPPORTED;
    if (batch == 0) return KDA_OK;
    if (!ring_d || !ring_k || !ring_a || !write_pos) return KDA_ERR_INVALID_ARG;
    if (!aligned16(ring_d) || !aligned16(ring_k) || !aligned16(ring_a)) return KDA_ERR_MISALIGNED;
    return from_cuda(kda::launch_replay(*p, gate_params(*p), q, k, v, g_raw, b_raw, A_log, dt_bias, batch,
                                        state_pool, num_slots, state_idx, ring_d, ring_k, ring_a, ring_len,
                                        write_pos, force_flush, out, (cudaStream_t)stream));
}

int32_t kda_recurrent_verify(const kda_params* p, const void* q, const void* k, const void* v,
                             const float* g_raw, const float* b_raw, const float* A_log,
                             const float* dt_bias, int32_t batch, int32_t t_draft,
                             const float* state_pool, int64_t num_slots,
                             const int32_t* state_idx, float* inter_states, void* out,
                             kda_stream_t stream)
{
    if (batch < 0 || t_draft < 1 || t_draft > 16) return KDA_ERR_INVALID_ARG;
    int32_t rc = check_common(p, q, k, v, g_raw, b_raw, A_log, dt_bias, (int64_t)batch * t_draft,
                              state_pool, num_slots, state_idx, out);
    if (rc != KDA_OK) return rc;
    if (!kda::recurrent_supported(*p)) return KDA_ERR_UNSUPPORTED;
    if (batch == 0) return KDA_OK;
    if (!inter_states) return KDA_ERR_INVALID_ARG;
    if (!aligned16(inter_states)) return KDA_ERR_MISALIGNED;
    return from_cuda(kda::launch_recurrent(*p, gate_params(*p), q, k, v, g_raw, b_raw, A_log, dt_bias,
                                           batch, t_draft, state_pool, nullptr, inter_states,
                                           num_slots, state_idx, out, (cudaStream_t)stream));
}

int32_t kda_check_device_errors(kda_stream_t stream, int32_t* code)
{
    if (!code) return KDA_ERR_INVALID_ARG;
    *code = 0;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return KDA_ERR_CUDA;
    int32_t c1 = 0, c2 = 0, c3 = 0;
    if (kda::recurrent_read_and_clear_error(&c1) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::prefill_read_and_clear_error(&c2) != cudaSuccess) return KDA_ERR_CUDA;
    if (kda::selftest_read_and_clear_error(&c3) != cudaSuccess) return KDA_ERR_CUDA;
    *code = c1 ? c1 : (c2 ? c2 : c3);
    return *code ? KDA_ERR_DEVICE_CHECK : KDA_OK;
}

int32_t kda_selftest_wait_timeout(uint32_t polls, int32_t* result, kda_stream_t stream)
{
    if (polls < 1u || polls > (1u << 24)) return KDA_ERR_INVALID_ARG;
    if (result && (reinterpret_cast<uintptr_t>(result) & 3u)) return KDA_ERR_MISALIGNED;
    return from_cuda(kda::launch_wait_selftest(polls, result, (cudaStream_t)stream));
}

}  // extern "C"
