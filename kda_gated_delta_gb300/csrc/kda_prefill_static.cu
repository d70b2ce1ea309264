// kda_prefill_static.cu -- kda_chunk_prefill_static_scratch: the chunk prefill for callers that
// cannot allocate device memory.
//
// The ordinary kda_chunk_prefill asks its caller for a workspace buffer.  Some callers have no
// way to get one: a plugin loaded into a serving process whose device memory is all reserved
// up front (state pools, KV caches) and handed out by someone else; a runtime with no binding to
// a CUDA allocator; a latency-critical loop that must not call cudaMalloc because that call can
// synchronise the whole device.  This entry point needs no workspace from the caller: its
// scratch is one array of fixed size compiled into the library (kda_static_scratch below), so
// every GPU that loads libkda holds KDA_STATIC_SCRATCH_BYTES of device memory for that array
// until the process exits.
//
// In host code the name kda_static_scratch is only a host-side handle for the device symbol,
// not a device address, so the address is looked up with cudaGetSymbolAddress, once per device,
// with that device current (the first call of this entry point on each device does it), and is
// then passed to the kernels like any other workspace pointer.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "kda.h"
#include "kda_internal.cuh"

namespace {

// The scratch shared by every call of kda_chunk_prefill_static_scratch on a device.
static __device__ __align__(256) unsigned char kda_static_scratch[KDA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of kda_static_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, kda_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int32_t kda_chunk_prefill_static_scratch(
    const kda_params* p, const void* q, const void* k, const void* v, const float* g_raw,
    const float* b_raw, const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
    int32_t num_seqs, int64_t total_tokens, float* state_pool, int64_t num_slots,
    const int32_t* state_idx, void* out, kda_stream_t stream)
{
    // Same host-side checks as kda_chunk_prefill, in the same order.
    if (!p || num_seqs < 0 || total_tokens < 0 || num_slots < 0 || p->num_heads <= 0 || p->head_dim <= 0)
        return KDA_ERR_INVALID_ARG;
    if (!(p->l2_eps >= 0.f) || !(p->softplus_threshold == p->softplus_threshold)) return KDA_ERR_INVALID_ARG;
    if (total_tokens > 0) {
        if (!q || !k || !v || !g_raw || !b_raw || !A_log || !state_pool || !state_idx || !out)
            return KDA_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(g_raw) || !aligned16(state_pool) ||
            !aligned16(out) || (dt_bias && !aligned16(dt_bias)))
            return KDA_ERR_MISALIGNED;
    }
    if (!kda::prefill_supported(*p)) return KDA_ERR_UNSUPPORTED;
    if (total_tokens == 0 || num_seqs == 0) return KDA_OK;
    if (!cu_seqlens) return KDA_ERR_INVALID_ARG;
    if (total_tokens >= ((int64_t)1 << 31) - 64) return KDA_ERR_UNSUPPORTED;
    // The problem must fit the fixed array; nothing is allocated to make room.
    const size_t need = kda::prefill_workspace_bytes(*p, num_seqs, total_tokens);
    if (need > (size_t)KDA_STATIC_SCRATCH_BYTES) return KDA_ERR_SCRATCH_LIMIT;

    kda::GateParams gp;
    gp.scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->head_dim);
    gp.l2_eps = p->l2_eps;
    gp.softplus_threshold = p->softplus_threshold;
    gp.lower_bound = p->lower_bound;
    gp.use_lower_bound = p->use_lower_bound ? 1 : 0;

    void* scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KDA_ERR_CUDA;
    // Nothing in the scratch has to start at zero: the chunk-table kernel writes every entry the
    // later kernels read, and each per-chunk record is written before it is read.
    const cudaError_t e = kda::launch_prefill(*p, gp, q, k, v, g_raw, b_raw, A_log, dt_bias, cu_seqlens,
                                              num_seqs, total_tokens, state_pool, num_slots, state_idx,
                                              out, scratch, (cudaStream_t)stream);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
