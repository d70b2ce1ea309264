// kda_prefill_static.cu -- kda_chunk_prefill_static_scratch: the chunk prefill for callers that
// cannot allocate device memory.
//
// The ordinary kda_chunk_prefill asks its caller for a workspace buffer.  Some callers have no
// way to get one: a plugin loaded into a serving process whose device memory is all reserved
// up front (state pools, KV caches) and handed out by someone else; a runtime with no binding to
// a CUDA allocator; a latency-critical loop that must not call cudaMalloc because that call can
// synchronise the whole device.  This entry point needs no workspace from the caller: its
// scratch is one array of fixed size compiled into the library (kda_static_scratch below).
// With CUDA's default lazy module loading a device holds the KDA_STATIC_SCRATCH_BYTES of that
// array from the first call of this entry point on it (the address lookup loads the module);
// with eager loading (CUDA_MODULE_LOADING=EAGER) from the creation of the context.  Either way
// it is held until the context is destroyed, normally at process exit.
//
// In host code the name kda_static_scratch is only a host-side handle for the device symbol,
// not a device address.  Every call looks the address up with cudaGetSymbolAddress on the
// current device and passes it to the kernels like any other workspace pointer.  Nothing is
// cached between calls, so a context that was torn down and created again (cudaDeviceReset, a
// reloaded module) can never leave a stale address behind.
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"
#include "kda_internal.cuh"

namespace {

// The scratch shared by every call of kda_chunk_prefill_static_scratch on a device.
static __device__ __align__(256) unsigned char kda_static_scratch[KDA_STATIC_SCRATCH_BYTES];

}  // namespace

extern "C" int32_t kda_chunk_prefill_static_scratch(
    const kda_params* p, const void* q, const void* k, const void* v, const float* g_raw,
    const float* b_raw, const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
    int32_t num_seqs, int64_t total_tokens, float* state_pool, int64_t num_slots,
    const int32_t* state_idx, void* out, kda_stream_t stream)
{
    // The same host-side checks as kda_chunk_prefill (one shared helper), then the size check
    // against the fixed array instead of the workspace check.
    bool noop = false;
    const int32_t rc = kda::check_prefill(p, q, k, v, g_raw, b_raw, A_log, dt_bias, cu_seqlens, num_seqs,
                                          total_tokens, state_pool, num_slots, state_idx, out, &noop);
    if (rc != KDA_OK || noop) return rc;
    // The problem must fit the fixed array; nothing is allocated to make room.
    const size_t need = kda::prefill_workspace_bytes(*p, num_seqs, total_tokens);
    if (need > (size_t)KDA_STATIC_SCRATCH_BYTES) return KDA_ERR_SCRATCH_LIMIT;

    // Device address of the array in the current device's context, looked up on every call.
    void* scratch = nullptr;
    if (cudaGetSymbolAddress(&scratch, kda_static_scratch) != cudaSuccess || scratch == nullptr)
        return KDA_ERR_CUDA;
    // Nothing in the scratch has to start at zero: the chunk-table kernel writes every entry the
    // later kernels read, and each per-chunk record is written before it is read.
    const cudaError_t e = kda::launch_prefill(*p, kda::gate_params(*p), q, k, v, g_raw, b_raw, A_log, dt_bias,
                                              cu_seqlens, num_seqs, total_tokens, state_pool, num_slots,
                                              state_idx, out, scratch, (cudaStream_t)stream);
    return e == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
