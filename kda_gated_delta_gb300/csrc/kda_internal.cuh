// kda_internal.cuh -- device helpers and launcher declarations shared by libkda's translation
// units.  Not part of the public ABI (include/kda.h is).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

// Device-side argument errors recorded by the kernels (first code wins).
enum DeviceError : int32_t {
    kDevErrNone = 0,
    kDevErrStateIndex = 1,   // state_idx[i] >= num_slots
    kDevErrSeqlens = 2,      // cu_seqlens not non-decreasing within [0, T]
    kDevErrTimeout = 3,      // a bounded wait inside a kernel gave up (the call's results are invalid)
    kDevErrAcceptLen = 4,    // accept_len outside [0, t_draft]
    kDevErrWritePos = 5,     // replay write_pos outside [0, ring_len)
};

// Scalar parameters every kernel needs, resolved on the host from kda_params.
struct GateParams {
    float scale;              // q scale after normalisation
    float l2_eps;
    float softplus_threshold;
    float lower_bound;
    int use_lower_bound;
};

// ---- element loads ---------------------------------------------------------------------------
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// ---- gate activation -------------------------------------------------------------------------
// softplus with the pages' guard: x above the threshold is returned as is, else log(1 + e^x)
// ("ReplaySSM -- buffered output-only decode", section 3.8).
__device__ __forceinline__ float softplus_f32(float x, float threshold) {
    return x > threshold ? x : log1pf(expf(x));
}

// Log-space decay g of one channel.  Default gate ("linear_attention", "Gated DeltaNet"/"KDA"):
//   g = -exp(A_log) * softplus(x);   safe gate ("linear_attention", "实例：Kimi K3"):
//   g = lower_bound * sigmoid(exp(A_log) * x),   with x = g_raw + dt_bias.
__device__ __forceinline__ float gate_log_decay(float x, float rate, const GateParams& gp) {
    if (gp.use_lower_bound) {
        return gp.lower_bound / (1.0f + expf(-rate * x));
    }
    return -rate * softplus_f32(x, gp.softplus_threshold);
}

__device__ __forceinline__ float sigmoid_f32(float x) { return 1.0f / (1.0f + expf(-x)); }

// ---- host-side argument handling (kda_api.cu) ----------------------------------------------------
GateParams gate_params(const kda_params& p);
// The host-side checks of a chunk-prefill call, in one place for every prefill entry point (the
// caller-workspace variants and the static-scratch one), so that they cannot drift apart.
// Returns KDA_OK or the negative status of the first failed check; *noop is set when the call is
// valid but has nothing to do (T = 0 or num_seqs = 0).  The workspace or scratch size is checked
// by the caller, after this.
int32_t check_prefill(const kda_params* p, const void* q, const void* k, const void* v, const float* g_raw,
                      const float* b_raw, const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
                      int32_t num_seqs, int64_t total_tokens, const void* state_pool, int64_t num_slots,
                      const int32_t* state_idx, const void* out, bool* noop);

// ---- launchers (implemented in kda_recurrent.cu / kda_prefill.cu) ------------------------------
cudaError_t launch_recurrent(const kda_params& p, const GateParams& gp, const void* q,
                             const void* k, const void* v, const float* g_raw,
                             const float* b_raw, const float* A_log, const float* dt_bias,
                             int32_t batch, int32_t t_draft, const float* pool_in,
                             float* pool_out, float* inter, int64_t num_slots,
                             const int32_t* state_idx, void* out, cudaStream_t stream);
bool recurrent_supported(const kda_params& p);
cudaError_t recurrent_read_and_clear_error(int32_t* code);
cudaError_t launch_replay(const kda_params& p, const GateParams& gp, const void* q, const void* k,
                          const void* v, const float* g_raw, const float* b_raw, const float* A_log,
                          const float* dt_bias, int32_t batch, float* pool, int64_t num_slots,
                          const int32_t* state_idx, float* ring_d, float* ring_k, float* ring_a,
                          int32_t ring_len, const int32_t* write_pos, const int32_t* force_flush,
                          void* out, cudaStream_t stream);
cudaError_t launch_commit(int H, int D, const float* inter, int32_t batch, int32_t t_draft,
                          const int32_t* accept_len, float* pool, int64_t num_slots,
                          const int32_t* state_idx, cudaStream_t stream);

size_t prefill_workspace_bytes(const kda_params& p, int32_t num_seqs, int64_t total_tokens);
cudaError_t launch_prefill(const kda_params& p, const GateParams& gp, const void* q,
                           const void* k, const void* v, const float* g_raw, const float* b_raw,
                           const float* A_log, const float* dt_bias, const int32_t* cu_seqlens,
                           int32_t num_seqs, int64_t total_tokens, float* pool,
                           int64_t num_slots, const int32_t* state_idx, void* out,
                           void* workspace, cudaStream_t stream,
                           const cudaEvent_t* events = nullptr,
                           float* chunk_states = nullptr, int64_t chunk_states_capacity = 0);
bool prefill_supported(const kda_params& p);
cudaError_t prefill_read_and_clear_error(int32_t* code);
cudaError_t launch_wait_selftest(uint32_t polls, int32_t* result, cudaStream_t stream);
cudaError_t selftest_read_and_clear_error(int32_t* code);

}  // namespace kda
