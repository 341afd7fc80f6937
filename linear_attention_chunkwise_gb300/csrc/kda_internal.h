// kda_internal.h -- launchers shared between the C-ABI front end and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/kda.h"

namespace kda {

constexpr int kChunk = 64;   // chunk length of the prefill
constexpr int kHeadDim = 128;  // dk = dv

// ---- decode ----
cudaError_t launch_decode(bool f32_io, const void* q, const void* k, const void* v, const float* log_alpha,
                          const float* beta, float* S, int32_t num_slots, const int32_t* state_indices,
                          int32_t N, int32_t H, void* o, int32_t* device_status, cudaStream_t stream);

// ---- prefill ----
struct PrefillArgs {
    const float* beta;
    const float* S0;
    const int32_t* cu_seqlens;
    const int32_t* order;     // schedule: longest sequences first (workspace)
    void* o;
    float* S_final;
    int32_t* device_status;
    int64_t total_tokens;
    int32_t num_seqs;
    int32_t H;
};

// Sequence schedule (longest first) + cu_seqlens validation.
cudaError_t launch_schedule(const int32_t* cu_seqlens, int32_t num_seqs, int64_t total_tokens, int32_t* order,
                            int32_t* device_status, cudaStream_t stream);

// fp32 -> bf16 copy (for fp32 q/k/v inputs).
cudaError_t launch_to_bf16(const float* src, void* dst, size_t n, cudaStream_t stream);

// The chunkwise prefill kernel; q/k/v/log_alpha are read through TMA maps.
cudaError_t launch_prefill(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                           const CUtensorMap& tm_la, const PrefillArgs& a, bool out_f32, cudaStream_t stream);

}  // namespace kda
