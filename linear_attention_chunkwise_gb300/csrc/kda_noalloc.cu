// kda_noalloc.cu -- kda_prefill for callers that cannot allocate device memory.
//
// kda_prefill needs a small device workspace (the longest-first sequence
// schedule).  Some callers cannot provide one: a plugin that an inference
// engine hands only the tensors it owns, after the engine has reserved all of
// HBM for its own caches; or a latency-critical path where cudaMalloc's
// implicit device synchronisation is not allowed.  This entry point takes its
// scratch from a fixed array in device global memory that is part of this
// library's image instead.  It allocates nothing itself and calls no
// allocating routine.
#include <cuda_runtime.h>

#include <mutex>

#include "kda_internal.h"

namespace {

// Scratch for the sequence schedule: one int32 per sequence.  Every GPU that
// loads libkda holds this array (256 KiB) until the process exits.
static __device__ __align__(256) int32_t g_prefill_scratch[KDA_NOALLOC_MAX_SEQS];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices];  // device address of g_prefill_scratch, per device

// Host code cannot use g_prefill_scratch's name as a device address (it names
// a host-side stand-in).  Look the real address up once per device, with that
// device current, and cache it.
kda_status scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return KDA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_prefill_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();  // clear the runtime's last-error slot for later calls
            return KDA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return KDA_OK;
}

}  // namespace

extern "C" KDA_API kda_status kda_prefill_noalloc(const void* q, const void* k, const void* v, kda_dtype qkv_dtype,
                                                  const float* log_alpha, const float* beta, const float* S0,
                                                  const int32_t* cu_seqlens, int32_t num_seqs,
                                                  int64_t total_tokens, int32_t H, int32_t dk, int32_t dv, void* o,
                                                  float* S_final, int32_t* device_status, kda_stream_t stream) {
    if (qkv_dtype != KDA_DTYPE_BF16) return KDA_ERR_UNSUPPORTED;  // fp32 inputs need token-sized scratch
    if (num_seqs > KDA_NOALLOC_MAX_SEQS) return KDA_ERR_WORKSPACE;
    // The same architecture check as kda_prefill, before the symbol lookup (which fails on a GPU
    // the library has no code for), so both entry points give the same status there.
    const kda_status dev = kda::device_check();
    if (dev != KDA_OK) return dev;
    void* scratch = nullptr;
    const kda_status st = scratch_for_current_device(&scratch);
    if (st != KDA_OK) return st;
    return kda_prefill(q, k, v, qkv_dtype, log_alpha, beta, S0, cu_seqlens, num_seqs, total_tokens, H, dk, dv, o,
                       S_final, scratch, sizeof(g_prefill_scratch), device_status, stream);
}
