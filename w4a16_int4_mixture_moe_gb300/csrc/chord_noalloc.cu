// moe_align_block_size for callers that cannot allocate device memory.
//
// chord_moe_align needs a caller-provided scratch buffer for its per-slice
// expert histograms.  Some callers cannot provide one: code that runs while a
// CUDA graph is being captured in a mode that forbids allocation, inference
// engine plugins that may only use the buffers the engine hands them, and
// latency-critical serving loops that avoid cudaMalloc / cudaFree because they
// synchronise the whole device.  This variant keeps that scratch in a
// fixed-size array in the library's own device memory instead.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/chord.h"
#include "chord_internal.h"

namespace chord {
namespace {

// Histogram scratch for chord_moe_align_noalloc: one int32 per (slice of 4096
// pairs, expert).  Every GPU that loads the library holds these 256 KiB until
// the process exits.
constexpr int64_t kStaticCountsEntries = CHORD_NOALLOC_ALIGN_SCRATCH_ENTRIES;
static __device__ __align__(256) int32_t g_align_scratch[kStaticCountsEntries];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int32_t* g_scratch_ptr[kMaxDevices];

// Device address of this device's copy of the array.  In host code the
// array's name stands for a host-side shadow, not a device address, so it must
// never be passed to a kernel; cudaGetSymbolAddress gives the real address.
// Runs once per device, with that device current.
cudaError_t scratch_for_current_device(int32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_align_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<int32_t*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace chord

using namespace chord;

extern "C" chord_status chord_moe_align_noalloc(const int32_t* topk_ids, int T, int topk, int E, int block_m,
                                                int32_t* sorted_ids, int32_t* expert_ids,
                                                int32_t* num_tokens_padded, int64_t capacity,
                                                const chord_opts* opts, void* stream) {
    if (T < 0 || topk <= 0 || E <= 0 || block_m <= 0) return CHORD_ERR_INVALID_ARG;
    if (E > 1024 || block_m > 256) return CHORD_ERR_UNSUPPORTED;
    if ((int64_t)T * topk >= INT32_MAX) return CHORD_ERR_UNSUPPORTED;
    const size_t need = chord_align_workspace_bytes(T, topk, E) / sizeof(int32_t);
    if ((int64_t)need > kStaticCountsEntries) return CHORD_ERR_BUFFER_TOO_SMALL;
    int32_t* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return CHORD_ERR_CUDA;
    // The histogram launch overwrites every scratch entry this call reads, so
    // nothing left by an earlier call needs clearing.
    return chord_moe_align(topk_ids, T, topk, E, block_m, sorted_ids, expert_ids, num_tokens_padded, capacity,
                           scratch, need * sizeof(int32_t), opts, stream);
}
