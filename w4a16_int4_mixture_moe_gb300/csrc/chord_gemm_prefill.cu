// Prefill-regime indexed W4A16 GEMM for sm_103a (tcgen05 MMA, TMEM accumulators).
#include <cuda_runtime.h>

#include "chord_common.cuh"
#include "chord_internal.h"

namespace chord {

bool prefill_available() { return false; }

cudaError_t launch_gemm_prefill(const GemmArgs& a, cudaStream_t stream) {
    (void)a;
    (void)stream;
    return cudaErrorNotSupported;
}

}  // namespace chord
