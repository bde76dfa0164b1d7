// Host-side launchers shared between the library's translation units.  Every
// launcher only enqueues on `stream` and returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace chord {

struct DeviceInfo {
    int sm_count = 0;
    int max_smem_optin = 0;
    int* err = nullptr;  // device address of this device's sticky error word
};

// Per-device facts, fetched once per device (thread-safe).
const DeviceInfo& device_info();

// Launch facts of one kernel on the current device, computed once per
// (device, kernel, arguments) and cached behind a mutex, so a launch costs no
// runtime query after the first: the kernel's dynamic shared-memory limit is
// raised to `smem_limit` and the resident CTAs per SM at `threads` x `smem`
// are stored in *ctas (at least 1).
cudaError_t kernel_ctas_per_sm(const void* func, int threads, size_t smem, size_t smem_limit, int* ctas);

// Raise a kernel's dynamic shared-memory limit once per (device, kernel, limit).
cudaError_t ensure_smem_limit(const void* func, size_t smem_limit);

// ---- pack / align / epilogues (chord_aux.cu) -------------------------------
cudaError_t launch_pack(const uint8_t* codes, const uint16_t* scales, int E, int N, int K, int layout,
                        uint8_t* packed, int* err, cudaStream_t stream);

int align_slices(int64_t P);
cudaError_t launch_align(const int32_t* topk_ids, int64_t P, int E, int block_m, int32_t* sorted_ids,
                         int32_t* expert_ids, int32_t* ntp, int64_t capacity, int32_t* counts, bool validate,
                         int* err, cudaStream_t stream);

cudaError_t launch_grouped_contiguous_index(const int32_t* m_indices, int64_t M, int E, int block_m,
                                            int32_t* sorted_ids, int32_t* expert_ids, int32_t* ntp,
                                            int64_t capacity, int* err, cudaStream_t stream);
cudaError_t launch_grouped_masked_index(const int32_t* masked_m, int G, int max_m, int block_m, int32_t* sorted_ids,
                                        int32_t* expert_ids, int32_t* ntp, int64_t capacity, int* err,
                                        cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(int* err, cudaStream_t stream);
cudaError_t launch_silu_mul(const uint16_t* C1, const int32_t* topk_ids, int64_t P, int E, int I, uint16_t* h,
                            cudaStream_t stream);
cudaError_t launch_combine(const void* C2, bool c2_f32, const int32_t* topk_ids, const float* topk_w, int T,
                           int topk, int E, int H, uint16_t* out, cudaStream_t stream);
// Fused combine: the per-pair plan before the down GEMM, and the weighted sum of
// the tokens with several local pairs (plus the +0 rows of tokens with none) after it.
cudaError_t launch_combine_plan(const int32_t* topk_ids, const float* topk_w, int T, int topk, int E, float* pair_w,
                                cudaStream_t stream);
cudaError_t launch_combine_finish(const float* C2, const int32_t* topk_ids, const float* topk_w, int T, int topk,
                                  int E, int H, uint16_t* out, cudaStream_t stream);

// ---- GEMMs ---------------------------------------------------------------
// GemmArgs::block_filter.  The valid rows of an align block are a prefix of
// its slots (align fills each expert's blocks from the front), so a block is
// small exactly when its slot CHORD_MIXED_SMALL_ROWS holds the sentinel (or
// the block has no such slot).
constexpr int kBlocksAll = 0;
constexpr int kBlocksSmall = 1;   // warp-level kernel, first 32-row sub-block only
constexpr int kBlocksLarge = 2;   // tcgen05 kernel
struct GemmArgs {
    const uint16_t* A;
    int64_t a_rows;
    int a_row_divisor;
    const uint8_t* packed;  // blob start (header at offset 0)
    int E, N, K;
    const int32_t* sorted_ids;
    const int32_t* expert_ids;
    const int32_t* ntp;
    int64_t capacity;
    int block_m;
    int64_t num_pairs;
    int64_t id_limit;   // pair ids below this are valid rows: min(num_pairs, a_rows * a_row_divisor)
    void* C;        // bf16 [num_pairs, N], or float when out_f32; bf16 [num_pairs, N/2] when silu
    int out_f32;
    uint32_t layout;   // packed layout the header must name: 2, or 3 with silu
    int silu;          // fused SiLU * up epilogue (rows interleaved gate/up by 8)
    int ksplit;        // K slices (warp-level kernel): > 1 writes FP32 partial sums to `partial`
    float* partial;    // warp-level: [ksplit, num_pairs, N], reduced by launch_splitk_reduce;
                       // tcgen05 tail split: [tail units, 128, tok_tile], reduced by launch_tc_tail_reduce
    size_t partial_bytes;
    int tail_split;    // tcgen05: cut the last partial wave's items into K slices (needs `partial`)
    int block_filter;  // kBlocksAll, or (mixed regime) only blocks with at most / more than
                       // CHORD_MIXED_SMALL_ROWS valid rows
    // Fused top-k combine (FP32 output only): a pair whose pair_w entry is a
    // number is its token's only local pair, and its weighted result
    // bf16(0 + w * sum) goes to out[pair / topk, n] instead of C; the others
    // (NaN) write their FP32 sums to C for chord_combine_finish.
    int tc_pairs;      // tcgen05 kernel in clusters of two CTAs (cta_group::2)
    int combine;
    int topk;
    const float* pair_w;
    uint16_t* out;
    int* err;
};

// Split-K reduction of the warp-level kernel: adds the S slices of partial
// [S, num_pairs, N] in slice order and applies the GEMM's epilogue (bf16,
// FP32, SiLU * up or the fused combine) for every valid row.
cudaError_t launch_splitk_reduce(const float* partial, int S, const GemmArgs& a, cudaStream_t stream);

// Warp-MMA kernel (decode regime, packed layout 2): tokens of a block in the N
// dimension of mma.sync m16n8k16, INT4 streamed through a bulk-copy pipeline.
// block_m % 8 == 0.
cudaError_t launch_gemm_decode(const GemmArgs& a, cudaStream_t stream);

// tcgen05 kernel (packed layout 2): dequantised weights in tensor memory as
// the MMA's A operand, tokens as its N side, FP32 accumulators in tensor
// memory.  block_m % 8 == 0, block_m <= 256, N % 128 == 0.
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t stream);

// Tail split of the tcgen05 kernel (see tail_plan): partial[u, r, j] of tail
// unit u = item_in_tail * S + slice, weight row r of the 128-row tile, token
// column j < tok_tile; slices added in order, then the GEMM's epilogue.
cudaError_t launch_tc_tail_reduce(const GemmArgs& a, int64_t grid, int kstages, int min_stages, int tok_tile,
                                  cudaStream_t stream);

}  // namespace chord
