// Packing, routing alignment and the element-wise epilogues (SiLU * up, top-k
// combine) of the W4A16 MoE library, sm_103a.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "chord_common.cuh"
#include "chord_internal.h"

namespace chord {

// ============================================================================
// Pack: canonical codes [E, N, K] + scales [E, N, K/32] -> layout 1 (the warp
// MMA kernel's A fragments) or layout 2 (one row per thread for the tcgen05
// kernel).  One thread writes one 32-bit word of the blob, so the writes are
// coalesced; the gathers from the canonical arrays are not, which is fine for
// a one-off load-time step.
// ============================================================================
// Layout 2: chunk (nt, kc) of 128 rows x 64 columns is 1152 words: words
// 0..1023 are codes (half h = w/512, row r = (w%512)/4, word j = w%4 holding
// columns 32h + 8j + m of the chunk, m = 2*(i%4) + i/4 in nibble i), words
// 1024..1151 the two group scales of each row.
// Layout 3 keeps layout 2's byte positions but reorders a gate_up weight's
// rows: packed row p holds gate row 8*(p/16) + p%16 when p%16 < 8, else the up
// row N/2 + 8*(p/16) + p%16 - 8 (each 16-row group: 8 gate rows, their up rows).
__device__ __forceinline__ int canonical_row(int p, int N, bool interleaved) {
    if (!interleaved) return p;
    const int g = p >> 4, i = p & 15;
    return i < 8 ? 8 * g + i : (N >> 1) + 8 * g + (i - 8);
}

// Header word 7 (written as 1 by header_kernel, earlier on the stream) drops
// to 0 when any scale lies outside [2^-126, 0.5); every writer stores the same
// 0, so the unordered stores agree.  `data` is the first word after the header.
__device__ __forceinline__ void clear_scale_range(uint32_t* data) {
    reinterpret_cast<volatile uint32_t*>(data - kHeaderBytes / 4)[kHdrScaleRangeWord] = 0u;
}

__global__ void pack2_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales, int E, int N,
                             int K, bool interleaved, uint32_t* __restrict__ out, int* err) {
    constexpr int kWords = 4608 / 4;
    const int kchunks = K / 64;
    const int64_t chunks_per_expert = (int64_t)(N / 128) * kchunks;
    const int64_t words = (int64_t)E * chunks_per_expert * kWords;
    const int G = K / kGroup;
    for (int64_t w = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; w < words; w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t chunk = w / kWords;
        const int wi = (int)(w % kWords);
        const int64_t e = chunk / chunks_per_expert;
        const int64_t cc = chunk % chunks_per_expert;
        const int nt = (int)(cc / kchunks), kc = (int)(cc % kchunks);
        uint32_t v = 0;
        if (wi < 1024) {
            const int h = wi / 512, r = (wi % 512) / 4, j = wi % 4;
            const int n = canonical_row(nt * 128 + r, N, interleaved);
            const uint8_t* p = codes + ((int64_t)e * N + n) * K + kc * 64 + h * 32 + j * 8;
            uint32_t bad = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t q = p[2 * (i & 3) + (i >> 2)];
                bad |= q >> 4;
                v |= (q & 0xFu) << (4 * i);
            }
            if (bad) set_error(err, CHORD_DEV_BAD_CODE);
        } else {
            const int r = wi - 1024;
            const int64_t row = (int64_t)e * N + canonical_row(nt * 128 + r, N, interleaved);
            v = (uint32_t)scales[row * G + 2 * kc] | ((uint32_t)scales[row * G + 2 * kc + 1] << 16);
            if (!scale_in_fma_range(v & 0xffffu) || !scale_in_fma_range(v >> 16)) clear_scale_range(out);
        }
        out[w] = v;
    }
}

__device__ __forceinline__ void write_header(uint8_t* packed, int64_t tid, int E, int N, int K, uint32_t layout) {
    if (tid < kHeaderBytes / 4) {
        const unsigned long long stride = (unsigned long long)N * (unsigned long long)K * 9ull / 16ull;
        uint32_t v = 0;
        switch ((int)tid) {
            case 0: v = kMagic; break;
            case 1: v = 1u; break;
            case 2: v = layout; break;
            case 3: v = (uint32_t)kGroup; break;
            case 4: v = (uint32_t)E; break;
            case 5: v = (uint32_t)N; break;
            case 6: v = (uint32_t)K; break;
            case kHdrScaleRangeWord: v = 1u; break;   // cleared by the pack kernel on an out-of-range scale
            case 8: v = (uint32_t)stride; break;
            case 9: v = (uint32_t)(stride >> 32); break;
            case 10: v = (uint32_t)kHeaderBytes; break;
            default: v = 0u;
        }
        reinterpret_cast<uint32_t*>(packed)[tid] = v;
    }
}

__global__ void header_kernel(uint8_t* packed, int E, int N, int K, uint32_t layout) {
    write_header(packed, threadIdx.x, E, N, K, layout);
}

__global__ void pack_kernel(const uint8_t* __restrict__ codes, const uint16_t* __restrict__ scales, int E, int N,
                            int K, uint8_t* __restrict__ packed, int* err) {
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int mtiles = N / 16;
    const int64_t chunks_per_expert = (int64_t)(K / 64) * mtiles;
    const int64_t words = (int64_t)E * chunks_per_expert * (kChunkBytes / 4);
    const int G = K / kGroup;
    uint32_t* out = reinterpret_cast<uint32_t*>(packed + kHeaderBytes);
    for (int64_t w = tid; w < words; w += (int64_t)gridDim.x * blockDim.x) {
        const int64_t chunk = w / (kChunkBytes / 4);
        const int wi = (int)(w % (kChunkBytes / 4));
        const int64_t e = chunk / chunks_per_expert;
        const int64_t cc = chunk % chunks_per_expert;
        const int kc = (int)(cc / mtiles);
        const int mt = (int)(cc % mtiles);
        uint32_t v = 0;
        if (wi < kChunkWeightBytes / 4) {
            const int lane = wi / 4, j = wi % 4;
            const int g = lane / 4, c = lane % 4;
            const int64_t r0 = (int64_t)e * N + mt * 16 + g;
            const int col = kc * 64 + 16 * j + 2 * c;
            const uint8_t* p0 = codes + r0 * K + col;
            const uint8_t* p1 = codes + (r0 + 8) * K + col;
            // nibble i of the word: i=0 (g, col), 1 (g+8, col), 2 (g, col+8), 3 (g+8, col+8),
            // i+4: the same with col+1.
            const uint32_t n[8] = {p0[0], p1[0], p0[8], p1[8], p0[1], p1[1], p0[9], p1[9]};
            uint32_t bad = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                bad |= n[i] >> 4;
                v |= (n[i] & 0xFu) << (4 * i);
            }
            if (bad) set_error(err, CHORD_DEV_BAD_CODE);
        } else {
            const int s = wi - kChunkWeightBytes / 4;
            const int h = s / 8, g = s % 8;
            const int64_t r0 = (int64_t)e * N + mt * 16 + g;
            const int grp = kc * 2 + h;
            v = (uint32_t)scales[r0 * G + grp] | ((uint32_t)scales[(r0 + 8) * G + grp] << 16);
            if (!scale_in_fma_range(v & 0xffffu) || !scale_in_fma_range(v >> 16)) clear_scale_range(out);
        }
        out[w] = v;
    }
}

cudaError_t launch_pack(const uint8_t* codes, const uint16_t* scales, int E, int N, int K, int layout,
                        uint8_t* packed, int* err, cudaStream_t stream) {
    header_kernel<<<1, kHeaderBytes / 4, 0, stream>>>(packed, E, N, K, (uint32_t)layout);
    cudaError_t st = cudaGetLastError();
    if (st != cudaSuccess || E == 0) return st;
    const int64_t words = (int64_t)E * (K / 64) * (N / 16) * (kChunkBytes / 4);  // same count for both layouts
    const int threads = 256;
    int64_t blocks = ceil_div64(words, threads);
    const int64_t cap = (int64_t)device_info().sm_count * 16;
    if (blocks > cap) blocks = cap;
    if (layout == 2 || layout == 3)
        pack2_kernel<<<(unsigned)blocks, threads, 0, stream>>>(codes, scales, E, N, K, layout == 3,
                                                               reinterpret_cast<uint32_t*>(packed + kHeaderBytes), err);
    else
        pack_kernel<<<(unsigned)blocks, threads, 0, stream>>>(codes, scales, E, N, K, packed, err);
    return cudaGetLastError();
}

// ============================================================================
// moe_align_block_size, deterministic: pairs of each expert in ascending pair
// id.  Up to kSlice pairs: one CTA does everything in one launch.  Above:
// three launches,
//   count:   per slice of kSlice pairs, an expert histogram; also fills
//            sorted_ids with the sentinel;
//   scan:    one CTA turns the histograms into each slice's starting offset per
//            expert, writes expert_ids and num_tokens_padded;
//   scatter: per slice, stable ranks within the slice (warp match + per-warp
//            counts, warps in order) place each pair.
// ============================================================================
constexpr int kSlice = 4096;
constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;

int align_slices(int64_t P) { return P > 0 ? (int)ceil_div64(P, kSlice) : 1; }

// Histogram of the local experts of pairs [base, min(base + kSlice, P)) into
// shared `hist` (zeroed by the caller).
__device__ __forceinline__ void slice_histogram(const int32_t* __restrict__ ids, int64_t P, int E, int64_t base,
                                                int32_t* hist, int validate, int* err) {
    for (int i = threadIdx.x; i < kSlice; i += blockDim.x) {
        const int64_t p = base + i;
        if (p >= P) break;
        const int e = ids[p];
        if (e >= 0 && e < E)
            atomicAdd(&hist[e], 1);
        else if (validate && e != -1)
            set_error(err, CHORD_DEV_BAD_EXPERT);
    }
}

// Thread e < E holds expert e's pair count `total`; returns the exclusive
// prefix sum of the block_m-padded counts (expert e's first slot), writes
// expert_ids for every block and -1 past the padded total, and the total to
// *ntp.  All kAlignThreads threads must call it.
__device__ __forceinline__ int32_t padded_offsets(int32_t total, int E, int block_m, int32_t* __restrict__ expert_ids,
                                                  int64_t nblocks_cap, int32_t* __restrict__ ntp) {
    __shared__ int32_t warp_sums[kAlignWarps];
    __shared__ int32_t total_padded;
    const int e = threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t padded = (e < E) ? (total + block_m - 1) / block_m * block_m : 0;
    int32_t x = padded;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        warp_sums[lane] = w;  // inclusive
        if (lane == 31) total_padded = w;
    }
    __syncthreads();
    const int32_t offset = x - padded + (warp > 0 ? warp_sums[warp - 1] : 0);
    if (e < E)
        for (int32_t b = offset / block_m; b < (offset + padded) / block_m; ++b) expert_ids[b] = e;
    const int32_t tp = total_padded;
    for (int64_t b = tp / block_m + threadIdx.x; b < nblocks_cap; b += blockDim.x) expert_ids[b] = -1;
    if (threadIdx.x == 0) *ntp = tp;
    return offset;
}

// Places the local pairs of slice [base, base + kSlice) at run[e], run[e] + 1,
// ... in ascending pair id (run: shared, next free slot per expert, advanced;
// wcnt: shared [kAlignWarps][E] scratch).
__device__ __forceinline__ void slice_scatter(const int32_t* __restrict__ ids, int64_t P, int E, int64_t base,
                                              int32_t* run, int32_t* wcnt, int32_t* __restrict__ sorted_ids) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    for (int r = 0; r < kSlice / kAlignThreads; ++r) {
        if (base + (int64_t)r * kAlignThreads >= P) break;   // uniform over the CTA
        for (int i = threadIdx.x; i < kAlignWarps * E; i += blockDim.x) wcnt[i] = 0;
        __syncthreads();
        const int64_t p = base + (int64_t)r * kAlignThreads + threadIdx.x;
        int e = (p < P) ? ids[p] : -1;
        const bool valid = (e >= 0 && e < E);
        if (!valid) e = -1;
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & lt_mask);
        if (valid && rank == 0) wcnt[warp * E + e] = __popc(peers);
        __syncthreads();
        for (int x = threadIdx.x; x < E; x += blockDim.x) {
            int32_t acc = run[x];
            for (int w = 0; w < kAlignWarps; ++w) {
                const int32_t v = wcnt[w * E + x];
                wcnt[w * E + x] = acc;
                acc += v;
            }
            run[x] = acc;
        }
        __syncthreads();
        if (valid) sorted_ids[wcnt[warp * E + e] + rank] = (int32_t)p;
        __syncthreads();
    }
}

// P <= kSlice: histogram, offsets, sentinel fill and placement in one CTA.
__global__ void __launch_bounds__(kAlignThreads) align_single_kernel(const int32_t* __restrict__ ids, int64_t P, int E,
                                                                     int block_m, int32_t* __restrict__ sorted_ids,
                                                                     int32_t* __restrict__ expert_ids,
                                                                     int64_t nblocks_cap, int32_t* __restrict__ ntp,
                                                                     int64_t capacity, int validate, int* err) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ int32_t sm[];
    int32_t* run = sm;        // [E] histogram, then next free slot per expert
    int32_t* wcnt = sm + E;   // [kAlignWarps][E]
    for (int i = threadIdx.x; i < E; i += blockDim.x) run[i] = 0;
    const int32_t sentinel = (int32_t)P;
    for (int64_t i = threadIdx.x; i < capacity; i += blockDim.x) sorted_ids[i] = sentinel;
    __syncthreads();
    slice_histogram(ids, P, E, 0, run, validate, err);
    __syncthreads();
    const int32_t total = threadIdx.x < E ? run[threadIdx.x] : 0;
    const int32_t offset = padded_offsets(total, E, block_m, expert_ids, nblocks_cap, ntp);
    if (threadIdx.x < E) run[threadIdx.x] = offset;
    __syncthreads();   // also orders the sentinel fill before the placement
    slice_scatter(ids, P, E, 0, run, wcnt, sorted_ids);
}

__global__ void __launch_bounds__(kAlignThreads) align_count_kernel(const int32_t* __restrict__ ids, int64_t P, int E,
                                                                    int32_t* __restrict__ counts,
                                                                    int32_t* __restrict__ sorted_ids,
                                                                    int64_t capacity, int validate, int* err) {
    extern __shared__ int32_t hist[];
    for (int i = threadIdx.x; i < E; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    slice_histogram(ids, P, E, (int64_t)blockIdx.x * kSlice, hist, validate, err);
    __syncthreads();
    for (int i = threadIdx.x; i < E; i += blockDim.x) counts[(int64_t)blockIdx.x * E + i] = hist[i];
    const int32_t sentinel = (int32_t)P;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < capacity;
         i += (int64_t)gridDim.x * blockDim.x)
        sorted_ids[i] = sentinel;
}

__global__ void __launch_bounds__(kAlignThreads) align_scan_kernel(int32_t* __restrict__ counts, int nslices, int E,
                                                                   int block_m, int32_t* __restrict__ expert_ids,
                                                                   int64_t nblocks_cap, int32_t* __restrict__ ntp) {
    const int e = threadIdx.x;
    int32_t total = 0;
    if (e < E) {
        for (int s = 0; s < nslices; ++s) {
            const int32_t v = counts[(int64_t)s * E + e];
            counts[(int64_t)s * E + e] = total;
            total += v;
        }
    }
    const int32_t offset = padded_offsets(total, E, block_m, expert_ids, nblocks_cap, ntp);
    if (e < E)
        for (int s = 0; s < nslices; ++s) counts[(int64_t)s * E + e] += offset;
}

__global__ void __launch_bounds__(kAlignThreads) align_scatter_kernel(const int32_t* __restrict__ ids, int64_t P,
                                                                      int E, const int32_t* __restrict__ counts,
                                                                      int32_t* __restrict__ sorted_ids) {
    extern __shared__ int32_t sm[];
    int32_t* run = sm;           // [E]   next free slot per expert
    int32_t* wcnt = sm + E;      // [kAlignWarps][E]
    for (int i = threadIdx.x; i < E; i += blockDim.x) run[i] = counts[(int64_t)blockIdx.x * E + i];
    slice_scatter(ids, P, E, (int64_t)blockIdx.x * kSlice, run, wcnt, sorted_ids);
}

cudaError_t launch_align(const int32_t* topk_ids, int64_t P, int E, int block_m, int32_t* sorted_ids,
                         int32_t* expert_ids, int32_t* ntp, int64_t capacity, int32_t* counts, bool validate, int* err,
                         cudaStream_t stream) {
    const int nslices = align_slices(P);
    const size_t hist_smem = (size_t)E * sizeof(int32_t);
    const size_t scatter_smem = (size_t)(E + kAlignWarps * E) * sizeof(int32_t);
    {
        const size_t most = (1024 + kAlignWarps * 1024) * sizeof(int32_t);
        cudaError_t e1 = ensure_smem_limit(reinterpret_cast<const void*>(align_scatter_kernel), most);
        if (e1 == cudaSuccess) e1 = ensure_smem_limit(reinterpret_cast<const void*>(align_single_kernel), most);
        if (e1 != cudaSuccess) return e1;
    }
    if (nslices == 1) {
        return launch_pdl(pdl_for(P), align_single_kernel, dim3(1), dim3(kAlignThreads), scatter_smem, stream, topk_ids, P, E,
                          block_m, sorted_ids, expert_ids, capacity / block_m, ntp, capacity, validate ? 1 : 0, err);
    }
    align_count_kernel<<<nslices, kAlignThreads, hist_smem, stream>>>(topk_ids, P, E, counts, sorted_ids, capacity,
                                                                      validate ? 1 : 0, err);
    cudaError_t st = cudaGetLastError();
    if (st != cudaSuccess) return st;
    align_scan_kernel<<<1, kAlignThreads, 0, stream>>>(counts, nslices, E, block_m, expert_ids, capacity / block_m,
                                                       ntp);
    st = cudaGetLastError();
    if (st != cudaSuccess) return st;
    align_scatter_kernel<<<nslices, kAlignThreads, scatter_smem, stream>>>(topk_ids, P, E, counts, sorted_ids);
    return cudaGetLastError();
}

// ============================================================================
// Grouped contracts -> the indexed GEMM's routing arrays (one row per pair,
// row id = pair id, sentinel = the row count).  Both contracts give each
// expert e a contiguous run of rows [start[e], start[e] + count[e]); its
// ceil(count[e] / block_m) blocks are laid out expert after expert, exactly as
// align lays out an expert's pairs, so the GEMM sees one block per expert when
// its rows fit.  One CTA (the expert tables live in shared memory):
//   contiguous: count and first row of each expert from m_indices (a row whose
//               expert's rows are not one run sets CHORD_DEV_BAD_ROW, an id
//               outside [-1, E) CHORD_DEV_BAD_EXPERT); padding rows (-1) are
//               in no block;
//   masked:     count = masked_m[g] (clamped to [0, max_m], CHORD_DEV_BAD_ROW
//               when outside), first row g * max_m.
// ============================================================================
constexpr int kGroupedThreads = 1024;

__device__ void grouped_fill(const int32_t* count, const int32_t* start, int32_t* first_block, int E, int block_m,
                             int32_t sentinel, int32_t* sorted_ids, int32_t* expert_ids, int32_t* ntp,
                             int64_t capacity) {
    if (threadIdx.x == 0) {
        int32_t acc = 0;
        for (int e = 0; e < E; ++e) {
            first_block[e] = acc;
            acc += (count[e] + block_m - 1) / block_m;
        }
        first_block[E] = acc;
        *ntp = acc * block_m;
    }
    __syncthreads();
    const int64_t total = (int64_t)first_block[E] * block_m;
    for (int64_t i = threadIdx.x; i < capacity; i += blockDim.x) {
        if (i >= total) {
            sorted_ids[i] = sentinel;
            continue;
        }
        const int32_t blk = (int32_t)(i / block_m);
        int lo = 0, hi = E - 1;   // the expert whose blocks contain blk (the last with first_block <= blk)
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (first_block[mid] <= blk) lo = mid; else hi = mid - 1;
        }
        const int32_t r = (blk - first_block[lo]) * block_m + (int32_t)(i % block_m);
        sorted_ids[i] = r < count[lo] ? start[lo] + r : sentinel;
        if (i % block_m == 0) expert_ids[blk] = lo;
    }
}

__global__ void grouped_contiguous_index_kernel(const int32_t* __restrict__ m_indices, int64_t M, int E,
                                                int block_m, int32_t* __restrict__ sorted_ids,
                                                int32_t* __restrict__ expert_ids, int32_t* __restrict__ ntp,
                                                int64_t capacity, int* err) {
    extern __shared__ int32_t tab[];   // count[E], start[E], first_block[E + 1]
    int32_t* count = tab;
    int32_t* start = tab + E;
    int32_t* first_block = tab + 2 * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        count[e] = 0;
        start[e] = INT32_MAX;
    }
    __syncthreads();
    for (int64_t m = threadIdx.x; m < M; m += blockDim.x) {
        const int32_t e = m_indices[m];
        if (e < -1 || e >= E) {
            set_error(err, CHORD_DEV_BAD_EXPERT);
        } else if (e >= 0) {
            atomicAdd(&count[e], 1);
            atomicMin(&start[e], (int32_t)m);
        }
    }
    __syncthreads();
    for (int64_t m = threadIdx.x; m < M; m += blockDim.x) {
        const int32_t e = m_indices[m];
        if (e >= 0 && e < E && (int64_t)m - start[e] >= count[e]) set_error(err, CHORD_DEV_BAD_ROW);
    }
    for (int e = threadIdx.x; e < E; e += blockDim.x)
        if (count[e] == 0) start[e] = 0;
    __syncthreads();
    grouped_fill(count, start, first_block, E, block_m, (int32_t)M, sorted_ids, expert_ids, ntp, capacity);
}

__global__ void grouped_masked_index_kernel(const int32_t* __restrict__ masked_m, int G, int max_m, int block_m,
                                            int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                                            int32_t* __restrict__ ntp, int64_t capacity, int* err) {
    extern __shared__ int32_t tab[];
    int32_t* count = tab;
    int32_t* start = tab + G;
    int32_t* first_block = tab + 2 * G;
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
        int32_t c = masked_m[g];
        if (c < 0 || c > max_m) {
            set_error(err, CHORD_DEV_BAD_ROW);
            c = c < 0 ? 0 : max_m;
        }
        count[g] = c;
        start[g] = g * max_m;
    }
    __syncthreads();
    grouped_fill(count, start, first_block, G, block_m, G * max_m, sorted_ids, expert_ids, ntp, capacity);
}

cudaError_t launch_grouped_contiguous_index(const int32_t* m_indices, int64_t M, int E, int block_m,
                                            int32_t* sorted_ids, int32_t* expert_ids, int32_t* ntp,
                                            int64_t capacity, int* err, cudaStream_t stream) {
    grouped_contiguous_index_kernel<<<1, kGroupedThreads, (size_t)(3 * E + 1) * sizeof(int32_t), stream>>>(
        m_indices, M, E, block_m, sorted_ids, expert_ids, ntp, capacity, err);
    return cudaGetLastError();
}

cudaError_t launch_grouped_masked_index(const int32_t* masked_m, int G, int max_m, int block_m, int32_t* sorted_ids,
                                        int32_t* expert_ids, int32_t* ntp, int64_t capacity, int* err,
                                        cudaStream_t stream) {
    grouped_masked_index_kernel<<<1, kGroupedThreads, (size_t)(3 * G + 1) * sizeof(int32_t), stream>>>(
        masked_m, G, max_m, block_m, sorted_ids, expert_ids, ntp, capacity, err);
    return cudaGetLastError();
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&r);
}

// ============================================================================
// Split-K reduction: C[p, n] = sum over slices s = 0 .. S-1, in that order,
// of partial[s, p, n] (the GEMM's FP32 partial sums of K slice s), for every
// pair p a block of the routing names; then the GEMM's epilogue: bf16 or FP32
// out, or with silu the fused SiLU * up of layout 3 (h column 8k + i from the
// packed rows 16k + i and 16k + 8 + i).  One thread per 4 output columns; the
// loads of up to 8 slices are issued before they are added, so the in-order
// sum costs one memory round trip per 8 slices.
// ============================================================================
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

template <bool kSilu>
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int S, const GemmArgs a) {
    pdl_trigger();
    pdl_wait();
    constexpr int kBatch = 8;
    const int N = a.N;
    const int out_cols = kSilu ? N / 2 : N;
    const int vpr = out_cols / 4;
    int64_t slots = *a.ntp;
    slots = slots < 0 ? 0 : (slots > a.capacity ? a.capacity : slots);
    const int64_t nvec = slots * vpr;
    const int64_t slice_stride = a.num_pairs * (int64_t)N / 4;   // in float4
    void* __restrict__ C = a.C;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += (int64_t)gridDim.x * blockDim.x) {
        int jv;
        const int32_t p = __ldg(a.sorted_ids + divmod_idx(v, vpr, jv));
        if (p < 0 || (int64_t)p >= a.id_limit) continue;
        const int j0 = jv * 4;
        // packed column of output column j0 (gate; up is 8 further)
        const int c0 = kSilu ? 16 * (j0 / 8) + j0 % 8 : j0;
        const float4* src = reinterpret_cast<const float4*>(partial + (int64_t)p * N + c0);
        float4 g = make_float4(0.f, 0.f, 0.f, 0.f), u = g;
        for (int s0 = 0; s0 < S; s0 += kBatch) {
            float4 gv[kBatch], uv[kBatch];
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (s0 + i < S) {
                    gv[i] = __ldcg(src + (int64_t)(s0 + i) * slice_stride);
                    if (kSilu) uv[i] = __ldcg(src + (int64_t)(s0 + i) * slice_stride + 2);
                }
            }
#pragma unroll
            for (int i = 0; i < kBatch; ++i) {
                if (s0 + i < S) {
                    g = add4(g, gv[i]);
                    if (kSilu) u = add4(u, uv[i]);
                }
            }
        }
        if (kSilu) {
            __nv_bfloat16 o[4] = {silu_mul_bf16(g.x, u.x), silu_mul_bf16(g.y, u.y), silu_mul_bf16(g.z, u.z),
                                  silu_mul_bf16(g.w, u.w)};
            *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(C) + (int64_t)p * out_cols + j0) =
                *reinterpret_cast<const uint2*>(o);
        } else if (a.combine) {
            const float w = __ldg(a.pair_w + p);
            const int64_t tok = p / a.topk;
            float* C2 = static_cast<float*>(C);
            combine_store(C2, a.out, N, p, tok, w, j0, g.x);
            combine_store(C2, a.out, N, p, tok, w, j0 + 1, g.y);
            combine_store(C2, a.out, N, p, tok, w, j0 + 2, g.z);
            combine_store(C2, a.out, N, p, tok, w, j0 + 3, g.w);
        } else if (a.out_f32) {
            *reinterpret_cast<float4*>(static_cast<float*>(C) + (int64_t)p * out_cols + j0) = g;
        } else {
            uint2 o;
            o.x = pack_bf16x2(g.x, g.y);
            o.y = pack_bf16x2(g.z, g.w);
            *reinterpret_cast<uint2*>(static_cast<uint16_t*>(C) + (int64_t)p * out_cols + j0) = o;
        }
    }
}

// ============================================================================
// SiLU * up: h[p, j] = bf16_rne(g / (1 + exp(-g)) * u), FP32 math.  One warp
// per pair row: lane 0's id decides for the whole row (a row of another GPU's
// expert costs one load), then the warp walks the row 8 columns per lane with
// 16-byte loads and stores, two vectors per lane in flight.
// ============================================================================
__device__ __forceinline__ uint4 silu_mul8(uint4 gv, uint4 uv) {
    uint4 o;
    o.x = pack_bf16x2(silu_times(bf16_lo(gv.x), bf16_lo(uv.x)), silu_times(bf16_hi(gv.x), bf16_hi(uv.x)));
    o.y = pack_bf16x2(silu_times(bf16_lo(gv.y), bf16_lo(uv.y)), silu_times(bf16_hi(gv.y), bf16_hi(uv.y)));
    o.z = pack_bf16x2(silu_times(bf16_lo(gv.z), bf16_lo(uv.z)), silu_times(bf16_hi(gv.z), bf16_hi(uv.z)));
    o.w = pack_bf16x2(silu_times(bf16_lo(gv.w), bf16_lo(uv.w)), silu_times(bf16_hi(gv.w), bf16_hi(uv.w)));
    return o;
}

__global__ void silu_mul_kernel(const uint16_t* __restrict__ C1, const int32_t* __restrict__ ids, int64_t P, int E,
                                int I, uint16_t* __restrict__ h) {
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int vpr = I / 8;
    for (int64_t p = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); p < P; p += warps) {
        int e = lane == 0 ? __ldg(ids + p) : 0;
        e = __shfl_sync(0xffffffffu, e, 0);
        if (e < 0 || e >= E) continue;
        const uint4* grow = reinterpret_cast<const uint4*>(C1 + p * 2 * I);
        const uint4* urow = reinterpret_cast<const uint4*>(C1 + p * 2 * I + I);
        uint4* hrow = reinterpret_cast<uint4*>(h + p * I);
        int j = lane;
        for (; j + 32 < vpr; j += 64) {
            const uint4 g0 = grow[j], u0 = urow[j], g1 = grow[j + 32], u1 = urow[j + 32];
            hrow[j] = silu_mul8(g0, u0);
            hrow[j + 32] = silu_mul8(g1, u1);
        }
        if (j < vpr) hrow[j] = silu_mul8(grow[j], urow[j]);
    }
}

// ============================================================================
// Self-test of the bounded pipeline wait: one thread initialises an mbarrier
// that nothing will ever arrive on and waits for its first phase through
// mbar_wait, the helper every GEMM pipeline waits with.  After the helper's
// bound (kWaitLimitCycles, about 2 s) the thread records CHORD_DEV_TIMEOUT in
// the error word and the kernel returns: a wait that cannot end becomes an
// error the host reads, with no fault and a context that stays usable.
// ============================================================================
__global__ void wait_timeout_selftest_kernel(int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
        if (!mbar_wait(&bar, 0)) set_error(err, CHORD_DEV_TIMEOUT);
    }
}

cudaError_t launch_wait_timeout_selftest(int* err, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

// ============================================================================
// Tail split of the tcgen05 kernel: for tail item i (item full + i of the
// launch's plan), weight row r of its 128-row tile and token column j of its
// block, C[id, 128 nt + r] = sum over slices s = 0 .. S-1, in that order, of
// partial[i S + s, r, j], for the valid pair id at slot j; then the GEMM's
// epilogue (bf16, FP32, or the layout-3 SiLU * up: gate row r, up row r + 8,
// h column 64 nt + 8 (r / 16) + r % 8).  The plan is recomputed from
// num_tokens_padded exactly as the GEMM computed it.  One thread per (item,
// row or gate row, token); tokens are the fastest index (contiguous partials).
// ============================================================================
template <bool kSilu>
__global__ void tc_tail_reduce_kernel(const GemmArgs a, int64_t G, int kstages, int min_stages, int tok_tile) {
    pdl_trigger();
    pdl_wait();
    int32_t ntp = *a.ntp;
    if (ntp < 0 || ntp > a.capacity || ntp % a.block_m) return;   // the GEMM reported it and ran nothing
    const int ntiles = a.N / 128;
    const TailPlan tp = tail_plan((int64_t)(ntp / a.block_m) * ntiles, G, kstages, min_stages, true);
    if (tp.S < 2) return;
    constexpr int kRows = kSilu ? 64 : 128;
    const int64_t per_item = (int64_t)kRows * tok_tile;
    const int64_t total = tp.tail * per_item;
    const int64_t slice = (int64_t)128 * tok_tile;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < total; v += (int64_t)gridDim.x * blockDim.x) {
        int rem;
        const int64_t i = divmod_idx(v, (int)per_item, rem);
        const int rr = rem / tok_tile, j = rem % tok_tile;
        if (j >= a.block_m) continue;
        const int64_t item = tp.full + i;
        const int nt = (int)(item % ntiles);
        const int64_t b = item / ntiles;
        const int e = a.expert_ids[b];
        if (e < 0 || e >= a.E) continue;
        // mixed regime: small blocks (sentinel in slot 32) were computed by the warp-level launch
        if (a.block_filter == kBlocksLarge &&
            a.sorted_ids[b * a.block_m + CHORD_MIXED_SMALL_ROWS] == (int32_t)a.num_pairs)
            continue;
        const int32_t id = a.sorted_ids[b * a.block_m + j];
        if (id < 0 || (int64_t)id >= a.id_limit) continue;
        const int r = kSilu ? 16 * (rr / 8) + rr % 8 : rr;
        const float* src = a.partial + (i * tp.S * 128 + r) * tok_tile + j;
        float g = 0.0f, u = 0.0f;
        for (int s = 0; s < tp.S; ++s) {
            g = __fadd_rn(g, __ldcg(src + s * slice));
            if (kSilu) u = __fadd_rn(u, __ldcg(src + s * slice + 8 * tok_tile));
        }
        if (kSilu) {
            const int h_col = nt * 64 + 8 * (r / 16) + r % 8;
            static_cast<__nv_bfloat16*>(a.C)[(int64_t)id * (a.N / 2) + h_col] = silu_mul_bf16(g, u);
        } else if (a.combine) {
            combine_store(static_cast<float*>(a.C), a.out, a.N, id, id / a.topk, __ldg(a.pair_w + id), nt * 128 + r,
                          g);
        } else if (a.out_f32) {
            static_cast<float*>(a.C)[(int64_t)id * a.N + nt * 128 + r] = g;
        } else {
            static_cast<__nv_bfloat16*>(a.C)[(int64_t)id * a.N + nt * 128 + r] = __float2bfloat16_rn(g);
        }
    }
}

cudaError_t launch_tc_tail_reduce(const GemmArgs& a, int64_t grid, int kstages, int min_stages, int tok_tile,
                                  cudaStream_t stream) {
    // the tail has fewer than `grid` items
    const int64_t total = (grid - 1) * (int64_t)(a.silu ? 64 : 128) * tok_tile;
    if (total <= 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = ceil_div64(total, threads);
    const int64_t cap = (int64_t)device_info().sm_count * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(pdl_for(a.num_pairs), a.silu ? tc_tail_reduce_kernel<true> : tc_tail_reduce_kernel<false>, dim3((unsigned)blocks),
                      dim3(threads), 0, stream, a, grid, kstages, min_stages, tok_tile);
}

cudaError_t launch_splitk_reduce(const float* partial, int S, const GemmArgs& a, cudaStream_t stream) {
    const int64_t nvec = a.capacity * ((a.silu ? a.N / 2 : a.N) / 4);
    if (nvec == 0) return cudaSuccess;
    const int threads = 128;
    int64_t blocks = ceil_div64(nvec, threads);
    const int64_t cap = (int64_t)device_info().sm_count * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(pdl_for(a.num_pairs), a.silu ? splitk_reduce_kernel<true> : splitk_reduce_kernel<false>,
                      dim3((unsigned)blocks), dim3(threads), 0, stream, partial, S, a);
}

cudaError_t launch_silu_mul(const uint16_t* C1, const int32_t* topk_ids, int64_t P, int E, int I, uint16_t* h,
                            cudaStream_t stream) {
    if (P == 0) return cudaSuccess;
    const int threads = 256;   // 8 warps = 8 rows per block and round
    int64_t blocks = ceil_div64(P, threads / 32);
    const int64_t cap = (int64_t)device_info().sm_count * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(pdl_for(P), silu_mul_kernel, dim3((unsigned)blocks), dim3(threads), 0, stream, C1, topk_ids, P, E, I, h);
}

// ============================================================================
// Top-k weighted combine: out[t, n] = bf16_rne(sum_k w[t,k] * C2[t*topk+k, n])
// over local k in ascending order, FP32 from +0, each product and each sum
// rounded separately (no fused multiply-add); C2 in bf16 or in FP32.
// ============================================================================
template <bool F32>
__device__ __forceinline__ void load4(const void* C2v, int64_t off, float (&c)[4]) {
    if constexpr (F32) {
        const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(C2v) + off);
        c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w;
    } else {
        const uint2 u = *reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(C2v) + off);
        c[0] = bf16_lo(u.x); c[1] = bf16_hi(u.x); c[2] = bf16_lo(u.y); c[3] = bf16_hi(u.y);
    }
}

// Many tokens: 8 columns per thread, one pair after the other; occupancy
// keeps enough rows in flight.
template <bool F32>
__global__ void combine_kernel(const void* __restrict__ C2v, const int32_t* __restrict__ ids,
                               const float* __restrict__ w, int T, int topk, int E, int H, uint16_t* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const int vpr = H / 8;
    const int64_t nvec = (int64_t)T * vpr;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += (int64_t)gridDim.x * blockDim.x) {
        int nv;
        const int64_t t = divmod_idx(v, vpr, nv);
        const int n = nv * 8;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (int k = 0; k < topk; ++k) {
            const int64_t p = t * topk + k;
            const int e = ids[p];
            if (e < 0 || e >= E) continue;
            const float wk = w[p];
            float c[8], d[4];
            load4<F32>(C2v, p * H + n, d);
            c[0] = d[0]; c[1] = d[1]; c[2] = d[2]; c[3] = d[3];
            load4<F32>(C2v, p * H + n + 4, d);
            c[4] = d[0]; c[5] = d[1]; c[6] = d[2]; c[7] = d[3];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(wk, c[i]));
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(out + t * H + n) = o;
    }
}

// Few tokens (latency-bound): 4 columns per thread, and the k loop in batches
// of kBatch: the ids and weights of a batch are loaded together, then the
// local pairs' rows together, then added in k order.
template <bool F32>
__global__ void combine_few_kernel(const void* __restrict__ C2v, const int32_t* __restrict__ ids,
                               const float* __restrict__ w, int T, int topk, int E, int H, uint16_t* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    constexpr int kBatch = 8;
    const int vpr = H / 4;
    const int64_t nvec = (int64_t)T * vpr;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += (int64_t)gridDim.x * blockDim.x) {
        int nv;
        const int64_t t = divmod_idx(v, vpr, nv);
        const int n = nv * 4;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int k0 = 0; k0 < topk; k0 += kBatch) {
            bool local[kBatch];
            float wk[kBatch];
#pragma unroll
            for (int j = 0; j < kBatch; ++j) {
                local[j] = false;
                wk[j] = 0.0f;
                if (k0 + j < topk) {
                    const int64_t p = t * topk + k0 + j;
                    const int e = __ldg(ids + p);
                    local[j] = e >= 0 && e < E;
                    wk[j] = __ldg(w + p);
                }
            }
            float c[kBatch][4];
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (local[j]) load4<F32>(C2v, (t * topk + k0 + j) * H + n, c[j]);
#pragma unroll
            for (int j = 0; j < kBatch; ++j)
                if (local[j])
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(wk[j], c[j][i]));
        }
        uint2 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        *reinterpret_cast<uint2*>(out + t * H + n) = o;
    }
}

cudaError_t launch_combine(const void* C2, bool c2_f32, const int32_t* topk_ids, const float* topk_w, int T,
                           int topk, int E, int H, uint16_t* out, cudaStream_t stream) {
    if ((int64_t)T * H == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t sms = device_info().sm_count;
    // one thread per 4 columns fits in about one wave of 256-thread blocks per SM
    const bool few = (int64_t)T * (H / 4) <= sms * threads;
    const int64_t nvec = few ? (int64_t)T * (H / 4) : (int64_t)T * (H / 8);
    int64_t blocks = ceil_div64(nvec, threads);
    if (blocks > sms * 8) blocks = sms * 8;
    auto kern = few ? (c2_f32 ? combine_few_kernel<true> : combine_few_kernel<false>)
                    : (c2_f32 ? combine_kernel<true> : combine_kernel<false>);
    return launch_pdl(pdl_for((int64_t)T * topk), kern, dim3((unsigned)blocks), dim3(threads), 0, stream, C2, topk_ids,
                      topk_w, T, topk, E, H, out);
}

// ============================================================================
// Fused top-k combine.  The down GEMM writes the output of a token whose only
// local pair it computes directly (bf16(0 + w * sum), what the combine would
// compute for one pair); the plan below tells it which pairs those are, and
// the finishing pass sums the tokens with several local pairs exactly as the
// combine does (FP32 from +0 over local k in ascending order, each product and
// sum rounded separately) and writes +0 for tokens with none.
// ============================================================================

// pair_w[p] = topk_w[p] for the local pair of a token with exactly one local
// pair; NaN for the local pairs of tokens with several.  One thread per token.
__global__ void combine_plan_kernel(const int32_t* __restrict__ ids, const float* __restrict__ w, int T, int topk,
                                    int E, float* __restrict__ pair_w) {
    pdl_trigger();
    pdl_wait();
    for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < T; t += (int64_t)gridDim.x * blockDim.x) {
        int cnt = 0;
        for (int k = 0; k < topk; ++k) {
            const int e = __ldg(ids + t * topk + k);
            cnt += (e >= 0 && e < E) ? 1 : 0;
        }
        for (int k = 0; k < topk; ++k) {
            const int64_t p = t * topk + k;
            const int e = __ldg(ids + p);
            if (e >= 0 && e < E) pair_w[p] = cnt == 1 ? __ldg(w + p) : __int_as_float(0x7fc00000);
        }
    }
}

// One thread per (token, 8 columns), as in the combine pass (one warp per
// token walked its columns serially and was latency-bound): a token with one
// local pair of finite weight was written by the GEMM and is skipped;
// otherwise its local pairs' FP32 rows are added in ascending k (+0 when it
// has none).  topk <= 32.
__global__ void combine_finish_kernel(const float* __restrict__ C2, const int32_t* __restrict__ ids,
                                      const float* __restrict__ w, int T, int topk, int E, int H,
                                      uint16_t* __restrict__ out) {
    pdl_trigger();
    pdl_wait();
    const int vpr = H / 8;
    const int64_t nvec = (int64_t)T * vpr;
    for (int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; v < nvec; v += (int64_t)gridDim.x * blockDim.x) {
        int nv;
        const int64_t t = divmod_idx(v, vpr, nv);
        const int n = nv * 8;
        uint32_t mask = 0;
        for (int k = 0; k < topk; ++k) {
            const int e = __ldg(ids + t * topk + k);
            if (e >= 0 && e < E) mask |= 1u << k;
        }
        if (__popc(mask) == 1) {
            const float w1 = __ldg(w + t * topk + (__ffs(mask) - 1));
            if (w1 == w1) continue;   // written by the down GEMM's epilogue
        }
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        for (uint32_t m = mask; m; m &= m - 1) {
            const int64_t p = t * topk + (__ffs(m) - 1);
            const float wv = __ldg(w + p);
            const float4 c0 = __ldcg(reinterpret_cast<const float4*>(C2 + p * H + n));
            const float4 c1 = __ldcg(reinterpret_cast<const float4*>(C2 + p * H + n + 4));
            const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], __fmul_rn(wv, c[i]));
        }
        uint4 o;
        o.x = pack_bf16x2(acc[0], acc[1]);
        o.y = pack_bf16x2(acc[2], acc[3]);
        o.z = pack_bf16x2(acc[4], acc[5]);
        o.w = pack_bf16x2(acc[6], acc[7]);
        *reinterpret_cast<uint4*>(out + t * H + n) = o;
    }
}

cudaError_t launch_combine_plan(const int32_t* topk_ids, const float* topk_w, int T, int topk, int E, float* pair_w,
                                cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = ceil_div64(T, threads);
    const int64_t cap = (int64_t)device_info().sm_count * 4;
    if (blocks > cap) blocks = cap;
    return launch_pdl(pdl_for((int64_t)T * topk), combine_plan_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                      stream, topk_ids, topk_w, T, topk, E, pair_w);
}

cudaError_t launch_combine_finish(const float* C2, const int32_t* topk_ids, const float* topk_w, int T, int topk,
                                  int E, int H, uint16_t* out, cudaStream_t stream) {
    if ((int64_t)T * H == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = ceil_div64((int64_t)T * (H / 8), threads);
    const int64_t cap = (int64_t)device_info().sm_count * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(pdl_for((int64_t)T * topk), combine_finish_kernel, dim3((unsigned)blocks), dim3(threads), 0,
                      stream, C2, topk_ids, topk_w, T, topk, E, H, out);
}

}  // namespace chord
