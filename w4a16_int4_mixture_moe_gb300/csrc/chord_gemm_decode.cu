// Decode-regime indexed W4A16 GEMM for sm_103a.
//
// Few routed rows per expert (tok_e of order 10) make this projection a
// weight stream: every packed INT4 byte is read once and used for at most a
// few dozen tokens.  The kernel therefore
//   * swaps the operands (the article's decode profile, section "H200 and
//     Blackwell indexed decode"): dequantised weights fill the 16-row M side
//     of a warp-level m16n8k16 BF16 MMA, the block's tokens its N side, so
//     8 tokens cost one MMA instead of a 128-row tile of padding;
//   * streams weights with bulk asynchronous copies (cp.async.bulk, completion
//     counted on mbarriers) into a STAGES-deep shared-memory ring, issued by
//     one producer warp, so tens of KB per SM are in flight;
//   * gathers the block's activation rows (one 256-byte row slice per token
//     and stage, row = pair id / a_row_divisor, sentinels skipped) into the
//     same stage;
//   * dequantises in registers: one 16-byte shared load gives a lane the codes
//     of four k16 steps of its A fragment (the packed layout is built for it),
//     0x4300|q gives 128+q, minus 136 gives q-8 exactly, one bf16x2 multiply
//     by the group scale rounds once ("subtract then scale");
//   * runs persistently: CTA i takes work items i, i + grid, ... where an item
//     is (align block, 8*NT-token sub-block, 128-row N tile), bounded on the
//     device by num_tokens_padded, so nothing is read back to the host.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "chord_common.cuh"
#include "chord_internal.h"

namespace chord {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kBN = kConsumerWarps * 32;          // 128 output rows per item
constexpr int kMtiles = kBN / 16;                 // 8 m16 tiles
constexpr int kKS = 128;                          // K columns per stage
constexpr int kChunkSpan = kMtiles * kChunkBytes; // 4608: one 64-column chunk of 8 m-tiles
constexpr int kWStageBytes = (kKS / 64) * kChunkSpan;
constexpr int kXStride = kKS * 2 + 16;            // padded token row: conflict-free ldmatrix

template <int NT>
struct Cfg {
    static constexpr int kTok = NT * 8;
    static constexpr int kStageBytes = kWStageBytes + kTok * kXStride;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n" : "=r"(r0), "=r"(r1) : "r"(addr));
}

// Per-item routing facts, computed identically by the producer and the
// consumers from the same global data.
struct ItemRows {
    int32_t id[2];    // pair id of token slots lane and lane + 32 (or -1)
    uint32_t vmask[2];
};

template <int NT>
__device__ __forceinline__ ItemRows load_item_rows(const GemmArgs& a, int64_t b, int sub, int lane, int* err) {
    ItemRows r;
#pragma unroll
    for (int s = 0; s < 2; ++s) {
        const int i = lane + 32 * s;
        int32_t id = -1;
        bool ok = false;
        if (i < Cfg<NT>::kTok) {
            id = a.sorted_ids[b * a.block_m + (int64_t)sub * Cfg<NT>::kTok + i];
            if (id != (int32_t)a.num_pairs) {
                ok = id >= 0 && (int64_t)id < a.num_pairs && (int64_t)(id / a.a_row_divisor) < a.a_rows;
                if (!ok) set_error(err, CHORD_DEV_BAD_ROW);
            }
        }
        r.id[s] = ok ? id : -1;
        r.vmask[s] = __ballot_sync(0xffffffffu, ok);
    }
    return r;
}

template <int NT, int STAGES>
__global__ void __launch_bounds__(kThreads) gemm_decode_kernel(const GemmArgs a) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kTok = Cfg<NT>::kTok;
    constexpr int kStage = Cfg<NT>::kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * kStage);
    uint64_t* empty = full + STAGES;
    volatile int* flags = reinterpret_cast<volatile int*>(empty + STAGES);  // [0] skip, [1] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        const bool ok = header_ok(a.packed, a.E, a.N, a.K);
        if (!ok) set_error(a.err, CHORD_DEV_BAD_HEADER);
        flags[0] = ok ? 0 : 1;
        flags[1] = 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    __syncthreads();
    if (flags[0]) return;

    int32_t ntp = *a.ntp;
    if (ntp < 0 || ntp > a.capacity || ntp % a.block_m) {
        if (threadIdx.x == 0) set_error(a.err, CHORD_DEV_BAD_PADDED);
        ntp = 0;
    }
    const int nsub = a.block_m / kTok;
    const int ntiles = a.N / kBN;
    const int64_t n_items = (int64_t)(ntp / a.block_m) * nsub * ntiles;
    const int kstages = (a.K + kKS - 1) / kKS;
    const int mt_total = a.N / 16;
    const uint64_t expert_bytes = (uint64_t)a.N * (uint64_t)a.K * 9ull / 16ull;
    const uint8_t* wbase = a.packed + kHeaderBytes;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        int64_t stage = 0;
        bool aborted = false;
        for (int64_t item = blockIdx.x; item < n_items && !aborted; item += gridDim.x) {
            const int nt = (int)(item % ntiles);
            const int64_t bs = item / ntiles;
            const int sub = (int)(bs % nsub);
            const int64_t b = bs / nsub;
            const int e = a.expert_ids[b];
            if (e < 0 || e >= a.E) {
                if (lane == 0) set_error(a.err, CHORD_DEV_BAD_EXPERT);
                continue;
            }
            const ItemRows rows = load_item_rows<NT>(a, b, sub, lane, nullptr);
            const int nvalid = __popc(rows.vmask[0]) + __popc(rows.vmask[1]);
            if (nvalid == 0) continue;
            const uint8_t* wexp = wbase + (uint64_t)e * expert_bytes;
            const uint16_t* arow[2];
#pragma unroll
            for (int s = 0; s < 2; ++s)
                arow[s] = rows.id[s] >= 0 ? a.A + (int64_t)(rows.id[s] / a.a_row_divisor) * a.K : nullptr;
            for (int ks = 0; ks < kstages; ++ks) {
                const int slot = (int)(stage % STAGES);
                const uint32_t par = (uint32_t)((stage / STAGES) & 1);
                if (!mbar_wait(&empty[slot], par ^ 1u) || flags[1]) {
                    if (lane == 0) set_error(a.err, CHORD_DEV_TIMEOUT);
                    flags[1] = 1;
                    aborted = true;
                    break;
                }
                const int nchunk = min(2, (a.K - ks * kKS) / 64);
                const uint32_t xbytes = (uint32_t)nchunk * 64u * 2u;
                uint8_t* sW = smem + slot * kStage;
                uint8_t* sX = sW + kWStageBytes;
                if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(nchunk * kChunkSpan) + nvalid * xbytes);
                __syncwarp();
                if (lane < nchunk) {
                    const int kc = ks * 2 + lane;
                    const uint8_t* src = wexp + ((uint64_t)kc * mt_total + (uint64_t)nt * kMtiles) * kChunkBytes;
                    bulk_g2s_hint(sW + lane * kChunkSpan, src, kChunkSpan, &full[slot], pol);
                }
#pragma unroll
                for (int s = 0; s < 2; ++s)
                    if (arow[s]) bulk_g2s(sX + (lane + 32 * s) * kXStride, arow[s] + ks * kKS, xbytes, &full[slot]);
                ++stage;
            }
        }
        // Leave only after every copy this warp issued has landed.
        if (lane == 0) {
            for (int s = 0; s < STAGES && s < stage; ++s) {
                const int64_t last = s + ((stage - 1 - s) / STAGES) * STAGES;
                if (!mbar_wait(&full[s], (uint32_t)((last / STAGES) & 1))) set_error(a.err, CHORD_DEV_TIMEOUT);
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int g = lane >> 2, c = lane & 3;
    int64_t stage = 0;
    // ldmatrix lane addressing: matrix q = lane / 8 (token tile +q/2, k half q%2), row lane % 8
    const int lm_q = lane >> 3, lm_r = lane & 7;
    for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
        const int nt = (int)(item % ntiles);
        const int64_t bs = item / ntiles;
        const int sub = (int)(bs % nsub);
        const int64_t b = bs / nsub;
        const int e = a.expert_ids[b];
        if (e < 0 || e >= a.E) continue;
        const ItemRows rows = load_item_rows<NT>(a, b, sub, lane, a.err);
        const uint64_t vm = (uint64_t)rows.vmask[0] | ((uint64_t)rows.vmask[1] << 32);
        if (vm == 0) continue;
        uint32_t tmask = 0;  // token tiles with at least one valid row
#pragma unroll
        for (int j = 0; j < NT; ++j)
            if ((vm >> (8 * j)) & 0xffull) tmask |= 1u << j;

        float acc[2][NT][4];
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[mi][j][q] = 0.0f;

        bool aborted = false;
        for (int ks = 0; ks < kstages; ++ks) {
            const int slot = (int)(stage % STAGES);
            const uint32_t par = (uint32_t)((stage / STAGES) & 1);
            if (!mbar_wait(&full[slot], par) || flags[1]) {
                if (lane == 0) set_error(a.err, CHORD_DEV_TIMEOUT);
                flags[1] = 1;
                aborted = true;
                break;
            }
            const int nchunk = min(2, (a.K - ks * kKS) / 64);
            const uint8_t* sW = smem + slot * kStage;
            const uint32_t sX = smem_u32(sW + kWStageBytes);
            for (int ch = 0; ch < nchunk; ++ch) {
                uint4 wv[2];
                uint32_t sc[2][2];
#pragma unroll
                for (int mi = 0; mi < 2; ++mi) {
                    const uint8_t* cp = sW + ch * kChunkSpan + (warp * 2 + mi) * kChunkBytes;
                    wv[mi] = *reinterpret_cast<const uint4*>(cp + lane * 16);
                    sc[mi][0] = *reinterpret_cast<const uint32_t*>(cp + kChunkWeightBytes + g * 4);
                    sc[mi][1] = *reinterpret_cast<const uint32_t*>(cp + kChunkWeightBytes + (8 + g) * 4);
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int kcol = ch * 64 + j * 16;
                    uint32_t bf[NT][2];
                    if constexpr (NT == 1) {
                        const int q = lm_q & 1;
                        ldmatrix_x2(sX + (uint32_t)(lm_r * kXStride + (kcol + 8 * q) * 2), bf[0][0], bf[0][1]);
                    } else {
#pragma unroll
                        for (int tp = 0; tp < NT / 2; ++tp) {
                            if (tmask & (3u << (2 * tp))) {
                                const int tile = 2 * tp + (lm_q >> 1);
                                const uint32_t addr =
                                    sX + (uint32_t)((8 * tile + lm_r) * kXStride + (kcol + 8 * (lm_q & 1)) * 2);
                                ldmatrix_x4(addr, bf[2 * tp][0], bf[2 * tp][1], bf[2 * tp + 1][0], bf[2 * tp + 1][1]);
                            }
                        }
                    }
#pragma unroll
                    for (int mi = 0; mi < 2; ++mi) {
                        const uint32_t word = j == 0 ? wv[mi].x : j == 1 ? wv[mi].y : j == 2 ? wv[mi].z : wv[mi].w;
                        uint32_t af[4];
                        dequant_frag(word, sc[mi][j >> 1], af);
#pragma unroll
                        for (int t = 0; t < NT; ++t)
                            if (tmask & (1u << t)) mma_bf16_16816(acc[mi][t], af, bf[t][0], bf[t][1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
            ++stage;
        }
        if (aborted) return;

        // ---- epilogue: C[p, n] = acc (bf16-rounded or FP32) for valid token columns
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            if (!(tmask & (1u << t))) continue;
            const int i0 = 8 * t + 2 * c;  // token slots i0, i0 + 1
            int32_t p[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u;
                const int32_t lo = __shfl_sync(0xffffffffu, rows.id[0], i & 31);
                const int32_t hi = __shfl_sync(0xffffffffu, rows.id[1], i & 31);
                p[u] = i < 32 ? lo : hi;
            }
#pragma unroll
            for (int mi = 0; mi < 2; ++mi) {
                const int n0 = nt * kBN + (warp * 2 + mi) * 16 + g;
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    if (p[u] < 0) continue;
                    if (a.out_f32) {
                        float* crow = static_cast<float*>(a.C) + (int64_t)p[u] * a.N;
                        crow[n0] = acc[mi][t][u];
                        crow[n0 + 8] = acc[mi][t][2 + u];
                    } else {
                        __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(a.C) + (int64_t)p[u] * a.N;
                        crow[n0] = __float2bfloat16_rn(acc[mi][t][u]);
                        crow[n0 + 8] = __float2bfloat16_rn(acc[mi][t][2 + u]);
                    }
                }
            }
        }
    }
}

template <int NT, int STAGES>
cudaError_t launch_nt(const GemmArgs& a, cudaStream_t stream) {
    constexpr int smem = STAGES * Cfg<NT>::kStageBytes + 2 * STAGES * 8 + 16;
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(gemm_decode_kernel<NT, STAGES>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_decode_kernel<NT, STAGES>, kThreads,
                                                                  smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    const int64_t items_cap = (a.capacity / a.block_m) * (a.block_m / (NT * 8)) * (a.N / kBN);
    int64_t grid = (int64_t)device_info().sm_count * per_sm;
    if (grid > items_cap) grid = items_cap;
    if (grid < 1) grid = 1;
    gemm_decode_kernel<NT, STAGES><<<(unsigned)grid, kThreads, smem, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_decode(const GemmArgs& a, cudaStream_t stream) {
    // Token sub-block of the MMA N side: the largest of 64/32/16/8 dividing block_m.
    if (a.block_m % 64 == 0) return launch_nt<8, 4>(a, stream);
    if (a.block_m % 32 == 0) return launch_nt<4, 5>(a, stream);
    if (a.block_m % 16 == 0) return launch_nt<2, 6>(a, stream);
    return launch_nt<1, 6>(a, stream);
}

}  // namespace chord
