// Decode-regime indexed W4A16 GEMM for sm_103a (warp-level tensor-core MMA).
//
// Few routed rows per expert (tok_e of order 10) make this projection a
// weight stream: every packed INT4 byte is read once and used for at most a
// few dozen tokens.  The kernel therefore
//   * swaps the operands (the article's decode profile, section "H200 and
//     Blackwell indexed decode"): dequantised weights fill the 16-row M side
//     of a warp-level m16n8k16 BF16 MMA, the block's tokens its N side, so
//     8 tokens cost one MMA instead of a 128-row tile of padding;
//   * streams the packed 128-row x 128-column weight stage (two contiguous
//     4608-byte chunks of the 128x64-chunk layout) with one bulk asynchronous
//     copy (cp.async.bulk, completion counted on an mbarrier) into a
//     STAGES-deep shared-memory ring, issued by one producer warp;
//   * gathers the block's activation rows (one 256-byte row slice per token
//     and stage, row = pair id / a_row_divisor, sentinels skipped) into the
//     same stage;
//   * dequantises in registers: lane (g, c) of a warp owns columns
//     [16c, 16c + 16) of every 64-column chunk for rows g and g + 8 of its
//     16-row tile.  The MMA's K order inside a chunk is permuted to match (the
//     k16 step s takes columns 16c + 4s .. 16c + 4s + 3 of each lane, for the
//     A and the B fragment alike), so one 8-byte shared load gives a lane the
//     codes of four k16 steps.  0x4300|q is 128+q, minus 136 gives q-8
//     exactly, one bf16x2 multiply by the group scale rounds once ("subtract
//     then scale"); when the blob's header says every scale lies in
//     [2^-126, 0.5), one bf16x2 FMA per pair computes the same value
//     (dequant_row8_fma);
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

constexpr int kBN = 128;                          // output rows per item
constexpr int kKS = 128;                          // K columns per stage
constexpr int kChunk2 = 4608;                     // one 128-row x 64-column packed chunk
constexpr int kWStageBytes = (kKS / 64) * kChunk2;
constexpr int kXStride = kKS * 2 + 16;            // padded token row: conflict-free 16-byte loads

// NT: 8-token MMA tiles per item; MI: 16-row tiles per consumer warp (the
// item's 128 rows are split over 8 / MI consumer warps).
template <int NT, int MI = 2>
struct Cfg {
    static constexpr int kTok = NT * 8;
    static constexpr int kStageBytes = kWStageBytes + kTok * kXStride;
    static constexpr int kConsumerWarps = 8 / MI;
    static constexpr int kThreads = (kConsumerWarps + 1) * 32;
};

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Epilogue of a launch, fixed at compile time so that each kernel carries
// only its own store path (the consumer loop is instantiated once per token
// tile count and dequantisation form; every store path inlined into each of
// those copies made the loop longer than the instruction cache holds).
enum Epi : int {
    kEpiStore = 0,     // C[pair, n]: bf16, or FP32 with out_f32
    kEpiSilu = 1,      // h[pair, j] = SiLU(gate) * up (packed layout 3)
    kEpiPartial = 2,   // FP32 partial sums of one K slice
    kEpiCombine = 3,   // fused top-k combine (FP32 sums of multi-pair tokens)
};

// Per-item routing facts, computed identically by the producer and the
// consumers from the same global data.  At most 32 token slots per item.
struct ItemRows {
    int32_t id;       // pair id of token slot `lane` (or -1)
    uint32_t vmask;   // slots holding a valid pair id
};

template <int NT>
__device__ __forceinline__ ItemRows load_item_rows(const GemmArgs& a, int64_t b, int sub, int lane, int* err) {
    static_assert(Cfg<NT>::kTok <= 32, "one token slot per lane");
    ItemRows r;
    int32_t id = -1;
    bool ok = false;
    const int slot_in_block = sub * Cfg<NT>::kTok + lane;
    if (lane < Cfg<NT>::kTok && slot_in_block < a.block_m) {
        id = a.sorted_ids[b * a.block_m + slot_in_block];
        if (id != (int32_t)a.num_pairs) {
            ok = id >= 0 && (int64_t)id < a.id_limit;
            if (!ok) set_error(err, CHORD_DEV_BAD_ROW);
        }
    }
    r.id = ok ? id : -1;
    r.vmask = __ballot_sync(0xffffffffu, ok);
    return r;
}

// One 64-column chunk: dequantise the warp's MI 16-row tiles (lane (g, c):
// rows g and g + 8, columns [16c, 16c + 16)) and accumulate them against NV
// 8-token tiles.  `row0` = the warp's first row + g; `xa` = shared address of
// token g's columns 16c.. of this chunk.  FD: the blob's scales all lie in
// [2^-126, 0.5) and each weight pair costs one FMA (dequant_row8_fma).  The
// B fragments are loaded first; each 16-row tile's MMAs follow its own
// dequantisation, so only one tile's A registers are live at a time
// (measured 3 % faster on EP8 decode than dequantising both tiles first).
template <int MI, int NV, bool FD>
__device__ __forceinline__ void chunk_mma(const uint8_t* cb, int row0, uint32_t code_off, uint32_t scale_sel,
                                          uint32_t xa, float (&acc)[MI][NV][4]) {
    // B fragments of token 8t + g, the same 16 columns
    uint32_t bv[NV][8];
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        const uint32_t x = xa + (uint32_t)(t * 8 * kXStride);
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(bv[t][0]), "=r"(bv[t][1]), "=r"(bv[t][2]), "=r"(bv[t][3])
                     : "r"(x));
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(bv[t][4]), "=r"(bv[t][5]), "=r"(bv[t][6]), "=r"(bv[t][7])
                     : "r"(x + 16));
    }
#pragma unroll
    for (int mi = 0; mi < MI; ++mi) {
        // av[r][p] = bf16x2 pair p (columns 16c + 2p, +1) of row g (r = 0) or g + 8 (r = 1)
        uint32_t av[2][8];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = row0 + mi * 16 + r * 8;
            const uint2 w = *reinterpret_cast<const uint2*>(cb + code_off + row * 16);
            const uint32_t sp = prmt(*reinterpret_cast<const uint32_t*>(cb + 4096 + row * 4), scale_sel);
            if (FD) {
                uint32_t b2, c2;
                fma_scale_pair(sp, b2, c2);
                dequant_row8_fma(w.x, b2, c2, av[r]);
                dequant_row8_fma(w.y, b2, c2, av[r] + 4);
            } else {
                dequant_row8(w.x, sp, av[r]);
                dequant_row8(w.y, sp, av[r] + 4);
            }
        }
        // k16 step st takes columns 16c + 4st .. + 3 of every lane, for A and B alike
#pragma unroll
        for (int st = 0; st < 4; ++st) {
#pragma unroll
            for (int t = 0; t < NV; ++t) {
                const uint32_t af[4] = {av[0][2 * st], av[1][2 * st], av[0][2 * st + 1], av[1][2 * st + 1]};
                mma_bf16_16816(acc[mi][t], af, bv[t][2 * st], bv[t][2 * st + 1]);
            }
        }
    }
}

// Consumer side of one item whose valid token slots lie in its first NV
// 8-token tiles (align fills a block's slots from the front): the K loop over
// the stage ring, then the epilogue.  Returns false when a wait gave up.
template <int NT, int STAGES, int MI, int NV, bool FD, int EPI>
__device__ __forceinline__ bool consume_item(const GemmArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                          volatile int* flags, int64_t& stage, int warp, int lane, int nt,
                                          int32_t my_id, int ks0, int ks1, int slice) {
    constexpr int kStage = Cfg<NT>::kStageBytes;
    const int g = lane >> 2, c = lane & 3;
    // lane (g, c) reads the two code words (c & 1) * 2, +1 of the 32-column
    // half c >> 1 of each of its rows, and that half's scale
    const uint32_t code_off = (uint32_t)((c >> 1) * 2048 + (c & 1) * 8);
    const uint32_t scale_sel = (c >> 1) ? 0x3232u : 0x1010u;   // prmt: that half's scale in both halves
    const int row0 = warp * MI * 16 + g;
    const uint32_t x_lane = (uint32_t)(g * kXStride + 32 * c);

    float acc[MI][NV][4];
#pragma unroll
    for (int mi = 0; mi < MI; ++mi)
#pragma unroll
        for (int t = 0; t < NV; ++t)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[mi][t][q] = 0.0f;

    const int ks_full = a.K / kKS;   // stages holding both 64-column chunks
    for (int ks = ks0; ks < ks1; ++ks, ++stage) {
        const int slot = (int)(stage % STAGES);
        const uint32_t par = (uint32_t)((stage / STAGES) & 1);
        // the abort flag is read only when the stage has not landed yet
        if (!mbar_try_wait(&full[slot], par) && (!mbar_wait(&full[slot], par) || flags[1])) {
            if (lane == 0) set_error(a.err, CHORD_DEV_TIMEOUT);
            flags[1] = 1;
            return false;
        }
        const uint8_t* sW = smem + slot * kStage;
        const uint32_t xa = smem_u32(sW + kWStageBytes) + x_lane;
        // both chunks' code in one block for a full stage, so the compiler can
        // schedule the second chunk's loads with the first chunk's math
        if (ks < ks_full) {
            chunk_mma<MI, NV, FD>(sW, row0, code_off, scale_sel, xa, acc);
            chunk_mma<MI, NV, FD>(sW + kChunk2, row0, code_off, scale_sel, xa + 128, acc);
        } else {
            chunk_mma<MI, NV, FD>(sW, row0, code_off, scale_sel, xa, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
    }

    // ---- epilogue: C[p, n] = acc (bf16-rounded or FP32) for valid token columns
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        int32_t p[2];
        float pw[2] = {0.0f, 0.0f};   // fused combine: the pair's weight when it is its token's only local pair
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            p[u] = __shfl_sync(0xffffffffu, my_id, 8 * t + 2 * c + u);
            if (EPI == kEpiCombine && p[u] >= 0) pw[u] = a.pair_w[p[u]];
        }
#pragma unroll
        for (int mi = 0; mi < MI; ++mi) {
            const int n0 = nt * kBN + (warp * MI + mi) * 16 + g;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                if (p[u] < 0) continue;
                if (EPI == kEpiPartial) {
                    // K slice `slice`: FP32 partial sums in packed row order
                    float* prow = a.partial + ((int64_t)slice * a.num_pairs + p[u]) * a.N;
                    prow[n0] = acc[mi][t][u];
                    prow[n0 + 8] = acc[mi][t][2 + u];
                } else if (EPI == kEpiSilu) {
                    // packed rows n0 = 16k + g and n0 + 8 hold gate and up of
                    // column j = 8k + g (layout 3)
                    __nv_bfloat16* hrow = static_cast<__nv_bfloat16*>(a.C) + (int64_t)p[u] * (a.N / 2);
                    hrow[8 * (n0 / 16) + g] = silu_mul_bf16(acc[mi][t][u], acc[mi][t][2 + u]);
                } else if (EPI == kEpiCombine) {
                    const int64_t tok = p[u] / a.topk;
                    combine_store(static_cast<float*>(a.C), a.out, a.N, p[u], tok, pw[u], n0, acc[mi][t][u]);
                    combine_store(static_cast<float*>(a.C), a.out, a.N, p[u], tok, pw[u], n0 + 8, acc[mi][t][2 + u]);
                } else if (a.out_f32) {
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
    return true;
}

// consume_item instantiated for the item's count of 8-token tiles.
template <int NT, int STAGES, int MI, bool FD, int EPI>
__device__ __forceinline__ bool consume_nv(const GemmArgs& a, uint8_t* smem, uint64_t* full, uint64_t* empty,
                                           volatile int* flags, int64_t& stage, int warp, int lane, int nt,
                                           int32_t my_id, int ks0, int ks1, int slice, int nv) {
    if (nv <= 1)
        return consume_item<NT, STAGES, MI, 1, FD, EPI>(a, smem, full, empty, flags, stage, warp, lane, nt, my_id, ks0,
                                                   ks1, slice);
    if (nv == 2 || NT == 2)
        return consume_item<NT, STAGES, MI, (NT >= 2 ? 2 : 1), FD, EPI>(a, smem, full, empty, flags, stage, warp, lane,
                                                                   nt, my_id, ks0, ks1, slice);
    if (nv == 3)
        return consume_item<NT, STAGES, MI, (NT >= 4 ? 3 : 1), FD, EPI>(a, smem, full, empty, flags, stage, warp, lane,
                                                                   nt, my_id, ks0, ks1, slice);
    return consume_item<NT, STAGES, MI, (NT >= 4 ? 4 : 1), FD, EPI>(a, smem, full, empty, flags, stage, warp, lane, nt,
                                                               my_id, ks0, ks1, slice);
}

// Mixed regime: whether align block b is one of the small blocks this launch
// takes (at most 32 valid rows; the valid rows of a block are a prefix).
__device__ __forceinline__ bool block_taken(const GemmArgs& a, int64_t b) {
    if (a.block_filter != kBlocksSmall || a.block_m <= CHORD_MIXED_SMALL_ROWS) return true;
    return a.sorted_ids[b * a.block_m + CHORD_MIXED_SMALL_ROWS] == (int32_t)a.num_pairs;
}

// Work unit -> (align block b, token sub-block, 128-row N tile, K slice and
// its stage range); 32-bit divisions while the unit index fits (always, in
// practice), no slice arithmetic when K is not split.
__device__ __forceinline__ int64_t unit_coords(int64_t unit, int S, int ntiles, int nsub, int kstages, int& slice,
                                               int& nt, int& sub, int& ks0, int& ks1) {
    int64_t item = unit;
    slice = 0;
    ks0 = 0;
    ks1 = kstages;
    if (S > 1) {
        item = divmod_idx(unit, S, slice);
        ks0 = slice * kstages / S;
        ks1 = (slice + 1) * kstages / S;
    }
    const int64_t bs = divmod_idx(item, ntiles, nt);
    return divmod_idx(bs, nsub, sub);
}

template <int NT, int STAGES, int MI, int MINB, int EPI>
__global__ void __launch_bounds__(Cfg<NT, MI>::kThreads, MINB) gemm_decode_kernel(const GemmArgs a) {
    pdl_trigger();
    pdl_wait();
    constexpr int kConsumerWarps = Cfg<NT, MI>::kConsumerWarps;
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kTok = Cfg<NT>::kTok;
    constexpr int kStage = Cfg<NT>::kStageBytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * kStage);
    uint64_t* empty = full + STAGES;
    // [0] skip, [1] abort, [2] num_tokens_padded, [3] every scale in the one-FMA dequantisation's range
    volatile int* flags = reinterpret_cast<volatile int*>(empty + STAGES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        const bool ok = header_ok_layout(a.packed, a.E, a.N, a.K, a.layout);
        if (!ok) set_error(a.err, CHORD_DEV_BAD_HEADER);
        flags[0] = ok ? 0 : 1;
        flags[1] = 0;
        flags[3] = ok && header_scales_in_fma_range(a.packed) ? 1 : 0;
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 33);        // the weight copy's expect_tx + one cp.async arrival per producer lane
            mbar_init(&empty[s], kConsumerWarps);
        }
        fence_barrier_init();
    }
    if (threadIdx.x == 32) flags[2] = *a.ntp;   // read while thread 0 checks the header
    __syncthreads();
    if (flags[0]) return;

    int32_t ntp = flags[2];
    if (ntp < 0 || ntp > a.capacity || ntp % a.block_m) {
        if (threadIdx.x == 0) set_error(a.err, CHORD_DEV_BAD_PADDED);
        ntp = 0;
    }
    // token sub-blocks (slots past block_m are empty); the mixed regime's small
    // blocks have all their rows in the first
    const int nsub = a.block_filter == kBlocksSmall ? 1 : (a.block_m + kTok - 1) / kTok;
    const int ntiles = a.N / kBN;
    const int64_t n_items = (int64_t)(ntp / a.block_m) * nsub * ntiles;
    const int kstages = (a.K + kKS - 1) / kKS;
    // Work unit = (item, K slice): slice s of S takes stages [s*kstages/S, (s+1)*kstages/S)
    const int S = a.ksplit > 1 ? a.ksplit : 1;
    const int64_t n_units = n_items * S;
    const int kchunks = a.K / 64;
    const uint64_t expert_bytes = (uint64_t)a.N * (uint64_t)a.K * 9ull / 16ull;
    const uint8_t* wbase = a.packed + kHeaderBytes;

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        const uint64_t pol = policy_evict_first();
        int64_t stage = 0;
        bool aborted = false;
        for (int64_t unit = blockIdx.x; unit < n_units && !aborted; unit += gridDim.x) {
            int slice, nt, sub, ks0, ks1;
            const int64_t b = unit_coords(unit, S, ntiles, nsub, kstages, slice, nt, sub, ks0, ks1);
            if (!block_taken(a, b)) continue;
            const int e = a.expert_ids[b];
            if (e < 0 || e >= a.E) {
                if (lane == 0) set_error(a.err, CHORD_DEV_BAD_EXPERT);
                continue;
            }
            const ItemRows rows = load_item_rows<NT>(a, b, sub, lane, nullptr);
            const int nvalid = __popc(rows.vmask);
            if (nvalid == 0) continue;
            const uint8_t* wexp = wbase + (uint64_t)e * expert_bytes;
            // Activation rows: lanes 0-15 copy the 16-byte pieces of token slot
            // 2i, lanes 16-31 those of slot 2i + 1 (valid slots are a prefix).
            // Each lane's source pieces are found once per item, so a stage
            // costs the producer one copy instruction per token and lane (its
            // loop paces the whole ring: a shuffle and an address per token and
            // stage made it issue a stage in about 1200 cycles on EP8 decode).
            const int npairs = (32 - __clz(rows.vmask) + 1) / 2;
            const int half_lane = lane >> 4, piece = lane & 15;
            const int32_t my_row = rows.id < 0 ? -1 : (a.a_row_divisor == 1 ? rows.id : rows.id / a.a_row_divisor);
            const uint16_t* src[kTok / 2];
#pragma unroll
            for (int i = 0; i < kTok / 2; ++i) {
                if (i >= npairs) break;   // npairs is the same in every lane
                const int32_t r = __shfl_sync(0xffffffffu, my_row, 2 * i + half_lane);
                src[i] = r >= 0 ? a.A + (int64_t)r * a.K + piece * 8 : nullptr;
            }
            const uint32_t xlane = (uint32_t)(half_lane * kXStride + piece * 16);
            for (int ks = ks0; ks < ks1; ++ks) {
                const int slot = (int)(stage % STAGES);
                const uint32_t par = (uint32_t)((stage / STAGES) & 1);
                // the abort flag is read only when the slot is not free yet
                if (!mbar_try_wait(&empty[slot], par ^ 1u) && (!mbar_wait(&empty[slot], par ^ 1u) || flags[1])) {
                    if (lane == 0) set_error(a.err, CHORD_DEV_TIMEOUT);
                    flags[1] = 1;
                    aborted = true;
                    break;
                }
                const int nchunk = min(2, (a.K - ks * kKS) / 64);
                uint8_t* sW = smem + slot * kStage;
                const uint32_t sX = smem_u32(sW + kWStageBytes);
                if (lane == 0) {
                    // chunks (nt, kc) of one expert are contiguous along kc
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(nchunk * kChunk2));
                    const uint8_t* src = wexp + ((uint64_t)nt * kchunks + (uint64_t)(2 * ks)) * kChunk2;
                    bulk_g2s_hint(sW, src, (uint32_t)(nchunk * kChunk2), &full[slot], pol);
                }
                if (piece < nchunk * 8) {   // a one-chunk stage has 8 pieces per row
                    const int off = ks * kKS;
#pragma unroll
                    for (int i = 0; i < kTok / 2; ++i) {
                        if (i >= npairs) break;
                        if (src[i]) cp_async16(sX + xlane + (uint32_t)(i * 2 * kXStride), src[i] + off);
                    }
                }
                cp_async_arrive_noinc(&full[slot]);
                ++stage;
            }
        }
        // Leave only after every copy this warp issued has landed.
        cp_async_wait<0>();
        if (lane == 0) {
            for (int s = 0; s < STAGES && s < stage; ++s) {
                const int64_t last = s + ((stage - 1 - s) / STAGES) * STAGES;
                if (!mbar_wait(&full[s], (uint32_t)((last / STAGES) & 1))) set_error(a.err, CHORD_DEV_TIMEOUT);
            }
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const bool fma_dequant = flags[3] != 0;
    int64_t stage = 0;
    for (int64_t unit = blockIdx.x; unit < n_units; unit += gridDim.x) {
        int slice, nt, sub, ks0, ks1;
        const int64_t b = unit_coords(unit, S, ntiles, nsub, kstages, slice, nt, sub, ks0, ks1);
        if (!block_taken(a, b)) continue;
        const int e = a.expert_ids[b];
        if (e < 0 || e >= a.E) continue;
        const ItemRows rows = load_item_rows<NT>(a, b, sub, lane, slice == 0 ? a.err : nullptr);
        if (rows.vmask == 0) continue;
        const int nv = (32 - __clz(rows.vmask) + 7) / 8;   // 8-token tiles up to the last valid slot
        const bool ok = fma_dequant
                            ? consume_nv<NT, STAGES, MI, true, EPI>(a, smem, full, empty, flags, stage, warp, lane, nt,
                                                               rows.id, ks0, ks1, slice, nv)
                            : consume_nv<NT, STAGES, MI, false, EPI>(a, smem, full, empty, flags, stage, warp, lane, nt,
                                                                rows.id, ks0, ks1, slice, nv);
        if (!ok) return;
    }
}

template <int NT, int STAGES, int MI, int MINB, int EPI>
cudaError_t launch_epi(const GemmArgs& a, cudaStream_t stream) {
    using C = Cfg<NT, MI>;
    constexpr int smem = STAGES * C::kStageBytes + 2 * STAGES * 8 + 16;
    auto kern = gemm_decode_kernel<NT, STAGES, MI, MINB, EPI>;
    int per_sm = 1;
    cudaError_t e = kernel_ctas_per_sm(reinterpret_cast<const void*>(kern), C::kThreads, smem, smem, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t nsub = a.block_filter == kBlocksSmall ? 1 : (a.block_m + NT * 8 - 1) / (NT * 8);
    const int64_t items_cap = (a.capacity / a.block_m) * nsub * (a.N / kBN) * (a.ksplit > 1 ? a.ksplit : 1);
    int64_t grid = (int64_t)device_info().sm_count * per_sm;
    if (grid > items_cap) grid = items_cap;
    if (grid < 1) grid = 1;
    return launch_pdl(pdl_for(a.num_pairs), kern, dim3((unsigned)grid), dim3(C::kThreads), (size_t)smem, stream, a);
}

template <int NT, int STAGES, int MI, int MINB>
cudaError_t launch_nt(const GemmArgs& a, cudaStream_t stream) {
    if (a.ksplit > 1) return launch_epi<NT, STAGES, MI, MINB, kEpiPartial>(a, stream);
    if (a.silu) return launch_epi<NT, STAGES, MI, MINB, kEpiSilu>(a, stream);
    if (a.combine) return launch_epi<NT, STAGES, MI, MINB, kEpiCombine>(a, stream);
    return launch_epi<NT, STAGES, MI, MINB, kEpiStore>(a, stream);
}

}  // namespace

cudaError_t launch_gemm_decode(const GemmArgs& a, cudaStream_t stream) {
    // Tokens per item: the smallest of 8/16/32 that holds the whole block
    // (larger blocks are split into 32-token sub-blocks, each re-streaming the
    // weights; the tcgen05 kernel serves those blocks by default).  Ring depth
    // and CTAs per SM as measured fastest on GB300 among 2-5 CTAs per SM and
    // 3-6 stages: three CTAs for 8- and 32-token items, four with four stages
    // for 16-token items (TP8 T=128 gate_up + down 289 -> 272 us).
    if (a.block_m <= 8) return launch_nt<1, 6, 2, 3>(a, stream);
    if (a.block_m <= 16) return launch_nt<2, 4, 2, 4>(a, stream);
    return launch_nt<4, 4, 2, 3>(a, stream);
}

}  // namespace chord
