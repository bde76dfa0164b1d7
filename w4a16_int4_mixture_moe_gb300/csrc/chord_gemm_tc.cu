// Indexed W4A16 GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// One work item is (align block b, 128-row tile of N).  The product is
// computed with the operands swapped, as the article's decode profile does
// (section "H200 and Blackwell indexed decode"): the 128 dequantised weight
// rows are the MMA's M side and the block's routed tokens its N side, so a
// block of 11 rows costs an N = 16 MMA instead of a padded 128-row tile, and
// a block of 176 rows an N = 176 MMA.  Per 128-column K stage:
//   * a producer warp streams the stage's two packed 128x64 weight chunks
//     (9216 contiguous bytes, one cp.async.bulk) into a shared-memory ring;
//   * gather warps copy the block's activation rows (row = pair id / divisor)
//     with 16-byte cp.async into a 128-byte-swizzled K-major tile, the MMA's B
//     operand; each lane's copies arrive on the stage's barrier when they land
//     (cp.async.mbarrier.arrive.noinc) and the MMA thread fences the async
//     proxy before reading the tile;
//   * dequantising warps (one row per thread, two warpgroups taking alternate
//     stages) turn 32 codes per 16-byte load into bf16((q - 8) * s) (one
//     bf16x2 FMA per pair when the blob's header says every scale lies in
//     [2^-126, 0.5), as in the warp-level kernel) and store them with
//     tcgen05.st into a tensor-memory stage, the MMA's A operand (no
//     shared-memory round trip for the dequantised weights);
//   * an MMA-issuing thread issues eight tcgen05.mma (M=128, N=tokens rounded
//     up to 16, K=16) into its FP32 accumulator in tensor memory and commits
//     the stage back to the producers (several issuers take alternate stages
//     when the blocks are small);
// after the item's last stage the dequantising warps read the accumulator
// with tcgen05.ld and write the pair rows of C.  Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "chord_common.cuh"
#include "chord_internal.h"

namespace chord {
namespace {

constexpr int kTileRows = 128;   // rows of N per item = MMA M
constexpr int kChunkK = 64;      // K columns of one packed chunk; a pipeline stage holds two
constexpr int kChunk2 = 4608;    // packed bytes of one 128 x 64 chunk (layout 2)
constexpr int kACols = 64;       // tensor-memory columns of one A stage (128 bf16 per lane)
constexpr int kStgWarpBytes = 2048;   // drain buffer of one dequantising warp: 16 tokens x 32 rows x FP32

// The A operand ring lives in tensor memory (64 columns per stage, as many
// stages as the columns left after the accumulators allow, sized at launch);
// GW: gather warps; MAXR: token rows one gather lane copies per stage
// (block rows / (GW * 4)).  Eight dequantising warps form two warpgroups
// that take alternate stages.  The B-tile and packed-weight rings live in
// shared memory and are sized at launch.
// NI: MMA-issuing warps.  A tcgen05.mma costs its issuing thread tens of
// cycles whatever N is, so with few tokens per item several issuers, each
// accumulating every NI-th stage of the item into its own accumulator, keep
// the tensor pipe fed; the epilogue adds the partial accumulators in issuer
// order.
template <int GW, int MAXR, int NI>
struct Cfg {
    static constexpr int kDQ = 8;             // dequantising warps
    static constexpr int kProducer = kDQ;     // warp index of the weight producer (owns TMEM)
    static constexpr int kMma0 = kDQ + 1;     // first MMA-issuing warp
    static constexpr int kGather0 = kDQ + 1 + NI;  // first gather warp
    static constexpr int kWarps = kDQ + 1 + NI + GW;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kMaxTokens = MAXR * GW * 4;
};

struct TcArgs {
    GemmArgs g;
    int tok_tile;      // rows of the B tile: block_m rounded up to 16
    uint32_t tmem_cols;
    int nsb;           // stages of the B-tile ring (shared memory)
    int nsw;           // stages of the packed-weight ring (shared memory)
    int nsa;           // stages of the A ring (tensor memory)
};

// ---- tcgen05 / cp.async wrappers --------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// D[128 x N] (+)= A[128 x 16] (tensor memory) * B[N x 16]^T (shared memory descriptor)
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
        "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
        "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- pairs of CTAs (cta_group::2) ------------------------------------------
// With PAIR, a cluster of two CTAs on neighbouring SMs computes one
// M = 256 product: every tcgen05 instruction of the kernel then names
// cta_group::2 (alloc, relinquish and dealloc by the producer warp of both
// CTAs; MMAs and their commits by the leader CTA's issuing thread, the commits
// arriving on the same barrier of both CTAs).
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc_g(uint32_t* slot, uint32_t ncols) {
    if constexpr (PAIR)
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                     "r"(ncols)
                     : "memory");
    else
        tmem_alloc(slot, ncols);
}
template <bool PAIR>
__device__ __forceinline__ void tmem_relinquish_g() {
    if constexpr (PAIR)
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    else
        tmem_relinquish();
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc_g(uint32_t taddr, uint32_t ncols) {
    if constexpr (PAIR)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
    else
        tmem_dealloc(taddr, ncols);
}
// Arrive on `bar` (the same barrier of both CTAs of a pair) once this
// thread's MMAs so far have completed.
template <bool PAIR>
__device__ __forceinline__ void tc_commit_g(uint64_t* bar) {
    if constexpr (PAIR)
        asm volatile(
            "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                smem_u32(bar)),
            "h"((uint16_t)3)
            : "memory");
    else
        tc_commit(bar);
}
template <bool PAIR>
__device__ __forceinline__ void tc_mma_ts_g(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    if constexpr (PAIR)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
            "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        tc_mma_ts(d_tmem, a_tmem, b_desc, idesc, accumulate);
}
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on the leader CTA's copy of `bar` (the same shared-memory offset in
// CTA 0 of the cluster), releasing this thread's writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_leader(uint64_t* bar) {
    uint32_t ra;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(ra) : "r"(smem_u32(bar)));
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}
// try_wait acquiring at cluster scope (for phases completed by the peer CTA's arrivals)
__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Shared-memory matrix descriptor of a K-major operand tile with 128-byte
// swizzle: rows of 64 bf16 (128 bytes), 8-row atoms of 1024 bytes.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1u << 16;               // leading byte offset (unused for swizzled K-major)
    d |= (uint64_t)(1024u >> 4) << 32;     // stride byte offset: next 8-row atom
    d |= (uint64_t)1u << 46;               // descriptor version of tcgen05
    d |= (uint64_t)2u << 61;               // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: D F32, A and B BF16, both K-major, M = 128
// (M = 256 for a pair of CTAs).
__device__ __forceinline__ uint32_t idesc_bf16(int n, int m = kTileRows) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Bounded wait that also gives up once another role has aborted.  The abort
// flag and the clock are checked every 64 polls only.  CL: acquire at cluster
// scope (a phase that the peer CTA's arrivals complete).
template <bool CL>
__device__ __forceinline__ bool try_wait_g(uint64_t* bar, uint32_t parity) {
    if constexpr (CL)
        return mbar_try_wait_cl(bar, parity);
    else
        return mbar_try_wait(bar, parity);
}

template <bool CL = false>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
    if (try_wait_g<CL>(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 1;; ++it) {
        if (try_wait_g<CL>(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort_flag) return false;
            if (clock64() - t0 > kWaitLimitCycles) {
                set_error(err, CHORD_DEV_TIMEOUT);
                *abort_flag = 1;
                return false;
            }
        }
    }
}

// Routing facts of one item, computed identically by every role from the
// same global data: whether any row is valid and the MMA's N (the tokens up
// to the last valid row, rounded up to 16).
struct ItemInfo {
    int e;
    int n_mma;   // 0: nothing to do
};

__device__ __forceinline__ bool row_valid(const GemmArgs& a, int32_t id) {
    return id >= 0 && (int64_t)id < a.id_limit;   // the sentinel num_pairs is never below id_limit
}

__device__ __forceinline__ ItemInfo item_info(const GemmArgs& a, int64_t b, int lane, bool report) {
    // All loads first (a block holds at most 256 rows: 8 per lane), so the
    // item's routing costs one memory latency, not one per row group.
    ItemInfo r;
    r.e = a.expert_ids[b];
    int32_t ids[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int i = lane + 32 * k;
        ids[k] = i < a.block_m ? a.sorted_ids[b * a.block_m + i] : (int32_t)a.num_pairs;
    }
    r.n_mma = 0;
    if (r.e < 0 || r.e >= a.E) {
        if (report && lane == 0) set_error(a.err, CHORD_DEV_BAD_EXPERT);
        return r;
    }
    int last = -1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int i = lane + 32 * k;
        const bool ok = row_valid(a, ids[k]);
        if (report && !ok && ids[k] != (int32_t)a.num_pairs) set_error(a.err, CHORD_DEV_BAD_ROW);
        if (ok) last = i;
    }
    last = __reduce_max_sync(0xffffffffu, last + 1);
    // mixed regime: a block whose slot 32 holds the sentinel has at most 32
    // valid rows (they are a prefix) and belongs to the warp-level launch
    if (a.block_filter == kBlocksLarge && __shfl_sync(0xffffffffu, ids[1], 0) == (int32_t)a.num_pairs) last = 0;
    r.n_mma = (last + 15) / 16 * 16;
    return r;
}

// Position in a ring of n stages: slot and the parity of the slot's current
// fill.  Producers wait for the previous fill's release (parity ^ 1),
// consumers for the fill itself (parity).  Advanced by one stage at a time, so
// no division on the hot path.
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
    __device__ __forceinline__ void prev(int n) {
        if (slot == 0) {
            slot = n - 1;
            phase ^= 1u;
        } else {
            --slot;
        }
    }
};

// A work unit: an item with the K stages [ks0, ks1) it covers; pidx >= 0
// marks a unit of the split tail (tail_plan), whose FP32 sums go to
// partial[pidx] instead of C.
struct Unit {
    int64_t item;
    int ks0, ks1;
    int64_t pidx;
};

__device__ __forceinline__ Unit unit_at(int64_t u, const TailPlan& tp, int kstages) {
    Unit r;
    if (u < tp.full || tp.S == 1) {
        r.item = u;
        r.ks0 = 0;
        r.ks1 = kstages;
        r.pidx = -1;
    } else {
        const int64_t v = u - tp.full;
        const int sl = (int)(v % tp.S);
        r.item = tp.full + v / tp.S;
        r.ks0 = sl * kstages / tp.S;
        r.ks1 = (sl + 1) * kstages / tp.S;
        r.pidx = v;
    }
    return r;
}

// Accumulator drain of one unit by a dequantising warp (its 32 tensor-memory
// lanes = weight rows, warpgroup wg taking tokens j with (j / 16) % 2 == wg):
// the FP32 sums of the issuers added in issuer order, then the split tail's
// partial slice, SiLU * up (layout 3), the fused combine (CMB), or the bf16 /
// FP32 output by pair id.  pre[k]: pair id of token wg*16 + 32*(2k + l/16) +
// l%16 held by lane l (-1: none).
template <bool CMB, int NI>
__device__ __forceinline__ void drain_item(const TcArgs& ta, const Unit& un, int n_mma, int nt, int wg, int lane,
                                           uint32_t acc_tmem, const int32_t (&pre)[4], uint8_t* stg) {
    const GemmArgs& a = ta.g;
    const int quarter = (threadIdx.x >> 5) & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const int n_out = nt * kTileRows + row;
    // fused SiLU * up (layout 3): rows 16k + i (i < 8) and 16k + i + 8 of
    // the tile hold gate and up of output column 64 * nt + 8k + i
    const int h_col = nt * (kTileRows / 2) + 8 * (row / 16) + (row % 8);
    const bool gate_row = (lane & 8) == 0;
    const int nst = un.ks1 - un.ks0;
    const int parts = nst < NI ? nst : NI;   // issuers that hold a share of this unit
    float prew[4];    // fused combine: the pair's weight (a number: its token's only local pair)
    int32_t pret[4];  // fused combine: the pair's token
    if (CMB) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            prew[k] = pre[k] >= 0 ? a.pair_w[pre[k]] : 0.0f;
            pret[k] = pre[k] >= 0 ? pre[k] / a.topk : 0;
        }
    }
#pragma unroll
    for (int it = 0; it < 8; ++it) {
        const int j0 = wg * 16 + 32 * it;
        if (j0 >= n_mma) continue;   // (not break: keeps the loop unrolled, pre[] in registers)
        uint32_t v[16];
        tmem_ld16(acc_tmem + lane_base + j0, v);
        for (int pi = 1; pi < parts; ++pi) {
            uint32_t w2[16];
            tc_wait_ld();
            tmem_ld16(acc_tmem + (uint32_t)(pi * ta.tok_tile) + lane_base + j0, w2);
            tc_wait_ld();
#pragma unroll
            for (int u = 0; u < 16; ++u) v[u] = __float_as_uint(__uint_as_float(v[u]) + __uint_as_float(w2[u]));
        }
        tc_wait_ld();
        if (un.pidx >= 0) {
            // a slice of a split tail item: its FP32 sums, row-major [row][token]
            float4* dst = reinterpret_cast<float4*>(a.partial + ((int64_t)un.pidx * kTileRows + row) * ta.tok_tile + j0);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                     __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            continue;
        }
        if (!CMB && !a.silu) {
            // Plain bf16 / FP32 output.  One warp store of a 32-row column
            // slice per token wrote 64 (128) bytes per instruction, and the
            // drain took longer than the item's MMAs it delays (the write
            // requests, not their bytes, are what an SM has few of in flight).
            // So the 16 x 32 tile goes through this warp's shared-memory
            // buffer, token-major, and leaves in 16-byte pieces: piece q
            // holds `per` consecutive rows of token q / (32 / per).
            const int esz = a.out_f32 ? 4 : 2;
            const int per = 16 / esz;              // rows per 16-byte piece
            const int pieces_tok = 32 / per;       // pieces per token
            const uint32_t sbase = smem_u32(stg);
#pragma unroll
            for (int u = 0; u < 16; ++u) {
                const uint32_t addr = sbase + (uint32_t)((u * 32 + lane) * esz);
                if (a.out_f32)
                    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v[u]) : "memory");
                else
                    asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr),
                                 "h"(__bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[u]))))
                                 : "memory");
            }
            __syncwarp();
            const int npieces = 16 * pieces_tok;   // 64 (bf16) or 128 (FP32) per warp
            for (int q = lane; q < npieces; q += 32) {
                const int u = q / pieces_tok;
                const int r0 = (q % pieces_tok) * per;
                const int32_t id = __shfl_sync(0xffffffffu, pre[it >> 1], u + 16 * (it & 1));
                uint4 w4;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(w4.x), "=r"(w4.y), "=r"(w4.z), "=r"(w4.w)
                             : "r"(sbase + (uint32_t)(q * 16))
                             : "memory");
                if (id >= 0) {
                    const int64_t col = (int64_t)nt * kTileRows + quarter * 32 + r0;
                    uint8_t* dst = static_cast<uint8_t*>(a.C) + ((int64_t)id * a.N + col) * esz;
                    *reinterpret_cast<uint4*>(dst) = w4;
                }
            }
            __syncwarp();
            continue;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (!CMB && a.silu) {
                // lanes l (gate row) and l ^ 8 (its up row) split the 16
                // tokens: the gate lane takes tokens 0-7, the up lane 8-15,
                // each receiving the partner's value for its tokens
                if (u < 8) {
                    const float lo = __uint_as_float(v[u]), hi = __uint_as_float(v[8 + u]);
                    const float mine = gate_row ? lo : hi;
                    const float other = __shfl_xor_sync(0xffffffffu, gate_row ? hi : lo, 8);
                    const int tok = gate_row ? u : 8 + u;
                    const int32_t id = __shfl_sync(0xffffffffu, pre[it >> 1], tok + 16 * (it & 1));
                    if (id >= 0)
                        static_cast<__nv_bfloat16*>(a.C)[(int64_t)id * (a.N / 2) + h_col] =
                            gate_row ? silu_mul_bf16(mine, other) : silu_mul_bf16(other, mine);
                }
                continue;
            }
            const int32_t id = __shfl_sync(0xffffffffu, pre[it >> 1], u + 16 * (it & 1));
            const float val = __uint_as_float(v[u]);
            if (CMB) {
                const float w = __shfl_sync(0xffffffffu, prew[it >> 1], u + 16 * (it & 1));
                const int32_t tok = __shfl_sync(0xffffffffu, pret[it >> 1], u + 16 * (it & 1));
                if (id >= 0) combine_store(static_cast<float*>(a.C), a.out, a.N, id, tok, w, n_out, val);
                continue;
            }
            if (id < 0) continue;
            if (a.out_f32)
                static_cast<float*>(a.C)[(int64_t)id * a.N + n_out] = val;
            else
                static_cast<__nv_bfloat16*>(a.C)[(int64_t)id * a.N + n_out] = __float2bfloat16_rn(val);
        }
    }
}

// The fused combine's drain, kept out of line: inlined next to the plain drain
// it made the dequantising warps' loop longer than the instruction cache holds
// (the EP8 prefill down GEMM, 2688 short items, measured 361 -> 423 us).
template <int NI>
__device__ __noinline__ void drain_item_combine(const TcArgs& ta, const Unit& un, int n_mma, int nt, int wg, int lane,
                                                uint32_t acc_tmem, const int32_t (&pre)[4]) {
    drain_item<true, NI>(ta, un, n_mma, nt, wg, lane, acc_tmem, pre, nullptr);
}

template <int GW, int MAXR, int NI, bool PAIR>
__global__ void __launch_bounds__(Cfg<GW, MAXR, NI>::kThreads, 1) gemm_tc_kernel(const TcArgs ta) {
    pdl_trigger();
    pdl_wait();
    using C = Cfg<GW, MAXR, NI>;
    const int SA = ta.nsa;
    const GemmArgs& a = ta.g;
    const int NSB = ta.nsb, NSW = ta.nsw;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled B tiles; plain pointer arithmetic on
    // the shared array keeps every access below a shared-memory access
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // PAIR: CTA `rank` of the cluster holds weight rows [128 rank, 128 rank + 128)
    // of the item's 256 and tokens [rank n / 2, (rank + 1) n / 2) of its B tile
    const uint32_t rank = PAIR ? cluster_rank() : 0u;
    const int b_sub = (PAIR ? ta.tok_tile / 2 : ta.tok_tile) * 128;   // one 64-column B sub-tile
    const int b_stage = 2 * b_sub;
    uint8_t* sB = smem;                               // NSB x 2 sub-tiles
    uint8_t* sW = sB + NSB * b_stage;                 // NSW x 2 packed chunks
    uint8_t* sStg = sW + NSW * 2 * kChunk2;           // the dequantising warps' drain buffers
    uint64_t* bars = reinterpret_cast<uint64_t*>(sStg + C::kDQ * kStgWarpBytes);
    uint64_t* w_full = bars;
    uint64_t* w_empty = w_full + NSW;
    uint64_t* b_full = w_empty + NSW;
    uint64_t* b_empty = b_full + NSB;
    uint64_t* a_full = b_empty + NSB;
    uint64_t* a_empty = a_full + SA;
    uint64_t* acc_full = a_empty + SA;
    uint64_t* acc_empty = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 1);
    // [0] skip, [1] abort, [2] every scale in the one-FMA dequantisation's range
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        const bool ok = header_ok_layout(a.packed, a.E, a.N, a.K, a.layout);
        if (!ok) set_error(a.err, CHORD_DEV_BAD_HEADER);
        flags[0] = ok ? 0 : 1;
        flags[1] = 0;
        flags[2] = ok && header_scales_in_fma_range(a.packed) ? 1 : 0;
        for (int s = 0; s < NSW; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], 4);        // the 4 warps of the warpgroup that took the stage
        }
        for (int s = 0; s < NSB; ++s) {
            // one cp.async-tracked arrival per gather lane (+ the peer's forwarded half in a pair's leader)
            mbar_init(&b_full[s], GW * 32 + (PAIR && rank == 0 ? 1 : 0));
            mbar_init(&b_empty[s], 1);
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(&a_full[s], PAIR ? 8 : 4);   // the warpgroup's 4 warps (of both CTAs in a pair)
            mbar_init(&a_empty[s], 1);
        }
        mbar_init(acc_full, NI);              // one arrival per MMA issuer
        mbar_init(acc_empty, PAIR ? 2 * C::kDQ : C::kDQ);
        fence_barrier_init();
    }
    __syncthreads();
    if (flags[0]) return;   // both CTAs of a pair read the same header
    // a pair's barriers must be initialised in both CTAs before any remote arrival
    if constexpr (PAIR) cluster_sync();
    if (warp == C::kProducer) {
        tmem_alloc_g<PAIR>(tmem_slot, ta.tmem_cols);
        tmem_relinquish_g<PAIR>();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t acc_tmem = tmem_base + SA * kACols;   // issuer i accumulates at acc_tmem + i * tok_tile

    int32_t ntp = *a.ntp;
    if (ntp < 0 || ntp > a.capacity || ntp % a.block_m) {
        if (threadIdx.x == 0) set_error(a.err, CHORD_DEV_BAD_PADDED);
        ntp = 0;
    }
    // An item is (align block, 128-row tile of N), or for a pair (align block,
    // 256-row tile) with CTA `rank` on its 128-row half; units run over the
    // CTAs (pairs) of the persistent grid in a static round robin.
    const int ntiles = a.N / (PAIR ? 2 * kTileRows : kTileRows);
    const int64_t G = PAIR ? gridDim.x / 2 : gridDim.x;
    const int64_t u0 = PAIR ? blockIdx.x / 2 : blockIdx.x;
    auto item_coords = [&](int64_t item, int& nt) {
        int q;
        const int64_t b = divmod_idx(item, ntiles, q);
        nt = PAIR ? 2 * q + (int)rank : q;
        return b;
    };
    const int kchunks = a.K / kChunkK;
    const int kstages = (kchunks + 1) / 2;   // the last stage holds one chunk when kchunks is odd
    const int64_t n_items = (int64_t)(ntp / a.block_m) * ntiles;
    const TailPlan tplan = tail_plan(n_items, G, kstages, NI, a.tail_split != 0);
    const int64_t n_units = tplan.full + tplan.tail * tplan.S;
    const uint64_t expert_bytes = (uint64_t)a.N * (uint64_t)a.K * 9ull / 16ull;

    if (warp == C::kProducer) {
        // ---------------------------------------------------------- weights
        const uint64_t pol = policy_evict_first();
        int64_t g = 0;   // stages lane 0 issued
        Ring wr;
        bool ok = true;
        for (int64_t wu = u0; wu < n_units && ok; wu += G) {
            const Unit un = unit_at(wu, tplan, kstages);
            int nt;
            const int64_t b = item_coords(un.item, nt);
            const ItemInfo inf = item_info(a, b, lane, false);
            if (inf.n_mma == 0) continue;
            if (lane == 0) {
                // chunks (nt, kc) of one expert are contiguous along kc
                const uint8_t* src = a.packed + kHeaderBytes + (uint64_t)inf.e * expert_bytes +
                                     (uint64_t)nt * (uint64_t)kchunks * kChunk2;
                for (int ks = un.ks0; ks < un.ks1; ++ks, ++g, wr.next(NSW)) {
                    const int nck = min(2, kchunks - 2 * ks);
                    if (!wait_or_abort(&w_empty[wr.slot], wr.phase ^ 1u, &flags[1], a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&w_full[wr.slot], nck * kChunk2);
                    bulk_g2s_hint(sW + wr.slot * 2 * kChunk2, src + (uint64_t)(2 * ks) * kChunk2, nck * kChunk2,
                                  &w_full[wr.slot], pol);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        // leave only after every copy issued here has landed
        if (lane == 0) {
            for (int i = 0; i < NSW && i < g; ++i) {
                wr.prev(NSW);
                if (!mbar_wait(&w_full[wr.slot], wr.phase)) set_error(a.err, CHORD_DEV_TIMEOUT);
            }
        }
        __syncwarp();
    } else if (warp >= C::kMma0 && warp < C::kGather0) {
        // ------------------------------------------------------------- MMA
        if (PAIR && rank == 1) {
            // The peer CTA issues no MMA: one thread forwards each B stage of
            // its gather warps (complete in this CTA) to the leader's barrier.
            if (warp == C::kMma0) {
                Ring br;
                bool ok = true;
                for (int64_t wu = u0; wu < n_units && ok; wu += G) {
                    const Unit un = unit_at(wu, tplan, kstages);
                    int nt_unused;
                    const ItemInfo inf = item_info(a, item_coords(un.item, nt_unused), lane, false);
                    if (inf.n_mma == 0) continue;
                    if (lane == 0) {
                        for (int ks = un.ks0; ks < un.ks1; ++ks, br.next(NSB)) {
                            if (!wait_or_abort(&b_full[br.slot], br.phase, &flags[1], a.err)) {
                                ok = false;
                                break;
                            }
                            // the tile was written by cp.async (generic proxy); the
                            // leader's MMA reads it through the async proxy
                            fence_proxy_async();
                            mbar_arrive_leader(&b_full[br.slot]);
                        }
                    }
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                }
            }
            __syncwarp();
        } else {
        // Issuer mi takes the item's stages ks with ks % NI == mi.
        const int mi = warp - C::kMma0;
        const uint32_t my_acc = acc_tmem + (uint32_t)(mi * ta.tok_tile);
        int64_t nitem = 0;
        int issued = 0;                 // stages whose MMAs this issuer committed
        Ring ar, br, last;
        bool ok = true;
        for (int64_t wu = u0; wu < n_units && ok; wu += G) {
            const Unit un = unit_at(wu, tplan, kstages);
            int nt_unused;
            const int64_t b = item_coords(un.item, nt_unused);
            const ItemInfo inf = item_info(a, b, lane, false);
            if (inf.n_mma == 0) continue;
            if (lane == 0) {
                if (!wait_or_abort<PAIR>(acc_empty, (uint32_t)((nitem & 1) ^ 1), &flags[1], a.err)) ok = false;
                tc_fence_after();
                const uint32_t idesc = idesc_bf16(inf.n_mma, PAIR ? 2 * kTileRows : kTileRows);
                bool any = false;
                for (int ks = un.ks0; ks < un.ks1 && ok; ++ks, ar.next(SA), br.next(NSB)) {
                    if (ks % NI != mi) continue;
                    const int nck = min(2, kchunks - 2 * ks);
                    if (!wait_or_abort<PAIR>(&a_full[ar.slot], ar.phase, &flags[1], a.err) ||
                        !wait_or_abort<PAIR>(&b_full[br.slot], br.phase, &flags[1], a.err)) {
                        ok = false;
                        break;
                    }
                    // the B tile was written by cp.async (generic proxy); the MMA
                    // reads it through the async proxy
                    fence_proxy_async();
                    tc_fence_after();
                    // Eight K = 16 steps per stage, unrolled: step kk reads A
                    // columns 8 kk of the stage and the B descriptor advanced by
                    // (kk / 4) sub-tiles and (kk % 4) 32-byte K slices (the
                    // descriptor's address field counts 16-byte units and stays
                    // below 2^14 inside the 227 KB of shared memory, so the sum
                    // never carries into the next field).
                    const uint64_t d0 = desc_sw128(smem_u32(sB + br.slot * b_stage));
                    const uint32_t a0 = tmem_base + ar.slot * kACols;
                    const uint32_t sub16 = (uint32_t)b_sub >> 4;
                    const uint32_t acc0 = any ? 1u : 0u;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        if (kk < 4 * nck)
                            tc_mma_ts_g<PAIR>(my_acc, a0 + kk * 8, d0 + (uint64_t)((kk >> 2) * sub16 + (kk & 3) * 2),
                                              idesc, kk > 0 ? 1u : acc0);
                    any = true;
                    tc_commit_g<PAIR>(&a_empty[ar.slot]);
                    tc_commit_g<PAIR>(&b_empty[br.slot]);
                    last = ar;
                    ++issued;
                }
                if (ok) {
                    // no share of this item: the commit arrives at once (on both
                    // CTAs' barrier in a pair)
                    if (any || PAIR)
                        tc_commit_g<PAIR>(acc_full);
                    else
                        mbar_arrive(acc_full);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            ++nitem;
        }
        // wait for this issuer's last MMAs before the tensor memory is released
        if (lane == 0 && issued > 0) mbar_wait(&a_empty[last.slot], last.phase);
        __syncwarp();
        }
    } else if (warp >= C::kGather0) {
        // ------------------------------------------------------ activations
        // Lane gl copies the 16-byte piece c = gl % 8 of token rows
        // j = gl / 8 + r * (GW * 4), r < MAXR, for both chunks of a stage;
        // their A row indices are read once per item.  Each lane's copies
        // arrive on the stage's barrier when they land, so a stage is full as
        // soon as its copies are (a warp-level arrival after waiting for the
        // previous stage's copies measured slower: it shortens the B ring by a
        // stage, and the ring holds only three at 224 tokens).
        const int gl = (warp - C::kGather0) * 32 + lane;
        const int c = gl & 7;
        constexpr int kRowStep = GW * 4;
        Ring br;
        bool ok = true;
        for (int64_t wu = u0; wu < n_units && ok; wu += G) {
            const Unit un = unit_at(wu, tplan, kstages);
            int nt_unused;
            const int64_t b = item_coords(un.item, nt_unused);
            const ItemInfo inf = item_info(a, b, lane, warp == C::kGather0 && un.ks0 == 0 && rank == 0);
            if (inf.n_mma == 0) continue;
            // a pair's CTA gathers its half of the block's first n_mma tokens
            const int rows = PAIR ? inf.n_mma / 2 : inf.n_mma;
            const int j0 = PAIR ? (int)rank * rows : 0;
            int32_t arow[MAXR];
#pragma unroll
            for (int r = 0; r < MAXR; ++r) {
                const int jl = (gl >> 3) + r * kRowStep;
                const int j = j0 + jl;
                arow[r] = -1;
                if (jl < rows && j < a.block_m) {
                    const int32_t id = a.sorted_ids[b * a.block_m + j];
                    if (row_valid(a, id)) arow[r] = a.a_row_divisor == 1 ? id : id / a.a_row_divisor;
                }
            }
            for (int ks = un.ks0; ks < un.ks1; ++ks, br.next(NSB)) {
                const int nck = min(2, kchunks - 2 * ks);
                if (!wait_or_abort<PAIR>(&b_empty[br.slot], br.phase ^ 1u, &flags[1], a.err)) {
                    ok = false;
                    break;
                }
                const uint32_t tile = smem_u32(sB + br.slot * b_stage);
                for (int ch = 0; ch < nck; ++ch) {
#pragma unroll
                    for (int r = 0; r < MAXR; ++r) {
                        if (arow[r] < 0) continue;
                        const int j = (gl >> 3) + r * kRowStep;
                        const uint16_t* src = a.A + (int64_t)arow[r] * a.K + (2 * ks + ch) * kChunkK + c * 8;
                        const uint32_t dst = tile + (uint32_t)(ch * b_sub + (j >> 3) * 1024 + (j & 7) * 128 +
                                                               ((c ^ (j & 7)) << 4));
                        cp_async16(dst, src);
                    }
                }
                cp_async_arrive_noinc(&b_full[br.slot]);
            }
        }
        // every copy must land before the CTA's shared memory goes away
        cp_async_wait<0>();
        __syncwarp();
    } else {
        // --------------------------------------- dequantisation and epilogue
        // Warpgroup wg takes the stages with (stage index & 1) == wg; each
        // thread dequantises its row's 128 columns of the stage.
        const int wg = warp >> 2;
        const int quarter = warp & 3;                  // tensor-memory lane quarter of this warp
        const int row = quarter * 32 + lane;           // weight row of the tile = TMEM lane
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        const bool fma_dequant = flags[2] != 0;   // the blob's header: one FMA per weight pair
        int64_t g = 0, nitem = 0;
        Ring wr, ar;
        bool ok = true;
        for (int64_t wu = u0; wu < n_units && ok; wu += G) {
            const Unit un = unit_at(wu, tplan, kstages);
            int nt;
            const int64_t b = item_coords(un.item, nt);
            const ItemInfo inf = item_info(a, b, lane, false);
            if (inf.n_mma == 0) continue;
            for (int ks = un.ks0; ks < un.ks1; ++ks, ++g, wr.next(NSW), ar.next(SA)) {
                if ((int)(g & 1) != wg) continue;
                const int nck = min(2, kchunks - 2 * ks);
                if (!wait_or_abort(&w_full[wr.slot], wr.phase, &flags[1], a.err) ||
                    !wait_or_abort<PAIR>(&a_empty[ar.slot], ar.phase ^ 1u, &flags[1], a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* wch = sW + wr.slot * 2 * kChunk2;
                uint4 q[4];
                uint32_t sc[2];
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    if (ch < nck) {
                        q[2 * ch] = *reinterpret_cast<const uint4*>(wch + ch * kChunk2 + row * 16);
                        q[2 * ch + 1] = *reinterpret_cast<const uint4*>(wch + ch * kChunk2 + 2048 + row * 16);
                        sc[ch] = *reinterpret_cast<const uint32_t*>(wch + ch * kChunk2 + 4096 + row * 4);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[wr.slot]);   // the packed chunks are in registers
#pragma unroll
                for (int ch = 0; ch < 2; ++ch) {
                    if (ch < nck) {
                        uint32_t v[32];
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            const uint32_t s16 = h ? (sc[ch] >> 16) : (sc[ch] & 0xffffu);
                            const uint32_t sp = s16 | (s16 << 16);
                            const uint4 qq = q[2 * ch + h];
                            if (fma_dequant) {
                                uint32_t b2, c2;
                                fma_scale_pair(sp, b2, c2);
                                dequant_row8_fma(qq.x, b2, c2, v + 16 * h + 0);
                                dequant_row8_fma(qq.y, b2, c2, v + 16 * h + 4);
                                dequant_row8_fma(qq.z, b2, c2, v + 16 * h + 8);
                                dequant_row8_fma(qq.w, b2, c2, v + 16 * h + 12);
                            } else {
                                dequant_row8(qq.x, sp, v + 16 * h + 0);
                                dequant_row8(qq.y, sp, v + 16 * h + 4);
                                dequant_row8(qq.z, sp, v + 16 * h + 8);
                                dequant_row8(qq.w, sp, v + 16 * h + 12);
                            }
                        }
                        tmem_st32(tmem_base + lane_base + ar.slot * kACols + ch * 32, v);
                    }
                }
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    // the stage's A rows are in this CTA's tensor memory; the MMA
                    // thread (the leader's, in a pair) may read them
                    if (PAIR && rank == 1)
                        mbar_arrive_leader(&a_full[ar.slot]);
                    else
                        mbar_arrive(&a_full[ar.slot]);
                }
            }
            if (!ok) break;
            // ---- epilogue: accumulator column j is token j of the block.
            // Pair ids first, before the accumulator is ready: lane l holds the
            // id of token wg*16 + 32*(2k + l/16) + l%16 in pre[k].
            int32_t pre[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int j = wg * 16 + 32 * (2 * k + (lane >> 4)) + (lane & 15);
                int32_t id = -1;
                if (j < inf.n_mma && j < a.block_m) {
                    id = a.sorted_ids[b * a.block_m + j];
                    if (!row_valid(a, id)) id = -1;
                }
                pre[k] = id;
            }
            if (!wait_or_abort<PAIR>(acc_full, (uint32_t)(nitem & 1), &flags[1], a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // the fused combine's drain is a separate instantiation, so the
            // plain drain carries none of its registers or branches
            if (a.combine)
                drain_item_combine<NI>(ta, un, inf.n_mma, nt, wg, lane, acc_tmem, pre);
            else
                drain_item<false, NI>(ta, un, inf.n_mma, nt, wg, lane, acc_tmem, pre, sStg + warp * kStgWarpBytes);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (PAIR && rank == 1)
                    mbar_arrive_leader(acc_empty);
                else
                    mbar_arrive(acc_empty);
            }
            ++nitem;
        }
    }

    // ------------------------------------------------------------ teardown
    // (every role reaches this point, also after an aborted wait, so the
    // cluster barrier below always completes)
    tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) cluster_sync();   // the leader's last MMAs into the peer's tensor memory are done
    tc_fence_after();
    if (warp == C::kProducer) tmem_dealloc_g<PAIR>(tmem_base, ta.tmem_cols);
}

uint32_t pow2_cols(uint32_t c) {
    uint32_t p = 32;
    while (p < c) p <<= 1;
    return p;
}

// Launch of a kernel in clusters of two CTAs (with programmatic stream
// serialization when `pdl`).
template <typename... KArgs, typename... Args>
cudaError_t launch_pairs(bool pdl, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                         Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Clusters of two CTAs of `kern` that can be resident at once on this device
// (cached per device, kernel and shared-memory size); 0 when the query fails.
int max_active_pairs(const void* kern, int threads, size_t smem) {
    struct Entry {
        int dev;
        const void* kern;
        size_t smem;
        int n;
    };
    static std::mutex mu;
    static Entry cache[64];
    static int ncache = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < ncache; ++i)
        if (cache[i].dev == dev && cache[i].kern == kern && cache[i].smem == smem) return cache[i].n;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 76);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    if (ncache < 64) cache[ncache++] = Entry{dev, kern, smem, n};
    return n;
}

template <int GW, int MAXR, int NI, bool PAIR>
cudaError_t launch_cfg(const GemmArgs& g, bool deep_weights, cudaStream_t stream) {
    using C = Cfg<GW, MAXR, NI>;
    auto kern = gemm_tc_kernel<GW, MAXR, NI, PAIR>;
    constexpr size_t kSmemBudget = 227 * 1024;   // the dynamic shared memory a CTA may use
    TcArgs ta;
    ta.g = g;
    ta.tok_tile = (g.block_m < 16 ? 16 : (g.block_m + 15) / 16 * 16);
    if (ta.tok_tile > C::kMaxTokens) return cudaErrorInvalidConfiguration;
    // A ring: every tensor-memory column the accumulators leave, at most 8 stages
    int nsa = (int)((512 - NI * ta.tok_tile) / kACols);
    nsa = nsa > 8 ? 8 : nsa;
    if (nsa < 2) return cudaErrorInvalidConfiguration;
    // Several issuers with a 3-stage A ring (two issuers, 160-token blocks, a
    // configuration the table below never picks) were seen to stall until the
    // bounded waits gave up; every configuration in use keeps >= 4 A stages.
    if (NI > 1 && nsa < 4) return cudaErrorInvalidConfiguration;
    ta.nsa = nsa;
    const uint32_t cols = nsa * kACols + NI * ta.tok_tile;
    ta.tmem_cols = pow2_cols(cols);
    // Ring depths.  Few tokens per item (HBM-bound): about 64 KB of B tiles and
    // the rest of the budget for packed weights, to keep enough HBM bytes in
    // flight.  Many tokens per item: four weight stages and the rest for B
    // tiles, whose gather from L2 has the longer latency per byte consumed.
    // (a pair's CTA holds half of each B tile)
    const size_t b_stage = (size_t)(PAIR ? ta.tok_tile / 2 : ta.tok_tile) * 256, w_stage = 2 * kChunk2;
    // 1 KB of alignment slack, the barriers' margin and the drain buffers
    const size_t fixed = 1024 + 64 + (size_t)C::kDQ * kStgWarpBytes;
    int nsb, nsw;
    if (deep_weights) {
        nsb = (int)((64 * 1024) / b_stage);
        nsb = nsb < 2 ? 2 : (nsb > 16 ? 16 : nsb);
        nsw = (int)((kSmemBudget - fixed - nsb * (b_stage + 16)) / (w_stage + 16));
        nsw = nsw > 32 ? 32 : nsw;
    } else {
        nsw = 4;
        nsb = (int)((kSmemBudget - fixed - nsw * (w_stage + 16)) / (b_stage + 16));
        nsb = nsb > 16 ? 16 : nsb;
    }
    if (nsw < 2 || nsb < 2) return cudaErrorInvalidConfiguration;
    ta.nsb = nsb;
    ta.nsw = nsw;
    size_t smem = fixed + (size_t)nsb * b_stage + (size_t)nsw * w_stage + (2 * nsw + 2 * nsb + 2 * nsa + 2) * 8 + 16;
    // A CTA that cannot get its tensor-memory columns waits in tcgen05.alloc
    // until a co-resident CTA exits.  When two CTAs' columns do not fit in the
    // SM's 512, ask for enough shared memory that only one CTA fits per SM.
    if (2 * ta.tmem_cols > 512 && smem < 120 * 1024) smem = 120 * 1024;
    int per_sm = 1;
    cudaError_t e = kernel_ctas_per_sm(reinterpret_cast<const void*>(kern), C::kThreads, smem, 227 * 1024, &per_sm);
    if (e != cudaSuccess) return e;
    const int tmem_fit = (int)(512 / ta.tmem_cols);
    if (per_sm > tmem_fit) per_sm = tmem_fit;
    if (per_sm < 1) per_sm = 1;
    const int64_t items_cap = (g.capacity / g.block_m) * (g.N / (PAIR ? 2 * kTileRows : kTileRows));
    int64_t grid = (int64_t)device_info().sm_count * per_sm / (PAIR ? 2 : 1);   // CTAs, or pairs of CTAs
    if (PAIR) {
        // only as many pairs as can be resident at once: a pair that starts
        // late would run its whole share of the static round robin late
        const int clusters = max_active_pairs(reinterpret_cast<const void*>(kern), C::kThreads, smem);
        if (clusters > 0 && grid > clusters) grid = clusters;
    }
    if (grid > items_cap) grid = items_cap;
    if (grid < 1) grid = 1;
    if (PAIR) {
        ta.g.tail_split = 0;   // the split tail is built for single CTAs
        return launch_pairs(pdl_for(g.num_pairs), kern, dim3((unsigned)(2 * grid)), dim3(C::kThreads), smem, stream,
                            ta);
    }
    // The split tail writes at most grid units of 128 x tok_tile FP32 sums (S * tail <= grid).
    const size_t tail_bytes = (size_t)grid * kTileRows * (size_t)ta.tok_tile * sizeof(float);
    ta.g.tail_split = (g.tail_split && g.partial && g.partial_bytes >= tail_bytes) ? 1 : 0;
    e = launch_pdl(pdl_for(g.num_pairs), kern, dim3((unsigned)grid), dim3(C::kThreads), smem, stream, ta);
    if (e != cudaSuccess || !ta.g.tail_split) return e;
    const int kstages = (g.K / kChunkK + 1) / 2;
    return launch_tc_tail_reduce(ta.g, grid, kstages, NI, ta.tok_tile, stream);
}

}  // namespace

bool tc_available() { return true; }


template <bool PAIR>
cudaError_t launch_tc_shape(const GemmArgs& a, cudaStream_t stream) {
    // Up to 64 tokens per item: four MMA issuers (a tcgen05.mma of N <= 64 costs
    // its issuing thread about as long as one of N = 128) and three gather warps
    // (measured on GB300: 360 -> 290 us for the EP8 decode gate_up against two
    // issuers and one gather warp).
    if (a.block_m <= 64) return launch_cfg<3, 6, 4, PAIR>(a, true, stream);
    // 65-128 tokens: two issuers (TP8 T=4096 gate_up 526 -> 363 us on GB300)
    if (a.block_m <= 128) return launch_cfg<4, 8, 2, PAIR>(a, false, stream);
    return launch_cfg<4, 16, 1, PAIR>(a, false, stream);                 // up to 256 tokens per item
}

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t stream) {
    if (a.block_m % 8 || a.block_m > 256 || a.N % kTileRows || a.K % kChunkK) return cudaErrorInvalidValue;
    // Pairs of CTAs on request only: measured on GB300 they lose on long-K items
    // (EP8 prefill gate_up, K = 7168: 562 -> 760 us) and gain little on short ones
    // (down, K = 2048: 421 -> 409 us): the cross-CTA hand-offs of every stage add
    // more latency than halving each SM's share of the activation gather saves.
    if (a.tc_pairs && a.N % (2 * kTileRows) == 0) return launch_tc_shape<true>(a, stream);
    return launch_tc_shape<false>(a, stream);
}

}  // namespace chord
