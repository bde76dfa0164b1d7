// Indexed W4A16 GEMM on the 5th-generation tensor cores (tcgen05) of sm_103a.
//
// One work item is (align block b, 128-row tile of N).  The product is
// computed with the operands swapped, as the article's decode profile does
// (section "H200 and Blackwell indexed decode"): the 128 dequantised weight
// rows are the MMA's M side and the block's routed tokens its N side, so a
// block of 11 rows costs an N = 16 MMA instead of a padded 128-row tile, and
// a block of 176 rows an N = 176 MMA.  Per 64-column K stage:
//   * a producer warp streams the packed 128x64 weight chunk (4608 bytes, one
//     cp.async.bulk) into a shared-memory ring;
//   * gather warps copy the block's activation rows (row = pair id / divisor)
//     with 16-byte cp.async into a 128-byte-swizzled K-major tile, the MMA's B
//     operand, and publish it after a proxy fence;
//   * dequantising warps (one row per thread) turn 32 codes per 16-byte load
//     into bf16((q - 8) * s) and store them with tcgen05.st into a tensor
//     memory stage, the MMA's A operand (no shared-memory round trip for the
//     dequantised weights);
//   * one thread issues four tcgen05.mma (M=128, N=tokens rounded up to 16,
//     K=16) into an FP32 accumulator in tensor memory and commits the stage
//     back to the producers;
// after the item's last stage the dequantising warps read the accumulator
// with tcgen05.ld and write the pair rows of C.  Every wait is bounded.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "chord_common.cuh"
#include "chord_internal.h"

namespace chord {
namespace {

constexpr int kTileRows = 128;   // rows of N per item = MMA M
constexpr int kBK = 64;          // K columns per stage
constexpr int kChunk2 = 4608;    // packed bytes of one 128 x 64 chunk (layout 2)
constexpr int kACols = 32;       // tensor-memory columns of one A stage (64 bf16 per lane)
constexpr uint32_t kLayoutTc = 2;

// SA: stages of the A (tensor memory) and B (shared memory) rings; SW: stages
// of the packed-weight ring (deeper, to keep enough HBM bytes in flight);
// DQ: dequantising warps (4 or 8); GW: gather warps; MAXR: token rows one
// gather lane copies per stage (block rows / (GW * 4)).
template <int SA, int SW, int DQ, int GW, int MAXR>
struct Cfg {
    static constexpr int kProducer = DQ;      // warp index of the weight producer (owns TMEM)
    static constexpr int kMma = DQ + 1;       // warp index of the MMA issuer
    static constexpr int kGather0 = DQ + 2;   // first gather warp
    static constexpr int kWarps = DQ + 2 + GW;
    static constexpr int kThreads = kWarps * 32;
    static constexpr int kLag = SA - 2;       // gather stages kept in flight before publishing
    static constexpr int kMaxTokens = MAXR * GW * 4;
};

struct TcArgs {
    GemmArgs g;
    int tok_tile;      // rows of the B tile: block_m rounded up to 16
    uint32_t tmem_cols;
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

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

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

// Instruction descriptor, kind::f16: D F32, A and B BF16, both K-major, M = 128.
__device__ __forceinline__ uint32_t idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTileRows >> 4) << 24);
}

// Bounded wait that also gives up once another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (*abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) {
            set_error(err, CHORD_DEV_TIMEOUT);
            *abort_flag = 1;
            return false;
        }
    }
    return true;
}

// Routing facts of one item, computed identically by every role from the
// same global data: whether any row is valid and the MMA's N (the tokens up
// to the last valid row, rounded up to 16).
struct ItemInfo {
    int e;
    int n_mma;   // 0: nothing to do
};

__device__ __forceinline__ bool row_valid(const GemmArgs& a, int32_t id) {
    return id != (int32_t)a.num_pairs && id >= 0 && (int64_t)id < a.num_pairs &&
           (int64_t)(id / a.a_row_divisor) < a.a_rows;
}

__device__ __forceinline__ ItemInfo item_info(const GemmArgs& a, int64_t b, int lane, bool report) {
    ItemInfo r;
    r.e = a.expert_ids[b];
    r.n_mma = 0;
    if (r.e < 0 || r.e >= a.E) {
        if (report && lane == 0) set_error(a.err, CHORD_DEV_BAD_EXPERT);
        return r;
    }
    int last = -1;
    for (int i = lane; i < a.block_m; i += 32) {
        const int32_t id = a.sorted_ids[b * a.block_m + i];
        const bool ok = row_valid(a, id);
        if (report && !ok && id != (int32_t)a.num_pairs) set_error(a.err, CHORD_DEV_BAD_ROW);
        if (ok) last = i;
    }
    last = __reduce_max_sync(0xffffffffu, last + 1);
    r.n_mma = (last + 15) / 16 * 16;
    return r;
}

template <int SA, int SW, int DQ, int GW, int MAXR>
__global__ void __launch_bounds__(Cfg<SA, SW, DQ, GW, MAXR>::kThreads, 1) gemm_tc_kernel(const TcArgs ta) {
    using C = Cfg<SA, SW, DQ, GW, MAXR>;
    const GemmArgs& a = ta.g;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled B tiles
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    const int b_tile_bytes = ta.tok_tile * 128;
    uint8_t* sB = smem;                                   // SA x tok_tile x 128 B
    uint8_t* sW = sB + SA * b_tile_bytes;                 // SW x 4608 B
    uint64_t* bars = reinterpret_cast<uint64_t*>(sW + SW * kChunk2);
    uint64_t* w_full = bars;
    uint64_t* w_empty = w_full + SW;
    uint64_t* b_full = w_empty + SW;
    uint64_t* a_full = b_full + SA;
    uint64_t* st_empty = a_full + SA;
    uint64_t* acc_full = st_empty + SA;
    uint64_t* acc_empty = acc_full + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 1);
    volatile int* flags = reinterpret_cast<volatile int*>(tmem_slot + 1);  // [0] skip, [1] abort

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        const bool ok = header_ok_layout(a.packed, a.E, a.N, a.K, kLayoutTc);
        if (!ok) set_error(a.err, CHORD_DEV_BAD_HEADER);
        flags[0] = ok ? 0 : 1;
        flags[1] = 0;
        for (int s = 0; s < SW; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], DQ);
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(&b_full[s], GW);
            mbar_init(&a_full[s], DQ);
            mbar_init(&st_empty[s], 1);
        }
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, DQ);
        fence_barrier_init();
    }
    __syncthreads();
    if (flags[0]) return;
    if (warp == C::kProducer) {
        tmem_alloc(tmem_slot, ta.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint32_t acc_tmem = tmem_base + SA * kACols;

    int32_t ntp = *a.ntp;
    if (ntp < 0 || ntp > a.capacity || ntp % a.block_m) {
        if (threadIdx.x == 0) set_error(a.err, CHORD_DEV_BAD_PADDED);
        ntp = 0;
    }
    const int ntiles = a.N / kTileRows;
    const int kchunks = a.K / kBK;
    const int64_t n_items = (int64_t)(ntp / a.block_m) * ntiles;
    const uint64_t expert_bytes = (uint64_t)a.N * (uint64_t)a.K * 9ull / 16ull;

    if (warp == C::kProducer) {
        // ---------------------------------------------------------- weights
        const uint64_t pol = policy_evict_first();
        int64_t g = 0;   // stages lane 0 issued
        bool ok = true;
        for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const int nt = (int)(item % ntiles);
            const int64_t b = item / ntiles;
            const ItemInfo inf = item_info(a, b, lane, false);
            if (inf.n_mma == 0) continue;
            if (lane == 0) {
                const uint8_t* src = a.packed + kHeaderBytes + (uint64_t)inf.e * expert_bytes +
                                     (uint64_t)nt * (uint64_t)kchunks * kChunk2;
                for (int kc = 0; kc < kchunks; ++kc, ++g) {
                    const int slot = (int)(g % SW);
                    const uint32_t par = (uint32_t)((g / SW) & 1);
                    if (!wait_or_abort(&w_empty[slot], par ^ 1u, &flags[1], a.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&w_full[slot], kChunk2);
                    bulk_g2s_hint(sW + slot * kChunk2, src + (uint64_t)kc * kChunk2, kChunk2, &w_full[slot], pol);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
        // leave only after every copy issued here has landed
        if (lane == 0) {
            for (int s = 0; s < SW && s < g; ++s) {
                const int64_t last = s + ((g - 1 - s) / SW) * SW;
                if (!mbar_wait(&w_full[s], (uint32_t)((last / SW) & 1))) set_error(a.err, CHORD_DEV_TIMEOUT);
            }
        }
        __syncwarp();
    } else if (warp == C::kMma) {
        // ------------------------------------------------------------- MMA
        int64_t g = 0, nitem = 0;   // g: stages whose MMAs lane 0 issued
        bool ok = true;
        for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const int64_t b = item / ntiles;
            const ItemInfo inf = item_info(a, b, lane, false);
            if (inf.n_mma == 0) continue;
            if (lane == 0) {
                if (!wait_or_abort(acc_empty, (uint32_t)((nitem & 1) ^ 1), &flags[1], a.err)) ok = false;
                tc_fence_after();
                const uint32_t idesc = idesc_bf16(inf.n_mma);
                for (int kc = 0; kc < kchunks && ok; ++kc, ++g) {
                    const int slot = (int)(g % SA);
                    const uint32_t par = (uint32_t)((g / SA) & 1);
                    if (!wait_or_abort(&a_full[slot], par, &flags[1], a.err) ||
                        !wait_or_abort(&b_full[slot], par, &flags[1], a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t b_base = smem_u32(sB + slot * b_tile_bytes);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        tc_mma_ts(acc_tmem, tmem_base + slot * kACols + kk * 8, desc_sw128(b_base + kk * 32), idesc,
                                  (kc > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(&st_empty[slot]);
                }
                if (ok) tc_commit(acc_full);
            }
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            ++nitem;
        }
        // wait for the last MMAs before the tensor memory is released
        if (lane == 0 && g > 0) {
            const int64_t last = g - 1;
            mbar_wait(&st_empty[last % SA], (uint32_t)((last / SA) & 1));
        }
        __syncwarp();
    } else if (warp >= C::kGather0) {
        // ------------------------------------------------------ activations
        // Lane gl copies the 16-byte piece c = gl % 8 of token rows
        // j = gl / 8 + r * (GW * 4), r < MAXR; their A row indices are read
        // once per item.
        const int gl = (warp - C::kGather0) * 32 + lane;
        const int c = gl & 7;
        constexpr int kRowStep = GW * 4;
        int64_t g = 0, published = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const int64_t b = item / ntiles;
            const ItemInfo inf = item_info(a, b, lane, warp == C::kGather0);
            if (inf.n_mma == 0) continue;
            int32_t arow[MAXR];
#pragma unroll
            for (int r = 0; r < MAXR; ++r) {
                const int j = (gl >> 3) + r * kRowStep;
                arow[r] = -1;
                if (j < inf.n_mma && j < a.block_m) {
                    const int32_t id = a.sorted_ids[b * a.block_m + j];
                    if (row_valid(a, id)) arow[r] = id / a.a_row_divisor;
                }
            }
            for (int kc = 0; kc < kchunks; ++kc, ++g) {
                const int slot = (int)(g % SA);
                const uint32_t par = (uint32_t)((g / SA) & 1);
                if (!wait_or_abort(&st_empty[slot], par ^ 1u, &flags[1], a.err)) {
                    ok = false;
                    break;
                }
                const uint32_t tile = smem_u32(sB + slot * b_tile_bytes);
#pragma unroll
                for (int r = 0; r < MAXR; ++r) {
                    if (arow[r] < 0) continue;
                    const int j = (gl >> 3) + r * kRowStep;
                    const uint16_t* src = a.A + (int64_t)arow[r] * a.K + kc * kBK + c * 8;
                    const uint32_t dst = tile + (uint32_t)((j >> 3) * 1024 + (j & 7) * 128 + ((c ^ (j & 7)) << 4));
                    cp_async16(dst, src);
                }
                cp_async_commit();
                if (g - published >= C::kLag) {
                    cp_async_wait<C::kLag>();
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&b_full[published % SA]);
                    ++published;
                }
            }
        }
        cp_async_wait<0>();
        fence_proxy_async();
        __syncwarp();
        for (; published < g; ++published)
            if (lane == 0) mbar_arrive(&b_full[published % SA]);
    } else {
        // --------------------------------------- dequantisation and epilogue
        const int quarter = warp & 3;                  // tensor-memory lane quarter of this warp
        const int row = quarter * 32 + lane;           // weight row of the tile = TMEM lane
        const int half0 = DQ == 8 ? (warp >> 2) : 0;   // 32-column halves this warp dequantises
        const int nhalf = DQ == 8 ? 1 : 2;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        int64_t g = 0, nitem = 0;
        bool ok = true;
        for (int64_t item = blockIdx.x; item < n_items && ok; item += gridDim.x) {
            const int nt = (int)(item % ntiles);
            const int64_t b = item / ntiles;
            const ItemInfo inf = item_info(a, b, lane, false);
            if (inf.n_mma == 0) continue;
            for (int kc = 0; kc < kchunks; ++kc, ++g) {
                const int wslot = (int)(g % SW), aslot = (int)(g % SA);
                if (!wait_or_abort(&w_full[wslot], (uint32_t)((g / SW) & 1), &flags[1], a.err) ||
                    !wait_or_abort(&st_empty[aslot], (uint32_t)(((g / SA) & 1) ^ 1), &flags[1], a.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* wch = sW + wslot * kChunk2;
                uint4 q[2];
                uint32_t sc[2];
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (i < nhalf) {
                        q[i] = *reinterpret_cast<const uint4*>(wch + (half0 + i) * 2048 + row * 16);
                        sc[i] = *reinterpret_cast<const uint16_t*>(wch + 4096 + row * 4 + (half0 + i) * 2);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[wslot]);   // the packed chunk is in registers
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (i < nhalf) {
                        const uint32_t sp = sc[i] | (sc[i] << 16);
                        uint32_t v[16];
                        dequant_row8(q[i].x, sp, v + 0);
                        dequant_row8(q[i].y, sp, v + 4);
                        dequant_row8(q[i].z, sp, v + 8);
                        dequant_row8(q[i].w, sp, v + 12);
                        tmem_st16(tmem_base + lane_base + aslot * kACols + (half0 + i) * 16, v);
                    }
                }
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&a_full[aslot]);
            }
            if (!ok) break;
            // ---- epilogue: accumulator column j is token j of the block
            if (!wait_or_abort(acc_full, (uint32_t)(nitem & 1), &flags[1], a.err)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int n_out = nt * kTileRows + row;
            const int col0 = DQ == 8 ? (warp >> 2) * 16 : 0;
            const int col_step = DQ == 8 ? 32 : 16;
            for (int j0 = col0; j0 < inf.n_mma; j0 += col_step) {
                uint32_t v[16];
                tmem_ld16(acc_tmem + lane_base + j0, v);
                // pair ids of tokens j0..j0+15: one load per lane, then shuffles
                int32_t my_id = -1;
                if (lane < 16 && j0 + lane < a.block_m) {
                    const int32_t id = a.sorted_ids[b * a.block_m + j0 + lane];
                    if (row_valid(a, id)) my_id = id;
                }
                tc_wait_ld();
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int32_t id = __shfl_sync(0xffffffffu, my_id, u);
                    if (id < 0) continue;
                    const float val = __uint_as_float(v[u]);
                    if (a.out_f32)
                        static_cast<float*>(a.C)[(int64_t)id * a.N + n_out] = val;
                    else
                        static_cast<__nv_bfloat16*>(a.C)[(int64_t)id * a.N + n_out] = __float2bfloat16_rn(val);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
            ++nitem;
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::kProducer) tmem_dealloc(tmem_base, ta.tmem_cols);
}

uint32_t pow2_cols(uint32_t c) {
    uint32_t p = 32;
    while (p < c) p <<= 1;
    return p;
}

template <int SA, int SW, int DQ, int GW, int MAXR>
cudaError_t launch_cfg(const GemmArgs& g, cudaStream_t stream) {
    using C = Cfg<SA, SW, DQ, GW, MAXR>;
    TcArgs ta;
    ta.g = g;
    ta.tok_tile = (g.block_m < 16 ? 16 : (g.block_m + 15) / 16 * 16);
    if (ta.tok_tile > C::kMaxTokens) return cudaErrorInvalidConfiguration;
    const uint32_t cols = SA * kACols + ta.tok_tile;
    if (cols > 512) return cudaErrorInvalidConfiguration;
    ta.tmem_cols = pow2_cols(cols);
    size_t smem = 1024 + (size_t)SA * ta.tok_tile * 128 + (size_t)SW * kChunk2 + (2 * SW + 3 * SA + 2) * 8 + 16;
    // A CTA that cannot get its tensor-memory columns waits in tcgen05.alloc
    // until a co-resident CTA exits.  When two CTAs' columns do not fit in the
    // SM's 512, ask for enough shared memory that only one CTA fits per SM.
    if (2 * ta.tmem_cols > 512 && smem < 120 * 1024) smem = 120 * 1024;
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<SA, SW, DQ, GW, MAXR>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemm_tc_kernel<SA, SW, DQ, GW, MAXR>,
                                                                  C::kThreads, smem);
    if (e != cudaSuccess) return e;
    const int tmem_fit = (int)(512 / ta.tmem_cols);
    if (per_sm > tmem_fit) per_sm = tmem_fit;
    if (per_sm < 1) per_sm = 1;
    const int64_t items_cap = (g.capacity / g.block_m) * (g.N / kTileRows);
    int64_t grid = (int64_t)device_info().sm_count * per_sm;
    if (grid > items_cap) grid = items_cap;
    if (grid < 1) grid = 1;
    gemm_tc_kernel<SA, SW, DQ, GW, MAXR><<<(unsigned)grid, C::kThreads, smem, stream>>>(ta);
    return cudaGetLastError();
}

}  // namespace

bool tc_available() { return true; }

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t stream) {
    if (a.block_m % 8 || a.block_m > 256 || a.N % kTileRows || a.K % kBK) return cudaErrorInvalidValue;
    if (a.block_m <= 64) return launch_cfg<8, 16, 8, 1, 16>(a, stream);   // up to 64 tokens per item
    return launch_cfg<4, 8, 8, 4, 16>(a, stream);                        // up to 256 tokens per item
}

}  // namespace chord
