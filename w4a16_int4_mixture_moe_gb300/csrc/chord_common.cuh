// Device helpers shared by the sm_103a kernels of the W4A16 MoE library:
// packed-layout constants, the sticky error word, mbarrier / bulk-copy
// wrappers (inline PTX), bounded waits.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdlib.h>

#include <utility>

#include "../../include/chord.h"

namespace chord {

// ---- packed weight layout 1 -------------------------------------------------
// 256-byte header, then per expert a grid of 576-byte chunks: chunk (kc, mt)
// at ((kc * N/16) + mt) * 576 covers 16 rows of N and 64 columns of K.  Bytes
// [0, 512) hold 128 words, word lane*4 + j (k16 step j) carrying the 8 codes of
// the m16n8k16 A fragment of that lane; bytes [512, 576) hold 16 words of
// scale pairs (row g, row g+8) for the two 32-column groups of the chunk.
constexpr int kHeaderBytes = 256;
constexpr uint32_t kMagic = 0x44524843u;  // "CHRD"
constexpr uint32_t kLayoutVersion = 1;
constexpr int kChunkBytes = 576;
constexpr int kChunkWeightBytes = 512;
constexpr int kGroup = 32;

// ---- error word -----------------------------------------------------------
__device__ __forceinline__ void set_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Wait bound for every spin on an mbarrier: after this many SM clocks the
// waiter records CHORD_DEV_TIMEOUT and gives up (about 2 s at 2 GHz).
constexpr long long kWaitLimitCycles = 4000000000LL;

// ---- programmatic dependent launch -------------------------------------------
// The layer's kernels are launched with programmatic stream serialization: a
// kernel may be scheduled while the previous kernel of the stream still runs
// (once every block of that kernel has started), and waits in
// griddepcontrol.wait until the previous kernel has finished and its memory
// is visible.  Every kernel launched this way calls pdl_wait() before its
// first access to global memory, so the order of reads and writes is the
// stream order; what overlaps is the launch and block scheduling.  Without
// the attribute both instructions return at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The attribute is used for calls of up to kPdlMaxPairs (token, expert) pairs,
// where launch latency is a visible share of the step (measured on GB300:
// one-token TP8 layer 32.6 -> 31.6 us, T=16 102.4 -> 100.9 us, the 16-token
// test layer 21.3 -> 19.6 us); larger calls measured slower with it (TP8
// T=1024 542 -> 561 us, T=4096 1326 -> 1361 us) and use plain launches.
// CHORD_PDL=0 in the environment turns it off everywhere.
constexpr int64_t kPdlMaxPairs = 4096;

inline bool pdl_enabled() {
    static const bool on = [] {
        const char* v = getenv("CHORD_PDL");
        return !(v && v[0] == '0');
    }();
    return on;
}

inline bool pdl_for(int64_t pairs) { return pairs <= kPdlMaxPairs && pdl_enabled(); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool on, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = on ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---- shared memory / mbarrier ------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false when
// the bound ran out (the caller records the error and leaves).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) return false;
    }
    return true;
}

// Bulk (non-tensor) async copy global -> this CTA's shared memory; completion
// is counted in bytes on `bar`.  Addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction-priority hint (weights are streamed once).
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(smem_dst)),
        "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 16-byte asynchronous copy global -> shared (cp.async, L2 only), both
// addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---- packed header check ----------------------------------------------------
// The header records the layout a blob was packed for; a kernel refuses a blob
// of another layout or shape (the article's prepared weights record their
// packing mode and a mismatch fails loudly at dispatch).
__device__ __forceinline__ bool header_ok_layout(const uint8_t* blob, int E, int N, int K, uint32_t layout) {
    const uint32_t* h = reinterpret_cast<const uint32_t*>(blob);
    const unsigned long long* h64 = reinterpret_cast<const unsigned long long*>(blob + 32);
    const unsigned long long stride = (unsigned long long)N * (unsigned long long)K * 9ull / 16ull;
    return h[0] == kMagic && h[1] == 1u && h[2] == layout && h[3] == (uint32_t)kGroup && h[4] == (uint32_t)E &&
           h[5] == (uint32_t)N && h[6] == (uint32_t)K && h64[0] == stride &&
           h64[1] == (unsigned long long)kHeaderBytes;
}

__device__ __forceinline__ bool header_ok(const uint8_t* blob, int E, int N, int K) {
    return header_ok_layout(blob, E, N, K, kLayoutVersion);
}

// ---- bf16 packing helpers ---------------------------------------------------
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t x, uint32_t mask, uint32_t magic) {
    uint32_t r;
    // (x & mask) | magic
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(x), "r"(mask), "r"(magic));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %1, %2;" : "=r"(r) : "r"(a), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t bf2_as_u32(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __nv_bfloat162 u32_as_bf2(uint32_t v) { return *reinterpret_cast<__nv_bfloat162*>(&v); }

// Four A-fragment registers (bf16x2) of one k16 step from the packed word `w`
// and the scale pair `sp` (low half: scale of row g, high half: row g+8).
// Each value is bf16_rne((q - 8) * s): 0x4300 | q is the bf16 number 128 + q,
// subtracting 136 gives q - 8 exactly, and one bf16x2 multiply rounds the
// exact product once, to nearest even.
__device__ __forceinline__ void dequant_frag(uint32_t w, uint32_t sp, uint32_t (&a)[4]) {
    const __nv_bfloat162 off = u32_as_bf2(0x43084308u);  // (136, 136)
    const __nv_bfloat162 s_lo = u32_as_bf2(prmt(sp, 0x1010u));
    const __nv_bfloat162 s_hi = u32_as_bf2(prmt(sp, 0x3232u));
    const uint32_t q0 = lop3_and_or(w, 0x000F000Fu, 0x43004300u);        // n0, n4: row g,   k 2c, 2c+1
    const uint32_t q1 = lop3_and_or(w >> 4, 0x000F000Fu, 0x43004300u);   // n1, n5: row g+8, k 2c, 2c+1
    const uint32_t q2 = lop3_and_or(w >> 8, 0x000F000Fu, 0x43004300u);   // n2, n6: row g,   k 2c+8, 2c+9
    const uint32_t q3 = lop3_and_or(w >> 12, 0x000F000Fu, 0x43004300u);  // n3, n7: row g+8, k 2c+8, 2c+9
    a[0] = bf2_as_u32(__hmul2(__hsub2(u32_as_bf2(q0), off), s_lo));
    a[1] = bf2_as_u32(__hmul2(__hsub2(u32_as_bf2(q1), off), s_hi));
    a[2] = bf2_as_u32(__hmul2(__hsub2(u32_as_bf2(q2), off), s_lo));
    a[3] = bf2_as_u32(__hmul2(__hsub2(u32_as_bf2(q3), off), s_hi));
}

// Eight consecutive columns of one row (layout 2: nibbles 0,4,1,5,2,6,3,7 of
// `w` hold columns +0..+7) to four bf16x2 registers in column order, with the
// row's group scale `sp` duplicated in both halves.  Same arithmetic as
// dequant_frag: 128 + q, minus 136, one rounding multiply.
__device__ __forceinline__ void dequant_row8(uint32_t w, uint32_t sp, uint32_t* out) {
    const __nv_bfloat162 off = u32_as_bf2(0x43084308u);  // (136, 136)
    const __nv_bfloat162 s2 = u32_as_bf2(sp);
    const uint32_t q0 = lop3_and_or(w, 0x000F000Fu, 0x43004300u);        // columns +0, +1
    const uint32_t q1 = lop3_and_or(w >> 4, 0x000F000Fu, 0x43004300u);   // +2, +3
    const uint32_t q2 = lop3_and_or(w >> 8, 0x000F000Fu, 0x43004300u);   // +4, +5
    const uint32_t q3 = lop3_and_or(w >> 12, 0x000F000Fu, 0x43004300u);  // +6, +7
    out[0] = bf2_as_u32(__hmul2(__hsub2(u32_as_bf2(q0), off), s2));
    out[1] = bf2_as_u32(__hmul2(__hsub2(u32_as_bf2(q1), off), s2));
    out[2] = bf2_as_u32(__hmul2(__hsub2(u32_as_bf2(q2), off), s2));
    out[3] = bf2_as_u32(__hmul2(__hsub2(u32_as_bf2(q3), off), s2));
}

// ---- one-instruction dequantisation for scales in [2^-126, 0.5) ---------------
// Header word 7 of a packed blob is 1 when every group scale is a positive
// normal bf16 below 0.5 (bit patterns 0x0080 .. 0x3EFF), else 0; the packer
// writes it.  For such scales a code q costs one bf16x2 FMA per pair:
//   * a nibble in bits 4..7 of a half-word whose other bits are zero is the
//     bf16 number q * 2^-129 exactly (exponent field 0 or 1: both have the
//     spacing 2^-133, so the value is linear in all four bits);
//   * b = s * 2^129 is exact and finite for s in range (an exponent add);
//   * c = -8 * s is exact;
//   * fma(a, b, c) = q*s - 8*s = (q - 8) * s exactly before its single
//     rounding to nearest even, i.e. bf16((q - 8) * s), the subtract-then-scale
//     value; q = 8 gives +0, as (q - 8) * s does for s > 0.
constexpr int kHdrScaleRangeWord = 7;

__host__ __device__ __forceinline__ bool scale_in_fma_range(uint32_t s16) {
    return s16 - 0x0080u <= 0x3EFFu - 0x0080u;
}

__device__ __forceinline__ bool header_scales_in_fma_range(const uint8_t* blob) {
    return reinterpret_cast<const uint32_t*>(blob)[kHdrScaleRangeWord] == 1u;
}

// (b, c) = (s * 2^129, -8 * s) in both halves, from the scale pair `sp`.
__device__ __forceinline__ void fma_scale_pair(uint32_t sp, uint32_t& b2, uint32_t& c2) {
    b2 = sp + 0x40804080u;   // exponent field + 129 in each half (normal s below 0.5: no carry out)
    c2 = bf2_as_u32(__hmul2(u32_as_bf2(sp), u32_as_bf2(0xC100C100u)));   // times -8, exact
}

// dequant_row8 for a blob whose header says every scale is in range: the
// same four bf16x2 registers, nibble i moved to bits 4..7 of each half.
__device__ __forceinline__ void dequant_row8_fma(uint32_t w, uint32_t b2u, uint32_t c2u, uint32_t* out) {
    const __nv_bfloat162 b2 = u32_as_bf2(b2u), c2 = u32_as_bf2(c2u);
    const uint32_t q0 = (w << 4) & 0x00F000F0u;   // columns +0, +1
    const uint32_t q1 = w & 0x00F000F0u;          // +2, +3
    const uint32_t q2 = (w >> 4) & 0x00F000F0u;   // +4, +5
    const uint32_t q3 = (w >> 8) & 0x00F000F0u;   // +6, +7
    out[0] = bf2_as_u32(__hfma2(u32_as_bf2(q0), b2, c2));
    out[1] = bf2_as_u32(__hfma2(u32_as_bf2(q1), b2, c2));
    out[2] = bf2_as_u32(__hfma2(u32_as_bf2(q2), b2, c2));
    out[3] = bf2_as_u32(__hfma2(u32_as_bf2(q3), b2, c2));
}

__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Tail split of a persistent launch of n_items items over G CTAs in a static
// round robin: the `full` = floor(n_items / G) * G items of the full waves run
// whole; the `tail` items of the last partial wave would keep `tail` CTAs busy
// for a whole item while the other G - tail idle, so each is cut into S K
// slices (S = G / tail, at most 16 and at most kstages / min_stages, so every
// slice holds >= min_stages stages), S = 1 when that gives fewer than two.
// Work units: u < full -> item u; else v = u - full, item full + v / S, slice
// v % S.  Computed from the device-side item count by every kernel that needs
// it, so no plan is stored.
struct TailPlan {
    int64_t full, tail;
    int S;
};

__host__ __device__ __forceinline__ TailPlan tail_plan(int64_t n_items, int64_t G, int kstages, int min_stages,
                                                       bool enabled) {
    TailPlan t;
    t.full = G > 0 ? n_items / G * G : n_items;
    t.tail = n_items - t.full;
    t.S = 1;
    if (enabled && t.tail > 0 && min_stages > 0) {
        int64_t S = G / t.tail;
        const int64_t cap = kstages / min_stages;
        if (S > cap) S = cap;
        if (S > 16) S = 16;
        t.S = S < 2 ? 1 : (int)S;
    }
    return t;
}

// q = v / d, r = v % d for v >= 0, d > 0: 32-bit division while v fits (the
// grid-stride element loops), 64-bit above.
__device__ __forceinline__ int64_t divmod_idx(int64_t v, int d, int& r) {
    if (v <= 0x7fffffffLL) {
        const uint32_t q = (uint32_t)v / (uint32_t)d;
        r = (int)((uint32_t)v - q * (uint32_t)d);
        return (int64_t)q;
    }
    const int64_t q = v / d;
    r = (int)(v - q * d);
    return q;
}

// SiLU(g) * u in FP32: g / (1 + exp(-g)), then times u, with the fast
// exponential and division intrinsics (a few float ulps from the correctly
// rounded forms, far below the bf16 rounding that follows).  Large -g gives
// exp(-g) = inf and a quotient of 0 where the exact value is a tiny negative.
__device__ __forceinline__ float silu_times(float g, float u) {
    const float s = __fdividef(g, __fadd_rn(1.0f, __expf(-g)));
    return __fmul_rn(s, u);
}

// The fused gate_up epilogue's value: the gate and up FP32 sums rounded to
// bf16 (the GEMM's output type), then bf16(SiLU(g) * u) — what the GEMM
// followed by the SiLU * up pass computes.
__device__ __forceinline__ __nv_bfloat16 silu_mul_bf16(float g_sum, float u_sum) {
    const float g = __bfloat162float(__float2bfloat16_rn(g_sum));
    const float u = __bfloat162float(__float2bfloat16_rn(u_sum));
    return __float2bfloat16_rn(silu_times(g, u));
}

// The fused combine's write for one FP32 result `v` of pair p, column n:
// when p is its token's only local pair (pair_w[p] a number) the token's
// output is the weighted sum over that one pair, bf16(0 + w * v) with the
// product and the sum rounded separately as in the combine pass; otherwise
// the FP32 value goes to C2 for the finishing sum.  Returns nothing.
__device__ __forceinline__ void combine_store(float* C2, uint16_t* out, int64_t N, int64_t p, int64_t t, float w,
                                              int n, float v) {
    if (w == w) {
        const float o = __fadd_rn(0.0f, __fmul_rn(w, v));
        out[t * N + n] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
    } else {
        C2[p * N + n] = v;
    }
}

}  // namespace chord
