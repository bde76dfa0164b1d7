/*
 * CPU oracle for the W4A16 INT4 mixture-of-experts expert GEMM described in
 * "vLLM x Novita AI: Chord, a faster INT4 MoE for Kimi K2.x" (sections
 * "Two kernel families", "Indexed kernels", "Grouped SM90 kernels").
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  It shares no code, header, table or
 * constant generator with the CUDA library, and neither includes the other.
 *
 * It is deliberately plain and slow: every result is the definition written
 * out, one output element at a time, with a sequential FP32 sum in ascending
 * k.  OpenMP only spreads independent output elements over threads; it never
 * splits or reorders a sum.  Build with -ffp-contract=off so that every
 * product and every sum is rounded exactly where the C source says.
 *
 * What is computed (the article fixes the data types; the reading of each
 * point the article leaves open is listed with the function):
 *   dequant   w = bf16_rne( (q - 8) * s ), q a uint4 code, s the BF16 scale of
 *             its group of 32 along K ("subtract then scale", section "H200 and
 *             Blackwell indexed decode"; weight and scale shapes [G,N,K] and
 *             [G,N,K/32] from the grouped operator example).
 *   align     vLLM moe_align_block_size contract: sorted_ids / expert_ids /
 *             num_tokens_padded, padding carried by sentinels in the index
 *             arrays, activations never padded (section "Grouped SM90
 *             kernels", figure 3, and the deployment notes on the indexed
 *             fast path).
 *   gemm      C[p, n] = bf16_rne( sum_k x[p / d, k] * w[e, n, k] ), FP32 sum
 *             (F16 accumulation is not implemented by either backend,
 *             deployment notes), BF16 output.
 *   act       h = bf16_rne( silu(g) * u ), gate rows 0..I-1, up rows I..2I-1.
 *   combine   out[t, n] = bf16_rne( sum over local k, ascending, of
 *             w[t, k] * C2[t * topk + k, n] ), C2 in bf16 or binary32.
 *   layer     the steps above, with the down projection's FP32 sums fed to
 *             the combine unrounded (see orc_moe_layer).
 *   f64 sums  a second valid evaluation of the same definitions: every dot
 *             product and the weighted sum in binary64, rounded to bf16 at the
 *             same points (orc_*_f64sum).  It is nearly the exact result, and
 *             the parity tests use it to measure how far two valid summation
 *             orders fall apart after a bf16 rounding.
 *   pack      the byte layout the CUDA library reads (its own specification,
 *             written out below), so the GPU packer can be checked byte for
 *             byte; and its inverse.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_EINVAL (-1)   /* bad shape or argument */
#define ORC_ELAYOUT (-2)  /* packed blob header does not match */
#define ORC_ERANGE (-3)   /* an index or code is out of range */
#define ORC_ENOMEM (-4)

#define ORC_GROUP 32

int orc_version(void) { return 1; }

/* ------------------------------------------------------------------------ */
/* BF16 <-> FP32.  A bf16 value is the upper half of an IEEE binary32.       */

static float f32_from_bf16(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to the nearest bf16, ties to even.  NaN stays NaN (quiet
 * bit set, sign kept); overflow rounds to infinity as IEEE rounding does. */
static uint16_t bf16_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u)))
        keep += 1u;
    return (uint16_t)keep;
}

uint16_t orc_bf16_round(float f) { return bf16_from_f32(f); }

/* Round a binary64 to the nearest bf16, ties to even, with one rounding.
 * (float)d rounds to the nearest binary32 first; that differs from rounding d
 * itself only when the binary32 result is exactly halfway between two bf16
 * values: d then lies on one side of that midpoint (or on it), and the sign of
 * the exact residual d - (float)d (exact by Sterbenz's lemma) says which.
 * Finite values in the binary32 range only (the layer's values are). */
static uint16_t bf16_from_f64(double d)
{
    float f = (float)d;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0xffffu) == 0x8000u && (u & 0x7fffffffu) < 0x7f800000u) {
        double r = d - (double)f;
        if (r != 0.0) {
            uint32_t keep = u >> 16;
            int away = (r > 0.0) == (f > 0.0);   /* |d| above the midpoint */
            return (uint16_t)(away ? keep + 1u : keep);
        }
    }
    return bf16_from_f32(f);
}

uint16_t orc_bf16_round_f64(double d) { return bf16_from_f64(d); }

/* ------------------------------------------------------------------------ */
/* Dequantisation: subtract the offset 8, then multiply by the group scale,
 * then round once to bf16.  (q - 8) is an integer in [-8, 7] and s carries 8
 * significant bits, so the binary32 product is exact and the only rounding is
 * the final one. */

uint16_t orc_dequant(uint8_t q, uint16_t s)
{
    float d = (float)((int)q - 8);
    float p = d * f32_from_bf16(s);
    return bf16_from_f32(p);
}

void orc_dequant_pairs(const uint8_t *q, const uint16_t *s, size_t n, uint16_t *out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = orc_dequant(q[i], s[i]);
}

/* ------------------------------------------------------------------------ */
/* Packed weight layouts.  The article records the packing mode in the
 * prepared weight and checks it when the weight is used; here the header
 * records the layout.
 *
 * blob  = 256-byte header, then E expert regions of N*K*9/16 bytes each.
 * header (little endian): u32 magic 0x44524843 ("CHRD"), u32 version 1,
 *        u32 layout (1, 2 or 3), u32 group 32, u32 E, u32 N, u32 K,
 *        u32 scale_range, u64 expert_stride = N*K*9/16, u64 data_offset = 256,
 *        then zeros.  scale_range is 1 when every scale of the blob is a
 *        positive normal bf16 below 0.5 (2^-126 <= s < 0.5), else 0: a fact
 *        about the weights that the header records so that a kernel may pick a
 *        dequantisation valid on that range; it does not change any value.
 *
 * Layout 1 ("m16 x k64 fragment chunks", N % 16 == 0, K % 64 == 0).
 * An expert region is a sequence of 576-byte chunks, chunk (kc, mt) at
 * ((kc * N/16) + mt) * 576, for kc < K/64 (64 columns of K) and mt < N/16
 * (16 rows of N).  Within a chunk:
 *   bytes [0, 512): 128 little-endian 32-bit words, word (lane*4 + j) for
 *       lane < 32 and j < 4 (16 columns each).  With g = lane/4, c = lane%4,
 *       nibble i (bits 4i..4i+3) of that word holds the code of
 *         i=0: row g,   col 16j+2c      i=4: row g,   col 16j+2c+1
 *         i=1: row g+8, col 16j+2c      i=5: row g+8, col 16j+2c+1
 *         i=2: row g,   col 16j+2c+8    i=6: row g,   col 16j+2c+9
 *         i=3: row g+8, col 16j+2c+8    i=7: row g+8, col 16j+2c+9
 *       (rows relative to 16*mt, columns relative to 64*kc).
 *   bytes [512, 576): 16 words, word (h*8 + g) for h < 2, g < 8 holds the bf16
 *       scale of row g in its low half and of row g+8 in its high half, for
 *       the group of 32 columns 64*kc + 32*h .. +31.
 *
 * Layout 2 ("128-row x k64 chunks", N % 128 == 0, K % 64 == 0).
 * An expert region is a sequence of 4608-byte chunks, chunk (nt, kc) at
 * ((nt * K/64) + kc) * 4608, for nt < N/128 (128 rows) and kc < K/64.  Within
 * a chunk, with r the row in the tile and c the column in the chunk:
 *   bytes [0, 4096): half h = c/32 at h*2048, then row r at r*16, then word
 *       j = (c%32)/8 at j*4 (little endian); column 8j + m of the half sits
 *       in nibble i of that word with m = 2*(i%4) + i/4, i.e. nibbles
 *       0,4,1,5,2,6,3,7 hold columns +0..+7.
 *   bytes [4096, 4608): the bf16 scale of row r, group h (columns 32h..32h+31
 *       of the chunk) at 4096 + r*4 + h*2.
 *
 * Layout 3 ("layout 2 with gate and up rows interleaved", for a gate_up weight
 * of N = 2I rows: gate rows 0..I-1, up rows I..2I-1; N % 128 == 0).  Layout 2
 * byte positions, where packed row p holds canonical row
 *   8*(p/16) + p%16            if p%16 < 8   (gate row j = 8*(p/16) + p%16)
 *   I + 8*(p/16) + p%16 - 8    otherwise     (the up row of the same j),
 * so each 16-row group holds gate rows 8g'..8g'+7 followed by their up rows.
 */

#define ORC_HDR 256u
#define ORC_MAGIC 0x44524843u
#define ORC_CHUNK1 576u
#define ORC_CHUNK2 4608u

static int layout_ok(int layout, int N, int K)
{
    if (N <= 0 || K <= 0 || K % 64)
        return 0;
    if (layout == 1)
        return N % 16 == 0;
    if (layout == 2 || layout == 3)
        return N % 128 == 0;
    return 0;
}

/* Layout 3: the packed row holding canonical row n (the inverse of the map in
 * the layout description); other layouts keep rows in place. */
static int packed_row(int layout, int N, int n)
{
    if (layout != 3)
        return n;
    int half = N / 2;
    if (n < half)
        return 16 * (n / 8) + n % 8;
    int m = n - half;
    return 16 * (m / 8) + 8 + m % 8;
}

size_t orc_packed_bytes(int E, int N, int K, int layout)
{
    if (E < 0 || !layout_ok(layout, N, K))
        return 0;
    return (size_t)ORC_HDR + (size_t)E * (size_t)N * (size_t)K * 9u / 16u;
}

static void put32(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}
static uint32_t get32(const uint8_t *p)
{
    return (uint32_t)p[0] | (uint32_t)p[1] << 8 | (uint32_t)p[2] << 16 | (uint32_t)p[3] << 24;
}
static void put64(uint8_t *p, uint64_t v) { put32(p, (uint32_t)v); put32(p + 4, (uint32_t)(v >> 32)); }
static uint64_t get64(const uint8_t *p) { return (uint64_t)get32(p) | (uint64_t)get32(p + 4) << 32; }

/* Byte offset (from the start of the expert region) and nibble shift of the
 * code of row n, column k. */
static void code_pos(int layout, int N, int K, int n, int k, size_t *byte, int *shift)
{
    n = packed_row(layout, N, n);
    if (layout == 1) {
        int mt = n / 16, r = n % 16, kc = k / 64, kk = k % 64;
        int j = kk / 16, kq = kk % 16;
        int g = r % 8, lower = r / 8;             /* lower: 0 = row g, 1 = row g+8 */
        int kpart = kq / 8, c = (kq % 8) / 2, odd = kq % 2;
        int lane = 4 * g + c;
        int word = lane * 4 + j;
        int i = kpart * 2 + lower + 4 * odd;
        *byte = ((size_t)kc * (size_t)(N / 16) + (size_t)mt) * ORC_CHUNK1 + (size_t)word * 4u + (size_t)(i / 2);
        *shift = (i % 2) * 4;
    } else {
        int nt = n / 128, r = n % 128, kc = k / 64, c = k % 64;
        int h = c / 32, j = (c % 32) / 8, m = c % 8;
        int i = (m % 2) * 4 + m / 2;              /* inverse of m = 2*(i%4) + i/4 */
        *byte = ((size_t)nt * (size_t)(K / 64) + (size_t)kc) * ORC_CHUNK2 + (size_t)h * 2048u
                + (size_t)r * 16u + (size_t)j * 4u + (size_t)(i / 2);
        *shift = (i % 2) * 4;
    }
}

/* Byte offset (from the start of the expert region) of the scale of row n,
 * group grp (columns 32*grp .. 32*grp+31). */
static size_t scale_pos(int layout, int N, int K, int n, int grp)
{
    n = packed_row(layout, N, n);
    if (layout == 1) {
        int mt = n / 16, r = n % 16, kc = grp / 2, h = grp % 2;
        int g = r % 8, lower = r / 8;
        return ((size_t)kc * (size_t)(N / 16) + (size_t)mt) * ORC_CHUNK1 + 512u
               + (size_t)(h * 8 + g) * 4u + (size_t)lower * 2u;
    } else {
        int nt = n / 128, r = n % 128, kc = grp / 2, h = grp % 2;
        return ((size_t)nt * (size_t)(K / 64) + (size_t)kc) * ORC_CHUNK2 + 4096u + (size_t)r * 4u
               + (size_t)h * 2u;
    }
}

/* 1 when every one of the n scales is a positive normal bf16 below 0.5, read
 * from its value: sign clear, biased exponent between 1 and 125. */
uint32_t orc_scale_range(const uint16_t *scales, size_t n)
{
    for (size_t i = 0; i < n; ++i) {
        unsigned sign = scales[i] >> 15, expo = (scales[i] >> 7) & 0xFFu;
        if (sign != 0 || expo < 1 || expo > 125)
            return 0u;
    }
    return 1u;
}

int orc_pack(const uint8_t *codes, const uint16_t *scales, int E, int N, int K, int layout,
             uint8_t *out, size_t out_bytes)
{
    size_t need = orc_packed_bytes(E, N, K, layout);
    if (need == 0 || out_bytes < need)
        return ORC_EINVAL;
    memset(out, 0, need);
    uint64_t stride = (uint64_t)N * (uint64_t)K * 9u / 16u;
    put32(out + 0, ORC_MAGIC);
    put32(out + 4, 1u);
    put32(out + 8, (uint32_t)layout);
    put32(out + 12, ORC_GROUP);
    put32(out + 16, (uint32_t)E);
    put32(out + 20, (uint32_t)N);
    put32(out + 24, (uint32_t)K);
    put32(out + 28, orc_scale_range(scales, (size_t)E * (size_t)N * (size_t)(K / ORC_GROUP)));
    put64(out + 32, stride);
    put64(out + 40, ORC_HDR);
    int G = K / ORC_GROUP;
    for (int e = 0; e < E; ++e) {
        uint8_t *reg = out + ORC_HDR + (size_t)e * stride;
        for (int n = 0; n < N; ++n) {
            for (int k = 0; k < K; ++k) {
                uint8_t q = codes[((size_t)e * N + n) * K + k];
                if (q > 15)
                    return ORC_ERANGE;
                size_t b; int sh;
                code_pos(layout, N, K, n, k, &b, &sh);
                reg[b] |= (uint8_t)(q << sh);
            }
            for (int grp = 0; grp < G; ++grp) {
                uint16_t s = scales[((size_t)e * N + n) * G + grp];
                size_t b = scale_pos(layout, N, K, n, grp);
                reg[b] = (uint8_t)s;
                reg[b + 1] = (uint8_t)(s >> 8);
            }
        }
    }
    return ORC_OK;
}

int orc_check_header(const uint8_t *blob, int E, int N, int K, int layout)
{
    if (get32(blob + 0) != ORC_MAGIC || get32(blob + 4) != 1u || get32(blob + 8) != (uint32_t)layout
        || get32(blob + 12) != ORC_GROUP || get32(blob + 16) != (uint32_t)E
        || get32(blob + 20) != (uint32_t)N || get32(blob + 24) != (uint32_t)K
        || get64(blob + 32) != (uint64_t)N * (uint64_t)K * 9u / 16u || get64(blob + 40) != ORC_HDR)
        return ORC_ELAYOUT;
    return ORC_OK;
}

int orc_unpack(const uint8_t *blob, size_t blob_bytes, int E, int N, int K, int layout,
               uint8_t *codes, uint16_t *scales)
{
    size_t need = orc_packed_bytes(E, N, K, layout);
    if (need == 0 || blob_bytes < need)
        return ORC_EINVAL;
    if (orc_check_header(blob, E, N, K, layout) != ORC_OK)
        return ORC_ELAYOUT;
    uint64_t stride = (uint64_t)N * (uint64_t)K * 9u / 16u;
    int G = K / ORC_GROUP;
    for (int e = 0; e < E; ++e) {
        const uint8_t *reg = blob + ORC_HDR + (size_t)e * stride;
        for (int n = 0; n < N; ++n) {
            for (int k = 0; k < K; ++k) {
                size_t b; int sh;
                code_pos(layout, N, K, n, k, &b, &sh);
                codes[((size_t)e * N + n) * K + k] = (uint8_t)((reg[b] >> sh) & 0xf);
            }
            for (int grp = 0; grp < G; ++grp) {
                size_t b = scale_pos(layout, N, K, n, grp);
                scales[((size_t)e * N + n) * G + grp] = (uint16_t)(reg[b] | (uint16_t)reg[b + 1] << 8);
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* moe_align_block_size.
 *
 * Pairs p = t*topk + k with topk_ids[p] = e in [0, E) are local; any other id
 * (the value -1 marks an expert on another GPU) is dropped.  Experts are laid
 * out in ascending order; within an expert its pair ids appear in ascending
 * order (the article does not fix this order; ascending makes the result
 * unique).  Each expert's run is padded with the sentinel P = T*topk up to a
 * multiple of block_m; an expert with no pair gets no block.  expert_ids[b]
 * names the expert of block b; num_tokens_padded is the padded total.  The
 * arrays are over-allocated to the capacity below; entries past the padded
 * total hold the sentinel (sorted_ids) and -1 (expert_ids). */

int64_t orc_align_capacity(int T, int topk, int E, int block_m)
{
    if (T < 0 || topk <= 0 || E <= 0 || block_m <= 0)
        return -1;
    int64_t P = (int64_t)T * topk;
    int64_t m = P < E ? P : E;
    int64_t c = P + m * (block_m - 1);
    return (c + block_m - 1) / block_m * block_m;
}

int orc_moe_align(const int32_t *topk_ids, int T, int topk, int E, int block_m,
                  int32_t *sorted_ids, int32_t *expert_ids, int32_t *num_tokens_padded,
                  int64_t capacity)
{
    int64_t cap = orc_align_capacity(T, topk, E, block_m);
    if (cap < 0 || capacity < cap)
        return ORC_EINVAL;
    int64_t P = (int64_t)T * topk;
    int32_t sentinel = (int32_t)P;
    int64_t pos = 0;
    for (int e = 0; e < E; ++e) {
        int64_t start = pos;
        for (int64_t p = 0; p < P; ++p)
            if (topk_ids[p] == e)
                sorted_ids[pos++] = (int32_t)p;
        if (pos == start)
            continue;
        while ((pos - start) % block_m)
            sorted_ids[pos++] = sentinel;
        for (int64_t b = start / block_m; b < pos / block_m; ++b)
            expert_ids[b] = e;
    }
    *num_tokens_padded = (int32_t)pos;
    for (int64_t i = pos; i < capacity; ++i)
        sorted_ids[i] = sentinel;
    for (int64_t b = pos / block_m; b < capacity / block_m; ++b)
        expert_ids[b] = -1;
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Indexed grouped GEMM.  For every block b below num_tokens_padded/block_m,
 * with e = expert_ids[b], and every non-sentinel pair id p in that block:
 *     C[p, n] = bf16_rne( sum_{k=0..K-1} float(A[p / d, k]) * float(w[e, n, k]) )
 * where w is the dequantised weight and d = a_row_divisor (topk when A holds
 * one row per token, 1 when it holds one row per pair).  The sum runs in
 * ascending k in binary32.  Each bf16 x bf16 product is exact in binary32.
 * Rows of C that no block names are left untouched. */

static void dequant_expert(const uint8_t *codes, const uint16_t *scales, int e, int N, int K,
                           float *wq, int nthreads)
{
    int G = K / ORC_GROUP;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int n = 0; n < N; ++n)
        for (int k = 0; k < K; ++k) {
            uint8_t q = codes[((size_t)e * N + n) * K + k];
            uint16_t s = scales[((size_t)e * N + n) * G + k / ORC_GROUP];
            wq[(size_t)n * K + k] = f32_from_bf16(orc_dequant(q, s));
        }
}

/* Shared body of the output precisions: exactly one of Cb (bf16, one
 * rounding of the sum), Cf (the FP32 sum itself) and Cd (the binary64 sum) is
 * non-NULL.  f64sum selects a binary64 sum (each bf16 x bf16 product is exact
 * in binary64 too) in the same ascending order; Cf goes with the FP32 sum
 * only, Cd with the binary64 sum only. */
static int gemm_indexed(const uint16_t *A, int64_t a_rows, int a_row_divisor,
                        const uint8_t *codes, const uint16_t *scales, int E, int N, int K,
                        const int32_t *sorted_ids, const int32_t *expert_ids, int32_t num_tokens_padded,
                        int block_m, int64_t num_pairs, uint16_t *Cb, float *Cf, double *Cd, int f64sum,
                        int nthreads)
{
    if (N <= 0 || K <= 0 || K % ORC_GROUP || block_m <= 0 || a_row_divisor <= 0
        || num_tokens_padded < 0 || num_tokens_padded % block_m)
        return ORC_EINVAL;
    int64_t nblocks = num_tokens_padded / block_m;
    for (int64_t b = 0; b < nblocks; ++b) {
        if (expert_ids[b] < 0 || expert_ids[b] >= E)
            return ORC_ERANGE;
        for (int i = 0; i < block_m; ++i) {
            int32_t p = sorted_ids[b * block_m + i];
            if (p == (int32_t)num_pairs)
                continue;
            if (p < 0 || p > num_pairs || (int64_t)(p / a_row_divisor) >= a_rows)
                return ORC_ERANGE;
        }
    }
    float *wq = (float *)malloc((size_t)N * (size_t)K * sizeof(float));
    int32_t *rows = (int32_t *)malloc((size_t)(num_tokens_padded > 0 ? num_tokens_padded : 1) * sizeof(int32_t));
    if (!wq || !rows) {
        free(wq); free(rows);
        return ORC_ENOMEM;
    }
    for (int e = 0; e < E; ++e) {
        int64_t nr = 0;
        for (int64_t b = 0; b < nblocks; ++b) {
            if (expert_ids[b] != e)
                continue;
            for (int i = 0; i < block_m; ++i) {
                int32_t p = sorted_ids[b * block_m + i];
                if (p != (int32_t)num_pairs)
                    rows[nr++] = p;
            }
        }
        if (nr == 0)
            continue;
        dequant_expert(codes, scales, e, N, K, wq, nthreads);
#pragma omp parallel for num_threads(nthreads) schedule(static) collapse(2)
        for (int64_t r = 0; r < nr; ++r)
            for (int n = 0; n < N; ++n) {
                int32_t p = rows[r];
                const uint16_t *a = A + (size_t)(p / a_row_divisor) * (size_t)K;
                const float *w = wq + (size_t)n * K;
                if (f64sum) {
                    double dacc = 0.0;
                    for (int k = 0; k < K; ++k)
                        dacc += (double)f32_from_bf16(a[k]) * (double)w[k];
                    if (Cb)
                        Cb[(size_t)p * N + n] = bf16_from_f64(dacc);
                    else
                        Cd[(size_t)p * N + n] = dacc;
                    continue;
                }
                float acc = 0.0f;
                for (int k = 0; k < K; ++k)
                    acc += f32_from_bf16(a[k]) * w[k];
                if (Cb)
                    Cb[(size_t)p * N + n] = bf16_from_f32(acc);
                else
                    Cf[(size_t)p * N + n] = acc;
            }
    }
    free(wq);
    free(rows);
    return ORC_OK;
}

/* BF16 output: the GEMM operation as the article's kernels expose it. */
int orc_moe_gemm(const uint16_t *A, int64_t a_rows, int a_row_divisor,
                 const uint8_t *codes, const uint16_t *scales, int E, int N, int K,
                 const int32_t *sorted_ids, const int32_t *expert_ids, int32_t num_tokens_padded,
                 int block_m, int64_t num_pairs, uint16_t *C, int nthreads)
{
    return gemm_indexed(A, a_rows, a_row_divisor, codes, scales, E, N, K, sorted_ids, expert_ids,
                        num_tokens_padded, block_m, num_pairs, C, NULL, NULL, 0, nthreads);
}

/* FP32 output: the sum before any rounding, for a consumer that keeps FP32
 * (the layer's down projection feeding the top-k weighted sum). */
int orc_moe_gemm_f32(const uint16_t *A, int64_t a_rows, int a_row_divisor,
                     const uint8_t *codes, const uint16_t *scales, int E, int N, int K,
                     const int32_t *sorted_ids, const int32_t *expert_ids, int32_t num_tokens_padded,
                     int block_m, int64_t num_pairs, float *C, int nthreads)
{
    return gemm_indexed(A, a_rows, a_row_divisor, codes, scales, E, N, K, sorted_ids, expert_ids,
                        num_tokens_padded, block_m, num_pairs, NULL, C, NULL, 0, nthreads);
}

/* The binary64-sum variant: C[p, n] = bf16_rne( binary64 sum ), one rounding. */
int orc_moe_gemm_f64sum(const uint16_t *A, int64_t a_rows, int a_row_divisor,
                        const uint8_t *codes, const uint16_t *scales, int E, int N, int K,
                        const int32_t *sorted_ids, const int32_t *expert_ids, int32_t num_tokens_padded,
                        int block_m, int64_t num_pairs, uint16_t *C, int nthreads)
{
    return gemm_indexed(A, a_rows, a_row_divisor, codes, scales, E, N, K, sorted_ids, expert_ids,
                        num_tokens_padded, block_m, num_pairs, C, NULL, NULL, 1, nthreads);
}

/* The binary64 sums themselves (the variant's down projection feeding its
 * weighted sum). */
int orc_moe_gemm_f64(const uint16_t *A, int64_t a_rows, int a_row_divisor,
                     const uint8_t *codes, const uint16_t *scales, int E, int N, int K,
                     const int32_t *sorted_ids, const int32_t *expert_ids, int32_t num_tokens_padded,
                     int block_m, int64_t num_pairs, double *C, int nthreads)
{
    return gemm_indexed(A, a_rows, a_row_divisor, codes, scales, E, N, K, sorted_ids, expert_ids,
                        num_tokens_padded, block_m, num_pairs, NULL, NULL, C, 1, nthreads);
}

/* ------------------------------------------------------------------------ */
/* Grouped contracts (the article's "Grouped SM90 kernels" section: a second
 * routing workload besides the indexed one).
 *
 * Contiguous (prefill): the rows of A [M, K] are concatenated per expert, each
 * expert's segment padded to a multiple of 128 rows; m_indices[m] is the
 * expert of row m, -1 on padding rows.
 *     C[m, n] = bf16_rne( sum_k A[m, k] * w[m_indices[m], n, k] )   (m_indices[m] >= 0)
 * Padding rows of C are not written.
 *
 * Masked (decode): A [G, max_m, K] holds a fixed row budget per group (expert)
 * g, of which the first masked_m[g] rows are valid; C is flat [G * max_m, N].
 *     C[g * max_m + r, n] = bf16_rne( sum_k A[g, r, k] * w[g, n, k] )   (r < masked_m[g])
 * Rows past a group's count are not written.
 *
 * Same dequantisation and sequential FP32 sum in ascending k as the indexed
 * GEMM. */
static void rows_times_expert(const uint16_t *A, const int64_t *rows, int64_t nr, const float *wq, int N, int K,
                              uint16_t *C, int nthreads)
{
#pragma omp parallel for num_threads(nthreads) schedule(static) collapse(2)
    for (int64_t r = 0; r < nr; ++r)
        for (int n = 0; n < N; ++n) {
            const uint16_t *a = A + (size_t)rows[r] * (size_t)K;
            const float *w = wq + (size_t)n * K;
            float acc = 0.0f;
            for (int k = 0; k < K; ++k)
                acc += f32_from_bf16(a[k]) * w[k];
            C[(size_t)rows[r] * N + n] = bf16_from_f32(acc);
        }
}

int orc_grouped_contiguous(const uint16_t *A, int64_t M, const int32_t *m_indices, const uint8_t *codes,
                           const uint16_t *scales, int E, int N, int K, uint16_t *C, int nthreads)
{
    if (M < 0 || N <= 0 || K <= 0 || K % ORC_GROUP || E <= 0)
        return ORC_EINVAL;
    for (int64_t m = 0; m < M; ++m)
        if (m_indices[m] < -1 || m_indices[m] >= E)
            return ORC_ERANGE;
    float *wq = (float *)malloc((size_t)N * (size_t)K * sizeof(float));
    int64_t *rows = (int64_t *)malloc((size_t)(M > 0 ? M : 1) * sizeof(int64_t));
    if (!wq || !rows) {
        free(wq); free(rows);
        return ORC_ENOMEM;
    }
    for (int e = 0; e < E; ++e) {
        int64_t nr = 0;
        for (int64_t m = 0; m < M; ++m)
            if (m_indices[m] == e)
                rows[nr++] = m;
        if (nr == 0)
            continue;
        dequant_expert(codes, scales, e, N, K, wq, nthreads);
        rows_times_expert(A, rows, nr, wq, N, K, C, nthreads);
    }
    free(wq);
    free(rows);
    return ORC_OK;
}

int orc_grouped_masked(const uint16_t *A, int G, int max_m, const int32_t *masked_m, const uint8_t *codes,
                       const uint16_t *scales, int N, int K, uint16_t *C, int nthreads)
{
    if (G <= 0 || max_m < 0 || N <= 0 || K <= 0 || K % ORC_GROUP)
        return ORC_EINVAL;
    for (int g = 0; g < G; ++g)
        if (masked_m[g] < 0 || masked_m[g] > max_m)
            return ORC_ERANGE;
    float *wq = (float *)malloc((size_t)N * (size_t)K * sizeof(float));
    int64_t *rows = (int64_t *)malloc((size_t)(max_m > 0 ? max_m : 1) * sizeof(int64_t));
    if (!wq || !rows) {
        free(wq); free(rows);
        return ORC_ENOMEM;
    }
    for (int g = 0; g < G; ++g) {
        if (masked_m[g] == 0)
            continue;
        for (int r = 0; r < masked_m[g]; ++r)
            rows[r] = (int64_t)g * max_m + r;
        dequant_expert(codes, scales, g, N, K, wq, nthreads);
        rows_times_expert(A, rows, masked_m[g], wq, N, K, C, nthreads);
    }
    free(wq);
    free(rows);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* SiLU * up.  C1 holds 2I columns per pair: gate in 0..I-1, up in I..2I-1
 * (the usual concatenation of w1 and w3; the article does not show it).
 *     h[p, j] = bf16_rne( (g / (1 + exp(-g))) * u ),  g = C1[p, j], u = C1[p, I + j]
 * in binary32, for the pairs whose id names a local expert. */

int orc_silu_mul(const uint16_t *C1, const int32_t *topk_ids, int64_t P, int E, int I,
                 uint16_t *h, int nthreads)
{
    if (I <= 0 || P < 0)
        return ORC_EINVAL;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int64_t p = 0; p < P; ++p) {
        if (topk_ids[p] < 0 || topk_ids[p] >= E)
            continue;
        for (int j = 0; j < I; ++j) {
            float g = f32_from_bf16(C1[(size_t)p * 2 * I + j]);
            float u = f32_from_bf16(C1[(size_t)p * 2 * I + I + j]);
            float s = g / (1.0f + expf(-g));
            h[(size_t)p * I + j] = bf16_from_f32(s * u);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Top-k weighted combine.
 *     out[t, n] = bf16_rne( sum over k ascending with topk_ids[t, k] local of
 *                           topk_w[t, k] * C2[t*topk + k, n] )
 * in binary32, starting from +0, C2 given in bf16 or in binary32.  A token
 * with no local pair outputs +0. */

static int combine_any(const uint16_t *C2b, const float *C2f, const int32_t *topk_ids,
                       const float *topk_w, int T, int topk, int E, int H, uint16_t *out, int nthreads)
{
    if (T < 0 || topk <= 0 || H <= 0)
        return ORC_EINVAL;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < H; ++n) {
            float acc = 0.0f;
            for (int k = 0; k < topk; ++k) {
                int64_t p = (int64_t)t * topk + k;
                if (topk_ids[p] < 0 || topk_ids[p] >= E)
                    continue;
                float v = C2b ? f32_from_bf16(C2b[(size_t)p * H + n]) : C2f[(size_t)p * H + n];
                acc += topk_w[p] * v;
            }
            out[(size_t)t * H + n] = bf16_from_f32(acc);
        }
    return ORC_OK;
}

int orc_combine(const uint16_t *C2, const int32_t *topk_ids, const float *topk_w,
                int T, int topk, int E, int H, uint16_t *out, int nthreads)
{
    return combine_any(C2, NULL, topk_ids, topk_w, T, topk, E, H, out, nthreads);
}

int orc_combine_f32(const float *C2, const int32_t *topk_ids, const float *topk_w,
                    int T, int topk, int E, int H, uint16_t *out, int nthreads)
{
    return combine_any(NULL, C2, topk_ids, topk_w, T, topk, E, H, out, nthreads);
}

/* The binary64-sum variant of the combine: the same weighted sum over local k
 * in ascending order from +0, in binary64 (each weight times value product is
 * exact there), rounded to bf16 once. */
int orc_combine_f64(const double *C2, const int32_t *topk_ids, const float *topk_w,
                    int T, int topk, int E, int H, uint16_t *out, int nthreads)
{
    if (T < 0 || topk <= 0 || H <= 0)
        return ORC_EINVAL;
#pragma omp parallel for num_threads(nthreads) schedule(static)
    for (int t = 0; t < T; ++t)
        for (int n = 0; n < H; ++n) {
            double acc = 0.0;
            for (int k = 0; k < topk; ++k) {
                int64_t p = (int64_t)t * topk + k;
                if (topk_ids[p] < 0 || topk_ids[p] >= E)
                    continue;
                acc += (double)topk_w[p] * C2[(size_t)p * H + n];
            }
            out[(size_t)t * H + n] = bf16_from_f64(acc);
        }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* One MoE layer: align -> gate_up GEMM (A = x, one row per token) -> SiLU*up
 * -> down GEMM (A = h, one row per pair) -> top-k combine.  The gate_up
 * result is rounded to bf16 (the GEMM's output type) and so is SiLU*up (the
 * bf16 activation operand of the down GEMM).  The down result of each pair
 * goes into the weighted sum in binary32 and the layer output is rounded to
 * bf16 once: the pages fix BF16 for the activations a GEMM consumes and for
 * the output, and say nothing of a rounding between the down projection and
 * the weighted sum.  Rounding there would let a last-place difference
 * between two valid FP32 summation orders flip a pair result by one bf16 ulp
 * (0.5 at magnitude 100) and move a combined output near zero by that ulp
 * times the pair's weight. */

int orc_moe_layer(const uint16_t *x, const int32_t *topk_ids, const float *topk_w,
                  int T, int topk, int E, int H, int I,
                  const uint8_t *codes13, const uint16_t *scales13,
                  const uint8_t *codes2, const uint16_t *scales2,
                  int block_m, uint16_t *out, int nthreads)
{
    int64_t cap = orc_align_capacity(T, topk, E, block_m);
    if (cap < 0 || H <= 0 || I <= 0 || H % ORC_GROUP || I % ORC_GROUP)
        return ORC_EINVAL;
    int64_t P = (int64_t)T * topk;
    int32_t *sorted_ids = (int32_t *)malloc((size_t)(cap > 0 ? cap : 1) * sizeof(int32_t));
    int32_t *expert_ids = (int32_t *)malloc((size_t)(cap / block_m > 0 ? cap / block_m : 1) * sizeof(int32_t));
    uint16_t *C1 = (uint16_t *)calloc((size_t)(P > 0 ? P : 1) * 2 * I, sizeof(uint16_t));
    uint16_t *hb = (uint16_t *)calloc((size_t)(P > 0 ? P : 1) * I, sizeof(uint16_t));
    float *C2 = (float *)calloc((size_t)(P > 0 ? P : 1) * H, sizeof(float));
    int rc = ORC_ENOMEM;
    int32_t ntp = 0;
    if (!sorted_ids || !expert_ids || !C1 || !hb || !C2)
        goto done;
    rc = orc_moe_align(topk_ids, T, topk, E, block_m, sorted_ids, expert_ids, &ntp, cap);
    if (rc) goto done;
    rc = orc_moe_gemm(x, T, topk, codes13, scales13, E, 2 * I, H, sorted_ids, expert_ids, ntp,
                      block_m, P, C1, nthreads);
    if (rc) goto done;
    rc = orc_silu_mul(C1, topk_ids, P, E, I, hb, nthreads);
    if (rc) goto done;
    rc = orc_moe_gemm_f32(hb, P, 1, codes2, scales2, E, H, I, sorted_ids, expert_ids, ntp,
                          block_m, P, C2, nthreads);
    if (rc) goto done;
    rc = orc_combine_f32(C2, topk_ids, topk_w, T, topk, E, H, out, nthreads);
done:
    free(sorted_ids); free(expert_ids); free(C1); free(hb); free(C2);
    return rc;
}

/* The layer with binary64 sums at the plain layer's rounding points: gate_up
 * rounded to bf16 from its binary64 sum, SiLU*up exactly as in the plain layer
 * (binary32, rounded to bf16), the down projection's binary64 sums fed to the
 * binary64 weighted sum unrounded, the output rounded to bf16 once. */
int orc_moe_layer_f64sum(const uint16_t *x, const int32_t *topk_ids, const float *topk_w,
                         int T, int topk, int E, int H, int I,
                         const uint8_t *codes13, const uint16_t *scales13,
                         const uint8_t *codes2, const uint16_t *scales2,
                         int block_m, uint16_t *out, int nthreads)
{
    int64_t cap = orc_align_capacity(T, topk, E, block_m);
    if (cap < 0 || H <= 0 || I <= 0 || H % ORC_GROUP || I % ORC_GROUP)
        return ORC_EINVAL;
    int64_t P = (int64_t)T * topk;
    int32_t *sorted_ids = (int32_t *)malloc((size_t)(cap > 0 ? cap : 1) * sizeof(int32_t));
    int32_t *expert_ids = (int32_t *)malloc((size_t)(cap / block_m > 0 ? cap / block_m : 1) * sizeof(int32_t));
    uint16_t *C1 = (uint16_t *)calloc((size_t)(P > 0 ? P : 1) * 2 * I, sizeof(uint16_t));
    uint16_t *hb = (uint16_t *)calloc((size_t)(P > 0 ? P : 1) * I, sizeof(uint16_t));
    double *C2 = (double *)calloc((size_t)(P > 0 ? P : 1) * H, sizeof(double));
    int rc = ORC_ENOMEM;
    int32_t ntp = 0;
    if (!sorted_ids || !expert_ids || !C1 || !hb || !C2)
        goto done;
    rc = orc_moe_align(topk_ids, T, topk, E, block_m, sorted_ids, expert_ids, &ntp, cap);
    if (rc) goto done;
    rc = orc_moe_gemm_f64sum(x, T, topk, codes13, scales13, E, 2 * I, H, sorted_ids, expert_ids, ntp,
                             block_m, P, C1, nthreads);
    if (rc) goto done;
    rc = orc_silu_mul(C1, topk_ids, P, E, I, hb, nthreads);
    if (rc) goto done;
    rc = orc_moe_gemm_f64(hb, P, 1, codes2, scales2, E, H, I, sorted_ids, expert_ids, ntp,
                          block_m, P, C2, nthreads);
    if (rc) goto done;
    rc = orc_combine_f64(C2, topk_ids, topk_w, T, topk, E, H, out, nthreads);
done:
    free(sorted_ids); free(expert_ids); free(C1); free(hb); free(C2);
    return rc;
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
