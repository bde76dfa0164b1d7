/*
 * chord.h - C ABI of the GB300 (sm_103a) W4A16 INT4 mixture-of-experts library.
 *
 * The operation is the expert GEMM of a mixture-of-experts layer with BF16
 * activations and INT4 weights ("vLLM x Novita AI: Chord, a faster INT4 MoE
 * for Kimi K2.x"):
 *   - weights are unsigned 4-bit codes q (offset 8) with one BF16 scale s per
 *     group of 32 consecutive K elements; a weight's value is
 *     bf16_rne((q - 8) * s), subtract first, then scale (section "H200 and
 *     Blackwell indexed decode"; logical shapes codes [G, N, K] and scales
 *     [G, N, K/32] from the grouped operator example in section "Grouped SM90
 *     kernels");
 *   - routed rows reach the GEMM through vLLM's moe_align_block_size buffers
 *     sorted_ids / expert_ids / num_tokens_padded; activations are never
 *     padded, padding lives in the index arrays as sentinels (section "Grouped
 *     SM90 kernels", figure 3 "where padding lives"); the buffers are
 *     over-allocated so no routed count is read back to the host and every
 *     call can be captured in a CUDA graph (deployment notes);
 *   - accumulation is FP32 (the F16-accumulation option is not implemented,
 *     deployment notes), outputs are BF16.
 *
 * Conventions for every call:
 *   - All tensor arguments are DEVICE pointers owned by the caller; the
 *     library never allocates device memory.  Sizes are element counts unless
 *     named *_bytes.  Matrices are row-major and densely packed.
 *   - BF16 buffers are passed as void* holding IEEE bfloat16 bit patterns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call only enqueues work on it and returns without synchronising, except
 *     chord_get_device_error and calls made with opts->validate != 0.
 *   - Argument errors are reported synchronously through the return value,
 *     before anything is enqueued.  Unsupported configurations (a group size
 *     other than 32, N not a multiple of 16 or K not a multiple of 64) return
 *     CHORD_ERR_UNSUPPORTED; nothing ever falls back to another kernel.
 *   - Problems found on the device (an expert id or pair id out of range, a
 *     packed blob whose header does not match the call, a pipeline wait that
 *     ran out) set a sticky per-device error word and the affected work is
 *     skipped; read and clear it with chord_get_device_error.
 *   - Pointers passed as A, C, x, out and the packed blob must be 16-byte
 *     aligned.
 */
#ifndef CHORD_H
#define CHORD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum chord_status {
    CHORD_OK = 0,
    CHORD_ERR_INVALID_ARG = 1,       /* null pointer, negative size, misaligned pointer */
    CHORD_ERR_UNSUPPORTED = 2,       /* shape or option this library does not implement */
    CHORD_ERR_LAYOUT_MISMATCH = 3,   /* packed blob size does not match E, N, K */
    CHORD_ERR_BUFFER_TOO_SMALL = 4,  /* a capacity or workspace below the required size */
    CHORD_ERR_CUDA = 5,              /* a CUDA runtime call failed */
    CHORD_ERR_DEVICE_VALIDATION = 6, /* validate mode: the device found bad routing or a bad blob */
    CHORD_ERR_TIMEOUT = 7            /* validate mode: a bounded device wait gave up */
} chord_status;

/* Device error word values (chord_get_device_error). */
#define CHORD_DEV_OK 0
#define CHORD_DEV_BAD_EXPERT 1   /* topk_ids / expert_ids entry outside its range */
#define CHORD_DEV_BAD_ROW 2      /* sorted_ids entry neither a pair id nor the sentinel */
#define CHORD_DEV_BAD_HEADER 3   /* packed blob header does not describe (E, N, K) */
#define CHORD_DEV_TIMEOUT 4      /* a pipeline wait exceeded its bound */
#define CHORD_DEV_BAD_CODE 5     /* pack: a code above 15 */
#define CHORD_DEV_BAD_PADDED 6   /* num_tokens_padded above capacity or not a multiple of block_m */

/* GEMM kernel family, picked from rows per expert (the article's two
 * regimes, section "Indexed kernels"): both take the block's tokens as the
 * MMA's N side (the operand swap of the article's decode profile) and read the
 * same packed layout.  CHORD_KERNEL_AUTO picks by block size and K
 * (chord_select_kernel). */
typedef enum chord_kernel {
    CHORD_KERNEL_AUTO = 0,      /* chord_select_kernel(block_m) */
    CHORD_KERNEL_TCGEN05 = 1,   /* tcgen05.mma, dequantised A in tensor memory, FP32 accumulators
                                   in tensor memory (prefill regime) */
    CHORD_KERNEL_WARP_MMA = 2   /* warp-level mma.sync m16n8k16 with register dequantisation
                                   (decode regime) */
} chord_kernel;

/* Packed weight layouts (recorded in the blob's header, checked on the device).
 * Both kernels read CHORD_LAYOUT_TCGEN05, and CHORD_LAYOUT_GATE_UP_INTERLEAVED
 * for the fused SiLU*up epilogue; layout 1 is packed for tests of the header
 * check only and no kernel accepts it. */
#define CHORD_LAYOUT_WARP_MMA 1   /* 16 x 64 chunks in m16n8k16 A-fragment order, N % 16 == 0 */
#define CHORD_LAYOUT_TCGEN05 2    /* 128 x 64 chunks, one row per 16-byte group, N % 128 == 0 */
#define CHORD_LAYOUT_GATE_UP_INTERLEAVED 3
    /* layout 2 of a gate_up weight (N = 2I, gate rows 0..I-1, up rows I..2I-1)
       with its rows reordered so that each 16-row group holds gate rows
       8g..8g+7 and then their up rows I+8g..I+8g+7: a thread that holds rows r
       and r+8 of an MMA tile holds a gate value and its up value */

/* GEMM epilogue. */
typedef enum chord_epilogue {
    CHORD_EPILOGUE_NONE = 0,      /* C = the projection */
    CHORD_EPILOGUE_SILU_MUL = 1   /* gate_up only: C = h = SiLU(gate) * up (see chord_w4a16_moe_gemm) */
} chord_epilogue;

typedef enum chord_dtype {
    CHORD_DTYPE_BF16 = 0,
    CHORD_DTYPE_F32 = 1
} chord_dtype;

typedef struct chord_opts {
    int32_t kernel;      /* chord_kernel (the packed blobs must have its layout) */
    int32_t validate;    /* nonzero: synchronise after the call and turn a set device
                            error word into CHORD_ERR_DEVICE_VALIDATION / _TIMEOUT
                            ("trusted routing validation" of the deployment notes) */
    int32_t split_k;     /* K slices of the warp-level kernel: 0 = automatic, 1 = off,
                            > 1 = that many (capped at K / 128 rounded up); < 0 is
                            refused.  tcgen05 kernel: 1 = no split tail, otherwise
                            the tail splits when the workspace holds it (> 1: an
                            error when it does not). */
    int32_t out_dtype;   /* GEMM output: CHORD_DTYPE_BF16 (default) or CHORD_DTYPE_F32,
                            the FP32 sums unrounded (for a consumer that keeps FP32) */
    int32_t epilogue;    /* chord_epilogue (GEMM and layer) */
    int32_t mixed;       /* per-block regime in the tcgen05 regime (the article's rule that
                            an expert's row count tok_e picks its kernel, section
                            "Indexed kernels"), decided on the device from the align
                            output: blocks holding at most CHORD_MIXED_SMALL_ROWS valid
                            rows run on the warp-level kernel (launched first), the
                            others on the tcgen05 kernel, for calls in the tcgen05
                            regime with block_m > CHORD_MIXED_SMALL_ROWS.  1 = on (also
                            with the kernel forced to tcgen05); 0 = the library's
                            choice, currently off (it pays only when many experts are
                            cold, which the host cannot see without a readback);
                            -1 = off. */
    int32_t fuse_combine; /* chord_moe_layer: 1 = the top-k combine fused into the down
                             GEMM (chord_combine_plan, chord_w4a16_moe_gemm_combine,
                             chord_combine_finish; topk <= 32); 0 (the library's
                             choice, measured faster on GB300) or -1 = the separate
                             chord_moe_combine pass.  The result is the same bit for
                             bit. */
    int32_t tc_pairs;    /* tcgen05 kernel: 1 = clusters of two CTAs on neighbouring SMs
                            computing M = 256 items with tcgen05 cta_group::2 (each CTA
                            dequantises its 128 weight rows into its own tensor memory and
                            gathers half of the block's tokens; N % 256 == 0, no split
                            tail); 0 (the library's choice) or -1 = one CTA per item.
                            Same results up to FP32 summation order. */
} chord_opts;

/* Blocks with at most this many valid rows count as small for opts.mixed. */
#define CHORD_MIXED_SMALL_ROWS 32

/* Library version (major * 10000 + minor * 100 + patch). */
int chord_version(void);

/* Human-readable name of a status. Never NULL. */
const char *chord_status_string(chord_status status);

/* ---------------------------------------------------------------- packing */

/* Bytes of the packed blob for E experts of an N x K weight in `layout`: a
 * 256-byte header followed by E * N * K * 9 / 16 bytes (4-bit codes plus one
 * BF16 scale per 32 codes).  Returns 0 when K % 64 is nonzero, N is not a
 * multiple of 16 (layout 1) or 128 (layout 2), a size is not positive or the
 * layout is unknown.  The byte layouts are the ones written out in the
 * library's packer (and in its CPU oracle): layout 1 places each 16 x 16 block
 * of codes so that one 32-bit load per lane yields an m16n8k16 A fragment;
 * layout 2 gives each thread of a 128-row tile its row's 32 consecutive codes
 * in one 16-byte load. */
size_t chord_packed_weight_bytes(int E, int N, int K, int layout);

/* Offline packing of canonical weights into an sm_103a layout (the article's
 * pack step, section "Grouped SM90 kernels": weights are prepared once at load
 * time, the mode is recorded in the prepared weight and checked when it is
 * used; a kernel given a blob of another layout refuses it on the device with
 * CHORD_DEV_BAD_HEADER).
 *   codes   device uint8 [E, N, K], each 0..15 (uint4, offset 8)
 *   scales  device bf16 [E, N, K / group_size]
 *   layout  CHORD_LAYOUT_TCGEN05 (default kernel) or CHORD_LAYOUT_WARP_MMA
 *   packed  device output of packed_bytes >= chord_packed_weight_bytes(E, N, K, layout)
 * group_size must be 32.  A code above 15 sets CHORD_DEV_BAD_CODE.
 * The header (little-endian 32-bit words) holds the magic "CHRD", version 1,
 * the layout, the group size, E, N, K, then in word 7 a 1 when every scale is
 * a positive normal bf16 below 0.5 (else 0), then the 64-bit expert stride
 * N * K * 9 / 16 and data offset 256.  Word 7 changes no result: with it set,
 * both GEMM kernels form each bf16((q - 8) * s) with one FMA per pair instead
 * of a subtract and a multiply (the same value, bit for bit). */
chord_status chord_pack_weights(const uint8_t *codes, const void *scales, int E, int N, int K,
                                int group_size, int layout, void *packed, size_t packed_bytes,
                                void *stream);

/* ---------------------------------------------------------------- routing */

/* Length of sorted_ids for moe_align_block_size: round_up(P + min(E, P) *
 * (block_m - 1), block_m) with P = T * topk; expert_ids has capacity / block_m
 * entries.  Returns -1 on bad arguments. */
int64_t chord_align_capacity(int T, int topk, int E, int block_m);

/* Scratch bytes chord_moe_align needs (per-slice expert histograms). */
size_t chord_align_workspace_bytes(int T, int topk, int E);

/* moe_align_block_size (the indexed routing contract of the article's
 * indexed family, section "Two kernel families", and figure 3):
 *   topk_ids  device int32 [T, topk]; entry e in [0, E) routes pair
 *             p = t * topk + k to local expert e; -1 marks an expert that
 *             lives on another GPU (dropped here, and in the combine).
 *   sorted_ids  device int32 [capacity]: for e = 0..E-1 the pair ids routed
 *             to e in ascending order, padded with the sentinel T * topk to a
 *             multiple of block_m; an expert with no pair gets no block;
 *             entries past num_tokens_padded hold the sentinel.
 *   expert_ids  device int32 [capacity / block_m]: expert of each block, -1
 *             past num_tokens_padded / block_m.
 *   num_tokens_padded  device int32 [1].
 * The result is unique (bit-for-bit deterministic).  1 <= block_m <= 256,
 * E <= 1024.  With opts->validate, an id outside [-1, E) is reported; without
 * it such ids are dropped like -1. */
chord_status chord_moe_align(const int32_t *topk_ids, int T, int topk, int E, int block_m,
                             int32_t *sorted_ids, int32_t *expert_ids,
                             int32_t *num_tokens_padded, int64_t capacity,
                             void *workspace, size_t workspace_bytes,
                             const chord_opts *opts, void *stream);

/* moe_align_block_size for callers that cannot allocate device memory.  The
 * article has no counterpart to this entry point; it exists for callers that
 * cannot hand the library a scratch buffer: code running while a CUDA graph is
 * captured in a mode that forbids allocation, inference-engine plugins limited
 * to the buffers the engine gives them, and serving loops that avoid
 * cudaMalloc / cudaFree because those synchronise the device.
 *
 * Same arguments, results and errors as chord_moe_align, without the
 * workspace: the per-slice histograms live in a fixed array of
 * CHORD_NOALLOC_ALIGN_SCRATCH_ENTRIES int32 (256 KiB) in the library's device
 * memory, which every GPU that loads the library holds until the process
 * exits.  The call needs ceil(T * topk / 4096) * E entries (at least E) and
 * returns CHORD_ERR_BUFFER_TOO_SMALL above the limit (for example E = 384
 * allows T * topk up to 696,320 pairs; E = 1024 up to 262,144).  It allocates
 * nothing.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current); make that first call before any
 *     stream capture.  The address is kept for the life of the process, so a
 *     cudaDeviceReset after the first call on that device is not supported
 *     (the library's module, and the array with it, is reloaded at a new
 *     address).
 *   - All calls on a device share the one array.  Calls whose work overlaps
 *     on the GPU (on different streams, or from several threads) race on it
 *     and may produce wrong routing; serialise them.
 *   - Each call overwrites every scratch entry it reads, so no state from an
 *     earlier call leaks into its result. */
#define CHORD_NOALLOC_ALIGN_SCRATCH_ENTRIES 65536
chord_status chord_moe_align_noalloc(const int32_t *topk_ids, int T, int topk, int E, int block_m,
                                     int32_t *sorted_ids, int32_t *expert_ids,
                                     int32_t *num_tokens_padded, int64_t capacity,
                                     const chord_opts *opts, void *stream);

/* Host-side block size choice from tokens per expert (the article's tok_e =
 * routed rows / experts rule, section "Indexed kernels"): tok_e = T * topk /
 * E_global is the expected number of rows per local expert, known without
 * reading anything back.  The block holds tok_e + 3 sqrt(tok_e) + 1 rows (a
 * Poisson count's mean plus three standard deviations) rounded up to 16, 8 when
 * that is at most 8, at most 256; 32 when that exceeds 32 but the mean plus two
 * standard deviations fits 32 (the warp-level kernel's largest block).
 * CHORD_BLOCK_M (environment) overrides.  Always returns a valid block_m. */
int chord_select_block_m(int T, int topk, int E_local, int E_global, int N, int K);

/* The kernel CHORD_KERNEL_AUTO runs for a GEMM of blocks of block_m rows and
 * an [N, K] weight: CHORD_KERNEL_WARP_MMA for decode blocks (block_m <= 32)
 * and for short K (K <= 512 with block_m <= 64, where the tcgen05 kernel's
 * fixed cost per block and N tile dominates), else CHORD_KERNEL_TCGEN05.
 * The environment variable CHORD_KERNEL (1 or 2), when set, overrides the
 * choice for every call whose opts leave the kernel at AUTO. */
int chord_select_kernel(int block_m, int N, int K);

/* ------------------------------------------------------------------- GEMM */

/* Kernel launches one chord_w4a16_moe_gemm call with these arguments makes,
 * from host arithmetic only (the same decisions the call takes, with a
 * 16-byte aligned workspace of workspace_bytes): the GEMM kernel, plus the
 * warp-level launch of the mixed regime (opts->mixed), plus the reduction of
 * its K slices or of the tcgen05 split tail when the workspace holds them.
 * 0 when the call would do nothing or be refused. */
int chord_gemm_launch_count(int64_t num_pairs, int N, int K, int block_m, size_t workspace_bytes,
                            const chord_opts *opts);

/* Scratch bytes chord_w4a16_moe_gemm needs for the given call shape.  Pure
 * host arithmetic (no device query).
 * Warp-level kernel: the FP32 partial sums of its K slices, S * num_pairs * N
 * * 4 bytes, 0 when S = 1.  The automatic S (opts->split_k = 0):
 * items = num_pairs * N / 128 bounds the launch's (align block, 128-row tile)
 * work items from above; when 2 * items < 456 (152 SMs x 3 resident CTAs)
 * S = min(ceil(456 / items), 16, ceil(K / 128) / 2), else 1.
 * tcgen05 kernel: 152 * 128 * tok_tile * 4 bytes (tok_tile = block_m rounded
 * up to 16), 0 with opts->split_k = 1.  The kernel runs its items on one
 * persistent CTA per SM; the items of the last partial wave (known only on
 * the device) are cut into S = min(CTAs / tail items, 16, K stages / MMA
 * issuers) K slices whose FP32 sums a second launch adds in order. */
size_t chord_gemm_workspace_bytes(int64_t num_pairs, int N, int K, int block_m,
                                  const chord_opts *opts);

/* Indexed W4A16 grouped GEMM, one projection (gate_up or down) -- the
 * article's indexed MoE GEMM ("Indexed kernels"; vLLM's moe_align_block_size
 * routing arrays):
 *   C[p, n] = bf16_rne( sum_k A[p / a_row_divisor, k] * w[e, n, k] )
 * for every block b < num_tokens_padded / block_m, e = expert_ids[b], and every
 * pair id p != num_pairs in sorted_ids[b * block_m .. + block_m); w is the
 * dequantised weight bf16_rne((q - 8) * s); the sum is FP32.
 *   A        device bf16 [a_rows, K]; a_row_divisor = topk when A has one row
 *            per token (gate_up), 1 when it has one row per pair (down).
 *   packed   blob from chord_pack_weights for (E, N, K) in CHORD_LAYOUT_TCGEN05.
 *   C        device bf16 [num_pairs, N] (float [num_pairs, N] with
 *            opts->out_dtype = CHORD_DTYPE_F32, the sum left unrounded);
 *            rows no block names are not written.
 * With opts->epilogue = CHORD_EPILOGUE_SILU_MUL (gate_up, SiLU*up fused):
 *   packed   in CHORD_LAYOUT_GATE_UP_INTERLEAVED, N = 2I;
 *   C        device bf16 [num_pairs, I]: h[p, j] = bf16_rne( g / (1 + exp(-g)) * u )
 *            with g, u the bf16-rounded gate and up sums of column j — the
 *            values this call without the epilogue followed by chord_silu_mul
 *            gives; out_dtype must be CHORD_DTYPE_BF16.
 *   capacity length of sorted_ids (expert_ids has capacity / block_m entries).
 * block_m must equal the value given to chord_moe_align, be a multiple of 8 and
 * at most 256; N % 128 == 0, K % 64 == 0.
 *   workspace  device, 16-byte aligned, >= chord_gemm_workspace_bytes(...) for
 *            K slices (warp-level) or the split tail (tcgen05; the same in-order
 *            reduction, results deterministic).  With S > 1 slices, slice s sums K stages
 *            [s * ks / S, (s + 1) * ks / S) (ks = ceil(K / 128)) into FP32
 *            partials, and a second launch adds slices 0 .. S-1 in order (FP32)
 *            and applies the output type or the SiLU * up epilogue; results
 *            are deterministic but differ from S = 1 by FP32 summation order.
 *            An automatic split with too small a workspace runs unsplit; an
 *            explicit one returns CHORD_ERR_BUFFER_TOO_SMALL. */
chord_status chord_w4a16_moe_gemm(const void *A, int64_t a_rows, int a_row_divisor,
                                  const void *packed, size_t packed_bytes, int E, int N, int K,
                                  const int32_t *sorted_ids, const int32_t *expert_ids,
                                  const int32_t *num_tokens_padded, int64_t capacity,
                                  int block_m, int64_t num_pairs, void *C,
                                  void *workspace, size_t workspace_bytes,
                                  const chord_opts *opts, void *stream);

/* --------------------------------------------------------- grouped GEMMs */

/* The article's two grouped contracts ("Grouped SM90 kernels"), served by the
 * same kernels through routing arrays built on the device (one row per pair).
 * Weights are packed as for chord_w4a16_moe_gemm (CHORD_LAYOUT_TCGEN05); the
 * epilogue, out_dtype and kernel options apply as there.  The workspace sizes
 * below hold the routing arrays (sorted ids, expert ids, padded count, each
 * 256-byte aligned) and, when the block size exceeds 32 rows (the tcgen05
 * kernel), the GEMM's split-tail partial sums (152 * 128 * tok_tile * 4
 * bytes); a workspace holding only the routing arrays is accepted and runs the
 * GEMM without the split tail.
 *
 * Contiguous (prefill): A [M, K] holds each expert's rows contiguously (the
 * article pads each expert's segment to a multiple of 128 rows); m_indices[m]
 * (device int32 [M]) is row m's expert, -1 on padding rows.
 *   C[m, n] = bf16_rne( sum_k A[m, k] * w[m_indices[m], n, k] )  for m_indices[m] >= 0
 * into C [M, N] (or [M, N/2] with the SiLU * up epilogue); padding rows are not
 * written.  An expert whose rows are not one contiguous run sets
 * CHORD_DEV_BAD_ROW, an id outside [-1, E) CHORD_DEV_BAD_EXPERT.  The block
 * size follows M / E as tok_e does.  E <= 4000.
 * workspace >= chord_grouped_contiguous_workspace_bytes(M, E). */
size_t chord_grouped_contiguous_workspace_bytes(int64_t M, int E);
chord_status chord_grouped_contiguous_gemm(const void *A, int64_t M, const int32_t *m_indices,
                                           const void *packed, size_t packed_bytes, int E, int N, int K,
                                           void *C, void *workspace, size_t workspace_bytes,
                                           const chord_opts *opts, void *stream);

/* Masked (decode): A [G, max_m, K] gives expert g a budget of max_m rows, of
 * which the first masked_m[g] (device int32 [G]) are valid; C is flat
 * [G * max_m, N] (or [G * max_m, N/2] with the SiLU * up epilogue):
 *   C[g * max_m + r, n] = bf16_rne( sum_k A[g, r, k] * w[g, n, k] )  for r < masked_m[g]
 * rows past a group's count are not written.  expected_m (> 0, a host value)
 * is the typical count; it picks the block size as tok_e does for the indexed
 * contract.  A count outside [0, max_m] sets CHORD_DEV_BAD_ROW (and is clamped).
 * G <= 4000.  workspace >= chord_grouped_masked_workspace_bytes(G, max_m, expected_m). */
size_t chord_grouped_masked_workspace_bytes(int G, int max_m, int expected_m);
chord_status chord_grouped_masked_gemm(const void *A, int G, int max_m, const int32_t *masked_m, int expected_m,
                                       const void *packed, size_t packed_bytes, int N, int K, void *C,
                                       void *workspace, size_t workspace_bytes, const chord_opts *opts,
                                       void *stream);

/* ------------------------------------------------------------- epilogues */

/* SiLU * up on the gate_up output:
 *   h[p, j] = bf16_rne( g / (1 + exp(-g)) * u ),  g = C1[p, j], u = C1[p, I + j]
 * (FP32 math), for every pair p whose topk_ids entry is a local expert.
 *   C1  device bf16 [P, 2 * I] (gate in columns 0..I-1, up in I..2I-1)
 *   h   device bf16 [P, I];  P = T * topk; I % 8 == 0. */
chord_status chord_silu_mul(const void *C1, const int32_t *topk_ids, int64_t P, int E, int I,
                            void *h, void *stream);

/* Top-k weighted combine (gather of each token's pair rows, weighted sum):
 *   out[t, n] = bf16_rne( sum over k ascending with topk_ids[t, k] in [0, E) of
 *                         topk_w[t, k] * C2[t * topk + k, n] ),  FP32, from +0,
 *               each product and each sum rounded separately (no fused multiply-add)
 *   C2 device [T * topk, H] of c2_dtype (CHORD_DTYPE_BF16 or CHORD_DTYPE_F32),
 *   topk_w device float [T, topk], out bf16 [T, H];
 * tokens with no local pair get +0.  H % 8 == 0. */
chord_status chord_moe_combine(const void *C2, int c2_dtype, const int32_t *topk_ids,
                               const float *topk_w, int T, int topk, int E, int H, void *out,
                               void *stream);

/* The top-k combine fused into the down GEMM (a scatter epilogue that applies
 * the top-k weights): the same out as chord_moe_combine of the down
 * GEMM's FP32 output, bit for bit, in three calls.  A token with exactly one
 * local pair gets its output straight from the GEMM's epilogue,
 * bf16(0 + w * sum), which is the weighted sum over that one pair; the FP32
 * rows of the other local pairs go to C2 and chord_combine_finish adds them
 * in ascending k as the combine does.  No atomics, so the result does not
 * depend on the order in which blocks finish.  topk <= 32.
 *
 * chord_combine_plan: pair_w device float [T * topk] (caller's scratch):
 *   pair_w[p] = topk_w[p] for the local pair of a token with one local pair,
 *   NaN for the local pairs of tokens with several; other entries untouched. */
chord_status chord_combine_plan(const int32_t *topk_ids, const float *topk_w, int T, int topk, int E,
                                float *pair_w, void *stream);

/* The down projection with the fused combine: chord_w4a16_moe_gemm with one A
 * row per pair (a_rows = num_pairs = T * topk, a_row_divisor = 1), FP32 sums,
 * opts->epilogue = CHORD_EPILOGUE_NONE (opts->out_dtype is ignored), and the
 * plan's pair_w: rows of pairs whose pair_w is a number are written to
 *   out[p / topk, n] = bf16_rne( 0 + pair_w[p] * sum )   (out bf16 [T, N])
 * and the others' FP32 sums to C2 [T * topk, N].  Same workspace, kernels,
 * splits, status codes and device errors as chord_w4a16_moe_gemm. */
chord_status chord_w4a16_moe_gemm_combine(const void *A, const void *packed, size_t packed_bytes, int E, int N,
                                          int K, const int32_t *sorted_ids, const int32_t *expert_ids,
                                          const int32_t *num_tokens_padded, int64_t capacity, int block_m, int T,
                                          int topk, const float *pair_w, float *C2, void *out, void *workspace,
                                          size_t workspace_bytes, const chord_opts *opts, void *stream);

/* Finishing pass of the fused combine: for every token with several local
 * pairs (or one whose weight is not a number),
 *   out[t, n] = bf16_rne( sum over local k ascending of topk_w[t, k] * C2[t * topk + k, n] )
 * (FP32 from +0, products and sums rounded separately); +0 for tokens with no
 * local pair; tokens with one local pair are left to the GEMM.  C2 device
 * float [T * topk, H], out bf16 [T, H], H % 8 == 0, topk <= 32. */
chord_status chord_combine_finish(const float *C2, const int32_t *topk_ids, const float *topk_w, int T, int topk,
                                  int E, int H, void *out, void *stream);

/* ------------------------------------------------------------------ layer */

/* Scratch bytes chord_moe_layer needs for this shape and block_m (0 = the
 * block size chord_select_block_m picks with E_global = E): the routing
 * arrays, the gate_up output, h, the down projection's FP32 rows, the fused
 * combine's per-pair weights (T * topk floats), and the larger of the two
 * GEMMs' automatic K-slice partial sums (an explicit
 * opts->split_k larger than that makes the layer call return
 * CHORD_ERR_BUFFER_TOO_SMALL). */
size_t chord_layer_workspace_bytes(int T, int topk, int E, int H, int I, int block_m);

/* One MoE expert layer on this GPU's E local experts:
 *   align -> gate_up GEMM (x rows gathered by pair id / topk) -> SiLU * up
 *   -> down GEMM -> top-k weighted combine, BF16 out [T, H].
 * The gate_up result and SiLU * up are rounded to BF16 (the GEMM output type
 * and the BF16 activation operand of the down GEMM); the down projection's
 * FP32 sums enter the weighted top-k sum unrounded and the output is rounded
 * to BF16 once.
 *   x          device bf16 [T, H]
 *   topk_ids   device int32 [T, topk] (local id or -1), topk_w device float [T, topk]
 *   packed_w13 blob for (E, 2 * I, H): rows 0..I-1 gate, I..2I-1 up, in
 *              CHORD_LAYOUT_TCGEN05, or in CHORD_LAYOUT_GATE_UP_INTERLEAVED with
 *              opts->epilogue = CHORD_EPILOGUE_SILU_MUL (SiLU * up then runs in
 *              the gate_up GEMM's epilogue, same results, one launch and the
 *              [T * topk, 2I] intermediate fewer)
 *   packed_w2  blob for (E, H, I) in CHORD_LAYOUT_TCGEN05
 *   E_global   number of experts the router chooses from (for tok_e)
 *   block_m    0 = chord_select_block_m(T, topk, E, E_global, 2 * I, H)
 *   workspace  >= chord_layer_workspace_bytes(T, topk, E, H, I, block_m) bytes
 * Tokens with no local pair get +0 (this GPU's partial sum of the layer). */
chord_status chord_moe_layer(const void *x, const int32_t *topk_ids, const float *topk_w,
                             int T, int topk, int E, int E_global, int H, int I,
                             const void *packed_w13, size_t w13_bytes,
                             const void *packed_w2, size_t w2_bytes, int block_m,
                             void *workspace, size_t workspace_bytes, void *out,
                             const chord_opts *opts, void *stream);

/* chord_moe_layer with its launches recorded once into a CUDA graph and
 * replayed: the host cost of a call becomes a lookup and one graph launch
 * (the article memoises its kernel resolution to remove host overhead from
 * small decode calls, section "Grouped SM90 kernels"; this removes the
 * per-kernel launch calls as well).  Same arguments, results and status codes
 * as chord_moe_layer, except:
 *   - opts->validate must be 0 (CHORD_ERR_UNSUPPORTED otherwise: validation
 *     synchronises, which a graph cannot record);
 *   - the first call with a given set of arguments (every pointer, size and
 *     option, on the current device) records the layer on a capture stream of
 *     the library and instantiates it: that call costs a capture, must not be
 *     made while the calling thread is capturing a stream itself, and leaves
 *     the graph cached; later calls with the same arguments replay it on
 *     `stream`, reading the buffers' current contents;
 *   - the library keeps at most 64 graphs (the least recently used is dropped)
 *     until chord_moe_layer_cache_clear.
 * Thread-safe; calls that overlap on the GPU race on the workspace as with
 * chord_moe_layer. */
chord_status chord_moe_layer_cached(const void *x, const int32_t *topk_ids, const float *topk_w,
                                    int T, int topk, int E, int E_global, int H, int I,
                                    const void *packed_w13, size_t w13_bytes,
                                    const void *packed_w2, size_t w2_bytes, int block_m,
                                    void *workspace, size_t workspace_bytes, void *out,
                                    const chord_opts *opts, void *stream);

/* Destroys every graph chord_moe_layer_cached holds; returns how many. */
int chord_moe_layer_cache_clear(void);

/* ------------------------------------------------------------------ errors */

/* Synchronises `stream`, returns the current device's sticky error word in
 * *code (CHORD_DEV_*) and clears it. */
chord_status chord_get_device_error(void *stream, int32_t *code);

/* Self-test of the device-side failure detection (no counterpart in the
 * article): launches one thread that waits, through the same bounded wait
 * every GEMM pipeline uses, on an mbarrier that nothing arrives on.  After the
 * bound (about 2 s) it sets CHORD_DEV_TIMEOUT in the device error word and
 * returns; the context stays usable.  A later chord_get_device_error reads the
 * code, and a call with opts->validate != 0 returns CHORD_ERR_TIMEOUT.
 * Asynchronous on `stream`; returns CHORD_ERR_CUDA if the launch fails. */
chord_status chord_selftest_wait_timeout(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* CHORD_H */
