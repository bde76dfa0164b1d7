// C ABI of the W4A16 MoE library (see include/chord.h): argument checks,
// schedule choice and launches.  No device memory is allocated here; every
// buffer, scratch included, belongs to the caller.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "../../include/chord.h"
#include "chord_common.cuh"
#include "chord_internal.h"

namespace chord {

// Sticky error word, one per device that loads the library.
__device__ int g_error_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_info_mu;
DeviceInfo g_info[kMaxDevices];
bool g_info_ok[kMaxDevices];

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

chord_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CHORD_OK : CHORD_ERR_CUDA; }

chord_opts opts_or_default(const chord_opts* o) {
    chord_opts d{};
    if (o) d = *o;
    return d;
}

// Blocks of at most this many rows (tok_e up to about 20) go to the
// warp-level MMA kernel, whose cost per stage does not depend on a tensor-core
// instruction's issue latency; larger blocks to the tcgen05 kernel, except
// for short K (few stages per item), where the tcgen05 kernel's fixed cost per
// item (pipeline fill, accumulator drain) dominates.
constexpr int kDecodeMaxBlockM = 32;
// opts.mixed = 0 (the library's choice) leaves the per-block split off.  The
// host cannot see the routing's skew without reading it back, and the split
// measured faster only where many experts are cold (GB300, 16384 tokens, 48
// of 384 experts: Zipf(2.0) routing 3606 -> 3373 us per layer; Zipf(1.2),
// three small blocks, 2359 -> 2427 us; uniform EP8 prefill 1034 -> 1048 us).
constexpr bool kMixedByDefault = false;
constexpr int kShortK = 512;
constexpr int kShortKMaxBlockM = 64;

int env_int(const char* name, int dflt) {
    const char* v = getenv(name);
    return v && *v ? atoi(v) : dflt;
}

// After a call in validate mode: wait for it and turn the error word into a status.
chord_status finish(const chord_opts& o, cudaStream_t stream) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return CHORD_ERR_CUDA;
    if (!o.validate) return CHORD_OK;
    int32_t code = 0;
    chord_status st = chord_get_device_error(stream, &code);
    if (st != CHORD_OK) return st;
    if (code == CHORD_DEV_TIMEOUT) return CHORD_ERR_TIMEOUT;
    return code ? CHORD_ERR_DEVICE_VALIDATION : CHORD_OK;
}
}  // namespace

const DeviceInfo& device_info() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) dev = 0;
    std::lock_guard<std::mutex> lk(g_info_mu);
    if (!g_info_ok[dev]) {
        DeviceInfo d;
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) == cudaSuccess) d.err = static_cast<int*>(p);
        if (d.sm_count <= 0) d.sm_count = 1;
        g_info[dev] = d;
        g_info_ok[dev] = d.err != nullptr;
    }
    return g_info[dev];
}

namespace {
struct LaunchFacts {
    int dev;
    const void* func;
    int threads;
    size_t smem, limit;
    int ctas;   // 0: only the limit was set
};
std::mutex g_facts_mu;
LaunchFacts g_facts[256];
int g_nfacts = 0;

// Entry for (device, func, threads, smem, limit), or nullptr; g_facts_mu held.
LaunchFacts* find_facts(int dev, const void* func, int threads, size_t smem, size_t limit) {
    for (int i = 0; i < g_nfacts; ++i) {
        LaunchFacts& f = g_facts[i];
        if (f.dev == dev && f.func == func && f.threads == threads && f.smem == smem && f.limit == limit) return &f;
    }
    return nullptr;
}
}  // namespace

cudaError_t ensure_smem_limit(const void* func, size_t smem_limit) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_facts_mu);
    if (find_facts(dev, func, 0, 0, smem_limit)) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit);
    if (e != cudaSuccess) return e;
    if (g_nfacts < 256) g_facts[g_nfacts++] = LaunchFacts{dev, func, 0, 0, smem_limit, 0};
    return cudaSuccess;
}

cudaError_t kernel_ctas_per_sm(const void* func, int threads, size_t smem, size_t smem_limit, int* ctas) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_facts_mu);
    if (const LaunchFacts* f = find_facts(dev, func, threads, smem, smem_limit)) {
        *ctas = f->ctas;
        return cudaSuccess;
    }
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_limit);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, func, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    if (g_nfacts < 256) g_facts[g_nfacts++] = LaunchFacts{dev, func, threads, smem, smem_limit, per_sm};
    *ctas = per_sm;
    return cudaSuccess;
}

}  // namespace chord

using namespace chord;

extern "C" {

int chord_version(void) { return 100; }

const char* chord_status_string(chord_status s) {
    switch (s) {
        case CHORD_OK: return "ok";
        case CHORD_ERR_INVALID_ARG: return "invalid argument";
        case CHORD_ERR_UNSUPPORTED: return "unsupported configuration";
        case CHORD_ERR_LAYOUT_MISMATCH: return "packed weight layout does not match the call";
        case CHORD_ERR_BUFFER_TOO_SMALL: return "buffer or workspace too small";
        case CHORD_ERR_CUDA: return "CUDA runtime error";
        case CHORD_ERR_DEVICE_VALIDATION: return "device-side validation failed";
        case CHORD_ERR_TIMEOUT: return "a bounded device wait timed out";
    }
    return "unknown status";
}

size_t chord_packed_weight_bytes(int E, int N, int K, int layout) {
    if (E < 0 || N <= 0 || K <= 0 || K % 64) return 0;
    const bool tile128 = layout == CHORD_LAYOUT_TCGEN05 || layout == CHORD_LAYOUT_GATE_UP_INTERLEAVED;
    if (!(layout == CHORD_LAYOUT_WARP_MMA && N % 16 == 0) && !(tile128 && N % 128 == 0)) return 0;
    return (size_t)kHeaderBytes + (size_t)E * (size_t)N * (size_t)K * 9u / 16u;
}

chord_status chord_pack_weights(const uint8_t* codes, const void* scales, int E, int N, int K, int group_size,
                                int layout, void* packed, size_t packed_bytes, void* stream) {
    if (group_size != kGroup) return CHORD_ERR_UNSUPPORTED;
    if (E < 0 || N <= 0 || K <= 0) return CHORD_ERR_INVALID_ARG;
    if (layout != CHORD_LAYOUT_WARP_MMA && layout != CHORD_LAYOUT_TCGEN05 && layout != CHORD_LAYOUT_GATE_UP_INTERLEAVED)
        return CHORD_ERR_INVALID_ARG;
    if (chord_packed_weight_bytes(E, N, K, layout) == 0) return CHORD_ERR_UNSUPPORTED;
    if (!packed || !aligned16(packed) || (E > 0 && (!codes || !scales))) return CHORD_ERR_INVALID_ARG;
    if (packed_bytes < chord_packed_weight_bytes(E, N, K, layout)) return CHORD_ERR_BUFFER_TOO_SMALL;
    const DeviceInfo& di = device_info();
    if (!di.err) return CHORD_ERR_CUDA;
    return cuda_status(launch_pack(codes, static_cast<const uint16_t*>(scales), E, N, K, layout,
                                   static_cast<uint8_t*>(packed), di.err, static_cast<cudaStream_t>(stream)));
}

int64_t chord_align_capacity(int T, int topk, int E, int block_m) {
    if (T < 0 || topk <= 0 || E <= 0 || block_m <= 0) return -1;
    const int64_t P = (int64_t)T * topk;
    const int64_t m = P < E ? P : E;
    const int64_t c = P + m * (block_m - 1);
    return (c + block_m - 1) / block_m * block_m;
}

size_t chord_align_workspace_bytes(int T, int topk, int E) {
    if (T < 0 || topk <= 0 || E <= 0) return 0;
    return (size_t)align_slices((int64_t)T * topk) * (size_t)E * sizeof(int32_t);
}

chord_status chord_moe_align(const int32_t* topk_ids, int T, int topk, int E, int block_m, int32_t* sorted_ids,
                             int32_t* expert_ids, int32_t* num_tokens_padded, int64_t capacity, void* workspace,
                             size_t workspace_bytes, const chord_opts* opts, void* stream) {
    if (T < 0 || topk <= 0 || E <= 0 || block_m <= 0) return CHORD_ERR_INVALID_ARG;
    if (E > 1024 || block_m > 256) return CHORD_ERR_UNSUPPORTED;
    if ((int64_t)T * topk >= INT32_MAX) return CHORD_ERR_UNSUPPORTED;
    const int64_t cap = chord_align_capacity(T, topk, E, block_m);
    if (capacity < cap) return CHORD_ERR_BUFFER_TOO_SMALL;
    if (capacity % block_m) return CHORD_ERR_INVALID_ARG;
    if (workspace_bytes < chord_align_workspace_bytes(T, topk, E)) return CHORD_ERR_BUFFER_TOO_SMALL;
    if (!num_tokens_padded || !workspace || (T > 0 && !topk_ids) || (capacity > 0 && (!sorted_ids || !expert_ids)))
        return CHORD_ERR_INVALID_ARG;
    const chord_opts o = opts_or_default(opts);
    const DeviceInfo& di = device_info();
    if (!di.err) return CHORD_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_align(topk_ids, (int64_t)T * topk, E, block_m, sorted_ids, expert_ids, num_tokens_padded,
                                 capacity, static_cast<int32_t*>(workspace), o.validate != 0, di.err, s);
    if (e != cudaSuccess) return CHORD_ERR_CUDA;
    return finish(o, s);
}

int chord_select_block_m(int T, int topk, int E_local, int E_global, int N, int K) {
    (void)N;
    (void)K;
    const int forced = env_int("CHORD_BLOCK_M", 0);
    if (forced > 0) return forced;
    const int eg = E_global > 0 ? E_global : (E_local > 0 ? E_local : 1);
    const double tok_e = (double)T * (double)(topk > 0 ? topk : 1) / (double)eg;
    // Rows per expert that a block should hold without splitting an expert in
    // two most of the time (every extra block of an expert re-streams and
    // re-dequantises that expert's weights): the mean plus three standard
    // deviations of a Poisson count, in steps of 16 (the MMA's N granularity),
    // at most 256 (the largest MMA N).  The kernels size each MMA to the rows a
    // block really holds, so a generous block costs only index padding.
    const double need = tok_e + 3.0 * sqrt(tok_e) + 1.0;
    if (need <= 8.0) return 8;
    // Blocks of up to 32 rows run on the warp-level kernel, which streams
    // weights faster than the tcgen05 kernel at these row counts (TP8 T=1024,
    // tok_e 21: 542 us per layer with 32-row blocks against 580 with 48): when
    // the mean plus two standard deviations still fits 32 rows, take 32 and let
    // the rare larger expert use a second block.
    if (need > 32.0 && tok_e + 2.0 * sqrt(tok_e) + 1.0 <= 32.0) return 32;
    int bm = (int)ceil(need / 16.0) * 16;
    if (bm > 256) bm = 256;
    return bm;
}

int chord_select_kernel(int block_m, int N, int K) {
    (void)N;
    const int forced = env_int("CHORD_KERNEL", 0);
    if (forced == CHORD_KERNEL_TCGEN05 || forced == CHORD_KERNEL_WARP_MMA) return forced;
    if (block_m <= kDecodeMaxBlockM || (K <= kShortK && block_m <= kShortKMaxBlockM)) return CHORD_KERNEL_WARP_MMA;
    return CHORD_KERNEL_TCGEN05;
}

}  // extern "C"

namespace {
// Split-K for the warp-level kernel.  Work units = items x K slices; a launch
// with fewer items than half of its resident CTAs (152 SMs x 3) leaves most
// SMs idle and each CTA streams a long K loop through a short pipeline, so the
// automatic choice cuts K into S slices until the units fill about one wave.
// Each nonempty align block holds at least one pair, so num_pairs x N / 128
// bounds the items from above without reading num_tokens_padded.
constexpr int64_t kSplitTargetUnits = 152 * 3;
constexpr int kSplitMax = 16;

int gemm_split(int64_t num_pairs, int N, int K, int block_m, const chord_opts& o) {
    const int kernel = o.kernel ? o.kernel : chord_select_kernel(block_m, N, K);
    if (kernel != CHORD_KERNEL_WARP_MMA || o.split_k == 1 || num_pairs <= 0 || N <= 0 || K <= 0) return 1;
    const int kstages = (K + 127) / 128;
    if (o.split_k > 1) return o.split_k < kstages ? o.split_k : kstages;
    if (o.split_k < 0) return 1;
    const int64_t items = num_pairs * (N / 128);
    if (items * 2 >= kSplitTargetUnits) return 1;
    int64_t S = items > 0 ? (kSplitTargetUnits + items - 1) / items : 1;
    if (S > kstages / 2) S = kstages / 2;
    if (S > kSplitMax) S = kSplitMax;
    return S < 2 ? 1 : (int)S;
}

size_t split_bytes(int S, int64_t num_pairs, int N) {
    return S > 1 ? (size_t)S * (size_t)num_pairs * (size_t)N * 4 : 0;
}

// tcgen05 tail split: at most one unit of 128 rows x tok_tile FP32 sums per
// CTA of the persistent grid (one CTA per SM for the configurations that use
// it; the launch turns the split off when the grid outgrows the workspace).
constexpr int64_t kTailSplitCtas = 152;

size_t tc_tail_bytes(int block_m) {
    const int64_t tok_tile = block_m < 16 ? 16 : (block_m + 15) / 16 * 16;
    return (size_t)kTailSplitCtas * 128 * (size_t)tok_tile * 4;
}

// Workspace of one GEMM call: the warp-level kernel's K-slice partial sums, or
// the tcgen05 kernel's split-tail partial sums.
size_t gemm_ws_bytes(int64_t num_pairs, int N, int K, int block_m, const chord_opts& o) {
    if (num_pairs <= 0 || N <= 0 || K <= 0 || block_m <= 0) return 0;
    const int kernel = o.kernel ? o.kernel : chord_select_kernel(block_m, N, K);
    if (kernel == CHORD_KERNEL_TCGEN05) return o.split_k == 1 || o.split_k < 0 ? 0 : tc_tail_bytes(block_m);
    return split_bytes(gemm_split(num_pairs, N, K, block_m, o), num_pairs, N);
}

// What one GEMM call launches, decided on the host from its arguments.
struct GemmPlan {
    chord_status status;
    int kernel;
    int S;        // K slices of the warp-level kernel
    bool tail;    // tcgen05 split tail (its reduction is a second launch)
    bool mixed;   // the small blocks on the warp-level kernel, launched first
};

GemmPlan plan_gemm(int64_t num_pairs, int N, int K, int block_m, bool ws_ok, size_t workspace_bytes,
                   const chord_opts& o) {
    GemmPlan p{CHORD_OK, o.kernel ? o.kernel : chord_select_kernel(block_m, N, K), 1, false, false};
    // Mixed regime: the small blocks of a tcgen05-regime call on the warp-level kernel.
    p.mixed = p.kernel == CHORD_KERNEL_TCGEN05 && block_m > CHORD_MIXED_SMALL_ROWS &&
              (o.mixed > 0 || (o.mixed == 0 && o.kernel == CHORD_KERNEL_AUTO && kMixedByDefault));
    // K slices: an explicit request needs its partial-sum workspace; the
    // automatic choice falls back to one slice when the caller gave none.
    p.S = gemm_split(num_pairs, N, K, block_m, o);
    if (p.S > 1 && (workspace_bytes < split_bytes(p.S, num_pairs, N) || !ws_ok)) {
        if (o.split_k > 1) {
            p.status = workspace_bytes < split_bytes(p.S, num_pairs, N) ? CHORD_ERR_BUFFER_TOO_SMALL
                                                                         : CHORD_ERR_INVALID_ARG;
            return p;
        }
        p.S = 1;
    }
    // tcgen05: the split tail, when the workspace holds its partial sums (one CTA per item only)
    const bool pairs = o.tc_pairs > 0 && N % 256 == 0;
    if (p.kernel == CHORD_KERNEL_TCGEN05 && o.split_k != 1 && !pairs) {
        const size_t need = tc_tail_bytes(block_m);
        if (ws_ok && workspace_bytes >= need)
            p.tail = true;
        else if (o.split_k > 1)
            p.status = workspace_bytes < need ? CHORD_ERR_BUFFER_TOO_SMALL : CHORD_ERR_INVALID_ARG;
    }
    return p;
}
}  // namespace

extern "C" {

int chord_gemm_launch_count(int64_t num_pairs, int N, int K, int block_m, size_t workspace_bytes,
                            const chord_opts* opts) {
    if (num_pairs <= 0 || N <= 0 || K <= 0 || block_m <= 0) return 0;
    const chord_opts o = opts_or_default(opts);
    const GemmPlan p = plan_gemm(num_pairs, N, K, block_m, workspace_bytes > 0, workspace_bytes, o);
    if (p.status != CHORD_OK) return 0;
    return 1 + (p.mixed ? 1 : 0) + (p.S > 1 ? 1 : 0) + (p.tail ? 1 : 0);
}

size_t chord_gemm_workspace_bytes(int64_t num_pairs, int N, int K, int block_m, const chord_opts* opts) {
    return gemm_ws_bytes(num_pairs, N, K, block_m, opts_or_default(opts));
}

}  // extern "C"

namespace {
// The fused combine's extra operands of a down-projection call (topk = 0: none).
struct CombineArgs {
    int topk = 0;
    const float* pair_w = nullptr;
    void* out = nullptr;
};

chord_status moe_gemm(const void* A, int64_t a_rows, int a_row_divisor, const void* packed, size_t packed_bytes,
                      int E, int N, int K, const int32_t* sorted_ids, const int32_t* expert_ids,
                      const int32_t* num_tokens_padded, int64_t capacity, int block_m, int64_t num_pairs, void* C,
                      void* workspace, size_t workspace_bytes, const chord_opts* opts, const CombineArgs& cmb,
                      void* stream) {
    if (E <= 0 || N <= 0 || K <= 0 || a_rows < 0 || a_row_divisor <= 0 || block_m <= 0 || capacity < 0 ||
        num_pairs < 0)
        return CHORD_ERR_INVALID_ARG;
    if (N % 128 || K % 64 || block_m % 8 || block_m > 256) return CHORD_ERR_UNSUPPORTED;
    if (num_pairs >= INT32_MAX) return CHORD_ERR_UNSUPPORTED;
    const chord_opts o = opts_or_default(opts);
    const int kernel = o.kernel ? o.kernel : chord_select_kernel(block_m, N, K);
    if (kernel != CHORD_KERNEL_TCGEN05 && kernel != CHORD_KERNEL_WARP_MMA) return CHORD_ERR_INVALID_ARG;
    if (packed_bytes != chord_packed_weight_bytes(E, N, K, CHORD_LAYOUT_TCGEN05)) return CHORD_ERR_LAYOUT_MISMATCH;
    if (!packed || !aligned16(packed) || !num_tokens_padded || (capacity > 0 && (!sorted_ids || !expert_ids)))
        return CHORD_ERR_INVALID_ARG;
    if (capacity % block_m) return CHORD_ERR_INVALID_ARG;
    if ((a_rows > 0 && (!A || !aligned16(A))) || (num_pairs > 0 && (!C || !aligned16(C))))
        return CHORD_ERR_INVALID_ARG;
    if (o.out_dtype != CHORD_DTYPE_BF16 && o.out_dtype != CHORD_DTYPE_F32) return CHORD_ERR_INVALID_ARG;
    if (o.epilogue != CHORD_EPILOGUE_NONE && o.epilogue != CHORD_EPILOGUE_SILU_MUL) return CHORD_ERR_INVALID_ARG;
    const bool silu = o.epilogue == CHORD_EPILOGUE_SILU_MUL;
    if (silu && o.out_dtype != CHORD_DTYPE_BF16) return CHORD_ERR_INVALID_ARG;
    if (o.split_k < 0) return CHORD_ERR_INVALID_ARG;
    if (o.mixed < -1 || o.mixed > 1 || o.tc_pairs < -1 || o.tc_pairs > 1) return CHORD_ERR_INVALID_ARG;
    const GemmPlan plan = plan_gemm(num_pairs, N, K, block_m, workspace && aligned16(workspace), workspace_bytes, o);
    if (plan.status != CHORD_OK) return plan.status;
    const int S = plan.S;
    const bool tail = plan.tail, mixed = plan.mixed;
    const DeviceInfo& di = device_info();
    if (!di.err) return CHORD_ERR_CUDA;
    if (capacity == 0 || num_pairs == 0) return CHORD_OK;
    GemmArgs g{};
    g.A = static_cast<const uint16_t*>(A);
    g.a_rows = a_rows;
    g.a_row_divisor = a_row_divisor;
    g.packed = static_cast<const uint8_t*>(packed);
    g.E = E;
    g.N = N;
    g.K = K;
    g.sorted_ids = sorted_ids;
    g.expert_ids = expert_ids;
    g.ntp = num_tokens_padded;
    g.capacity = capacity;
    g.block_m = block_m;
    g.num_pairs = num_pairs;
    g.id_limit = a_rows * (int64_t)a_row_divisor < num_pairs ? a_rows * (int64_t)a_row_divisor : num_pairs;
    g.C = C;
    g.out_f32 = o.out_dtype == CHORD_DTYPE_F32 ? 1 : 0;
    g.silu = silu ? 1 : 0;
    g.layout = silu ? CHORD_LAYOUT_GATE_UP_INTERLEAVED : CHORD_LAYOUT_TCGEN05;
    g.tc_pairs = o.tc_pairs > 0 ? 1 : 0;
    g.combine = cmb.topk > 0 ? 1 : 0;
    g.topk = cmb.topk;
    g.pair_w = cmb.pair_w;
    g.out = static_cast<uint16_t*>(cmb.out);
    g.err = di.err;
    g.ksplit = S;
    g.partial = (S > 1 || tail) ? static_cast<float*>(workspace) : nullptr;
    g.partial_bytes = workspace_bytes;
    g.tail_split = tail ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaSuccess;
    if (mixed) {
        GemmArgs gs = g;
        gs.block_filter = kBlocksSmall;
        gs.ksplit = 1;
        gs.partial = nullptr;
        gs.partial_bytes = 0;
        gs.tail_split = 0;
        e = launch_gemm_decode(gs, s);
        g.block_filter = kBlocksLarge;
    }
    if (e == cudaSuccess) e = kernel == CHORD_KERNEL_TCGEN05 ? launch_gemm_tc(g, s) : launch_gemm_decode(g, s);
    if (e == cudaSuccess && S > 1)
        e = launch_splitk_reduce(g.partial, S, g, s);
    if (e != cudaSuccess) return CHORD_ERR_CUDA;
    return finish(o, s);
}
}  // namespace

extern "C" {

chord_status chord_w4a16_moe_gemm(const void* A, int64_t a_rows, int a_row_divisor, const void* packed,
                                  size_t packed_bytes, int E, int N, int K, const int32_t* sorted_ids,
                                  const int32_t* expert_ids, const int32_t* num_tokens_padded, int64_t capacity,
                                  int block_m, int64_t num_pairs, void* C, void* workspace, size_t workspace_bytes,
                                  const chord_opts* opts, void* stream) {
    return moe_gemm(A, a_rows, a_row_divisor, packed, packed_bytes, E, N, K, sorted_ids, expert_ids,
                    num_tokens_padded, capacity, block_m, num_pairs, C, workspace, workspace_bytes, opts,
                    CombineArgs{}, stream);
}

chord_status chord_combine_plan(const int32_t* topk_ids, const float* topk_w, int T, int topk, int E, float* pair_w,
                                void* stream) {
    if (T < 0 || topk <= 0 || E <= 0) return CHORD_ERR_INVALID_ARG;
    if (topk > 32) return CHORD_ERR_UNSUPPORTED;
    if (T > 0 && (!topk_ids || !topk_w || !pair_w)) return CHORD_ERR_INVALID_ARG;
    return cuda_status(launch_combine_plan(topk_ids, topk_w, T, topk, E, pair_w, static_cast<cudaStream_t>(stream)));
}

chord_status chord_w4a16_moe_gemm_combine(const void* A, const void* packed, size_t packed_bytes, int E, int N, int K,
                                          const int32_t* sorted_ids, const int32_t* expert_ids,
                                          const int32_t* num_tokens_padded, int64_t capacity, int block_m, int T,
                                          int topk, const float* pair_w, float* C2, void* out, void* workspace,
                                          size_t workspace_bytes, const chord_opts* opts, void* stream) {
    if (T < 0 || topk <= 0) return CHORD_ERR_INVALID_ARG;
    if (topk > 32) return CHORD_ERR_UNSUPPORTED;
    chord_opts o = opts_or_default(opts);
    if (o.epilogue != CHORD_EPILOGUE_NONE) return CHORD_ERR_INVALID_ARG;
    if (T > 0 && (!pair_w || !out || !aligned16(out))) return CHORD_ERR_INVALID_ARG;
    o.out_dtype = CHORD_DTYPE_F32;
    const int64_t P = (int64_t)T * topk;
    CombineArgs cmb;
    cmb.topk = topk;
    cmb.pair_w = pair_w;
    cmb.out = out;
    return moe_gemm(A, P, 1, packed, packed_bytes, E, N, K, sorted_ids, expert_ids, num_tokens_padded, capacity,
                    block_m, P, C2, workspace, workspace_bytes, &o, cmb, stream);
}

chord_status chord_combine_finish(const float* C2, const int32_t* topk_ids, const float* topk_w, int T, int topk,
                                  int E, int H, void* out, void* stream) {
    if (T < 0 || topk <= 0 || E <= 0 || H <= 0) return CHORD_ERR_INVALID_ARG;
    if (topk > 32) return CHORD_ERR_UNSUPPORTED;
    if (H % 8) return CHORD_ERR_UNSUPPORTED;
    if (T > 0 && (!C2 || !topk_ids || !topk_w || !out || !aligned16(C2) || !aligned16(out)))
        return CHORD_ERR_INVALID_ARG;
    return cuda_status(launch_combine_finish(C2, topk_ids, topk_w, T, topk, E, H, static_cast<uint16_t*>(out),
                                             static_cast<cudaStream_t>(stream)));
}

chord_status chord_silu_mul(const void* C1, const int32_t* topk_ids, int64_t P, int E, int I, void* h, void* stream) {
    if (P < 0 || E <= 0 || I <= 0) return CHORD_ERR_INVALID_ARG;
    if (I % 8) return CHORD_ERR_UNSUPPORTED;
    if (P > 0 && (!C1 || !topk_ids || !h || !aligned16(C1) || !aligned16(h))) return CHORD_ERR_INVALID_ARG;
    return cuda_status(launch_silu_mul(static_cast<const uint16_t*>(C1), topk_ids, P, E, I, static_cast<uint16_t*>(h),
                                       static_cast<cudaStream_t>(stream)));
}

chord_status chord_moe_combine(const void* C2, int c2_dtype, const int32_t* topk_ids, const float* topk_w, int T,
                               int topk, int E, int H, void* out, void* stream) {
    if (T < 0 || topk <= 0 || E <= 0 || H <= 0) return CHORD_ERR_INVALID_ARG;
    if (c2_dtype != CHORD_DTYPE_BF16 && c2_dtype != CHORD_DTYPE_F32) return CHORD_ERR_INVALID_ARG;
    if (H % 8) return CHORD_ERR_UNSUPPORTED;
    if (T > 0 && (!C2 || !topk_ids || !topk_w || !out || !aligned16(C2) || !aligned16(out)))
        return CHORD_ERR_INVALID_ARG;
    return cuda_status(launch_combine(C2, c2_dtype == CHORD_DTYPE_F32, topk_ids, topk_w, T, topk, E, H,
                                      static_cast<uint16_t*>(out), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
struct LayerWs {
    size_t counts, sorted, experts, ntp, c1, h, c2, pair_w, split, total;
};

size_t up256(size_t x) { return (x + 255) & ~(size_t)255; }

bool layer_ws(int T, int topk, int E, int H, int I, int block_m, LayerWs* w) {
    const int64_t cap = chord_align_capacity(T, topk, E, block_m);
    if (cap < 0) return false;
    const size_t P = (size_t)T * (size_t)topk;
    size_t off = 0;
    w->counts = off;
    off = up256(off + chord_align_workspace_bytes(T, topk, E));
    w->sorted = off;
    off = up256(off + (size_t)cap * 4);
    w->experts = off;
    off = up256(off + (size_t)(cap / block_m) * 4);
    w->ntp = off;
    off = up256(off + 4);
    w->c1 = off;
    off = up256(off + P * 2 * (size_t)I * 2);
    w->h = off;
    off = up256(off + P * (size_t)I * 2);
    w->c2 = off;
    off = up256(off + P * (size_t)H * 4);
    w->pair_w = off;   // the fused combine's per-pair weights
    off = up256(off + P * 4);
    // FP32 partial sums of the K-sliced GEMMs (default options), shared by
    // the gate_up and the down projection, which run one after the other
    w->split = off;
    const chord_opts o = opts_or_default(nullptr);
    const size_t s13 = gemm_ws_bytes((int64_t)P, 2 * I, H, block_m, o);
    const size_t s2 = gemm_ws_bytes((int64_t)P, H, I, block_m, o);
    off = up256(off + (s13 > s2 ? s13 : s2));
    w->total = off;
    return true;
}
}  // namespace

extern "C" {

size_t chord_layer_workspace_bytes(int T, int topk, int E, int H, int I, int block_m) {
    if (T < 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return 0;
    if (block_m <= 0) block_m = chord_select_block_m(T, topk, E, E, 2 * I, H);
    LayerWs w;
    return layer_ws(T, topk, E, H, I, block_m, &w) ? w.total : 0;
}

chord_status chord_moe_layer(const void* x, const int32_t* topk_ids, const float* topk_w, int T, int topk, int E,
                             int E_global, int H, int I, const void* packed_w13, size_t w13_bytes,
                             const void* packed_w2, size_t w2_bytes, int block_m, void* workspace,
                             size_t workspace_bytes, void* out, const chord_opts* opts, void* stream) {
    if (T < 0 || topk <= 0 || E <= 0 || H <= 0 || I <= 0) return CHORD_ERR_INVALID_ARG;
    if (E_global <= 0) E_global = E;
    if (block_m <= 0) block_m = chord_select_block_m(T, topk, E, E_global, 2 * I, H);
    LayerWs w;
    if (!layer_ws(T, topk, E, H, I, block_m, &w)) return CHORD_ERR_INVALID_ARG;
    if (workspace_bytes < w.total) return CHORD_ERR_BUFFER_TOO_SMALL;
    if (!workspace || !aligned16(workspace)) return CHORD_ERR_INVALID_ARG;
    if (T == 0) return CHORD_OK;
    if (!x || !topk_ids || !topk_w || !out) return CHORD_ERR_INVALID_ARG;
    chord_opts o = opts_or_default(opts);
    const int validate = o.validate;
    o.validate = 0;  // validate once, at the end
    o.out_dtype = CHORD_DTYPE_BF16;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* counts = reinterpret_cast<int32_t*>(ws + w.counts);
    int32_t* sorted = reinterpret_cast<int32_t*>(ws + w.sorted);
    int32_t* experts = reinterpret_cast<int32_t*>(ws + w.experts);
    int32_t* ntp = reinterpret_cast<int32_t*>(ws + w.ntp);
    void* c1 = ws + w.c1;
    void* h = ws + w.h;
    void* c2 = ws + w.c2;
    void* split = ws + w.split;
    const size_t split_len = w.total - w.split;
    const int64_t P = (int64_t)T * topk;
    const int64_t cap = chord_align_capacity(T, topk, E, block_m);
    chord_status st;
    st = chord_moe_align(topk_ids, T, topk, E, block_m, sorted, experts, ntp, cap, counts,
                         chord_align_workspace_bytes(T, topk, E), &o, stream);
    if (st != CHORD_OK) return st;
    if (o.epilogue == CHORD_EPILOGUE_SILU_MUL) {
        // w13 in layout 3: SiLU * up in the gate_up GEMM's epilogue, h written directly
        st = chord_w4a16_moe_gemm(x, T, topk, packed_w13, w13_bytes, E, 2 * I, H, sorted, experts, ntp, cap, block_m,
                                  P, h, split, split_len, &o, stream);
        if (st != CHORD_OK) return st;
    } else {
        if (o.epilogue != CHORD_EPILOGUE_NONE) return CHORD_ERR_INVALID_ARG;
        st = chord_w4a16_moe_gemm(x, T, topk, packed_w13, w13_bytes, E, 2 * I, H, sorted, experts, ntp, cap, block_m,
                                  P, c1, split, split_len, &o, stream);
        if (st != CHORD_OK) return st;
        st = chord_silu_mul(c1, topk_ids, P, E, I, h, stream);
        if (st != CHORD_OK) return st;
    }
    chord_opts o_down = o;
    o_down.out_dtype = CHORD_DTYPE_F32;
    o_down.epilogue = CHORD_EPILOGUE_NONE;
    if (o.fuse_combine < -1 || o.fuse_combine > 1) return CHORD_ERR_INVALID_ARG;
    if (o.fuse_combine > 0 && topk <= 32) {
        // top-k combine fused into the down GEMM: tokens with one local pair are
        // written by its epilogue, the others summed by the finishing pass
        float* pair_w = reinterpret_cast<float*>(ws + w.pair_w);
        st = chord_combine_plan(topk_ids, topk_w, T, topk, E, pair_w, stream);
        if (st != CHORD_OK) return st;
        st = chord_w4a16_moe_gemm_combine(h, packed_w2, w2_bytes, E, H, I, sorted, experts, ntp, cap, block_m, T,
                                          topk, pair_w, static_cast<float*>(c2), out, split, split_len, &o_down,
                                          stream);
        if (st != CHORD_OK) return st;
        st = chord_combine_finish(static_cast<const float*>(c2), topk_ids, topk_w, T, topk, E, H, out, stream);
        if (st != CHORD_OK) return st;
    } else {
        st = chord_w4a16_moe_gemm(h, P, 1, packed_w2, w2_bytes, E, H, I, sorted, experts, ntp, cap, block_m, P, c2,
                                  split, split_len, &o_down, stream);
        if (st != CHORD_OK) return st;
        st = chord_moe_combine(c2, CHORD_DTYPE_F32, topk_ids, topk_w, T, topk, E, H, out, stream);
        if (st != CHORD_OK) return st;
    }
    o.validate = validate;
    return finish(o, static_cast<cudaStream_t>(stream));
}

// ---- the layer replayed from a CUDA graph (chord_moe_layer_cached)
}  // extern "C"

namespace {
// One recorded layer: the call's arguments (the graph reads the same buffers
// every replay) and the instantiated graph.  The key is compared as bytes, so
// it is zero-filled before its fields are set.
struct LayerKey {
    int dev;
    const void* x;
    const int32_t* topk_ids;
    const float* topk_w;
    int T, topk, E, E_global, H, I, block_m;
    const void* w13;
    size_t w13_bytes;
    const void* w2;
    size_t w2_bytes;
    void* workspace;
    size_t workspace_bytes;
    void* out;
    chord_opts opts;
};
struct LayerGraph {
    LayerKey key;
    cudaGraphExec_t exec;
    uint64_t last_use;
};
constexpr int kMaxLayerGraphs = 64;
std::mutex g_graph_mu;
LayerGraph g_graphs[kMaxLayerGraphs];
int g_ngraphs = 0;
uint64_t g_graph_clock = 0;
cudaStream_t g_capture_stream[kMaxDevices];
}  // namespace

extern "C" {

chord_status chord_moe_layer_cached(const void* x, const int32_t* topk_ids, const float* topk_w, int T, int topk,
                                    int E, int E_global, int H, int I, const void* packed_w13, size_t w13_bytes,
                                    const void* packed_w2, size_t w2_bytes, int block_m, void* workspace,
                                    size_t workspace_bytes, void* out, const chord_opts* opts, void* stream) {
    const chord_opts o = opts_or_default(opts);
    if (o.validate) return CHORD_ERR_UNSUPPORTED;   // validation synchronises, which a graph cannot record
    if (T == 0) return chord_moe_layer(x, topk_ids, topk_w, T, topk, E, E_global, H, I, packed_w13, w13_bytes,
                                       packed_w2, w2_bytes, block_m, workspace, workspace_bytes, out, &o, stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CHORD_ERR_CUDA;
    LayerKey key;
    memset(&key, 0, sizeof key);
    key.dev = dev;
    key.x = x;
    key.topk_ids = topk_ids;
    key.topk_w = topk_w;
    key.T = T;
    key.topk = topk;
    key.E = E;
    key.E_global = E_global;
    key.H = H;
    key.I = I;
    key.block_m = block_m;
    key.w13 = packed_w13;
    key.w13_bytes = w13_bytes;
    key.w2 = packed_w2;
    key.w2_bytes = w2_bytes;
    key.workspace = workspace;
    key.workspace_bytes = workspace_bytes;
    key.out = out;
    key.opts = o;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lk(g_graph_mu);
    for (int i = 0; i < g_ngraphs; ++i) {
        if (memcmp(&g_graphs[i].key, &key, sizeof key) == 0) {
            g_graphs[i].last_use = ++g_graph_clock;
            return cudaGraphLaunch(g_graphs[i].exec, s) == cudaSuccess ? CHORD_OK : CHORD_ERR_CUDA;
        }
    }
    // first call with these arguments: record the layer's launches on a
    // capture stream of this device, instantiate, keep
    if (!g_capture_stream[dev] && cudaStreamCreateWithFlags(&g_capture_stream[dev], cudaStreamNonBlocking) != cudaSuccess)
        return CHORD_ERR_CUDA;
    cudaStream_t cs = g_capture_stream[dev];
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return CHORD_ERR_CUDA;
    const chord_status st = chord_moe_layer(x, topk_ids, topk_w, T, topk, E, E_global, H, I, packed_w13, w13_bytes,
                                            packed_w2, w2_bytes, block_m, workspace, workspace_bytes, out, &o, cs);
    cudaGraph_t graph = nullptr;
    const cudaError_t ce = cudaStreamEndCapture(cs, &graph);
    if (st != CHORD_OK || ce != cudaSuccess || !graph) {
        if (graph) cudaGraphDestroy(graph);
        cudaGetLastError();
        return st != CHORD_OK ? st : CHORD_ERR_CUDA;
    }
    cudaGraphExec_t exec = nullptr;
    const cudaError_t ie = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (ie != cudaSuccess) return CHORD_ERR_CUDA;
    int slot = g_ngraphs;
    if (g_ngraphs == kMaxLayerGraphs) {   // full: the least recently used graph goes
        slot = 0;
        for (int i = 1; i < g_ngraphs; ++i)
            if (g_graphs[i].last_use < g_graphs[slot].last_use) slot = i;
        cudaGraphExecDestroy(g_graphs[slot].exec);
    } else {
        ++g_ngraphs;
    }
    g_graphs[slot].key = key;
    g_graphs[slot].exec = exec;
    g_graphs[slot].last_use = ++g_graph_clock;
    return cudaGraphLaunch(exec, s) == cudaSuccess ? CHORD_OK : CHORD_ERR_CUDA;
}

int chord_moe_layer_cache_clear(void) {
    std::lock_guard<std::mutex> lk(g_graph_mu);
    const int n = g_ngraphs;
    for (int i = 0; i < g_ngraphs; ++i) cudaGraphExecDestroy(g_graphs[i].exec);
    g_ngraphs = 0;
    return n;
}

// ---- grouped contracts: routing arrays built on the device, then the
// indexed GEMM with one row per pair (a_row_divisor = 1).
static size_t grouped_ws(int64_t cap, int block_m) {
    size_t off = up256((size_t)cap * 4);
    off = up256(off + (size_t)(cap / block_m) * 4);
    return up256(off + 4);
}

// Routing arrays plus, for blocks the tcgen05 kernel takes (more than 32
// rows), room for its split tail; a workspace with only the routing arrays
// runs the GEMM without the split.
static size_t grouped_ws_total(int64_t cap, int block_m) {
    return grouped_ws(cap, block_m) + (block_m > kDecodeMaxBlockM ? tc_tail_bytes(block_m) : 0);
}

static int masked_block_m(int expected_m, int N, int K) {
    return chord_select_block_m(expected_m, 1, 1, 1, N, K);
}

// Contiguous: block size from the rows per expert (padding included), like
// tok_e; capacity bounds sum_e ceil(count_e / bm) * bm.
static int contiguous_block_m(int64_t M, int E) {
    return chord_select_block_m((int)(M < INT32_MAX ? M : INT32_MAX), 1, E, E, 0, 0);
}
static int64_t contiguous_capacity(int64_t M, int E, int bm) { return ((M + bm - 1) / bm + E) * bm; }

constexpr int kGroupedMaxExperts = 4000;   // the index builder's per-expert tables fit in 48 KB of shared memory

size_t chord_grouped_contiguous_workspace_bytes(int64_t M, int E) {
    if (M < 0 || E <= 0 || E > kGroupedMaxExperts) return 0;
    const int bm = contiguous_block_m(M, E);
    return grouped_ws_total(contiguous_capacity(M, E, bm), bm);
}

chord_status chord_grouped_contiguous_gemm(const void* A, int64_t M, const int32_t* m_indices, const void* packed,
                                           size_t packed_bytes, int E, int N, int K, void* C, void* workspace,
                                           size_t workspace_bytes, const chord_opts* opts, void* stream) {
    if (M < 0 || E <= 0 || N <= 0 || K <= 0) return CHORD_ERR_INVALID_ARG;
    if (M >= INT32_MAX || E > kGroupedMaxExperts) return CHORD_ERR_UNSUPPORTED;
    const int bm = contiguous_block_m(M, E);
    const int64_t cap = contiguous_capacity(M, E, bm);
    if (workspace_bytes < grouped_ws(cap, bm)) return CHORD_ERR_BUFFER_TOO_SMALL;
    if (!workspace || !aligned16(workspace) || (M > 0 && !m_indices)) return CHORD_ERR_INVALID_ARG;
    const DeviceInfo& di = device_info();
    if (!di.err) return CHORD_ERR_CUDA;
    if (M == 0) return CHORD_OK;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* sorted = reinterpret_cast<int32_t*>(ws);
    int32_t* experts = reinterpret_cast<int32_t*>(ws + up256((size_t)cap * 4));
    int32_t* ntp = reinterpret_cast<int32_t*>(ws + up256(up256((size_t)cap * 4) + (size_t)(cap / bm) * 4));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_grouped_contiguous_index(m_indices, M, E, bm, sorted, experts, ntp, cap, di.err, s) != cudaSuccess)
        return CHORD_ERR_CUDA;
    const size_t idx = grouped_ws(cap, bm);
    return chord_w4a16_moe_gemm(A, M, 1, packed, packed_bytes, E, N, K, sorted, experts, ntp, cap, bm, M, C, ws + idx,
                                workspace_bytes - idx, opts, stream);
}

size_t chord_grouped_masked_workspace_bytes(int G, int max_m, int expected_m) {
    if (G <= 0 || G > kGroupedMaxExperts || max_m < 0 || expected_m <= 0) return 0;
    const int bm = masked_block_m(expected_m, 0, 0);
    return grouped_ws_total((int64_t)G * ((max_m + bm - 1) / bm) * bm, bm);
}

chord_status chord_grouped_masked_gemm(const void* A, int G, int max_m, const int32_t* masked_m, int expected_m,
                                       const void* packed, size_t packed_bytes, int N, int K, void* C,
                                       void* workspace, size_t workspace_bytes, const chord_opts* opts,
                                       void* stream) {
    if (G <= 0 || max_m < 0 || expected_m <= 0 || N <= 0 || K <= 0) return CHORD_ERR_INVALID_ARG;
    if (G > kGroupedMaxExperts || (int64_t)G * max_m >= INT32_MAX) return CHORD_ERR_UNSUPPORTED;
    const int bm = masked_block_m(expected_m, N, K);
    const int64_t cap = (int64_t)G * ((max_m + bm - 1) / bm) * bm;
    if (workspace_bytes < grouped_ws(cap, bm)) return CHORD_ERR_BUFFER_TOO_SMALL;
    if (!workspace || !aligned16(workspace) || !masked_m) return CHORD_ERR_INVALID_ARG;
    const DeviceInfo& di = device_info();
    if (!di.err) return CHORD_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    int32_t* sorted = reinterpret_cast<int32_t*>(ws);
    int32_t* experts = reinterpret_cast<int32_t*>(ws + up256((size_t)cap * 4));
    int32_t* ntp = reinterpret_cast<int32_t*>(ws + up256(up256((size_t)cap * 4) + (size_t)(cap / bm) * 4));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cap == 0) return CHORD_OK;
    if (launch_grouped_masked_index(masked_m, G, max_m, bm, sorted, experts, ntp, cap, di.err, s) != cudaSuccess)
        return CHORD_ERR_CUDA;
    const int64_t rows = (int64_t)G * max_m;
    const size_t idx = grouped_ws(cap, bm);
    return chord_w4a16_moe_gemm(A, rows, 1, packed, packed_bytes, G, N, K, sorted, experts, ntp, cap, bm, rows, C,
                                ws + idx, workspace_bytes - idx, opts, stream);
}

chord_status chord_selftest_wait_timeout(void* stream) {
    const DeviceInfo& di = device_info();
    if (!di.err) return CHORD_ERR_CUDA;
    return cuda_status(launch_wait_timeout_selftest(di.err, static_cast<cudaStream_t>(stream)));
}

chord_status chord_get_device_error(void* stream, int32_t* code) {
    if (!code) return CHORD_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return CHORD_ERR_CUDA;
    int32_t v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof v) != cudaSuccess) return CHORD_ERR_CUDA;
    const int32_t zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero) != cudaSuccess) return CHORD_ERR_CUDA;
    *code = v;
    return CHORD_OK;
}

}  // extern "C"
