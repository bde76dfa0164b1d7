"""CPU-side checks of the C ABI: the library builds for sm_103a, loads, exports
every function include/chord.h declares, and its host-only logic (sizes,
capacities, block size choice, argument checks that return before any CUDA
call) behaves as documented.  No GPU is touched."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

import w4a16_int4_mixture_moe_gb300 as chord

HEADER = os.path.join(ROOT, "include", "chord.h")


@pytest.fixture(scope="module")
def lib():
    chord.build()
    return chord.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(chord_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ["chord_pack_weights", "chord_moe_align", "chord_w4a16_moe_gemm", "chord_moe_layer"]:
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
        assert n in chord._SIGS, f"binding lacks {n}"


def test_sizes_and_capacity(lib):
    for layout in (1, 2, 3):
        assert chord.chord_packed_weight_bytes(48, 4096, 7168, layout) == 256 + 48 * 4096 * 7168 * 9 // 16
        assert chord.chord_packed_weight_bytes(1, 8, 64, layout) == 0
        assert chord.chord_packed_weight_bytes(1, 128, 96, layout) == 0
    assert chord.chord_packed_weight_bytes(1, 16, 64, 1) == 256 + 16 * 64 * 9 // 16
    assert chord.chord_packed_weight_bytes(1, 16, 64, 2) == 0
    assert chord.chord_packed_weight_bytes(1, 16, 64, 3) == 0
    assert chord.chord_packed_weight_bytes(1, 128, 64, 4) == 0
    P = 512 * 8
    assert chord.chord_align_capacity(512, 8, 48, 16) == -(-(P + 48 * 15) // 16) * 16
    assert chord.chord_align_capacity(1, 8, 384, 8) == -(-(8 + 8 * 7) // 8) * 8
    assert chord.chord_align_capacity(0, 8, 48, 16) == 0
    assert chord.chord_align_capacity(1, 0, 48, 16) == -1
    assert chord.chord_align_workspace_bytes(16384, 8, 48) == 32 * 48 * 4


def test_status_strings(lib):
    for s in range(8):
        assert chord.chord_status_string(s)
    assert chord.chord_status_string(99) == "unknown status"


def test_select_block_m(lib):
    # tokens per expert (tok_e = T * topk / E_global) decides, not the token count
    assert chord.chord_select_block_m(512, 8, 48, 384, 4096, 7168) in (16, 32)   # tok_e ~ 10.7
    assert chord.chord_select_block_m(1, 8, 384, 384, 512, 7168) == 8
    # tok_e 21.3: mean + 3 sd = 36.2 rows, mean + 2 sd = 31.6 -> the 32-row warp-level block
    assert chord.chord_select_block_m(1024, 8, 384, 384, 512, 7168) == 32
    # tok_e 24: mean + 2 sd = 34.8 -> 48
    assert chord.chord_select_block_m(1152, 8, 384, 384, 512, 7168) == 48
    assert chord.chord_select_block_m(16, 2, 8, 8, 256, 256) in (8, 16)          # tok_e = 4
    prev = 0
    for T in (1, 16, 128, 512, 1024, 4096, 8192, 16384):
        bm = chord.chord_select_block_m(T, 8, 48, 384, 4096, 7168)
        assert bm % 8 == 0 and 8 <= bm <= 256
        assert bm >= prev, "block size must not shrink as tokens per expert grow"
        assert bm >= min(T * 8 / 384, 64)
        prev = bm


def test_select_kernel_by_regime(lib, monkeypatch):
    """Decode blocks (at most 32 rows) and short-K GEMMs with blocks up to 64
    rows go to the warp-level kernel, the rest to the tcgen05 kernel; the
    decode workload's block and the prefill workload's block land on
    different sides."""
    monkeypatch.delenv("CHORD_KERNEL", raising=False)
    W, T = chord.KERNEL_WARP_MMA, chord.KERNEL_TCGEN05
    for bm in (8, 16, 24, 32):
        assert chord.chord_select_kernel(bm, 4096, 7168) == W
    for bm in (40, 64, 128, 256):
        assert chord.chord_select_kernel(bm, 4096, 7168) == T
    assert chord.chord_select_kernel(48, 7168, 256) == W       # TP8 down, T = 1024
    assert chord.chord_select_kernel(64, 7168, 256) == W
    assert chord.chord_select_kernel(128, 7168, 256) == T      # TP8 down, T = 4096
    assert chord.chord_select_kernel(256, 7168, 256) == T
    assert chord.chord_select_kernel(64, 7168, 1024) == T
    bm_dec = chord.chord_select_block_m(512, 8, 48, 384, 4096, 7168)
    bm_pre = chord.chord_select_block_m(8192, 8, 48, 384, 4096, 7168)
    assert chord.chord_select_kernel(bm_dec, 4096, 7168) == W and chord.chord_select_kernel(bm_dec, 7168, 2048) == W
    assert chord.chord_select_kernel(bm_pre, 4096, 7168) == T and chord.chord_select_kernel(bm_pre, 7168, 2048) == T
    monkeypatch.setenv("CHORD_KERNEL", "1")
    assert chord.chord_select_kernel(8, 4096, 7168) == T
    monkeypatch.setenv("CHORD_KERNEL", "2")
    assert chord.chord_select_kernel(256, 4096, 7168) == W
    monkeypatch.setenv("CHORD_KERNEL", "7")        # not a kernel: ignored
    assert chord.chord_select_kernel(256, 4096, 7168) == T


def test_grouped_workspace_and_argument_errors(lib):
    """Grouped contracts: workspace = sorted ids + expert ids + padded count,
    each 256-byte aligned, plus the tcgen05 split tail (152 x 128 x tok_tile
    FP32) for blocks of more than 32 rows; bad arguments are refused before
    any launch."""
    up = lambda x: (x + 255) // 256 * 256
    tail = lambda bm: 152 * 128 * ((bm + 15) // 16 * 16) * 4 if bm > 32 else 0
    for M, E in ((0, 4), (1, 1), (128, 2), (12288, 48)):
        bmc = chord.chord_select_block_m(M, 1, E, E, 0, 0)
        cap = (-(-M // bmc) + E) * bmc
        assert chord.chord_grouped_contiguous_workspace_bytes(M, E) == (up(up(up(cap * 4) + cap // bmc * 4) + 4)
                                                                         + tail(bmc))
    assert chord.chord_select_block_m(12288, 1, 48, 48, 0, 0) > 32   # the EP8 prefill case carries the tail
    assert chord.chord_grouped_contiguous_workspace_bytes(128, 5000) == 0
    G, max_m, em = 48, 40, 11
    bm = chord.chord_select_block_m(em, 1, 1, 1, 4096, 7168)
    cap = G * -(-max_m // bm) * bm
    assert chord.chord_grouped_masked_workspace_bytes(G, max_m, em) == up(up(up(cap * 4) + cap // bm * 4) + 4) + tail(bm)
    assert chord.chord_grouped_masked_workspace_bytes(0, 8, 4) == 0
    vp = ctypes.c_void_p
    big = vp(1 << 20)
    # contiguous: workspace too small, negative M
    assert lib.chord_grouped_contiguous_gemm(big, 256, big, big, 10 ** 6, 2, 128, 64, big, big, 16, None,
                                             None) == 4
    assert lib.chord_grouped_contiguous_gemm(big, -1, big, big, 10 ** 6, 2, 128, 64, big, big, 10 ** 6, None,
                                             None) == 1
    # masked: expected_m <= 0, too many groups, workspace too small
    assert lib.chord_grouped_masked_gemm(big, 4, 8, big, 0, big, 10 ** 6, 128, 64, big, big, 10 ** 6, None,
                                         None) == 1
    assert lib.chord_grouped_masked_gemm(big, 4001, 8, big, 4, big, 10 ** 6, 128, 64, big, big, 10 ** 6, None,
                                         None) == 2
    assert lib.chord_grouped_masked_gemm(big, 4, 8, big, 4, big, 10 ** 6, 128, 64, big, big, 8, None, None) == 4


def test_layer_workspace_formula(lib):
    T, topk, E, H, I, bm = 512, 8, 48, 7168, 2048, 16
    P = T * topk
    cap = chord.chord_align_capacity(T, topk, E, bm)
    up = lambda x: (x + 255) // 256 * 256
    want = up(chord.chord_align_workspace_bytes(T, topk, E))
    want = up(want + cap * 4)
    want = up(want + cap // bm * 4)
    want = up(want + 4)
    want = up(want + P * 2 * I * 2)
    want = up(want + P * I * 2)
    want = up(want + P * H * 4)   # the down projection's FP32 sums
    want = up(want + P * 4)       # the fused combine's per-pair weights
    # 4096 pairs fill the GPU: no K slices, no partial-sum space
    assert chord.chord_layer_workspace_bytes(T, topk, E, H, I, bm) == want
    # one token, TP8 shapes: the gate_up projection is cut into 15 K slices
    T, topk, E, H, I, bm = 1, 8, 384, 7168, 256, 8
    P = T * topk
    cap = chord.chord_align_capacity(T, topk, E, bm)
    want = up(chord.chord_align_workspace_bytes(T, topk, E))
    for b in (cap * 4, cap // bm * 4, 4, P * 2 * I * 2, P * I * 2, P * H * 4, P * 4):
        want = up(want + b)
    want = up(want + max(chord.chord_gemm_workspace_bytes(P, 2 * I, H, bm),
                         chord.chord_gemm_workspace_bytes(P, H, I, bm)))
    assert chord.chord_gemm_workspace_bytes(P, 2 * I, H, bm) == 15 * P * 2 * I * 4
    assert chord.chord_layer_workspace_bytes(T, topk, E, H, I, bm) == want


def test_split_k_choice(lib, monkeypatch):
    """K slices of the warp-level kernel: the automatic choice cuts K only
    when num_pairs x N / 128 items fill less than half of 456 resident CTAs,
    into ceil(456 / items) slices, at most 16 and at most half the 128-column
    K stages; an explicit count is capped at the number of stages.  The
    workspace holds S x num_pairs x N FP32 partial sums.  The tcgen05 kernel
    splits only its last partial wave; its workspace is 152 units of
    128 x tok_tile FP32 sums (tok_tile = block_m rounded up to 16), none with
    split_k = 1."""
    monkeypatch.delenv("CHORD_KERNEL", raising=False)
    ws = chord.chord_gemm_workspace_bytes
    assert ws(8, 512, 7168, 8) == 15 * 8 * 512 * 4          # 32 items -> 15 slices
    assert ws(1, 128, 7168, 8) == 16 * 1 * 128 * 4          # 1 item -> capped at 16
    assert ws(1, 128, 512, 8) == 2 * 1 * 128 * 4            # 4 stages -> at most 2
    assert ws(1, 128, 256, 8) == 0                          # 2 stages -> 1 slice
    assert ws(8, 7168, 256, 8) == 0                         # 448 items fill the GPU
    assert ws(128, 512, 7168, 8) == 0                       # 512 items
    assert ws(40, 512, 7168, 8) == 3 * 40 * 512 * 4         # 160 items -> 3 slices
    assert ws(8, 512, 7168, 256) == 152 * 128 * 256 * 4     # tcgen05: the split tail
    assert ws(8, 512, 7168, 200) == 152 * 128 * 208 * 4
    assert ws(8, 512, 7168, 256, chord.ChordOpts(split_k=1)) == 0
    opts = chord.ChordOpts(split_k=1)
    assert ws(8, 512, 7168, 8, opts) == 0
    opts = chord.ChordOpts(split_k=7)
    assert ws(4096, 4096, 7168, 16, opts) == 7 * 4096 * 4096 * 4
    opts = chord.ChordOpts(split_k=99)
    assert ws(8, 512, 384, 8, opts) == 3 * 8 * 512 * 4      # 3 stages
    opts = chord.ChordOpts(split_k=4, kernel=chord.KERNEL_TCGEN05)
    assert ws(8, 512, 7168, 8, opts) == 152 * 128 * 16 * 4
    monkeypatch.setenv("CHORD_KERNEL", "1")
    assert ws(8, 512, 7168, 8) == 152 * 128 * 16 * 4
    # an explicit split without its workspace is refused before any launch
    vp = ctypes.c_void_p
    big = vp(1 << 20)
    o = chord.ChordOpts(split_k=4, kernel=chord.KERNEL_WARP_MMA)
    nbytes = chord.chord_packed_weight_bytes(2, 128, 512)
    assert lib.chord_w4a16_moe_gemm(big, 8, 1, big, nbytes, 2, 128, 512, big, big, big, 8, 8, 8, big, big, 16,
                                    ctypes.byref(o), None) == 4
    o = chord.ChordOpts(split_k=-1)
    assert lib.chord_w4a16_moe_gemm(big, 8, 1, big, nbytes, 2, 128, 512, big, big, big, 8, 8, 8, big, None, 0,
                                    ctypes.byref(o), None) == 1
    o = chord.ChordOpts(split_k=2, kernel=chord.KERNEL_TCGEN05)
    assert lib.chord_w4a16_moe_gemm(big, 8, 1, big, nbytes, 2, 128, 512, big, big, big, 256, 256, 8, big, big,
                                    1024, ctypes.byref(o), None) == 4


def test_argument_errors_before_any_launch(lib):
    """Unsupported shapes and bad sizes are refused synchronously, before the
    library touches CUDA (so this runs without a GPU)."""
    vp = ctypes.c_void_p
    big = vp(1 << 20)
    # group size other than 32
    assert lib.chord_pack_weights(big, big, 1, 128, 64, 64, 2, big, 10 ** 6, None) == 2
    # N not a multiple of 16 (layout 1) / 128 (layout 2)
    assert lib.chord_pack_weights(big, big, 1, 8, 64, 32, 1, big, 10 ** 6, None) == 2
    assert lib.chord_pack_weights(big, big, 1, 16, 64, 32, 2, big, 10 ** 6, None) == 2
    # unknown layout
    assert lib.chord_pack_weights(big, big, 1, 128, 64, 32, 7, big, 10 ** 6, None) == 1
    # packed buffer too small
    assert lib.chord_pack_weights(big, big, 1, 128, 64, 32, 2, big, 100, None) == 4
    # GEMM: packed size does not match (E, N, K) -> layout mismatch
    args = [big, 16, 1, big, 12345, 2, 128, 64, big, big, big, 16, 8, 16, big, None, 0, None, None]
    assert lib.chord_w4a16_moe_gemm(*args) == 3
    # GEMM: K not a multiple of 64 -> unsupported
    args = [big, 16, 1, big, 12345, 2, 128, 96, big, big, big, 16, 8, 16, big, None, 0, None, None]
    assert lib.chord_w4a16_moe_gemm(*args) == 2
    # align: capacity too small
    assert lib.chord_moe_align(big, 4, 2, 4, 8, big, big, big, 8, big, 10 ** 6, None, None) == 4
    # align: too many experts for the scan
    assert lib.chord_moe_align(big, 4, 2, 2000, 8, big, big, big, 10 ** 6, big, 10 ** 8, None, None) == 2
    # misaligned activation pointer
    nb = chord.chord_packed_weight_bytes(2, 128, 64, 2)
    args = [vp((1 << 20) + 2), 16, 1, big, nb, 2, 128, 64, big, big, big, 16, 8, 16, big, None, 0, None, None]
    assert lib.chord_w4a16_moe_gemm(*args) == 1
    # fused SiLU * up: an unknown epilogue, or FP32 output with the epilogue
    args = [big, 16, 1, big, nb, 2, 128, 64, big, big, big, 16, 8, 16, big, None, 0, None, None]
    for epi, dt in [(2, 0), (1, 1)]:
        o = chord.ChordOpts(epilogue=epi, out_dtype=dt)
        args[17] = ctypes.byref(o)
        assert lib.chord_w4a16_moe_gemm(*args) == 1, (epi, dt)
    # layout 3 (gate_up rows interleaved) has layout 2's size and needs N % 128 == 0
    assert chord.chord_packed_weight_bytes(2, 256, 64, 3) == chord.chord_packed_weight_bytes(2, 256, 64, 2)
    assert chord.chord_packed_weight_bytes(2, 64, 64, 3) == 0
    assert lib.chord_pack_weights(big, big, 1, 64, 64, 32, 3, big, 10 ** 6, None) == 2
