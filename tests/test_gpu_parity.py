"""Parity of the CUDA path (through the C ABI) with the CPU oracle, at sizes
the oracle finishes in seconds: several N tiles, several K stages, ragged
blocks, every block size, edge-case routing.  Pack and align must match byte
for byte; GEMM, SiLU*up and the layer within |gpu - ref| <= 1e-2 + 1e-2|ref|
(bit for bit where every summation order gives the same FP32 value)."""
import numpy as np
import pytest
import torch

import oracle
import w4a16_int4_mixture_moe_gb300 as chord
import workloads as wl
from gpu_util import (DEV, KERNELS, align, assert_close, check_h_from_gpu_c1, check_layer_chain, dbf, dev, f64, gemm,
                      host_bits, run_layer_steps,
                      layer, pack, valid_rows)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    chord.build()
    chord.load()
    oracle.build()
    chord.chord_get_device_error()
    yield
    assert chord.chord_get_device_error() == 0, "a test left the device error word set"


# --------------------------------------------------------------------- pack

@pytest.mark.parametrize("layout,shape", [(1, (8, 256, 256)), (1, (8, 256, 128)), (1, (3, 32, 128)),
                                          (1, (2, 144, 192)), (1, (1, 4096, 7168)),
                                          (2, (8, 256, 256)), (2, (8, 256, 128)), (2, (3, 384, 192)),
                                          (2, (1, 4096, 7168)), (2, (2, 7168, 256)),
                                          (3, (8, 256, 256)), (3, (3, 384, 192)), (3, (1, 4096, 7168))])
def test_pack_byte_exact(layout, shape):
    E, N, K = shape
    codes = wl.random_codes(sum(shape), shape)
    scales = wl.random_scales(sum(shape) + 1, (E, N, K // 32))
    got = pack(codes, scales, layout).cpu().numpy()
    want = oracle.pack(codes, scales, layout)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("layout", [1, 2, 3])
@pytest.mark.parametrize("planted", [0x3C00, 0x3EFF, 0x0080, 0x3F00, 0x0040, 0x0000, 0x8000, 0xBC00, 0x7FC0])
def test_pack_scale_range_word_byte_exact(layout, planted):
    """Header word 7 (every scale in [2^-126, 0.5)) is set by the packer that
    sees all scales: one planted scale in the last expert decides it, on the
    GPU as in the oracle, and the rest of the blob is unchanged."""
    E, N, K = 3, 256, 128
    codes = wl.random_codes(7, (E, N, K))
    scales = wl.random_scales(8, (E, N, K // 32))
    scales[E - 1, N - 3, 1] = planted
    got = pack(codes, scales, layout).cpu().numpy()
    want = oracle.pack(codes, scales, layout)
    np.testing.assert_array_equal(got, want)
    assert int(got[28:32].view(np.uint32)[0]) == int(planted in (0x3C00, 0x3EFF, 0x0080))


@pytest.mark.parametrize("layout", [1, 2, 3])
def test_pack_bad_code_sets_error_word(layout):
    codes = np.zeros((1, 128, 64), np.uint8)
    codes[0, 5, 7] = 17
    pack(codes, np.zeros((1, 128, 2), np.uint16), layout)
    assert chord.chord_get_device_error() == 5  # CHORD_DEV_BAD_CODE
    assert chord.chord_get_device_error() == 0


# -------------------------------------------------------------------- align

ALIGN_CASES = [
    (16, 2, 8, 4, 0.0), (33, 8, 48, 16, 0.5), (7, 3, 5, 8, 0.2), (64, 8, 384, 8, 0.0), (1, 8, 384, 16, 0.0),
    (128, 4, 6, 64, 0.3), (200, 6, 12, 256, 0.1), (4096, 8, 384, 32, 0.0), (2048, 8, 48, 256, 0.875),
    (1000, 1, 1024, 8, 0.0), (5000, 2, 3, 1, 0.0),
]


@pytest.mark.parametrize("T,topk,E,bm,pnl", ALIGN_CASES)
def test_align_bit_exact(T, topk, E, bm, pnl):
    ids = wl.random_ids(T * 7 + E, T, topk, E, p_nonlocal=pnl)
    s, e, n = align(ids, E, bm)
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    assert int(n.item()) == n2
    np.testing.assert_array_equal(s.cpu().numpy(), s2)
    np.testing.assert_array_equal(e.cpu().numpy(), e2)


@pytest.mark.parametrize("wl_name", ["ep8_decode", "ep8_prefill", "skewed", "tp8_4096"])
def test_align_workload_routing_bit_exact(wl_name):
    w = {"ep8_decode": wl.EP8_DECODE, "ep8_prefill": wl.EP8_PREFILL, "skewed": wl.SKEWED,
         "tp8_4096": wl.tp8(4096)}[wl_name]
    ids, _ = wl.make_routing(w)
    for bm in (16, 64, 256):
        s, e, n = align(ids, w.E, bm)
        s2, e2, n2 = oracle.moe_align(ids, w.E, bm)
        assert int(n.item()) == n2
        np.testing.assert_array_equal(s.cpu().numpy(), s2)
        np.testing.assert_array_equal(e.cpu().numpy(), e2)


def test_align_edge_counts_and_empty():
    bm = 8
    flat = [1] + [2] * 2 + [3] * (bm - 1) + [4] * bm + [5] * (bm + 1) + [-1, -1]
    rng = np.random.default_rng(3)
    flat = np.array(flat, np.int32)[rng.permutation(len(flat))]
    flat = np.append(flat, np.int32(-1)) if flat.size % 2 else flat
    ids = flat.astype(np.int32).reshape(-1, 2)
    s, e, n = align(ids, 6, bm)
    s2, e2, n2 = oracle.moe_align(ids, 6, bm)
    assert int(n.item()) == n2
    np.testing.assert_array_equal(s.cpu().numpy(), s2)
    np.testing.assert_array_equal(e.cpu().numpy(), e2)
    # no tokens at all
    s, e, n = align(np.zeros((0, 8), np.int32), 48, 16)
    assert int(n.item()) == 0 and s.numel() == 0
    # nothing local
    s, e, n = align(np.full((9, 4), -1, np.int32), 8, 4)
    assert int(n.item()) == 0 and bool((s == 36).all()) and bool((e == -1).all())


def test_align_validate_reports_bad_ids():
    ids = wl.random_ids(5, 20, 4, 8)
    ids[3, 1] = 11
    with pytest.raises(chord.ChordError) as ei:
        align(ids, 8, 8, opts=chord.ChordOpts(validate=1))
    assert ei.value.status == 6
    # without validation the id is dropped like a non-local one
    s, e, n = align(ids, 8, 8)
    s2, e2, n2 = oracle.moe_align(ids, 8, 8)
    np.testing.assert_array_equal(s.cpu().numpy(), s2)
    assert chord.chord_get_device_error() == 0


# --------------------------------------------------------------------- GEMM

def run_gemm_case(T, topk, E, N, K, bm, seed, div=None, pnl=0.2, kernel="tcgen05", exact=False, x=None,
                  codes=None, scales=None, ids=None):
    div = topk if div is None else div
    a_rows = T if div == topk else T * topk
    if x is None:
        x = wl.random_bf16(seed, (a_rows, K))
    if codes is None:
        codes = wl.random_codes(seed + 1, (E, N, K))
    if scales is None:
        scales = wl.random_scales(seed + 2, (E, N, K // 32))
    if ids is None:
        ids = wl.random_ids(seed + 3, T, topk, E, p_nonlocal=pnl)
    P = T * topk
    kid, layout = KERNELS[kernel]
    packed = pack(codes, scales, layout)
    s, e, n = align(ids, E, bm)
    C = gemm(x, div, packed, E, N, K, s, e, n, bm, P, kernel=kid)
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    ref = oracle.moe_gemm(x, div, codes, scales, s2, e2, n2, bm, P,
                          C=np.full((P, N), 0xFFFF, np.uint16))
    got = host_bits(C)
    rows = valid_rows(ids, E)
    other = np.setdiff1d(np.arange(P), rows)
    assert (got[other] == 0xFFFF).all(), "rows of non-local pairs were written"
    if exact:
        np.testing.assert_array_equal(got[rows], ref[rows])
    else:
        assert_close(got[rows], ref[rows], f"{kernel} gemm T={T} E={E} N={N} K={K} bm={bm}")
    return got, ref


BOTH = pytest.mark.parametrize("kernel", ["tcgen05", "warp_mma"])


@BOTH
@pytest.mark.parametrize("bm", [8, 16, 24, 32, 64, 128, 256])
@pytest.mark.parametrize("K", [256, 2048])
@pytest.mark.parametrize("scale", [0x3F80, 0x3E80])
def test_gemm_exact_integer_regime_bit_exact(kernel, bm, K, scale):
    """x in {-1, 0, 1}, scales 1.0 or 0.25: sums are exact multiples of the
    scale in any order, so the GPU must match the oracle bit for bit (catches
    any wrong index, lost or doubled K chunk, or token/row mix-up).  Scale 1.0
    lies outside [2^-126, 0.5) and takes the subtract-then-scale instructions,
    0.25 the one-FMA dequantisation (both kernels)."""
    T, topk, E, N = 40, 4, 5, 256
    rng = np.random.default_rng(bm * 100 + K)
    xi = rng.integers(-1, 2, size=(T, K)).astype(np.float32)
    x = wl._bf16(xi)
    scales = np.full((E, N, K // 32), scale, np.uint16)
    run_gemm_case(T, topk, E, N, K, bm, seed=bm + K, x=x, scales=scales, exact=True, kernel=kernel)


@BOTH
@pytest.mark.parametrize("bm", [8, 16, 32, 64, 128])
def test_gemm_dequant_bit_exact_one_hot(kernel, bm):
    """One-hot activation rows make C the dequantised weight column itself:
    C[t, n] = bf16((q[n, t] - 8) * s[n, t/32]) exactly.  Every code and a wide
    range of scale exponents go through the kernel's subtract-then-scale path."""
    K, N, E = 128, 256, 1
    T = K
    x = np.zeros((T, K), np.float32)
    x[np.arange(T), np.arange(K)] = 1.0
    x = wl._bf16(x)
    codes = wl.random_codes(90 + bm, (E, N, K))
    rng = np.random.default_rng(91)
    sc = (rng.standard_normal((E, N, K // 32)) * np.exp2(rng.integers(-20, 20, size=(E, N, K // 32))))
    scales = wl._bf16(sc.astype(np.float32))
    ids = np.zeros((T, 1), np.int32)
    got, ref = run_gemm_case(T, 1, E, N, K, bm, seed=0, div=1, x=x, codes=codes, scales=scales, ids=ids,
                             exact=True, kernel=kernel)
    deq = oracle.dequant_pairs(codes[0].T.copy().ravel(),
                               np.repeat(scales[0], 32, axis=1).T.copy().ravel()).reshape(K, N)
    # a zero weight times a negative scale is -0; a sum that starts from +0 returns +0
    deq = np.where(deq == 0x8000, np.uint16(0), deq)
    np.testing.assert_array_equal(got, deq)


@BOTH
@pytest.mark.parametrize("bm", [8, 16, 32, 64, 128])
def test_gemm_dequant_bit_exact_one_hot_fma_range(kernel, bm):
    """As above with every scale a positive bf16 in [2^-126, 0.5): the packer
    sets header word 7 and both kernels take the one-FMA dequantisation, which
    must equal subtract-then-scale.  Exponents over that whole range, random mantissas, and both ends
    (2^-126 and the largest bf16 below 0.5).  Every code times every such scale
    must equal the oracle's bf16((q - 8) * s), q = 8 giving +0."""
    K, N, E = 128, 256, 1
    T = K
    x = np.zeros((T, K), np.float32)
    x[np.arange(T), np.arange(K)] = 1.0
    x = wl._bf16(x)
    codes = wl.random_codes(95 + bm, (E, N, K))
    rng = np.random.default_rng(96)
    expo = rng.integers(1, 126, size=(E, N, K // 32)).astype(np.uint16)
    mant = rng.integers(0, 128, size=(E, N, K // 32)).astype(np.uint16)
    scales = (expo << 7) | mant
    scales[0, 0, :] = [0x0080, 0x3EFF, 0x0080, 0x3EFF]
    scales[0, 1, :] = [0x3EFF, 0x0080, 0x00FF, 0x3E80]
    ids = np.zeros((T, 1), np.int32)
    packed = pack(codes, scales, KERNELS[kernel][1])
    assert int(packed[28:32].cpu().numpy().view(np.uint32)[0]) == 1
    got, ref = run_gemm_case(T, 1, E, N, K, bm, seed=0, div=1, x=x, codes=codes, scales=scales, ids=ids,
                             exact=True, kernel=kernel)
    deq = oracle.dequant_pairs(codes[0].T.copy().ravel(),
                               np.repeat(scales[0], 32, axis=1).T.copy().ravel()).reshape(K, N)
    np.testing.assert_array_equal(got, deq)


@BOTH
@pytest.mark.parametrize("bm", [8, 32, 64, 256])
def test_gemm_f32_output(kernel, bm):
    """FP32 output: exact integers in the exact-integer regime (bit-exact with the
    oracle's unrounded sum), within tolerance on random data."""
    T, topk, E, N, K = 24, 4, 5, 256, 1024
    kid, layout = KERNELS[kernel]
    rng = np.random.default_rng(bm)
    xi = rng.integers(-1, 2, size=(T, K)).astype(np.float32)
    codes = wl.random_codes(bm + 1, (E, N, K))
    ids = wl.random_ids(bm + 2, T, topk, E, p_nonlocal=0.2)
    rows = valid_rows(ids, E)
    s, e, n = align(ids, E, bm)
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    for x, scales, exact in [(wl._bf16(xi), np.full((E, N, K // 32), 0x3F80, np.uint16), True),
                             (wl.random_bf16(bm + 3, (T, K)), wl.random_scales(bm + 4, (E, N, K // 32)), False)]:
        packed = pack(codes, scales, layout)
        C = torch.full((T * topk, N), float("nan"), dtype=torch.float32, device=DEV)
        chord.chord_w4a16_moe_gemm(dbf(x), topk, packed, E, N, K, s, e, n, bm, T * topk, C,
                                   opts=chord.ChordOpts(kernel=kid, out_dtype=chord.DTYPE_F32))
        got = C.cpu().numpy()
        ref = oracle.moe_gemm_f32(x, topk, codes, scales, s2, e2, n2, bm, T * topk)
        if exact:
            np.testing.assert_array_equal(got[rows], ref[rows])
        else:
            err = np.abs(got[rows].astype(np.float64) - ref[rows])
            assert (err <= 1e-2 + 1e-2 * np.abs(ref[rows])).all(), err.max()
        other = np.setdiff1d(np.arange(T * topk), rows)
        assert np.isnan(got[other]).all()


@BOTH
@pytest.mark.parametrize("bm", [8, 16, 32, 64, 96, 256])
@pytest.mark.parametrize("shape", [(3, 128, 64), (4, 384, 320), (6, 256, 1024)])
def test_gemm_random_vs_oracle(kernel, bm, shape):
    E, N, K = shape
    run_gemm_case(37, 3, E, N, K, bm, seed=E * N + K + bm, kernel=kernel)


@BOTH
def test_gemm_many_rows_per_expert(kernel):
    """Blocks full up to 256 rows and experts spanning several blocks (the
    prefill case): 600 pairs on 3 experts, block sizes 128 and 256."""
    T, topk, E = 300, 2, 3
    ids = wl.random_ids(61, T, topk, E)
    for bm in (128, 256):
        run_gemm_case(T, topk, E, 256, 512, bm, seed=62 + bm, ids=ids, kernel=kernel)


@BOTH
def test_gemm_down_projection_row_per_pair(kernel):
    """a_row_divisor = 1: A holds one row per pair (the down projection)."""
    run_gemm_case(30, 4, 5, 256, 256, 16, seed=77, div=1, kernel=kernel)


@BOTH
def test_gemm_edge_routing(kernel):
    """Experts with 0, 1, 2, bm-1, bm, bm+1 and 3*bm+5 rows in one call."""
    bm = 16
    counts = [0, 1, 2, bm - 1, bm, bm + 1, 3 * bm + 5]
    flat = np.concatenate([np.full(c, e, np.int32) for e, c in enumerate(counts)])
    flat = flat[np.random.default_rng(4).permutation(flat.size)]
    pad = (-flat.size) % 2
    flat = np.concatenate([flat, np.full(pad, -1, np.int32)])
    ids = flat.reshape(-1, 2)
    run_gemm_case(ids.shape[0], 2, len(counts), 128, 192, bm, seed=5, ids=ids, kernel=kernel)


@BOTH
def test_gemm_nothing_local_writes_nothing(kernel):
    ids = np.full((12, 4), -1, np.int32)
    run_gemm_case(12, 4, 3, 128, 64, 8, seed=6, ids=ids, kernel=kernel)


def test_bounded_wait_times_out_and_context_survives():
    """Failure detection without a fault: a pipeline wait that can never end
    (an mbarrier nothing arrives on, waited on through the helper every GEMM
    pipeline uses) gives up after its bound, leaves CHORD_DEV_TIMEOUT in the
    error word, and the context keeps working; a validating call reports the
    code as CHORD_ERR_TIMEOUT."""
    assert chord.chord_get_device_error() == 0
    chord.chord_selftest_wait_timeout()
    assert chord.chord_get_device_error() == 4          # CHORD_DEV_TIMEOUT, read and cleared
    assert chord.chord_get_device_error() == 0
    # the context still computes: an exact-integer GEMM matches the oracle bit for bit
    T, topk, E, N, K, bm = 12, 2, 3, 256, 256, 16
    rng = np.random.default_rng(77)
    x = wl._bf16(rng.integers(-1, 2, size=(T, K)).astype(np.float32))
    scales = np.full((E, N, K // 32), 0x3F80, np.uint16)
    run_gemm_case(T, topk, E, N, K, bm, seed=77, x=x, scales=scales, exact=True, kernel="warp_mma")
    # a validating call reads the word and maps the timeout to CHORD_ERR_TIMEOUT
    chord.chord_selftest_wait_timeout()
    codes = wl.random_codes(78, (E, N, K))
    packed = pack(codes, scales)
    ids = wl.random_ids(79, T, topk, E)
    s, e, n = align(ids, E, bm)
    C = torch.empty((T * topk, N), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(chord.ChordError) as ei:
        chord.chord_w4a16_moe_gemm(dbf(x), topk, packed, E, N, K, s, e, n, bm, T * topk, C,
                                   opts=chord.ChordOpts(kernel=chord.KERNEL_WARP_MMA, validate=1))
    assert ei.value.status == 7                           # CHORD_ERR_TIMEOUT
    assert chord.chord_get_device_error() == 0


def test_gemm_header_mismatch_is_reported():
    """A blob packed for (E, N, K) = (2, 128, 128) passed as (2, 256, 64) has the
    right size but the wrong header, and a blob of packed layout 1 has the wrong
    layout for either kernel: the device refuses each and writes nothing."""
    E = 2
    codes = wl.random_codes(1, (E, 128, 128))
    scales = wl.random_scales(2, (E, 128, 4))
    ids = wl.random_ids(3, 8, 2, E)
    s, e, n = align(ids, E, 8)
    for layout, N, K, kernel in [(2, 256, 64, chord.KERNEL_TCGEN05), (2, 256, 64, chord.KERNEL_WARP_MMA),
                                 (1, 128, 128, chord.KERNEL_TCGEN05), (1, 128, 128, chord.KERNEL_WARP_MMA)]:
        packed = pack(codes, scales, layout)
        x = wl.random_bf16(4, (8, K))
        C = torch.full((16, N), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        with pytest.raises(chord.ChordError) as ei:
            chord.chord_w4a16_moe_gemm(dbf(x), 2, packed, E, N, K, s, e, n, 8, 16, C,
                                       opts=chord.ChordOpts(kernel=kernel, validate=1))
        assert ei.value.status == 6
        assert (host_bits(C) == 0xFFFF).all()


# ------------------------------------------------------------------ split-K

WARP = chord.KERNEL_WARP_MMA


@pytest.mark.parametrize("bm", [8, 16, 32])
@pytest.mark.parametrize("S", [2, 3, 7, 16])
def test_split_k_exact_integer_regime_bit_exact(bm, S):
    """K slices with FP32 partials and an in-order reduction: in the
    exact-integer regime every sum is exact, so the split result equals the
    oracle bit for bit, and rows of non-local pairs stay unwritten."""
    T, topk, E, N, K = 12, 4, 5, 256, 2048
    rng = np.random.default_rng(S * 10 + bm)
    x = wl._bf16(rng.integers(-1, 2, size=(T, K)).astype(np.float32))
    codes = wl.random_codes(S + bm, (E, N, K))
    scales = np.full((E, N, K // 32), 0x3F80, np.uint16)
    ids = wl.random_ids(S + bm + 1, T, topk, E, p_nonlocal=0.2)
    P = T * topk
    s, e, n = align(ids, E, bm)
    got = host_bits(gemm(x, topk, pack(codes, scales), E, N, K, s, e, n, bm, P, kernel=WARP, split_k=S))
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    ref = oracle.moe_gemm(x, topk, codes, scales, s2, e2, n2, bm, P, C=np.full((P, N), 0xFFFF, np.uint16))
    rows = valid_rows(ids, E)
    np.testing.assert_array_equal(got[rows], ref[rows])
    assert (got[np.setdiff1d(np.arange(P), rows)] == 0xFFFF).all()


@pytest.mark.parametrize("S", [2, 5, 99])
@pytest.mark.parametrize("shape", [(3, 128, 320), (4, 384, 1024), (2, 256, 7168)])
def test_split_k_random_vs_oracle(S, shape):
    """Random data, bf16 and FP32 outputs, ragged K (the last 64-column stage
    of K = 320 lands in the last slice; S = 99 is capped at the stage count)."""
    E, N, K = shape
    T, topk, bm = 9, 4, 8
    x = wl.random_bf16(S + K, (T, K))
    codes = wl.random_codes(S + K + 1, (E, N, K))
    scales = wl.random_scales(S + K + 2, (E, N, K // 32))
    ids = wl.random_ids(S + K + 3, T, topk, E, p_nonlocal=0.2)
    P = T * topk
    packed = pack(codes, scales)
    s, e, n = align(ids, E, bm)
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    rows = valid_rows(ids, E)
    got = host_bits(gemm(x, topk, packed, E, N, K, s, e, n, bm, P, kernel=WARP, split_k=S))
    ref = oracle.moe_gemm(x, topk, codes, scales, s2, e2, n2, bm, P, C=np.full((P, N), 0xFFFF, np.uint16))
    assert_close(got[rows], ref[rows], f"split-K S={S} E={E} N={N} K={K}")
    C = torch.full((P, N), float("nan"), dtype=torch.float32, device=DEV)
    gemm(x, topk, packed, E, N, K, s, e, n, bm, P, kernel=WARP, C=C, split_k=S, out_dtype=chord.DTYPE_F32)
    got32 = C.cpu().numpy()
    ref32 = oracle.moe_gemm_f32(x, topk, codes, scales, s2, e2, n2, bm, P)
    err = np.abs(got32[rows].astype(np.float64) - ref32[rows])
    assert (err <= 1e-2 + 1e-2 * np.abs(ref32[rows])).all(), err.max()
    assert np.isnan(got32[np.setdiff1d(np.arange(P), rows)]).all()


@pytest.mark.parametrize("S", [3, 8])
def test_split_k_fused_silu_mul(S):
    """The reduction applies the SiLU * up epilogue: bit-identical to the split
    GEMM without it followed by chord_silu_mul, close to the oracle."""
    T, topk, E, I, K, bm = 11, 3, 4, 192, 1024, 16
    x = wl.random_bf16(70 + S, (T, K))
    codes = wl.random_codes(71 + S, (E, 2 * I, K))
    scales = wl.random_scales(72 + S, (E, 2 * I, K // 32))
    ids = wl.random_ids(73 + S, T, topk, E, p_nonlocal=0.2)
    P = T * topk
    s, e, n = align(ids, E, bm)
    h = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    gemm(x, topk, pack(codes, scales, chord.LAYOUT_GATE_UP_INTERLEAVED), E, 2 * I, K, s, e, n, bm, P,
         kernel=WARP, C=h, split_k=S, epilogue=chord.EPILOGUE_SILU_MUL)
    got = host_bits(h)
    C1 = gemm(x, topk, pack(codes, scales), E, 2 * I, K, s, e, n, bm, P, kernel=WARP, split_k=S)
    h2 = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    chord.chord_silu_mul(C1, dev(ids.ravel().copy()), E, h2)
    rows = valid_rows(ids, E)
    np.testing.assert_array_equal(got[rows], host_bits(h2)[rows])
    assert (got[np.setdiff1d(np.arange(P), rows)] == 0xFFFF).all()
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    c1 = oracle.moe_gemm(x, topk, codes, scales, s2, e2, n2, bm, P, C=np.zeros((P, 2 * I), np.uint16))
    check_h_from_gpu_c1(got, host_bits(C1), c1, ids.ravel(), E, rows, f"split-K fused S={S}")


def test_split_k_automatic_one_token():
    """One token, TP8 gate_up shape (N = 512, K = 7168): the automatic choice
    splits K (15 slices) when given its workspace, runs unsplit without one,
    and both agree with the oracle."""
    T, topk, E, N, K, bm = 1, 8, 16, 512, 7168, 8
    assert chord.chord_gemm_workspace_bytes(T * topk, N, K, bm) == 15 * 8 * N * 4
    x = wl.random_bf16(80, (T, K))
    codes = wl.random_codes(81, (E, N, K))
    scales = wl.random_scales(82, (E, N, K // 32))
    ids = wl.random_ids(83, T, topk, E, p_nonlocal=0.0)
    P = T * topk
    packed = pack(codes, scales)
    s, e, n = align(ids, E, bm)
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    ref = oracle.moe_gemm(x, topk, codes, scales, s2, e2, n2, bm, P, C=np.zeros((P, N), np.uint16))
    rows = valid_rows(ids, E)
    split = host_bits(gemm(x, topk, packed, E, N, K, s, e, n, bm, P, split_k=0))
    plain = host_bits(gemm(x, topk, packed, E, N, K, s, e, n, bm, P))
    assert_close(split[rows], ref[rows], "automatic split-K, one token")
    assert_close(plain[rows], ref[rows], "no workspace, one token")
    assert chord.chord_get_device_error() == 0


def test_layer_one_token_split_k_vs_oracle():
    """The layer with one token and TP8 widths (H = 7168, I = 256) on 16 local
    experts: its workspace carries the gate_up split's partial sums."""
    T, topk, E, H, I = 1, 8, 16, 7168, 256
    ids = wl.random_ids(90, T, topk, E, p_nonlocal=0.0)
    wts = wl.random_weights(91, T, topk)
    x = wl.random_bf16(92, (T, H))
    c13, s13 = wl.random_codes(93, (E, 2 * I, H)), wl.random_scales(94, (E, 2 * I, H // 32))
    c2, s2 = wl.random_codes(95, (E, H, I)), wl.random_scales(96, (E, H, I // 32))
    for fused in (False, True):
        p13 = pack(c13, s13, chord.LAYOUT_GATE_UP_INTERLEAVED if fused else chord.LAYOUT_TCGEN05)
        opts = chord.ChordOpts(epilogue=chord.EPILOGUE_SILU_MUL if fused else chord.EPILOGUE_NONE)
        out, bm = layer(x, ids, wts, E, 384, I, p13, pack(c2, s2), opts=opts)
        assert bm == 8
        ref = oracle.moe_layer(x, ids, wts, (c13, s13), (c2, s2), E, block_m=bm)
        assert_close(host_bits(out), ref, f"one-token layer fused={fused}")


# ------------------------------------------------- tcgen05 split tail

TC = chord.KERNEL_TCGEN05


def tail_case(bm, K, seed, exact, T=100, topk=8, E=8, N=2560):
    """8 experts x 20 N tiles = 160 items (320 with two blocks per expert) on
    152 persistent CTAs: whole waves plus a tail that the kernel cuts into K
    slices."""
    rng = np.random.default_rng(seed)
    if exact:
        x = wl._bf16(rng.integers(-1, 2, size=(T, K)).astype(np.float32))
        scales = np.full((E, N, K // 32), 0x3F80, np.uint16)
    else:
        x = wl.random_bf16(seed, (T, K))
        scales = wl.random_scales(seed + 2, (E, N, K // 32))
    codes = wl.random_codes(seed + 1, (E, N, K))
    ids = wl.random_ids(seed + 3, T, topk, E, p_nonlocal=0.1)
    return x, codes, scales, ids


@pytest.mark.parametrize("bm,K,exact", [(256, 512, True), (256, 320, True), (256, 1024, False), (128, 1024, True),
                                        (128, 640, False), (64, 2048, True)])
def test_tc_tail_split_vs_oracle(bm, K, exact):
    """The last partial wave's items in K slices (FP32 partials, in-order
    reduction): bit-exact with the oracle in the exact-integer regime, within
    tolerance on random data; bf16 and FP32 outputs; rows of non-local pairs
    untouched; the same as the unsplit launch up to FP32 order."""
    T, topk, E, N = 100, 8, 8, 2560
    x, codes, scales, ids = tail_case(bm, K, bm + K, exact)
    P = T * topk
    packed = pack(codes, scales)
    s, e, n = align(ids, E, bm)
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    assert chord.chord_gemm_workspace_bytes(P, N, K, bm) == 152 * 128 * ((bm + 15) // 16 * 16) * 4
    got = host_bits(gemm(x, topk, packed, E, N, K, s, e, n, bm, P, kernel=TC, split_k=0))
    ref = oracle.moe_gemm(x, topk, codes, scales, s2, e2, n2, bm, P, C=np.full((P, N), 0xFFFF, np.uint16))
    rows = valid_rows(ids, E)
    assert (got[np.setdiff1d(np.arange(P), rows)] == 0xFFFF).all()
    if exact:
        np.testing.assert_array_equal(got[rows], ref[rows])
    else:
        assert_close(got[rows], ref[rows], f"tail split bm={bm} K={K}")
    plain = host_bits(gemm(x, topk, packed, E, N, K, s, e, n, bm, P, kernel=TC, split_k=1))
    if exact:
        np.testing.assert_array_equal(plain[rows], got[rows])
    C = torch.full((P, N), float("nan"), dtype=torch.float32, device=DEV)
    gemm(x, topk, packed, E, N, K, s, e, n, bm, P, kernel=TC, C=C, split_k=0, out_dtype=chord.DTYPE_F32)
    got32 = C.cpu().numpy()
    ref32 = oracle.moe_gemm_f32(x, topk, codes, scales, s2, e2, n2, bm, P)
    if exact:
        np.testing.assert_array_equal(got32[rows], ref32[rows])
    else:
        err = np.abs(got32[rows].astype(np.float64) - ref32[rows])
        assert (err <= 1e-2 + 1e-2 * np.abs(ref32[rows])).all(), err.max()
    assert chord.chord_get_device_error() == 0


@pytest.mark.parametrize("bm", [256, 128])
@pytest.mark.parametrize("exact", [True, False])
def test_tc_tail_split_fused_silu_mul(bm, exact):
    """SiLU * up applied by the tail reduction (layout 3).  Layout 3 puts other
    rows in each N tile than layout 2, so the two GEMMs split different
    items and sum some rows in another FP32 order: bit-identical to the layout-2
    GEMM followed by chord_silu_mul in the exact-integer regime (every order
    gives the same sums), close to the oracle on random data."""
    T, topk, E, I, K = 100, 8, 8, 1280, 512
    x, codes, scales, ids = tail_case(bm, K, 7 + bm, exact, N=2 * I)
    P = T * topk
    s, e, n = align(ids, E, bm)
    h = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    gemm(x, topk, pack(codes, scales, chord.LAYOUT_GATE_UP_INTERLEAVED), E, 2 * I, K, s, e, n, bm, P, kernel=TC,
         C=h, split_k=0, epilogue=chord.EPILOGUE_SILU_MUL)
    got = host_bits(h)
    C1 = gemm(x, topk, pack(codes, scales), E, 2 * I, K, s, e, n, bm, P, kernel=TC, split_k=0)
    h2 = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    chord.chord_silu_mul(C1, dev(ids.ravel().copy()), E, h2)
    rows = valid_rows(ids, E)
    if exact:
        np.testing.assert_array_equal(got[rows], host_bits(h2)[rows])
    assert (got[np.setdiff1d(np.arange(P), rows)] == 0xFFFF).all()
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    c1 = oracle.moe_gemm(x, topk, codes, scales, s2, e2, n2, bm, P, C=np.zeros((P, 2 * I), np.uint16))
    check_h_from_gpu_c1(got, host_bits(C1), c1, ids.ravel(), E, rows, f"tail split fused bm={bm}")


def test_layer_tc_tail_split_vs_oracle():
    """A layer whose gate_up GEMM (tcgen05, 160 items) splits its tail through
    the layer workspace."""
    T, topk, E, H, I, bm = 100, 8, 8, 1024, 1280, 256
    ids = wl.random_ids(30, T, topk, E, p_nonlocal=0.1)
    wts = wl.random_weights(31, T, topk)
    x = wl.random_bf16(32, (T, H))
    c13, s13 = wl.random_codes(33, (E, 2 * I, H)), wl.random_scales(34, (E, 2 * I, H // 32))
    c2, s2 = wl.random_codes(35, (E, H, I)), wl.random_scales(36, (E, H, I // 32))
    assert chord.chord_layer_workspace_bytes(T, topk, E, H, I, bm) > 152 * 128 * 256 * 4
    p13, p2 = pack(c13, s13), pack(c2, s2)
    out, _ = layer(x, ids, wts, E, E, I, p13, p2, bm=bm, opts=chord.ChordOpts(kernel=TC))
    st = run_layer_steps(x, ids, wts, E, I, p13, p2, bm, fused=False, kernel=TC)
    assert torch.equal(out.view(torch.int16), st["out"].view(torch.int16)), "layer call differs from its steps"
    check_layer_chain(x, ids, wts, (c13, s13), (c2, s2), E, host_bits(st["C1"]), host_bits(st["h"]),
                      st["C2"].cpu().numpy(), host_bits(st["out"]), "layer with a split tail")


# ---------------------------------------------------------- fused SiLU * up

def run_fused_case(T, topk, E, I, K, bm, seed, kernel, pnl=0.2):
    """The gate_up GEMM with the SiLU * up epilogue on a layout-3 blob, against
    the oracle's GEMM followed by its SiLU * up, and bit for bit against this
    library's unfused path (same sums, same rounding points)."""
    x = wl.random_bf16(seed, (T, K))
    codes = wl.random_codes(seed + 1, (E, 2 * I, K))
    scales = wl.random_scales(seed + 2, (E, 2 * I, K // 32))
    ids = wl.random_ids(seed + 3, T, topk, E, p_nonlocal=pnl)
    P = T * topk
    kid, layout = KERNELS[kernel]
    s, e, n = align(ids, E, bm)
    h = torch.full((max(P, 1), I), -1, dtype=torch.int16, device=DEV)[:P].view(torch.bfloat16)
    chord.chord_w4a16_moe_gemm(dbf(x), topk, pack(codes, scales, chord.LAYOUT_GATE_UP_INTERLEAVED), E, 2 * I, K,
                               s, e, n, bm, P, h, opts=chord.ChordOpts(kernel=kid, epilogue=chord.EPILOGUE_SILU_MUL))
    got = host_bits(h)
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    c1 = oracle.moe_gemm(x, topk, codes, scales, s2, e2, n2, bm, P, C=np.zeros((P, 2 * I), np.uint16))
    rows = valid_rows(ids, E)
    other = np.setdiff1d(np.arange(P), rows)
    assert (got[other] == 0xFFFF).all(), "rows of non-local pairs were written"
    C1 = gemm(x, topk, pack(codes, scales, layout), E, 2 * I, K, s, e, n, bm, P, kernel=kid)
    check_h_from_gpu_c1(got, host_bits(C1), c1, ids.ravel(), E, rows,
                        f"{kernel} fused gate_up T={T} E={E} I={I} K={K} bm={bm}")
    h2 = torch.full((max(P, 1), I), -1, dtype=torch.int16, device=DEV)[:P].view(torch.bfloat16)
    chord.chord_silu_mul(C1, dev(ids.ravel().copy()), E, h2)
    np.testing.assert_array_equal(got[rows], host_bits(h2)[rows])


@BOTH
@pytest.mark.parametrize("bm", [8, 16, 32, 64, 128, 256])
@pytest.mark.parametrize("shape", [(3, 64, 128), (4, 192, 320), (2, 128, 1024)])
def test_fused_silu_mul_vs_oracle(kernel, bm, shape):
    E, I, K = shape
    run_fused_case(37, 3, E, I, K, bm, seed=E * I + K + bm, kernel=kernel)


def test_fused_silu_mul_needs_layout3_and_vice_versa():
    """A layout-2 blob with the epilogue, and a layout-3 blob without it, are
    refused on the device and write nothing."""
    E, I, K = 2, 64, 128
    codes = wl.random_codes(1, (E, 2 * I, K))
    scales = wl.random_scales(2, (E, 2 * I, K // 32))
    ids = wl.random_ids(3, 8, 2, E)
    s, e, n = align(ids, E, 8)
    x = wl.random_bf16(4, (8, K))
    for layout, epi, width in [(2, chord.EPILOGUE_SILU_MUL, I), (3, chord.EPILOGUE_NONE, 2 * I)]:
        for kid in (chord.KERNEL_TCGEN05, chord.KERNEL_WARP_MMA):
            C = torch.full((16, width), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
            with pytest.raises(chord.ChordError) as ei:
                chord.chord_w4a16_moe_gemm(dbf(x), 2, pack(codes, scales, layout), E, 2 * I, K, s, e, n, 8, 16, C,
                                           opts=chord.ChordOpts(kernel=kid, validate=1, epilogue=epi))
            assert ei.value.status == 6
            assert (host_bits(C) == 0xFFFF).all()


# ----------------------------------------------------------- grouped GEMMs

def contiguous_rows(counts):
    """m_indices of experts' segments padded to 128-row multiples."""
    return np.concatenate([np.concatenate([np.full(c, e), np.full(-(-c // 128) * 128 - c, -1)])
                           for e, c in enumerate(counts)]).astype(np.int32)


@BOTH
@pytest.mark.parametrize("counts", [[70, 0, 128, 5], [1, 200, 33], [128, 128]])
@pytest.mark.parametrize("NK", [(256, 320), (128, 1024)])
def test_grouped_contiguous_vs_oracle(kernel, counts, NK):
    N, K = NK
    E = len(counts)
    m_idx = contiguous_rows(counts)
    M = m_idx.size
    seed = sum(counts) + N + K
    x = wl.random_bf16(seed, (M, K))
    codes, scales = wl.random_codes(seed + 1, (E, N, K)), wl.random_scales(seed + 2, (E, N, K // 32))
    ws = torch.empty(chord.chord_grouped_contiguous_workspace_bytes(M, E), dtype=torch.uint8, device=DEV)
    C = torch.full((M, N), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    chord.chord_grouped_contiguous_gemm(dbf(x), dev(m_idx), pack(codes, scales), E, N, K, C, ws,
                                        opts=chord.ChordOpts(kernel=KERNELS[kernel][0]))
    ref = oracle.grouped_contiguous(x, m_idx, codes, scales, C=np.full((M, N), 0xFFFF, np.uint16))
    got = host_bits(C)
    assert (got[m_idx < 0] == 0xFFFF).all(), "padding rows were written"
    assert_close(got[m_idx >= 0], ref[m_idx >= 0], f"{kernel} grouped contiguous {counts} N={N} K={K}")


def test_grouped_contiguous_split_tail_exact():
    """Eight experts of 100 rows (128-row segments, one block each) x 20 N
    tiles = 160 tcgen05 items on 152 CTAs: the tail splits through the grouped
    workspace.  Exact-integer regime: bit-exact with the oracle, and with a
    workspace that holds only the routing arrays (no split)."""
    counts = [100] * 8
    E, N, K = 8, 2560, 1024
    m_idx = contiguous_rows(counts)
    M = m_idx.size
    rng = np.random.default_rng(5)
    x = wl._bf16(rng.integers(-1, 2, size=(M, K)).astype(np.float32))
    codes = wl.random_codes(6, (E, N, K))
    scales = np.full((E, N, K // 32), 0x3F80, np.uint16)
    packed = pack(codes, scales)
    ref = oracle.grouped_contiguous(x, m_idx, codes, scales, C=np.full((M, N), 0xFFFF, np.uint16))
    full = chord.chord_grouped_contiguous_workspace_bytes(M, E)
    bm = chord.chord_select_block_m(M, 1, E, E, 0, 0)
    assert 128 <= bm <= 256
    for nbytes in (full, full - 152 * 128 * ((bm + 15) // 16 * 16) * 4):
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        C = torch.full((M, N), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        chord.chord_grouped_contiguous_gemm(dbf(x), dev(m_idx), packed, E, N, K, C, ws)
        got = host_bits(C)
        assert (got[m_idx < 0] == 0xFFFF).all()
        np.testing.assert_array_equal(got[m_idx >= 0], ref[m_idx >= 0])
    assert chord.chord_get_device_error() == 0


def test_grouped_contiguous_split_expert_is_reported():
    """An expert whose rows are not one contiguous run breaks the contract: the
    device error word says so (validate mode turns it into a status)."""
    E, N, K = 2, 128, 64
    m_idx = np.array([0] * 60 + [1] * 40 + [0] * 28, np.int32)
    x = wl.random_bf16(1, (128, K))
    codes, scales = wl.random_codes(2, (E, N, K)), wl.random_scales(3, (E, N, K // 32))
    ws = torch.empty(chord.chord_grouped_contiguous_workspace_bytes(128, E), dtype=torch.uint8, device=DEV)
    C = torch.empty((128, N), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(chord.ChordError) as ei:
        chord.chord_grouped_contiguous_gemm(dbf(x), dev(m_idx), pack(codes, scales), E, N, K, C, ws,
                                            opts=chord.ChordOpts(validate=1))
    assert ei.value.status == 6


@BOTH
@pytest.mark.parametrize("masked,max_m,expected_m", [([3, 0, 9, 1], 9, 4), ([17, 40, 2, 33, 0, 64], 64, 20),
                                                     ([200, 5, 256], 256, 150)])
def test_grouped_masked_vs_oracle(kernel, masked, max_m, expected_m):
    N, K = 256, 512
    G = len(masked)
    masked_m = np.array(masked, np.int32)
    seed = sum(masked) + max_m
    x = wl.random_bf16(seed, (G, max_m, K))
    codes, scales = wl.random_codes(seed + 1, (G, N, K)), wl.random_scales(seed + 2, (G, N, K // 32))
    ws = torch.empty(chord.chord_grouped_masked_workspace_bytes(G, max_m, expected_m), dtype=torch.uint8,
                     device=DEV)
    C = torch.full((G * max_m, N), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    chord.chord_grouped_masked_gemm(dbf(x), dev(masked_m), expected_m, pack(codes, scales), N, K, C, ws,
                                    opts=chord.ChordOpts(kernel=KERNELS[kernel][0]))
    ref = oracle.grouped_masked(x, masked_m, codes, scales, C=np.full((G * max_m, N), 0xFFFF, np.uint16))
    got = host_bits(C)
    valid = np.array([r < masked[g] for g in range(G) for r in range(max_m)])
    assert (got[~valid] == 0xFFFF).all(), "rows past a group's count were written"
    assert_close(got[valid], ref[valid], f"{kernel} grouped masked {masked} max_m={max_m}")


def test_grouped_masked_count_out_of_range_is_reported():
    G, max_m, N, K = 2, 8, 128, 64
    x = wl.random_bf16(1, (G, max_m, K))
    codes, scales = wl.random_codes(2, (G, N, K)), wl.random_scales(3, (G, N, K // 32))
    ws = torch.empty(chord.chord_grouped_masked_workspace_bytes(G, max_m, 4), dtype=torch.uint8, device=DEV)
    C = torch.empty((G * max_m, N), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(chord.ChordError) as ei:
        chord.chord_grouped_masked_gemm(dbf(x), dev(np.array([3, 9], np.int32)), 4, pack(codes, scales), N, K, C,
                                        ws, opts=chord.ChordOpts(validate=1))
    assert ei.value.status == 6


# ---------------------------------------------------------------- epilogues

@pytest.mark.parametrize("P,I", [(50, 192), (3, 8), (17, 264), (9, 2048), (12000, 64)])
def test_silu_mul_vs_oracle(P, I):
    """One warp per pair row: rows of 1, 24, 33 and 256 vectors of 8 columns
    (one partial round of lanes, one full and one partial, several full) and
    more rows than the grid's warps."""
    E = 4
    C1 = wl.random_bf16(8, (P, 2 * I), std=4.0)
    ids = wl.random_ids(9, P, 1, E, p_nonlocal=0.3)
    h = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    chord.chord_silu_mul(dbf(C1), dev(ids.ravel().copy()), E, h)
    ref = oracle.silu_mul(C1, ids.ravel(), E, h=np.full((P, I), 0xFFFF, np.uint16))
    got = host_bits(h)
    rows = valid_rows(ids, E)
    assert_close(got[rows], ref[rows], "silu_mul")
    other = np.setdiff1d(np.arange(P), rows)
    assert (got[other] == 0xFFFF).all()
    # expf may differ from the C library's by an ulp; nearly all results are identical
    assert np.mean(got[rows] == ref[rows]) > 0.99


@pytest.mark.parametrize("T,topk,H", [(33, 8, 1792), (130, 8, 1792), (1, 8, 7168), (3, 20, 1024), (5, 1, 256)])
def test_combine_bit_exact(T, topk, H):
    """Same FP32 operations in the same order as the oracle: bit-exact, on both
    the few-token kernel (batched top-k loads, T * H / 4 up to one wave of
    threads) and the many-token kernel, with top-k above the batch of 8."""
    E = 16
    C2 = wl.random_bf16(10, (T * topk, H), std=30.0)
    ids = wl.random_ids(11, T, topk, E, p_nonlocal=0.4)
    ids[0, :] = -1
    w = wl.random_weights(12, T, topk)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    chord.chord_moe_combine(dbf(C2), dev(ids), dev(w), E, out)
    ref = oracle.combine(C2, ids, w, E)
    np.testing.assert_array_equal(host_bits(out), ref)
    # FP32 pair results (the layer's down projection output)
    C2f = (np.random.default_rng(13).standard_normal((T * topk, H)) * 80).astype(np.float32)
    chord.chord_moe_combine(dev(C2f), dev(ids), dev(w), E, out)
    np.testing.assert_array_equal(host_bits(out), oracle.combine(C2f, ids, w, E))


# -------------------------------------------------------------------- layer

@BOTH
@pytest.mark.parametrize("bm", [0, 8, 16, 32, 64, 256])
@pytest.mark.parametrize("fused", [False, True])
def test_layer_tiny_vs_oracle(kernel, bm, fused):
    w = wl.TINY
    ids, wts = wl.make_routing(w)
    x = wl.make_x(w)
    c13, s13 = wl.make_w13(w)
    c2, s2 = wl.make_w2(w)
    kid, layout = KERNELS[kernel]
    p13 = pack(c13, s13, chord.LAYOUT_GATE_UP_INTERLEAVED if fused else layout)
    epi = chord.EPILOGUE_SILU_MUL if fused else chord.EPILOGUE_NONE
    out, used_bm = layer(x, ids, wts, w.E, w.E_global, w.I, p13, pack(c2, s2, layout), bm=bm,
                         opts=chord.ChordOpts(kernel=kid, epilogue=epi))
    ref = oracle.moe_layer(x, ids, wts, (c13, s13), (c2, s2), w.E, block_m=used_bm)
    assert_close(host_bits(out), ref, f"tiny layer bm={used_bm}")


@pytest.mark.parametrize("fused", [False, True])
def test_layer_ep_partial_and_empty_tokens(fused):
    """EP-style routing with most pairs non-local; tokens with no local pair are +0."""
    T, topk, E, H, I = 24, 8, 6, 256, 128
    ids = wl.random_ids(20, T, topk, 48)
    ids = np.where(ids < E, ids, -1).astype(np.int32)
    ids[5, :] = -1
    wts = wl.random_weights(21, T, topk)
    x = wl.random_bf16(22, (T, H))
    c13, s13 = wl.random_codes(23, (E, 2 * I, H)), wl.random_scales(24, (E, 2 * I, H // 32))
    c2, s2 = wl.random_codes(25, (E, H, I)), wl.random_scales(26, (E, H, I // 32))
    p13 = pack(c13, s13, chord.LAYOUT_GATE_UP_INTERLEAVED if fused else chord.LAYOUT_TCGEN05)
    opts = chord.ChordOpts(epilogue=chord.EPILOGUE_SILU_MUL if fused else chord.EPILOGUE_NONE)
    out, bm = layer(x, ids, wts, E, 48, I, p13, pack(c2, s2), opts=opts)
    ref = oracle.moe_layer(x, ids, wts, (c13, s13), (c2, s2), E, block_m=bm)
    got = host_bits(out)
    assert_close(got, ref, "ep partial layer")
    assert (got[5] == 0).all()


def test_layer_zero_tokens():
    E, H, I = 4, 128, 64
    p13 = pack(np.zeros((E, 2 * I, H), np.uint8), np.zeros((E, 2 * I, H // 32), np.uint16))
    p2 = pack(np.zeros((E, H, I), np.uint8), np.zeros((E, H, I // 32), np.uint16))
    ws = torch.empty(4096, dtype=torch.uint8, device=DEV)
    out = torch.empty((0, H), dtype=torch.bfloat16, device=DEV)
    chord.chord_moe_layer(torch.empty((0, H), dtype=torch.bfloat16, device=DEV),
                          torch.empty((0, 2), dtype=torch.int32, device=DEV),
                          torch.empty((0, 2), dtype=torch.float32, device=DEV), E, E, I, p13, p2, ws, out,
                          block_m=8)


def test_layer_cuda_graph_replay():
    """The layer enqueues no host synchronisation, so it captures into a CUDA
    graph; replays give the eager result."""
    w = wl.TINY
    ids, wts = wl.make_routing(w)
    x = wl.make_x(w)
    c13, s13 = wl.make_w13(w)
    c2, s2 = wl.make_w2(w)
    p13, p2 = pack(c13, s13), pack(c2, s2)
    bm = 16
    ws = torch.empty(chord.chord_layer_workspace_bytes(w.T, w.topk, w.E, w.H, w.I, bm), dtype=torch.uint8,
                     device=DEV)
    xd, idd, wd = dbf(x), dev(ids), dev(wts)
    eager = torch.empty((w.T, w.H), dtype=torch.bfloat16, device=DEV)
    chord.chord_moe_layer(xd, idd, wd, w.E, w.E_global, w.I, p13, p2, ws, eager, block_m=bm)
    out = torch.zeros((w.T, w.H), dtype=torch.bfloat16, device=DEV)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            chord.chord_moe_layer(xd, idd, wd, w.E, w.E_global, w.I, p13, p2, ws, out, block_m=bm, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(out), host_bits(eager))


# ------------------------------------------------- mixed regime (per-block kernel)

def skewed_ids(seed, T, topk, E, s=2.0):
    """Zipf-skewed routing without replacement (Gumbel top-k over log rank^-s):
    a few hot experts with hundreds of rows and a cold tail with a handful."""
    rng = np.random.default_rng(seed)
    logp = -s * np.log(np.arange(1, E + 1, dtype=np.float64))
    keys = logp[None, :] - np.log(-np.log(rng.random((T, E))))
    return np.ascontiguousarray(np.argsort(-keys, axis=1)[:, :topk].astype(np.int32))


@pytest.mark.parametrize("bm,K,exact,silu", [(128, 1024, True, False), (128, 1024, False, False),
                                             (256, 640, True, False), (64, 2048, False, False),
                                             (128, 1024, False, True), (256, 1024, True, True)])
def test_mixed_regime_vs_oracle(bm, K, exact, silu):
    """Skewed routing (hot experts over several blocks, cold experts with 1-20
    rows) in the tcgen05 regime with the per-block split on: blocks of at most
    32 valid rows run on the warp-level kernel, the rest on tcgen05 with its
    split tail (the reduction must leave the small blocks' rows alone).
    Bit-exact with the oracle and with the split off in the exact-integer
    regime; within tolerance on random data; FP32 output and the fused SiLU * up
    epilogue; rows of non-local pairs untouched."""
    T, topk, E, N = 300, 4, 24, 1024 if not silu else 512
    ids = skewed_ids(bm + K, T, topk, E)
    ids = np.where(np.random.default_rng(bm).random(ids.shape) < 0.05, -1, ids).astype(np.int32)
    counts = np.bincount(ids[ids >= 0], minlength=E)
    assert (counts > bm).any() and ((counts > 0) & (counts <= 32)).sum() >= 5
    rng = np.random.default_rng(K + bm)
    if exact:
        x = wl._bf16(rng.integers(-1, 2, size=(T, K)).astype(np.float32))
        scales = np.full((E, N, K // 32), 0x3F80, np.uint16)
    else:
        x = wl.random_bf16(K + 1, (T, K))
        scales = wl.random_scales(K + 2, (E, N, K // 32))
    codes = wl.random_codes(K + 3, (E, N, K))
    P = T * topk
    s, e, n = align(ids, E, bm)
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    rows = valid_rows(ids, E)
    other = np.setdiff1d(np.arange(P), rows)
    ref = oracle.moe_gemm(x, topk, codes, scales, s2, e2, n2, bm, P, C=np.full((P, N), 0xFFFF, np.uint16))
    if silu:
        I = N // 2
        p3 = pack(codes, scales, chord.LAYOUT_GATE_UP_INTERLEAVED)
        h = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        gemm(x, topk, p3, E, N, K, s, e, n, bm, P, C=h, split_k=0, epilogue=chord.EPILOGUE_SILU_MUL, mixed=1)
        got = host_bits(h)
        assert (got[other] == 0xFFFF).all()
        C1 = gemm(x, topk, pack(codes, scales), E, N, K, s, e, n, bm, P, split_k=0, mixed=1)
        check_h_from_gpu_c1(got, host_bits(C1), ref, ids.ravel(), E, rows, f"mixed fused bm={bm}")
        if exact:
            # exact sums in any order: the fused epilogue equals the SiLU * up pass on the same C1
            h2 = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
            chord.chord_silu_mul(C1, dev(ids.ravel().copy()), E, h2)
            np.testing.assert_array_equal(got[rows], host_bits(h2)[rows])
        return
    packed = pack(codes, scales)
    got = host_bits(gemm(x, topk, packed, E, N, K, s, e, n, bm, P, split_k=0, mixed=1))
    off = host_bits(gemm(x, topk, packed, E, N, K, s, e, n, bm, P, split_k=0, mixed=-1))
    assert (got[other] == 0xFFFF).all(), "rows of non-local pairs were written"
    if exact:
        np.testing.assert_array_equal(got[rows], ref[rows])
        np.testing.assert_array_equal(off[rows], ref[rows])
    else:
        assert_close(got[rows], ref[rows], f"mixed bm={bm} K={K}")
        assert_close(off[rows], ref[rows], f"mixed off bm={bm} K={K}")
    C = torch.full((P, N), float("nan"), dtype=torch.float32, device=DEV)
    gemm(x, topk, packed, E, N, K, s, e, n, bm, P, C=C, split_k=0, out_dtype=chord.DTYPE_F32, mixed=1)
    got32 = C.cpu().numpy()
    ref32 = oracle.moe_gemm_f32(x, topk, codes, scales, s2, e2, n2, bm, P)
    if exact:
        np.testing.assert_array_equal(got32[rows], ref32[rows])
    else:
        err = np.abs(got32[rows].astype(np.float64) - ref32[rows])
        assert (err <= 1e-2 + 1e-2 * np.abs(ref32[rows])).all(), err.max()
    assert np.isnan(got32[other]).all()
    assert chord.chord_get_device_error() == 0


def test_mixed_regime_option_is_checked():
    """opts.mixed outside -1..1 is refused before anything is enqueued."""
    E, N, K, bm = 2, 256, 1024, 64
    codes = wl.random_codes(1, (E, N, K))
    scales = wl.random_scales(2, (E, N, K // 32))
    ids = wl.random_ids(3, 8, 2, E)
    s, e, n = align(ids, E, bm)
    with pytest.raises(chord.ChordError) as ei:
        gemm(wl.random_bf16(4, (8, K)), 2, pack(codes, scales), E, N, K, s, e, n, bm, 16, mixed=2)
    assert ei.value.status == 1


# ------------------------------------------------- top-k combine fused into the down GEMM

def _combine_case(seed, T, topk, E, none_token=3):
    ids = wl.random_ids(seed, T, topk, 4 * E)
    ids = np.where(ids < E, ids, -1).astype(np.int32)     # about 1/4 of the pairs local
    ids[none_token, :] = -1                               # a token with no local pair
    ids[none_token + 1, :] = -1
    ids[none_token + 1, 2] = 0                            # a token with exactly one
    ids[none_token + 2, :] = np.arange(topk) % E          # a token with all pairs local
    return np.ascontiguousarray(ids)


@pytest.mark.parametrize("kernel,bm,K,split", [("warp_mma", 16, 1024, None), ("warp_mma", 8, 2048, 0),
                                               ("tcgen05", 64, 1024, 0), ("tcgen05", 128, 512, None),
                                               ("auto", 256, 1024, 0)])
def test_fused_combine_matches_the_separate_pass(kernel, bm, K, split):
    """chord_combine_plan -> chord_w4a16_moe_gemm_combine -> chord_combine_finish
    gives exactly what the down GEMM's FP32 output followed by the combine pass
    gives (bit for bit, also against the oracle's combine of that output), on
    routing with tokens that have no, one and several local pairs; with K
    slices (warp-level), the tcgen05 split tail, and the mixed regime (auto,
    256-row blocks)."""
    T, topk, E, N = 120, 8, 6, 512
    ids = _combine_case(bm + K, T, topk, E)
    w = wl.random_weights(K, T, topk)
    P = T * topk
    A = wl.random_bf16(bm, (P, K))
    codes = wl.random_codes(bm + 1, (E, N, K))
    scales = wl.random_scales(bm + 2, (E, N, K // 32))
    packed = pack(codes, scales)
    kid = 0 if kernel == "auto" else KERNELS[kernel][0]
    s, e, n = align(ids, E, bm)
    idd, wd = dev(ids), dev(w)
    opts = chord.ChordOpts(kernel=kid, split_k=split or 0, out_dtype=chord.DTYPE_F32,
                           mixed=1 if kernel == "auto" else 0)
    nb = chord.chord_gemm_workspace_bytes(P, N, K, bm, opts) if split is not None else 0
    ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=DEV) if split is not None else None
    # the separate path
    C2 = torch.full((P, N), float("nan"), dtype=torch.float32, device=DEV)
    chord.chord_w4a16_moe_gemm(dbf(A), 1, packed, E, N, K, s, e, n, bm, P, C2, workspace=ws, opts=opts)
    out_sep = torch.empty((T, N), dtype=torch.bfloat16, device=DEV)
    chord.chord_moe_combine(C2, idd, wd, E, out_sep)
    # the fused path
    pair_w = torch.full((P,), 7.0, dtype=torch.float32, device=DEV)
    chord.chord_combine_plan(idd, wd, E, pair_w)
    flat = ids.ravel()
    local = (flat >= 0) & (flat < E)
    cnt = local.reshape(T, topk).sum(axis=1)
    pw = pair_w.cpu().numpy()
    single = local & (np.repeat(cnt, topk) == 1)
    multi = local & (np.repeat(cnt, topk) > 1)
    np.testing.assert_array_equal(pw[single], w.ravel()[single])
    assert np.isnan(pw[multi]).all() and (pw[~local] == 7.0).all()
    C2f = torch.full((P, N), float("nan"), dtype=torch.float32, device=DEV)
    out = torch.full((T, N), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    chord.chord_w4a16_moe_gemm_combine(dbf(A), packed, E, N, K, s, e, n, bm, topk, pair_w, C2f, out, workspace=ws,
                                       opts=opts)
    c2 = C2.cpu().numpy()
    c2f = C2f.cpu().numpy()
    np.testing.assert_array_equal(c2f[multi], c2[multi])       # several local pairs: FP32 rows as before
    assert np.isnan(c2f[~multi]).all()                          # the others: nothing written to C2
    chord.chord_combine_finish(C2f, idd, wd, E, out)
    got = host_bits(out)
    np.testing.assert_array_equal(got, host_bits(out_sep))
    np.testing.assert_array_equal(got, oracle.combine(c2, ids, w, E))
    assert (got[cnt == 0] == 0).all()
    assert chord.chord_get_device_error() == 0


@BOTH
@pytest.mark.parametrize("silu", [False, True])
def test_layer_fused_combine_bit_identical(kernel, silu):
    """chord_moe_layer with the fused combine (opts.fuse_combine = 1) equals
    the layer with the separate combine pass bit for bit; EP-like routing with tokens
    that have no, one and several local pairs."""
    T, topk, E, H, I = 40, 8, 6, 256, 128
    ids = _combine_case(9, T, topk, E)
    wts = wl.random_weights(10, T, topk)
    x = wl.random_bf16(11, (T, H))
    c13, s13 = wl.random_codes(12, (E, 2 * I, H)), wl.random_scales(13, (E, 2 * I, H // 32))
    c2, s2 = wl.random_codes(14, (E, H, I)), wl.random_scales(15, (E, H, I // 32))
    kid, layout = KERNELS[kernel]
    p13 = pack(c13, s13, chord.LAYOUT_GATE_UP_INTERLEAVED if silu else layout)
    p2 = pack(c2, s2, layout)
    epi = chord.EPILOGUE_SILU_MUL if silu else chord.EPILOGUE_NONE
    a, bm = layer(x, ids, wts, E, 4 * E, I, p13, p2, bm=16,
                  opts=chord.ChordOpts(kernel=kid, epilogue=epi, fuse_combine=1))
    b, _ = layer(x, ids, wts, E, 4 * E, I, p13, p2, bm=16,
                 opts=chord.ChordOpts(kernel=kid, epilogue=epi, fuse_combine=-1))
    np.testing.assert_array_equal(host_bits(a), host_bits(b))
    got = host_bits(a)
    none = ~((ids >= 0) & (ids < E)).any(axis=1)
    assert (got[none] == 0).all()


def test_fused_combine_rejects_bad_arguments():
    """topk above 32 and an out pointer that is not 16-byte aligned are refused
    before anything is enqueued."""
    ids = torch.zeros((4, 33), dtype=torch.int32, device=DEV)
    w = torch.zeros((4, 33), dtype=torch.float32, device=DEV)
    pw = torch.zeros(4 * 33, dtype=torch.float32, device=DEV)
    with pytest.raises(chord.ChordError) as ei:
        chord.chord_combine_plan(ids, w, 2, pw)
    assert ei.value.status == 2
    C2 = torch.zeros((4 * 33, 256), dtype=torch.float32, device=DEV)
    out = torch.zeros((4, 256), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(chord.ChordError) as ei:
        chord.chord_combine_finish(C2, ids, w, 2, out)
    assert ei.value.status == 2


# ------------------------------------------------- tcgen05 in clusters of two CTAs

@pytest.mark.parametrize("bm,K,exact", [(256, 1024, True), (256, 320, True), (128, 640, True), (64, 2048, True),
                                        (256, 1024, False), (128, 512, False), (24, 256, True)])
def test_tc_pairs_vs_oracle(bm, K, exact):
    """opts.tc_pairs = 1 (cta_group::2: a cluster of two CTAs per 256-row item,
    each CTA's 128 dequantised rows in its own tensor memory, each gathering half
    of the block's tokens): bit-exact with the oracle in the exact-integer
    regime, within tolerance on random data, bf16 and FP32 outputs, the fused
    SiLU * up and the mixed regime; one, two and four MMA issuers (blocks of up
    to 256, 128 and 64 rows); a ragged last K stage."""
    T, topk, E, N = 100, 8, 8, 1024
    x, codes, scales, ids = tail_case(bm, K, 11 + bm + K, exact, N=N)
    P = T * topk
    packed = pack(codes, scales)
    s, e, n = align(ids, E, bm)
    s2, e2, n2 = oracle.moe_align(ids, E, bm)
    rows = valid_rows(ids, E)
    other = np.setdiff1d(np.arange(P), rows)
    ref = oracle.moe_gemm(x, topk, codes, scales, s2, e2, n2, bm, P, C=np.full((P, N), 0xFFFF, np.uint16))
    for mixed in (0, 1):
        got = host_bits(gemm(x, topk, packed, E, N, K, s, e, n, bm, P, kernel=TC, split_k=0, mixed=mixed,
                             tc_pairs=1))
        assert (got[other] == 0xFFFF).all(), "rows of non-local pairs were written"
        if exact:
            np.testing.assert_array_equal(got[rows], ref[rows])
        else:
            assert_close(got[rows], ref[rows], f"pairs bm={bm} K={K} mixed={mixed}")
    C = torch.full((P, N), float("nan"), dtype=torch.float32, device=DEV)
    gemm(x, topk, packed, E, N, K, s, e, n, bm, P, kernel=TC, C=C, split_k=0, out_dtype=chord.DTYPE_F32, tc_pairs=1)
    got32 = C.cpu().numpy()
    ref32 = oracle.moe_gemm_f32(x, topk, codes, scales, s2, e2, n2, bm, P)
    if exact:
        np.testing.assert_array_equal(got32[rows], ref32[rows])
    else:
        err = np.abs(got32[rows].astype(np.float64) - ref32[rows])
        assert (err <= 1e-2 + 1e-2 * np.abs(ref32[rows])).all(), err.max()
    # the fused SiLU * up epilogue (layout 3), against this library's SiLU * up of the pairs' C1
    I = N // 2
    h = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    gemm(x, topk, pack(codes, scales, chord.LAYOUT_GATE_UP_INTERLEAVED), E, N, K, s, e, n, bm, P, kernel=TC, C=h,
         split_k=0, epilogue=chord.EPILOGUE_SILU_MUL, tc_pairs=1)
    C1 = gemm(x, topk, packed, E, N, K, s, e, n, bm, P, kernel=TC, split_k=0, tc_pairs=1)
    check_h_from_gpu_c1(host_bits(h), host_bits(C1), ref, ids.ravel(), E, rows, f"pairs fused bm={bm}")
    if exact:
        h2 = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
        chord.chord_silu_mul(C1, dev(ids.ravel().copy()), E, h2)
        np.testing.assert_array_equal(host_bits(h)[rows], host_bits(h2)[rows])
    assert chord.chord_get_device_error() == 0


def test_layer_tc_pairs_and_fused_combine():
    """A layer on the tcgen05 kernel in clusters of two CTAs, with the top-k
    combine fused into the down GEMM, checked through the chain of definitions
    against the oracle (its ABI steps with the same options give the same
    output bit for bit)."""
    T, topk, E, H, I, bm = 100, 8, 8, 1024, 1280, 256
    ids = wl.random_ids(40, T, topk, E, p_nonlocal=0.1)
    wts = wl.random_weights(41, T, topk)
    x = wl.random_bf16(42, (T, H))
    c13, s13 = wl.random_codes(43, (E, 2 * I, H)), wl.random_scales(44, (E, 2 * I, H // 32))
    c2, s2 = wl.random_codes(45, (E, H, I)), wl.random_scales(46, (E, H, I // 32))
    p13, p2 = pack(c13, s13), pack(c2, s2)
    out, _ = layer(x, ids, wts, E, E, I, p13, p2, bm=bm,
                   opts=chord.ChordOpts(kernel=TC, tc_pairs=1, fuse_combine=1))
    sep, _ = layer(x, ids, wts, E, E, I, p13, p2, bm=bm, opts=chord.ChordOpts(kernel=TC, tc_pairs=1))
    np.testing.assert_array_equal(host_bits(out), host_bits(sep))
    s, e, n = align(ids, E, bm)
    P = T * topk
    C1 = gemm(x, topk, p13, E, 2 * I, H, s, e, n, bm, P, kernel=TC, tc_pairs=1)
    h = torch.full((P, I), -1, dtype=torch.int16, device=DEV).view(torch.bfloat16)
    chord.chord_silu_mul(C1, dev(ids), E, h)
    C2 = torch.full((P, H), float("nan"), dtype=torch.float32, device=DEV)
    gemm(h, 1, p2, E, H, I, s, e, n, bm, P, kernel=TC, C=C2, out_dtype=chord.DTYPE_F32, tc_pairs=1)
    check_layer_chain(x, ids, wts, (c13, s13), (c2, s2), E, host_bits(C1), host_bits(h), C2.cpu().numpy(),
                      host_bits(out), "layer on CTA pairs")


# ------------------------------------------------- the layer replayed from a CUDA graph

def test_layer_cached_matches_eager_and_rereads_inputs():
    """chord_moe_layer_cached records the layer once per argument set and
    replays the graph: bit for bit the eager layer on calls whose input
    contents change at the same addresses (the replay reads the buffers
    anew), for two argument sets (each its own graph) used alternately, on
    another stream than the one it recorded on; validation is refused; the
    cache is cleared at the end."""
    chord.chord_moe_layer_cache_clear()
    cases = []
    for T, topk, E, H, I, fused in ((24, 4, 6, 256, 128, True), (40, 8, 6, 256, 256, False)):
        c13, s13 = wl.random_codes(T + 1, (E, 2 * I, H)), wl.random_scales(T + 2, (E, 2 * I, H // 32))
        c2, s2 = wl.random_codes(T + 3, (E, H, I)), wl.random_scales(T + 4, (E, H, I // 32))
        p13 = pack(c13, s13, chord.LAYOUT_GATE_UP_INTERLEAVED if fused else chord.LAYOUT_TCGEN05)
        p2 = pack(c2, s2)
        bm = 16
        ws = torch.empty(chord.chord_layer_workspace_bytes(T, topk, E, H, I, bm), dtype=torch.uint8, device=DEV)
        xd = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        idd = torch.empty((T, topk), dtype=torch.int32, device=DEV)
        wd = torch.empty((T, topk), dtype=torch.float32, device=DEV)
        out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
        opts = chord.ChordOpts(epilogue=chord.EPILOGUE_SILU_MUL if fused else chord.EPILOGUE_NONE)
        cases.append((T, topk, E, H, I, p13, p2, bm, ws, xd, idd, wd, out, opts))
    s = torch.cuda.Stream()
    for rnd in range(3):
        for (T, topk, E, H, I, p13, p2, bm, ws, xd, idd, wd, out, opts) in cases:
            ids = wl.random_ids(100 * rnd + T, T, topk, 4 * E)
            ids = np.where(ids < E, ids, -1).astype(np.int32)
            xd.copy_(dbf(wl.random_bf16(100 * rnd + T + 1, (T, H))))
            idd.copy_(dev(ids))
            wd.copy_(dev(wl.random_weights(100 * rnd + T + 2, T, topk)))
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                chord.chord_moe_layer_cached(xd, idd, wd, E, 4 * E, I, p13, p2, ws, out, block_m=bm, opts=opts,
                                             stream=s)
            s.synchronize()
            got = host_bits(out).copy()
            ref = torch.empty_like(out)
            chord.chord_moe_layer(xd, idd, wd, E, 4 * E, I, p13, p2, ws, ref, block_m=bm, opts=opts)
            torch.cuda.synchronize()
            np.testing.assert_array_equal(got, host_bits(ref))
    T, topk, E, H, I, p13, p2, bm, ws, xd, idd, wd, out, opts = cases[0]
    with pytest.raises(chord.ChordError) as ei:
        chord.chord_moe_layer_cached(xd, idd, wd, E, 4 * E, I, p13, p2, ws, out, block_m=bm,
                                     opts=chord.ChordOpts(validate=1))
    assert ei.value.status == 2
    assert chord.chord_moe_layer_cache_clear() == 2
    assert chord.chord_get_device_error() == 0
