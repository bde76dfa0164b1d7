"""Pins of the CPU oracle against things other than itself.

Every check compares the oracle with an independent source: a value printed on
the pages or derived by hand (tests/golden/), a library routine (torch's
float32 -> bf16 conversion, numpy integer and float64 matmul, scipy's expit,
Python's sort), exact integer arithmetic, a closed form, or an invariant.
Each test names the mistake it is there to catch.
"""
import numpy as np
import pytest
import torch
from scipy.special import expit

import workloads as wl
from conftest import read_golden

GROUP = 32


# --- independent helpers (library routines, not the oracle's code) --------

def to_bf16(f):
    """float32 values -> bf16 bits via torch's round-to-nearest-even conversion."""
    t = torch.from_numpy(np.ascontiguousarray(np.asarray(f, dtype=np.float32)))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f64(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16r(v):
    """Round float64 values to bf16 (through an exact-or-nearest float32) and widen."""
    return f64(to_bf16(np.asarray(v, np.float64).astype(np.float32)))


def dequant_ref(codes, scales):
    """(q - 8) * s in float64 (exact), rounded to bf16 by torch."""
    s = np.repeat(f64(scales), GROUP, axis=-1)
    return to_bf16(((codes.astype(np.float64) - 8.0) * s).astype(np.float32))


# --- bf16 rounding ----------------------------------------------------------

def test_bf16_round_page_example(orc):
    """Worked example of the rounding table on the MI355X page: 256.5 -> 256."""
    rows = read_golden("bf16_rounding.txt")
    for r in rows:
        if len(r) == 2:
            assert orc.bf16_round(float(r[0])) == int(r[1], 16)
        else:
            a, b, d_fp32, d_bf16 = map(float, r)
            assert np.float32(a) - np.float32(b) == d_fp32
            assert f64([orc.bf16_round(a)])[0] - f64([orc.bf16_round(b)])[0] == d_bf16


def test_bf16_round_matches_torch(orc):
    """Catches a wrong tie rule, a truncation, or mishandled subnormals/overflow."""
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # add exact ties, near-ties, subnormals, overflow boundary, infinities
    extra = [0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001, 0x00008000, 0x00018000,
             0x7F7FFFFF, 0x7F7F7FFF, 0x7F7F8000, 0xFF7F8000, 0x7F800000, 0xFF800000, 0, 0x80000000]
    bits = np.concatenate([bits, np.array(extra, np.uint32)])
    vals = bits.view(np.float32)
    vals = vals[~np.isnan(vals)]
    want = to_bf16(vals)
    got = np.array([orc.bf16_round(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, want)


# --- dequantisation ---------------------------------------------------------

def test_dequant_closed_forms(orc):
    for q, s, want, *_ in read_golden("dequant_closed_forms.txt"):
        assert orc.dequant(int(q), int(s, 16)) == int(want, 16), (q, s)


def test_dequant_exhaustive(orc):
    """All 16 codes x all 65536 bf16 scale patterns against an exact float64
    product rounded by torch.  Catches a missing offset, add-instead-of-subtract,
    scale-then-subtract order, double rounding, a wrong NaN/Inf path."""
    q = np.repeat(np.arange(16, dtype=np.uint8), 65536)
    s = np.tile(np.arange(65536, dtype=np.uint32).astype(np.uint16), 16)
    got = orc.dequant_pairs(q, s)
    prod = (q.astype(np.float64) - 8.0) * f64(s)
    with np.errstate(invalid="ignore", over="ignore"):
        want = to_bf16(prod.astype(np.float32))
    nan_g = np.isnan(f64(got))
    nan_w = np.isnan(f64(want))
    np.testing.assert_array_equal(nan_g, nan_w)
    np.testing.assert_array_equal(got[~nan_w], want[~nan_w])


# --- packing ----------------------------------------------------------------

def test_packed_bytes_closed_form(orc):
    for E, N, K in [(1, 128, 64), (8, 256, 256), (8, 256, 128), (48, 4096, 7168), (384, 7168, 256)]:
        for layout in (1, 2, 3):
            assert orc.packed_bytes(E, N, K, layout) == 256 + E * N * K * 9 // 16
    for bad in [(1, 8, 64, 1), (1, 16, 32, 1), (1, 0, 64, 1), (1, 16, 64, 2), (1, 128, 96, 2), (1, 64, 64, 3),
                (1, 128, 64, 4)]:
        assert orc.packed_bytes(*bad) == 0


@pytest.mark.parametrize("layout", [1, 2, 3])
def test_pack_header(orc, layout):
    codes = wl.random_codes(1, (3, 128, 128))
    scales = wl.random_scales(2, (3, 128, 4))
    blob = orc.pack(codes, scales, layout)
    h = blob[:256]
    u32 = h[:32].view(np.uint32)
    assert bytes(h[:4]) == b"CHRD"
    # word 7: every random scale (|N(0, 0.02)| + 1e-3) is a positive normal bf16 below 0.5
    assert list(u32[1:8]) == [1, layout, 32, 3, 128, 128, 1]
    assert list(h[32:48].view(np.uint64)) == [128 * 128 * 9 // 16, 256]
    assert not h[48:].any()
    assert orc.check_header(blob, 3, 128, 128, layout)
    for other in {1, 2, 3} - {layout}:
        assert not orc.check_header(blob, 3, 128, 128, other)
    assert not orc.check_header(blob, 3, 64, 256, layout)


# (one scale planted among scales of 2^-7, header word 7 expected): the bf16
# bit patterns by hand — 0.5 = 0x3F00 (exponent 126), the largest bf16 below
# 0.5 = 0x3EFF (exponent 125, mantissa 127), the smallest normal 2^-126 =
# 0x0080, 2^-127 is subnormal (0x0040).
SCALE_RANGE_CASES = [(0x3C00, 1), (0x3EFF, 1), (0x0080, 1), (0x3F00, 0), (0x3F80, 0), (0x0040, 0), (0x0000, 0),
                     (0x8000, 0), (0xBC00, 0), (0x8080, 0), (0x7F80, 0), (0x7FC0, 0)]


@pytest.mark.parametrize("layout", [1, 2, 3])
@pytest.mark.parametrize("planted,flag", SCALE_RANGE_CASES)
def test_pack_header_scale_range(orc, layout, planted, flag):
    """Header word 7 is 1 exactly when every scale lies in [2^-126, 0.5) and is
    positive; one planted scale anywhere decides it, and nothing else in the
    blob depends on it (codes and scales unpack unchanged)."""
    assert wl._bf16(np.array([0.5, 0.498046875, 2.0 ** -126, 2.0 ** -127, 2.0 ** -7], np.float32)).tolist() == [
        0x3F00, 0x3EFF, 0x0080, 0x0040, 0x3C00]
    codes = wl.random_codes(3, (2, 128, 128))
    scales = np.full((2, 128, 4), 0x3C00, np.uint16)
    scales[1, 77, 2] = planted
    blob = orc.pack(codes, scales, layout)
    assert int(blob[28:32].view(np.uint32)[0]) == flag
    c2, s2 = orc.unpack(blob, 2, 128, 128, layout)
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(s2, scales)


@pytest.mark.parametrize("layout,N,K", [(1, 32, 128), (2, 256, 128), (3, 256, 128)])
def test_pack_positions_golden(orc, layout, N, K):
    """Hand-derived byte/nibble positions of each layout's specification."""
    E = 1
    for r in read_golden(f"layout_v{layout}_positions.txt"):
        codes = np.zeros((E, N, K), np.uint8)
        scales = np.zeros((E, N, K // GROUP), np.uint16)
        if len(r) == 4:
            n, k, off, sh = map(int, r)
            codes[0, n, k] = 0xF
            data = orc.pack(codes, scales, layout)[256:]
            nz = np.nonzero(data)[0]
            assert list(nz) == [off], (n, k, list(nz))
            assert data[off] == (0xF << sh), (n, k)
        else:
            n, grp, off = map(int, r)
            scales[0, n, grp] = 0xABCD
            data = orc.pack(codes, scales, layout)[256:]
            assert list(np.nonzero(data)[0]) == [off, off + 1], (n, grp)
            assert data[off] == 0xCD and data[off + 1] == 0xAB


@pytest.mark.parametrize("layout,shape", [(1, (1, 16, 64)), (1, (3, 32, 128)), (1, (2, 256, 256)),
                                          (1, (2, 128, 192)), (2, (1, 128, 64)), (2, (2, 256, 192)),
                                          (2, (1, 384, 128)), (3, (1, 128, 64)), (3, (2, 256, 192)),
                                          (3, (1, 512, 128))])
def test_pack_roundtrip_and_coverage(orc, layout, shape):
    """unpack(pack(x)) == x for random data, and all-ones data fills the data region
    completely: together the placement is a bijection (no overlap, no gap)."""
    E, N, K = shape
    codes = wl.random_codes(3, shape)
    scales = wl.random_scales(4, (E, N, K // GROUP))
    blob = orc.pack(codes, scales, layout)
    c2, s2 = orc.unpack(blob, E, N, K, layout)
    np.testing.assert_array_equal(c2, codes)
    np.testing.assert_array_equal(s2, scales)
    full = orc.pack(np.full(shape, 15, np.uint8), np.full((E, N, K // GROUP), 0xFFFF, np.uint16), layout)
    assert (full[256:] == 0xFF).all()
    assert full.size == 256 + E * N * K * 9 // 16


def test_layout3_is_layout2_of_interleaved_rows(orc):
    """Layout 3 of a gate_up weight equals layout 2 of the same weight with its
    rows reordered gate 0-7, up 0-7, gate 8-15, up 8-15, ... (except for the
    layout word of the header)."""
    E, N, K = 2, 256, 128
    codes = wl.random_codes(5, (E, N, K))
    scales = wl.random_scales(6, (E, N, K // GROUP))
    I = N // 2
    order = np.concatenate([np.concatenate([np.arange(8 * g, 8 * g + 8), I + np.arange(8 * g, 8 * g + 8)])
                            for g in range(I // 8)])
    b3 = orc.pack(codes, scales, 3)
    b2 = orc.pack(codes[:, order], scales[:, order], 2)
    assert b3[8] == 3 and b2[8] == 2
    np.testing.assert_array_equal(b3[12:], b2[12:])


def test_pack_rejects_bad_codes_and_header(orc):
    codes = np.zeros((1, 128, 64), np.uint8)
    codes[0, 3, 5] = 16
    with pytest.raises(orc.OracleError):
        orc.pack(codes, np.zeros((1, 128, 2), np.uint16))
    blob = orc.pack(np.zeros((1, 128, 64), np.uint8), np.zeros((1, 128, 2), np.uint16))
    blob[0] ^= 1
    with pytest.raises(orc.OracleError):
        orc.unpack(blob, 1, 128, 64)
    blob = orc.pack(np.zeros((1, 128, 64), np.uint8), np.zeros((1, 128, 2), np.uint16), 2)
    with pytest.raises(orc.OracleError):
        orc.unpack(blob, 1, 128, 64, 1)


# --- align ------------------------------------------------------------------

def align_by_sort(ids, E, bm):
    """Independent construction with Python's sort over (expert, pair id)."""
    T, topk = ids.shape
    P = T * topk
    pairs = sorted((int(e), p) for p, e in enumerate(ids.ravel()) if 0 <= e < E)
    sorted_ids, expert_ids = [], []
    i = 0
    while i < len(pairs):
        e = pairs[i][0]
        seg = []
        while i < len(pairs) and pairs[i][0] == e:
            seg.append(pairs[i][1])
            i += 1
        while len(seg) % bm:
            seg.append(P)
        sorted_ids += seg
        expert_ids += [e] * (len(seg) // bm)
    ntp = len(sorted_ids)
    cap = -(-(P + min(E, P) * (bm - 1)) // bm) * bm
    sorted_ids += [P] * (cap - ntp)
    expert_ids += [-1] * (cap // bm - len(expert_ids))
    return np.array(sorted_ids, np.int32), np.array(expert_ids, np.int32), ntp


@pytest.mark.parametrize("T,topk,E,bm,pnl", [(16, 2, 8, 4, 0.0), (33, 8, 48, 16, 0.5), (7, 3, 5, 1, 0.2),
                                             (64, 8, 384, 8, 0.0), (1, 8, 384, 16, 0.0),
                                             (128, 4, 6, 64, 0.3), (200, 6, 12, 256, 0.1)])
def test_align_vs_sort(orc, T, topk, E, bm, pnl):
    ids = wl.random_ids(T * 31 + E, T, topk, E, p_nonlocal=pnl)
    s, e, ntp = orc.moe_align(ids, E, bm)
    s2, e2, ntp2 = align_by_sort(ids, E, bm)
    assert ntp == ntp2
    np.testing.assert_array_equal(s, s2)
    np.testing.assert_array_equal(e, e2)


def test_align_edge_counts(orc):
    """Experts with 0, 1, 2, bm-1, bm, bm+1 rows; ids >= E and -1 are dropped."""
    bm = 8
    counts = {0: 0, 1: 1, 2: 2, 3: bm - 1, 4: bm, 5: bm + 1}
    E = 6
    flat = []
    for e, c in counts.items():
        flat += [e] * c
    flat += [-1, -1, E, E + 3]
    rng = np.random.default_rng(0)
    flat = np.array(flat, np.int32)[rng.permutation(len(flat))]
    if flat.size % 2:
        flat = np.append(flat, -1)
    ids = flat.astype(np.int32).reshape(-1, 2)
    s, e, ntp = orc.moe_align(ids, E, bm)
    P = ids.size
    want_ntp = sum(-(-c // bm) * bm for c in counts.values())
    assert ntp == want_ntp
    s2, e2, _ = align_by_sort(ids, E, bm)
    np.testing.assert_array_equal(s, s2)
    np.testing.assert_array_equal(e, e2)
    assert 0 not in e[: ntp // bm]
    assert (s[ntp:] == P).all()


def test_align_empty_and_all_nonlocal(orc):
    s, e, ntp = orc.moe_align(np.zeros((0, 8), np.int32), 48, 16)
    assert ntp == 0 and s.size == 0 and e.size == 0
    ids = np.full((5, 4), -1, np.int32)
    s, e, ntp = orc.moe_align(ids, 8, 4)
    assert ntp == 0 and (s == 20).all() and (e == -1).all()
    assert s.size == orc.align_capacity(5, 4, 8, 4)


def test_align_invariants_large(orc):
    """Every local pair exactly once, each segment ascending, padding only at
    segment ends, capacity formula."""
    w = wl.EP8_DECODE
    ids, _ = wl.make_routing(w)
    bm = 16
    s, e, ntp = orc.moe_align(ids, w.E, bm)
    P = w.P
    assert s.size == -(-(P + min(P, w.E) * (bm - 1)) // bm) * bm
    local = np.nonzero((ids.ravel() >= 0) & (ids.ravel() < w.E))[0]
    valid = s[:ntp][s[:ntp] != P]
    np.testing.assert_array_equal(np.sort(valid), local)
    for b in range(ntp // bm):
        blk = s[b * bm:(b + 1) * bm]
        v = blk[blk != P]
        assert (ids.ravel()[v] == e[b]).all()
        assert (np.diff(v) > 0).all()
        if v.size < bm:
            assert (blk[v.size:] == P).all()
    assert (np.diff(e[: ntp // bm]) >= 0).all()


# --- GEMM -------------------------------------------------------------------

def _gemm_via_align(orc, A, div, codes, scales, ids, bm=8):
    E = codes.shape[0]
    s, e, ntp = orc.moe_align(ids, E, bm)
    C = np.full((ids.size, codes.shape[1]), 0xFFFF, np.uint16)
    return orc.moe_gemm(A, div, codes, scales, s, e, ntp, bm, ids.size, C)


@pytest.mark.parametrize("K", [256, 2048])
def test_gemm_exact_integer_regime(orc, K):
    """x in {-1,0,1}, scale 1: every partial sum is an integer below 2^24, so the
    result is exact in any order; compare with numpy's integer matmul.  Catches a
    wrong sign, a transposed operand, a wrong row index or a dropped term."""
    T, topk, E, N = 12, 2, 3, 48
    rng = np.random.default_rng(K)
    xi = rng.integers(-1, 2, size=(T, K))
    x = to_bf16(xi.astype(np.float32))
    codes = wl.random_codes(K + 1, (E, N, K))
    scales = np.full((E, N, K // GROUP), 0x3F80, np.uint16)
    ids = wl.random_ids(K + 2, T, topk, E, p_nonlocal=0.25)
    C = _gemm_via_align(orc, x, topk, codes, scales, ids)
    Wi = codes.astype(np.int64) - 8
    for p in range(T * topk):
        e = ids.ravel()[p]
        if e < 0:
            assert (C[p] == 0xFFFF).all()
            continue
        exact = Wi[e] @ xi[p // topk]
        np.testing.assert_array_equal(C[p], to_bf16(exact.astype(np.float32)))


def test_grouped_contiguous_exact_integer_and_padding(orc):
    """Grouped contiguous: x in {-1,0,1}, scale 1, against numpy's integer
    matmul row by row with the row's own expert; padding rows (m_indices -1)
    keep the fill pattern.  Segments of 128 rows per expert, one expert empty."""
    K, N, E = 256, 48, 4
    counts = [70, 0, 128, 5]
    m_idx = np.concatenate([np.concatenate([np.full(c, e), np.full(-(-c // 128) * 128 - c, -1)])
                            for e, c in enumerate(counts)]).astype(np.int32)
    M = m_idx.size
    rng = np.random.default_rng(7)
    xi = rng.integers(-1, 2, size=(M, K))
    x = to_bf16(xi.astype(np.float32))
    codes = wl.random_codes(8, (E, N, K))
    scales = np.full((E, N, K // GROUP), 0x3F80, np.uint16)
    C = orc.grouped_contiguous(x, m_idx, codes, scales, C=np.full((M, N), 0xFFFF, np.uint16))
    Wi = codes.astype(np.int64) - 8
    for m in range(M):
        if m_idx[m] < 0:
            assert (C[m] == 0xFFFF).all(), m
        else:
            np.testing.assert_array_equal(C[m], to_bf16((Wi[m_idx[m]] @ xi[m]).astype(np.float32)))


def test_grouped_masked_exact_integer_and_budget(orc):
    """Grouped masked: group g's first masked_m[g] rows against numpy's integer
    matmul with expert g (flat output row g * max_m + r); rows past the count
    keep the fill pattern, including a group with no rows and a full one."""
    K, N, G, max_m = 128, 32, 4, 9
    masked_m = np.array([3, 0, 9, 1], np.int32)
    rng = np.random.default_rng(9)
    xi = rng.integers(-1, 2, size=(G, max_m, K))
    x = to_bf16(xi.astype(np.float32))
    codes = wl.random_codes(10, (G, N, K))
    scales = np.full((G, N, K // GROUP), 0x3F80, np.uint16)
    C = orc.grouped_masked(x, masked_m, codes, scales, C=np.full((G * max_m, N), 0xFFFF, np.uint16))
    Wi = codes.astype(np.int64) - 8
    for g in range(G):
        for r in range(max_m):
            row = C[g * max_m + r]
            if r >= masked_m[g]:
                assert (row == 0xFFFF).all(), (g, r)
            else:
                np.testing.assert_array_equal(row, to_bf16((Wi[g] @ xi[g, r]).astype(np.float32)))


def test_grouped_contracts_match_indexed_gemm(orc):
    """With real-valued data both grouped contracts equal the indexed GEMM given
    the equivalent routing (one row per pair, block size 8), bit for bit: same
    dequantisation, same sequential sums."""
    K, N, E = 320, 64, 3
    codes = wl.random_codes(11, (E, N, K))
    scales = wl.random_scales(12, (E, N, K // GROUP))
    m_idx = np.array([0] * 5 + [-1] * 3 + [2] * 8 + [1] * 2 + [-1] * 6, np.int32)
    x = wl.random_bf16(13, (m_idx.size, K))
    got = orc.grouped_contiguous(x, m_idx, codes, scales)
    ids = m_idx.reshape(-1, 1)
    want = _gemm_via_align(orc, x, 1, codes, scales, ids)
    rows = m_idx >= 0
    np.testing.assert_array_equal(got[rows], want[rows])
    masked_m = np.array([4, 0, 7], np.int32)
    x3 = wl.random_bf16(14, (E, 7, K))
    got3 = orc.grouped_masked(x3, masked_m, codes, scales)
    ids3 = np.array([[g if r < masked_m[g] else -1] for g in range(E) for r in range(7)], np.int32)
    want3 = _gemm_via_align(orc, x3.reshape(-1, K), 1, codes, scales, ids3)
    rows3 = ids3.ravel() >= 0
    np.testing.assert_array_equal(got3[rows3], want3[rows3])


def test_gemm_identity(orc):
    """Code 9 on the diagonal, 8 elsewhere, scale 1: W = I, so C = x exactly."""
    T, topk, E, K = 5, 2, 2, 64
    codes = np.full((E, K, K), 8, np.uint8)
    for e in range(E):
        np.fill_diagonal(codes[e], 9)
    scales = np.full((E, K, K // GROUP), 0x3F80, np.uint16)
    x = wl.random_bf16(11, (T, K))
    ids = wl.random_ids(12, T, topk, E)
    C = _gemm_via_align(orc, x, topk, codes, scales, ids, bm=4)
    for p in range(T * topk):
        np.testing.assert_array_equal(C[p], x[p // topk])
    # one row per pair (down projection): A indexed by pair id directly
    A = wl.random_bf16(13, (T * topk, K))
    C = _gemm_via_align(orc, A, 1, codes, scales, ids, bm=4)
    np.testing.assert_array_equal(C, A)


def test_gemm_float_bound(orc):
    """Random data against a float64 matmul of independently dequantised
    weights: |C - ref| <= half a bf16 ulp of ref plus the FP32 summation bound
    K * 2^-24 * sum|x*w|.  Catches a wrong group index (scales differ per
    group), a wrong expert, an off-by-one in K."""
    T, topk, E, N, K = 9, 3, 4, 64, 320
    x = wl.random_bf16(21, (T, K))
    codes = wl.random_codes(22, (E, N, K))
    scales = wl.random_scales(23, (E, N, K // GROUP))
    ids = wl.random_ids(24, T, topk, E, p_nonlocal=0.2)
    C = _gemm_via_align(orc, x, topk, codes, scales, ids)
    W = f64(dequant_ref(codes, scales))
    X = f64(x)
    for p in range(T * topk):
        e = ids.ravel()[p]
        if e < 0:
            continue
        ref = W[e] @ X[p // topk]
        mag = np.abs(W[e]) @ np.abs(X[p // topk])
        tol = np.abs(ref) * 2.0 ** -8 + K * 2.0 ** -24 * mag + 1e-30
        assert (np.abs(f64(C[p]) - ref) <= tol).all()


def test_gemm_f32_exact_integer_and_bf16_consistency(orc):
    """FP32 output: in the exact-integer regime it equals numpy's integer
    matmul exactly (no rounding at all), and rounding it with torch gives the
    bf16-output GEMM bit for bit (same sum, one rounding)."""
    T, topk, E, N, K = 10, 3, 4, 64, 512
    rng = np.random.default_rng(5)
    xi = rng.integers(-1, 2, size=(T, K))
    x = to_bf16(xi.astype(np.float32))
    codes = wl.random_codes(6, (E, N, K))
    ones = np.full((E, N, K // GROUP), 0x3F80, np.uint16)
    ids = wl.random_ids(7, T, topk, E, p_nonlocal=0.2)
    s, e, ntp = orc.moe_align(ids, E, 8)
    Cf = orc.moe_gemm_f32(x, topk, codes, ones, s, e, ntp, 8, T * topk)
    for p in range(T * topk):
        if ids.ravel()[p] >= 0:
            exact = (codes[ids.ravel()[p]].astype(np.int64) - 8) @ xi[p // topk]
            np.testing.assert_array_equal(Cf[p], exact.astype(np.float32))
    x = wl.random_bf16(8, (T, K))
    scales = wl.random_scales(9, (E, N, K // GROUP))
    Cf = orc.moe_gemm_f32(x, topk, codes, scales, s, e, ntp, 8, T * topk)
    Cb = orc.moe_gemm(x, topk, codes, scales, s, e, ntp, 8, T * topk, C=np.zeros((T * topk, N), np.uint16))
    rows = np.nonzero(ids.ravel() >= 0)[0]
    np.testing.assert_array_equal(to_bf16(Cf[rows]), Cb[rows])


def test_combine_f32_one_hot_and_bound(orc):
    """FP32 input: a one-hot weight gives bf16(C2 row) (torch rounding); a
    general case stays within the FP32 bound of a float64 sum."""
    T, topk, E, H = 7, 4, 5, 96
    rng = np.random.default_rng(10)
    C2 = (rng.standard_normal((T * topk, H)) * 100).astype(np.float32)
    ids = wl.random_ids(11, T, topk, E)
    w = np.zeros((T, topk), np.float32)
    pick = rng.integers(0, topk, size=T)
    w[np.arange(T), pick] = 1.0
    out = orc.combine(C2, ids, w, E)
    for t in range(T):
        np.testing.assert_array_equal(out[t], to_bf16(C2[t * topk + pick[t]]))
    w = wl.random_weights(12, T, topk)
    out = f64(orc.combine(C2, ids, w, E))
    Y = C2.astype(np.float64).reshape(T, topk, H)
    ref = (w.astype(np.float64)[:, :, None] * Y).sum(1)
    mag = (np.abs(w.astype(np.float64))[:, :, None] * np.abs(Y)).sum(1)
    assert (np.abs(out - ref) <= np.abs(ref) * 2.0 ** -8 + topk * 2.0 ** -23 * mag).all()


# --- activation -------------------------------------------------------------

def test_silu_mul_vs_expit(orc):
    """silu(g) * u against scipy's expit in float64: catches swapped gate/up
    halves, a missing factor g, exp(+g) instead of exp(-g)."""
    P, I, E = 40, 96, 4
    C1 = wl.random_bf16(31, (P, 2 * I), std=3.0)
    ids = wl.random_ids(32, P, 1, E, p_nonlocal=0.2).ravel()
    h = np.full((P, I), 0xFFFF, np.uint16)
    h = orc.silu_mul(C1, ids, E, h)
    g, u = f64(C1[:, :I]), f64(C1[:, I:])
    ref = g * expit(g) * u
    for p in range(P):
        if ids[p] < 0:
            assert (h[p] == 0xFFFF).all()
            continue
        err = np.abs(f64(h[p]) - ref[p])
        assert (err <= np.abs(ref[p]) * 2.0 ** -7 + 1e-30).all()


def test_silu_mul_closed_forms(orc):
    g = np.array([0.0, 100.0, -100.0, 2.0, 5.0], np.float32)
    u = np.array([3.0, 0.5, 4.0, 0.0, -1.0], np.float32)
    C1 = np.concatenate([to_bf16(g), to_bf16(u)])[None, :]
    h = f64(orc.silu_mul(C1, np.zeros(1, np.int32), 1)[0])
    assert h[0] == 0.0                      # silu(0) = 0
    assert h[1] == f64(to_bf16([100.0 * 0.5]))[0]   # silu(g) -> g for large g
    assert h[2] == 0.0                      # silu(g) -> 0 for very negative g
    assert h[3] == 0.0                      # u = 0
    assert h[4] == f64(to_bf16([-5.0 * expit(5.0)]))[0]


# --- combine ----------------------------------------------------------------

def test_combine_one_hot_and_nonlocal(orc):
    """A one-hot weight reproduces that pair's row exactly; tokens with no local
    pair give +0; non-local pairs never contribute even with a weight."""
    T, topk, E, H = 6, 4, 5, 64
    C2 = wl.random_bf16(41, (T * topk, H))
    ids = wl.random_ids(42, T, topk, E)
    ids[5, :] = -1
    w = np.zeros((T, topk), np.float32)
    pick = np.array([0, 1, 2, 3, 1, 0])
    w[np.arange(T), pick] = 1.0
    ids[2, 0] = -1            # weight on a non-local pair must not count
    w[2, 0] = 5.0
    out = orc.combine(C2, ids, w, E)
    for t in range(5):
        np.testing.assert_array_equal(out[t], C2[t * topk + pick[t]])
    assert (out[5] == 0).all()


def test_combine_float_bound(orc):
    T, topk, E, H = 10, 8, 16, 128
    C2 = wl.random_bf16(51, (T * topk, H), std=50.0)
    ids = wl.random_ids(52, T, topk, E, p_nonlocal=0.3)
    w = wl.random_weights(53, T, topk)
    out = f64(orc.combine(C2, ids, w, E))
    Y = f64(C2).reshape(T, topk, H)
    mask = (ids >= 0)[:, :, None]
    ref = (w.astype(np.float64)[:, :, None] * Y * mask).sum(1)
    mag = (np.abs(w.astype(np.float64))[:, :, None] * np.abs(Y) * mask).sum(1)
    assert (np.abs(out - ref) <= np.abs(ref) * 2.0 ** -8 + topk * 2.0 ** -23 * mag + 1e-30).all()


# --- layer ------------------------------------------------------------------

def layer_dense_reference(x, ids, w, c13, s13, c2, s2, E):
    """Dense per-token loop over each token's experts in float64, with bf16
    rounding (torch) after gate_up and after SiLU*up; the down result enters
    the weighted sum unrounded and the output is rounded once."""
    W13 = f64(dequant_ref(c13, s13))
    W2 = f64(dequant_ref(c2, s2))
    X = f64(x)
    T, topk = ids.shape
    I = c2.shape[2]
    out = np.zeros((T, X.shape[1]))
    for t in range(T):
        acc = np.zeros(X.shape[1])
        for k in range(topk):
            e = ids[t, k]
            if not 0 <= e < E:
                continue
            gu = bf16r(W13[e] @ X[t])
            h = bf16r(gu[:I] * expit(gu[:I]) * gu[I:])
            y = W2[e] @ h
            acc += float(w[t, k]) * y
        out[t] = bf16r(acc)
    return out


def test_layer_tiny_vs_dense_loop(orc):
    w = wl.TINY
    ids, wts = wl.make_routing(w)
    x = wl.make_x(w)
    c13, s13 = wl.make_w13(w)
    c2, s2 = wl.make_w2(w)
    got = f64(orc.moe_layer(x, ids, wts, (c13, s13), (c2, s2), w.E, block_m=4))
    ref = layer_dense_reference(x, ids, wts, c13, s13, c2, s2, w.E)
    err = np.abs(got - ref)
    assert (err <= 1e-2 + 1e-2 * np.abs(ref)).all(), err.max()
    # the two differ only by FP32-vs-FP64 summation order near rounding ties
    assert np.mean(got == ref) > 0.9


def test_layer_block_m_invariance(orc):
    """The layer result does not depend on the align block size."""
    w = wl.TINY
    ids, wts = wl.make_routing(w)
    x = wl.make_x(w)
    w13, w2 = wl.make_w13(w), wl.make_w2(w)
    a = orc.moe_layer(x, ids, wts, w13, w2, w.E, block_m=1)
    b = orc.moe_layer(x, ids, wts, w13, w2, w.E, block_m=16)
    np.testing.assert_array_equal(a, b)


# --- the binary64-sum variant -----------------------------------------------
# A second valid evaluation of the same definitions (dot products and the
# weighted sum in binary64, bf16 at the same rounding points).  Pinned against
# exact rational arithmetic (Python's fractions: every bf16 and binary32 value
# is a dyadic rational, so sums of their products are exact there) and against
# a hand-worked table of one-rounding cases.

from fractions import Fraction  # noqa: E402


def bf16_rne_exact(fr):
    """bf16 bits of the exact rational `fr`, rounded once to nearest even
    (normal range): pure integer arithmetic, independent of the oracle."""
    if fr == 0:
        return 0
    sign = 0x8000 if fr < 0 else 0
    m = abs(fr)
    e = m.numerator.bit_length() - m.denominator.bit_length()
    if Fraction(2) ** e > m:
        e -= 1
    if m >= Fraction(2) ** (e + 1):
        e += 1
    assert -126 <= e <= 127
    ulp = Fraction(2) ** (e - 7)
    q = m / ulp
    n = q.numerator // q.denominator
    r = q - n
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and n % 2 == 1):
        n += 1
    val = n * ulp
    return sign | int(np.array([float(val)], np.float32).view(np.uint32)[0] >> 16)


def test_bf16_round_f64_hand_table(orc):
    """One rounding from binary64, including values that a binary32 step would
    put exactly on a midpoint (catches rounding through binary32 twice)."""
    for r in read_golden("bf16_round_f64.txt"):
        v = float.fromhex(r[0]) if "0x" in r[0] else float(r[0])
        assert orc.bf16_round_f64(v) == int(r[1], 16), r
        assert bf16_rne_exact(Fraction(v)) == int(r[1], 16), r


def test_bf16_round_f64_matches_exact_rounding(orc):
    """Random binary64 values, and values a few binary64 ulps from bf16
    midpoints, against the exact rounding of the rational value."""
    rng = np.random.default_rng(11)
    vals = list(rng.standard_normal(2000) * 10.0 ** rng.integers(-20, 20, 2000))
    lo = rng.integers(0x0080, 0x7f00, 500, dtype=np.uint16)
    mids = ((f64(lo) + f64(lo + 1)) / 2.0).tolist()   # midpoints of neighbouring bf16 values (exact in binary64)
    for m in mids:
        vals += [np.nextafter(m, np.inf), m, np.nextafter(m, -np.inf), -m]
    for v in vals:
        assert orc.bf16_round_f64(float(v)) == bf16_rne_exact(Fraction(float(v))), v


def _small_gemm_case(seed, T=5, topk=2, E=2, N=16, K=256):
    x = wl.random_bf16(seed, (T, K))
    codes = wl.random_codes(seed + 1, (E, N, K))
    scales = wl.random_scales(seed + 2, (E, N, K // GROUP))
    ids = wl.random_ids(seed + 3, T, topk, E, p_nonlocal=0.2)
    return x, codes, scales, ids


def test_gemm_f64sum_against_exact_sums(orc):
    """Every output of the binary64-sum GEMM is the exact sum rounded once to
    bf16 (fractions), and its binary64 output is within the binary64
    summation bound K * 2^-53 * sum|x w| of the exact sum.  Catches a binary32
    accumulator, a second rounding, or a dropped / shifted term."""
    x, codes, scales, ids = _small_gemm_case(21)
    T, K = x.shape
    E, N, _ = codes.shape
    topk = ids.shape[1]
    P = T * topk
    s, e, n = orc.moe_align(ids, E, 4)
    got = orc.moe_gemm_f64sum(x, topk, codes, scales, s, e, n, 4, P, C=np.zeros((P, N), np.uint16))
    got64 = orc.moe_gemm_f64(x, topk, codes, scales, s, e, n, 4, P)
    W = f64(dequant_ref(codes, scales))
    X = f64(x)
    checked = 0
    for p in range(P):
        ex = ids.ravel()[p]
        if ex < 0:
            continue
        t = p // topk
        for j in range(N):
            terms = [Fraction(float(X[t, k])) * Fraction(float(W[ex, j, k])) for k in range(K)]
            exact = sum(terms, Fraction(0))
            assert got[p, j] == bf16_rne_exact(exact), (p, j)
            bound = K * 2.0 ** -53 * float(sum(abs(a) for a in terms))
            assert abs(Fraction(float(got64[p, j])) - exact) <= Fraction(bound), (p, j)
            checked += 1
    assert checked > 100


def test_gemm_f64sum_cancellation(orc):
    """x = (2^24, 1, -2^24, 0, ...) against unit weights: the exact sum is 1.
    A binary32 sum in ascending k loses the 1 (2^24 + 1 rounds to 2^24); the
    binary64 sum keeps it.  Catches a binary32 accumulator in the variant."""
    K, N, E = 64, 16, 1
    x = np.zeros((1, K), np.uint16)
    x[0, 0], x[0, 1], x[0, 2] = to_bf16([2.0 ** 24, 1.0, -(2.0 ** 24)])
    codes = np.full((E, N, K), 9, np.uint8)                # q - 8 = 1
    scales = np.full((E, N, K // GROUP), 0x3F80, np.uint16)  # 1.0
    ids = np.zeros((1, 1), np.int32)
    s, e, n = orc.moe_align(ids, E, 1)
    v64 = orc.moe_gemm_f64sum(x, 1, codes, scales, s, e, n, 1, 1, C=np.zeros((1, N), np.uint16))
    v32 = orc.moe_gemm(x, 1, codes, scales, s, e, n, 1, 1, C=np.zeros((1, N), np.uint16))
    assert (v64 == 0x3F80).all() and (v32 == 0).all()
    d64 = orc.moe_gemm_f64(x, 1, codes, scales, s, e, n, 1, 1)
    assert (d64 == 1.0).all()


def test_gemm_f64sum_exact_integer_regime_equals_plain(orc):
    """x in {-1, 0, 1}, scale 1, K = 2048: every partial sum is an integer
    below 2^24, so both evaluations are exact and agree bit for bit."""
    rng = np.random.default_rng(3)
    T, topk, E, N, K = 6, 2, 3, 32, 2048
    x = to_bf16(rng.integers(-1, 2, (T, K)).astype(np.float32))
    codes = wl.random_codes(5, (E, N, K))
    scales = np.full((E, N, K // GROUP), 0x3F80, np.uint16)
    ids = wl.random_ids(6, T, topk, E)
    s, e, n = orc.moe_align(ids, E, 8)
    a = orc.moe_gemm(x, topk, codes, scales, s, e, n, 8, T * topk, C=np.zeros((T * topk, N), np.uint16))
    b = orc.moe_gemm_f64sum(x, topk, codes, scales, s, e, n, 8, T * topk, C=np.zeros((T * topk, N), np.uint16))
    np.testing.assert_array_equal(a, b)


def test_combine_f64_against_exact_sums(orc):
    """The binary64 weighted sum over local k, rounded once: against exact
    fractions of w * C2 (C2 binary64 values with many significant bits)."""
    rng = np.random.default_rng(8)
    T, topk, E, H = 6, 4, 5, 16
    ids = wl.random_ids(9, T, topk, E, p_nonlocal=0.3)
    ids[2, :] = -1
    w = wl.random_weights(10, T, topk)
    C2 = rng.standard_normal((T * topk, H)) * 37.0
    out = orc.combine_f64(C2, ids, w, E)
    for t in range(T):
        for j in range(H):
            ex = sum((Fraction(float(w[t, k])) * Fraction(float(C2[t * topk + k, j]))
                      for k in range(topk) if 0 <= ids[t, k] < E), Fraction(0))
            assert out[t, j] == bf16_rne_exact(ex), (t, j)
    assert (out[2] == 0).all()


def test_layer_f64sum_is_the_composition_and_close_to_dense(orc):
    """The variant's layer equals align -> binary64-sum gate_up (bf16) -> SiLU*up
    -> binary64 down sums -> binary64 combine, bit for bit (catches a rounding
    of the down sums or a wrong stage order), and agrees with the float64
    dense per-token loop within the tolerance."""
    w = wl.TINY
    ids, wts = wl.make_routing(w)
    x = wl.make_x(w)
    c13, s13 = wl.make_w13(w)
    c2, s2 = wl.make_w2(w)
    got = orc.moe_layer_f64sum(x, ids, wts, (c13, s13), (c2, s2), w.E, block_m=4)
    P = w.P
    s, e, n = orc.moe_align(ids, w.E, 4)
    C1 = orc.moe_gemm_f64sum(x, w.topk, c13, s13, s, e, n, 4, P, C=np.zeros((P, 2 * w.I), np.uint16))
    h = orc.silu_mul(C1, ids.ravel(), w.E, h=np.zeros((P, w.I), np.uint16))
    C2 = orc.moe_gemm_f64(h, 1, c2, s2, s, e, n, 4, P, C=np.zeros((P, w.H), np.float64))
    np.testing.assert_array_equal(got, orc.combine_f64(C2, ids, wts, w.E))
    ref = layer_dense_reference(x, ids, wts, c13, s13, c2, s2, w.E)
    err = np.abs(f64(got) - ref)
    assert (err <= 1e-2 + 1e-2 * np.abs(ref)).all(), err.max()


def test_plain_sums_within_the_summation_bound_of_f64_sums(orc):
    """At the Kimi-K2 gate_up depth (K = 7168, x ~ N(0,1), the workloads'
    weights) the plain oracle's binary32 sums (before the bf16 rounding) lie
    within Higham's bound for recursive summation, gamma_(K-1) * sum_k |x_k w_k|
    with gamma_n = n u / (1 - n u), u = 2^-24, of the binary64 sums (whose own
    error, K * 2^-53 * sum|x w|, is added).  Catches a lower-precision
    accumulator in the plain oracle (bf16 or binary16 partial sums)."""
    T, topk, E, N, K = 4, 2, 2, 256, 7168
    x = wl.random_bf16(41, (T, K))
    codes = wl.random_codes(42, (E, N, K))
    scales = wl.random_scales(43, (E, N, K // GROUP))
    ids = wl.random_ids(44, T, topk, E)
    s, e, n = orc.moe_align(ids, E, 8)
    P = T * topk
    a = orc.moe_gemm_f32(x, topk, codes, scales, s, e, n, 8, P).astype(np.float64)
    b = orc.moe_gemm_f64(x, topk, codes, scales, s, e, n, 8, P)
    W = np.abs(f64(dequant_ref(codes, scales)))
    X = np.abs(f64(x))
    u = 2.0 ** -24
    g = (K - 1) * u / (1 - (K - 1) * u)
    for p in range(P):
        ex = ids.ravel()[p]
        mag = W[ex] @ X[p // topk]
        assert (np.abs(a[p] - b[p]) <= g * mag + K * 2.0 ** -53 * mag).all(), p


def bf16_order(bits):
    """bf16 bit patterns -> integers in value order (one step per representable value; +0 = -0 = 0)."""
    b = np.asarray(bits, np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def test_layer_closed_form_down_sum_needs_binary64(orc):
    """A layer built so that every down sum is exactly 1 + 2^-8 + 2^-30:
    x = (128, 0, ...); gate rows j < 3 have weight 1 on k = 0, so g = 128 and
    SiLU(g) = 128 (exp(-128) underflows in binary32); up rows j < 3 have
    weight 2^-14, 2^-22, 2^-44 on k = 0, so h = 128 * 128 * w = 1, 2^-8, 2^-30;
    every down row has weight 1 on j < 3.  The weighted sum (weight 1) of
    1 + 2^-8 + 2^-30 lies just above the bf16 midpoint of 1 and 1 + 2^-7:
    the binary64 layer rounds it to 1 + 2^-7 (0x3f81); the plain layer's
    binary32 down sum is 1 + 2^-8 (a tie) and rounds to the even 1 (0x3f80).
    Catches a binary32 step anywhere in the variant's down sum or combine."""
    H, I, E = 64, 64, 1
    x = np.zeros((1, H), np.uint16)
    x[0, 0] = to_bf16([128.0])[0]
    c13 = np.full((E, 2 * I, H), 8, np.uint8)
    s13 = np.full((E, 2 * I, H // GROUP), 0x3F80, np.uint16)
    up_scale = to_bf16([2.0 ** -14, 2.0 ** -22, 2.0 ** -44])
    for j in range(3):
        c13[0, j, 0] = 9                     # gate weight 1
        c13[0, I + j, 0] = 9                 # up weight = its group's scale
        s13[0, I + j, 0] = up_scale[j]
    c2 = np.full((E, H, I), 8, np.uint8)
    c2[0, :, :3] = 9
    s2 = np.full((E, H, I // GROUP), 0x3F80, np.uint16)
    ids = np.zeros((1, 1), np.int32)
    wts = np.ones((1, 1), np.float32)
    got64 = orc.moe_layer_f64sum(x, ids, wts, (c13, s13), (c2, s2), E, block_m=1)
    got32 = orc.moe_layer(x, ids, wts, (c13, s13), (c2, s2), E, block_m=1)
    assert (got64 == 0x3F81).all(), got64
    assert (got32 == 0x3F80).all(), got32
