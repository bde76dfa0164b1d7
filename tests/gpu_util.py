"""Helpers for the GPU parity tests: device copies, calls through the C ABI
binding, the element-wise tolerance check |gpu - ref| <= 1e-2 + 1e-2 |ref|,
and the chain check of a whole layer against the oracle (every stage against
the oracle's result on the GPU's own previous stage)."""
import numpy as np
import torch

import oracle
import w4a16_int4_mixture_moe_gb300 as chord
import workloads as wl

DEV = "cuda:0"
ATOL = 1e-2
RTOL = 1e-2


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def dbf(bits):
    return dev(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def host_bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def f64(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def assert_close(got_bits, ref_bits, what=""):
    g, r = f64(got_bits), f64(ref_bits)
    err = np.abs(g - r)
    bad = ~(err <= ATOL + RTOL * np.abs(r))
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside "
                             f"{ATOL} + {RTOL}|ref|; max err {np.nanmax(err):.4g}; first {idx}; "
                             f"got {g[bad][:5]} ref {r[bad][:5]}")
    return float(err.max()) if err.size else 0.0


def bf16_order(bits):
    """bf16 bit patterns -> integers in value order (one step per representable
    value; +0 and -0 both 0)."""
    b = np.asarray(bits, np.uint16).astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def assert_close_f32(got, ref, what=""):
    """FP32 values (the down projection's sums) within 1e-2 + 1e-2|ref|."""
    err = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    bad = ~(err <= ATOL + RTOL * np.abs(ref))
    if bad.any():
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance, "
                             f"max err {np.nanmax(err):.4g}")


def oracle_align8(ids, E):
    return oracle.moe_align(ids, E, 8)


def steps_apart(a_bits, b_bits):
    """Number of elements whose bf16 values differ, and the largest distance
    in bf16 steps (reported, not bounded: near zero the steps are far smaller
    than an FP32 sum's error, so valid orders can be many steps apart there)."""
    d = np.abs(bf16_order(a_bits) - bf16_order(b_bits))
    return int((d > 0).sum()), int(d.max()) if d.size else 0


def check_h_from_gpu_c1(h_bits, C1_bits, C1_ref_bits, ids_flat, E, rows, what=""):
    """A GPU SiLU * up output h (fused into the gate_up GEMM, or a separate
    pass) checked through the chain it is defined by: the GPU's own gate_up
    output C1 within the tolerance of the oracle's gate_up, and h within the
    tolerance of the oracle's SiLU * up applied to that C1 (a sum that two
    valid FP32 orders round to neighbouring bf16 values moves h by the same
    propagation in both)."""
    assert_close(C1_bits[rows], C1_ref_bits[rows], f"{what}: gate_up")
    P, I2 = C1_bits.shape
    h_ref = oracle.silu_mul(C1_bits, ids_flat, E, h=np.zeros((P, I2 // 2), np.uint16))
    assert_close(h_bits[rows], h_ref[rows], f"{what}: SiLU*up of the GPU's gate_up")


def check_layer_chain(x, ids, wts, w13, w2, E, C1g, hg, C2g, outg, what="", with_f64=True):
    """The whole layer checked on every element of the given tokens (their rows
    of x, ids and weights, and the GPU's intermediates of their pairs, in pair
    order), through the chain of definitions, each stage against the oracle's
    result on the GPU's own previous stage:
      gate_up  C1g within 1e-2 + 1e-2|ref| of the oracle's and of the
               binary64-sum oracle's (nearly the exact sums);
      SiLU*up  hg within the tolerance of the oracle's SiLU*up of C1g;
      down     C2g (FP32 sums) within the tolerance of the oracle's down
               projection of hg;
      combine  outg bit for bit the oracle's weighted sum of C2g;
      layer    outg within the tolerance of the oracle's layer evaluated from
               C1g (the end-to-end result given the GPU's gate_up), and, against
               the plain oracle's layer from x, within the tolerance plus the
               deviation the oracle itself shows between its layer from x and
               its layer from C1g.  No element is exempt and no constant is
               chosen: where the GPU's gate_up rounded a sum to the
               neighbouring bf16 value, the oracle fed that value moves the
               output by the same propagation.
    Returns counts for reporting."""
    topk = ids.shape[1]
    T, H = x.shape
    I = w2[0].shape[2]
    P = T * topk
    flat = ids.ravel()
    rows = np.nonzero((flat >= 0) & (flat < E))[0]
    s, e, n = oracle_align8(ids, E)
    C1r = oracle.moe_gemm(x, topk, w13[0], w13[1], s, e, n, 8, P, C=np.zeros((P, 2 * I), np.uint16))
    assert_close(C1g[rows], C1r[rows], f"{what}: gate_up")
    flips = steps_apart(C1g[rows], C1r[rows])
    flips64 = None
    if with_f64:
        C1d = oracle.moe_gemm_f64sum(x, topk, w13[0], w13[1], s, e, n, 8, P, C=np.zeros((P, 2 * I), np.uint16))
        assert_close(C1g[rows], C1d[rows], f"{what}: gate_up vs the binary64-sum oracle")
        flips64 = steps_apart(C1g[rows], C1d[rows])
        del C1d
    h_of_c1g = oracle.silu_mul(C1g, flat, E, h=np.zeros((P, I), np.uint16))
    assert_close(hg[rows], h_of_c1g[rows], f"{what}: SiLU*up of the GPU's gate_up")
    C2_of_hg = oracle.moe_gemm_f32(hg, 1, w2[0], w2[1], s, e, n, 8, P, C=np.zeros((P, H), np.float32))
    assert_close_f32(C2g[rows], C2_of_hg[rows], f"{what}: down projection of the GPU's h")
    del C2_of_hg
    np.testing.assert_array_equal(outg, oracle.combine(C2g, ids, wts, E), err_msg=f"{what}: combine")
    C2_of_c1g = oracle.moe_gemm_f32(h_of_c1g, 1, w2[0], w2[1], s, e, n, 8, P, C=np.zeros((P, H), np.float32))
    out_of_c1g = oracle.combine(C2_of_c1g, ids, wts, E)
    del C2_of_c1g
    assert_close(outg, out_of_c1g, f"{what}: layer from the GPU's gate_up")
    hr = oracle.silu_mul(C1r, flat, E, h=np.zeros((P, I), np.uint16))
    C2r = oracle.moe_gemm_f32(hr, 1, w2[0], w2[1], s, e, n, 8, P, C=np.zeros((P, H), np.float32))
    out_ref = oracle.combine(C2r, ids, wts, E)
    del C2r
    g, r, rc = f64(outg), f64(out_ref), f64(out_of_c1g)
    bound = ATOL + RTOL * np.abs(r) + np.abs(rc - r)
    bad = np.abs(g - r) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs beyond tolerance + the oracle's own deviation"
    outside = int((np.abs(g - r) > ATOL + RTOL * np.abs(r)).sum())
    return {"c1_flips": flips, "c1_flips_vs_f64": flips64, "out_outside_plain_tol": outside, "outputs": g.size,
            "pairs": int(rows.size)}


KERNELS = {"tcgen05": (chord.KERNEL_TCGEN05, chord.LAYOUT_TCGEN05),
           "warp_mma": (chord.KERNEL_WARP_MMA, chord.LAYOUT_TCGEN05)}


def pack(codes, scales, layout=chord.LAYOUT_TCGEN05):
    E, N, K = codes.shape
    out = torch.empty(chord.chord_packed_weight_bytes(E, N, K, layout), dtype=torch.uint8, device=DEV)
    chord.chord_pack_weights(dev(codes), dbf(scales), out, layout=layout)
    return out


def align(ids, E, bm, opts=None):
    ids_d = ids if isinstance(ids, torch.Tensor) else dev(ids)
    T, topk = ids_d.shape
    cap = chord.chord_align_capacity(T, topk, E, bm)
    s = torch.empty(max(cap, 1), dtype=torch.int32, device=DEV)[:cap]
    e = torch.empty(max(cap // bm, 1), dtype=torch.int32, device=DEV)[:cap // bm]
    n = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(chord.chord_align_workspace_bytes(T, topk, E), 4), dtype=torch.uint8, device=DEV)
    chord.chord_moe_align(ids_d, E, bm, s, e, n, ws, opts=opts)
    return s, e, n


def gemm(A_bits, div, packed, E, N, K, s, e, n, bm, P, kernel=0, C=None, split_k=None, epilogue=0,
         out_dtype=0, mixed=0, tc_pairs=0):
    """C rows that no block names keep the fill pattern 0xFFFF (a NaN).
    split_k=None passes no workspace (the GEMM runs unsplit); otherwise the
    option is set and the workspace sized by chord_gemm_workspace_bytes."""
    A = A_bits if isinstance(A_bits, torch.Tensor) else dbf(A_bits)
    if C is None:
        C = torch.full((max(P, 1), N), -1, dtype=torch.int16, device=DEV)[:P].view(torch.bfloat16)
    opts = chord.ChordOpts(kernel=kernel, split_k=split_k or 0, epilogue=epilogue, out_dtype=out_dtype, mixed=mixed,
                           tc_pairs=tc_pairs)
    ws = None
    if split_k is not None:
        nb = chord.chord_gemm_workspace_bytes(P, N, K, bm, opts)
        ws = torch.empty(max(nb, 16), dtype=torch.uint8, device=DEV)
    chord.chord_w4a16_moe_gemm(A, div, packed, E, N, K, s, e, n, bm, P, C, workspace=ws, opts=opts)
    return C


def layer(x_bits, ids, wts, E, E_global, I, p13, p2, bm=0, opts=None):
    T, H = x_bits.shape
    topk = ids.shape[1]
    if bm <= 0:
        bm = chord.chord_select_block_m(T, topk, E, E_global, 2 * I, H)
    ws = torch.empty(chord.chord_layer_workspace_bytes(T, topk, E, H, I, bm), dtype=torch.uint8, device=DEV)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    chord.chord_moe_layer(dbf(x_bits), dev(ids), dev(wts), E, E_global, I, p13, p2, ws, out, block_m=bm,
                          opts=opts)
    return out, bm


def valid_rows(ids, E):
    flat = ids.ravel()
    return np.nonzero((flat >= 0) & (flat < E))[0]


def run_layer_steps(x_bits, ids, wts, E, I, p13, p2, bm, fused, kernel=0, split=True, mixed=0):
    """The layer as the benchmark's step runs it, every call through the C ABI:
    align -> gate_up (SiLU * up fused when `fused`, w13 then in layout 3) ->
    SiLU * up pass (unfused) -> down with FP32 output -> combine.  Each GEMM
    gets its workspace (K slices or the split tail as the benchmark runs
    them) unless split is False.  Returns the device tensors."""
    T, H = x_bits.shape
    topk = ids.shape[1]
    P = T * topk
    xd, idd, wd = dbf(x_bits), dev(ids), dev(wts)
    s, e, n = align(idd, E, bm)
    epi = chord.EPILOGUE_SILU_MUL if fused else chord.EPILOGUE_NONE
    h = torch.full((max(P, 1), I), -1, dtype=torch.int16, device=DEV)[:P].view(torch.bfloat16)
    C1 = None
    if fused:
        gemm(xd, topk, p13, E, 2 * I, H, s, e, n, bm, P, kernel=kernel, C=h, split_k=0 if split else None,
             epilogue=epi, mixed=mixed)
    else:
        C1 = gemm(xd, topk, p13, E, 2 * I, H, s, e, n, bm, P, kernel=kernel, split_k=0 if split else None,
                  mixed=mixed)
        chord.chord_silu_mul(C1, idd, E, h)
    C2 = torch.full((max(P, 1), H), float("nan"), dtype=torch.float32, device=DEV)[:P]
    gemm(h, 1, p2, E, H, I, s, e, n, bm, P, kernel=kernel, C=C2, split_k=0 if split else None,
         out_dtype=chord.DTYPE_F32, mixed=mixed)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=DEV)
    chord.chord_moe_combine(C2, idd, wd, E, out)
    return {"sorted": s, "experts": e, "ntp": n, "C1": C1, "h": h, "C2": C2, "out": out}


def pair_rows(t, pairs):
    """Rows `pairs` (numpy int64) of a device tensor, copied to the host."""
    return t[torch.from_numpy(np.ascontiguousarray(pairs)).to(t.device)]
