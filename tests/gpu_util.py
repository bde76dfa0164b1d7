"""Helpers for the GPU parity tests: device copies, calls through the C ABI
binding, and the element-wise tolerance check |gpu - ref| <= 1e-2 + 1e-2 |ref|."""
import numpy as np
import torch

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


def assert_close_layer(got_bits, ref_bits, what=""):
    """A whole layer against the oracle's: the tolerance 1e-2 + 1e-2|ref| for at
    least 99.5% of the elements; the rest may differ by the propagation of
    one-ulp BF16 flips of the gate_up output and of SiLU*up (two valid FP32
    summation orders round an intermediate differently; the oracle recomputed
    with float64 sums shows the same effect), bounded by 5% of the token's
    output RMS, with the error RMS below 0.2% of the output RMS."""
    g, r = f64(got_bits), f64(ref_bits)
    err = np.abs(g - r)
    inside = err <= ATOL + RTOL * np.abs(r)
    rms = np.sqrt((r ** 2).mean(axis=1, keepdims=True)) + 1e-30
    msg = (f"{what}: {int((~inside).sum())} of {inside.size} outside the per-element tolerance, "
           f"max err {err.max():.4g}, max err/rms {(err / rms).max():.4g}")
    assert inside.mean() >= 0.995, msg
    assert (err <= ATOL + RTOL * np.abs(r) + 0.05 * rms).all(), msg
    assert np.sqrt((err ** 2).mean()) <= 2e-3 * np.sqrt((r ** 2).mean()) + 1e-6, msg


def assert_close_h(got_bits, ref_bits, what=""):
    """For h = bf16(SiLU(g) * u) computed from this library's own bf16 gate and
    up sums: a last-place flip of one of those roundings (an FP32 summation
    order effect) moves h by a few bf16 ulps, more where SiLU is steep (g well
    below zero).  The exact checks are elsewhere: the fused result equals the
    unfused path bit for bit, whose GEMM and SiLU * up stages are each checked
    against the oracle on the oracle's own inputs.  Here at most 0.1 % of the
    elements may fall outside the GEMM tolerance."""
    g, r = f64(got_bits), f64(ref_bits)
    err = np.abs(g - r)
    bad = ~(err <= ATOL + RTOL * np.abs(r))
    assert bad.sum() <= max(1, bad.size // 1000), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance, "
                                                   f"max err {np.nanmax(err):.4g}")


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
         out_dtype=0):
    """C rows that no block names keep the fill pattern 0xFFFF (a NaN).
    split_k=None passes no workspace (the GEMM runs unsplit); otherwise the
    option is set and the workspace sized by chord_gemm_workspace_bytes."""
    A = A_bits if isinstance(A_bits, torch.Tensor) else dbf(A_bits)
    if C is None:
        C = torch.full((max(P, 1), N), -1, dtype=torch.int16, device=DEV)[:P].view(torch.bfloat16)
    opts = chord.ChordOpts(kernel=kernel, split_k=split_k or 0, epilogue=epilogue, out_dtype=out_dtype)
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
