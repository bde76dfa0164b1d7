"""CPU oracle for the W4A16 INT4 mixture-of-experts expert GEMM.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The CUDA library never calls it and shares no code with it.

The arithmetic lives in ``chord_oracle.c`` (plain C, built here with gcc,
``-ffp-contract=off`` so every rounding happens where the source says).  This
module only builds it and marshals numpy arrays.  Every function cites the
passage it follows in the C source.

Parity status per function (see the pins in ``tests/test_oracle_pins.py``):
dequant, pack/unpack, align, gemm, silu_mul, combine and the layer are pinned
against closed forms, library routines, exact integer arithmetic or brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "chord_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liborc.so")
CFLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-std=c11"]

_lock = threading.Lock()
_lib = None

OK, EINVAL, ELAYOUT, ERANGE, ENOMEM = 0, -1, -2, -3, -4
GROUP = 32


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liborc.so`` (gcc, OpenMP).

    ``CHORD_ORACLE_LIB`` names an already-built library to load instead; the
    mutation tests use it to run the pins against deliberately broken copies.
    """
    alt = os.environ.get("CHORD_ORACLE_LIB")
    if alt:
        return alt
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _P(t):
    return ctypes.POINTER(t)


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u8p, u16p, i32p, f32p = _P(ctypes.c_uint8), _P(ctypes.c_uint16), _P(ctypes.c_int32), _P(ctypes.c_float)
            f64p = _P(ctypes.c_double)
            c_int, c_i64, c_sz = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
            sig = {
                "orc_version": (c_int, []),
                "orc_max_threads": (c_int, []),
                "orc_bf16_round": (ctypes.c_uint16, [ctypes.c_float]),
                "orc_dequant": (ctypes.c_uint16, [ctypes.c_uint8, ctypes.c_uint16]),
                "orc_dequant_pairs": (None, [u8p, u16p, c_sz, u16p]),
                "orc_packed_bytes": (c_sz, [c_int, c_int, c_int, c_int]),
                "orc_pack": (c_int, [u8p, u16p, c_int, c_int, c_int, c_int, u8p, c_sz]),
                "orc_check_header": (c_int, [u8p, c_int, c_int, c_int, c_int]),
                "orc_unpack": (c_int, [u8p, c_sz, c_int, c_int, c_int, c_int, u8p, u16p]),
                "orc_align_capacity": (c_i64, [c_int, c_int, c_int, c_int]),
                "orc_moe_align": (c_int, [i32p, c_int, c_int, c_int, c_int, i32p, i32p, i32p, c_i64]),
                "orc_moe_gemm": (c_int, [u16p, c_i64, c_int, u8p, u16p, c_int, c_int, c_int,
                                         i32p, i32p, ctypes.c_int32, c_int, c_i64, u16p, c_int]),
                "orc_moe_gemm_f32": (c_int, [u16p, c_i64, c_int, u8p, u16p, c_int, c_int, c_int,
                                             i32p, i32p, ctypes.c_int32, c_int, c_i64, f32p, c_int]),
                "orc_grouped_contiguous": (c_int, [u16p, c_i64, i32p, u8p, u16p, c_int, c_int, c_int, u16p, c_int]),
                "orc_grouped_masked": (c_int, [u16p, c_int, c_int, i32p, u8p, u16p, c_int, c_int, u16p, c_int]),
                "orc_silu_mul": (c_int, [u16p, i32p, c_i64, c_int, c_int, u16p, c_int]),
                "orc_combine": (c_int, [u16p, i32p, f32p, c_int, c_int, c_int, c_int, u16p, c_int]),
                "orc_combine_f32": (c_int, [f32p, i32p, f32p, c_int, c_int, c_int, c_int, u16p, c_int]),
                "orc_moe_layer": (c_int, [u16p, i32p, f32p, c_int, c_int, c_int, c_int, c_int,
                                          u8p, u16p, u8p, u16p, c_int, u16p, c_int]),
                "orc_bf16_round_f64": (ctypes.c_uint16, [ctypes.c_double]),
                "orc_moe_gemm_f64sum": (c_int, [u16p, c_i64, c_int, u8p, u16p, c_int, c_int, c_int,
                                                i32p, i32p, ctypes.c_int32, c_int, c_i64, u16p, c_int]),
                "orc_moe_gemm_f64": (c_int, [u16p, c_i64, c_int, u8p, u16p, c_int, c_int, c_int,
                                             i32p, i32p, ctypes.c_int32, c_int, c_i64, f64p, c_int]),
                "orc_combine_f64": (c_int, [f64p, i32p, f32p, c_int, c_int, c_int, c_int, u16p, c_int]),
                "orc_moe_layer_f64sum": (c_int, [u16p, i32p, f32p, c_int, c_int, c_int, c_int, c_int,
                                                 u8p, u16p, u8p, u16p, c_int, u16p, c_int]),
            }
            for name, (res, args) in sig.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


def _ptr(a, t):
    return a.ctypes.data_as(_P(t))


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {a.dtype}")
    return a


def _check(rc, what):
    if rc != OK:
        raise OracleError(f"{what} failed with code {rc}")


def threads(n=None) -> int:
    return int(n) if n else lib().orc_max_threads()


# --- dequantisation -------------------------------------------------------

def bf16_round(f: float) -> int:
    return int(lib().orc_bf16_round(float(f)))


def dequant(q: int, s_bits: int) -> int:
    """bf16 bits of (q - 8) * s, rounded once to nearest even."""
    return int(lib().orc_dequant(q, s_bits))


def dequant_pairs(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    q = _c(q, np.uint8).ravel()
    s = _c(s, np.uint16).ravel()
    assert q.size == s.size
    out = np.empty(q.size, np.uint16)
    lib().orc_dequant_pairs(_ptr(q, ctypes.c_uint8), _ptr(s, ctypes.c_uint16), q.size,
                            _ptr(out, ctypes.c_uint16))
    return out


# --- packing --------------------------------------------------------------

def packed_bytes(E: int, N: int, K: int, layout: int = 2) -> int:
    return int(lib().orc_packed_bytes(E, N, K, layout))


def pack(codes: np.ndarray, scales: np.ndarray, layout: int = 2) -> np.ndarray:
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    E, N, K = codes.shape
    assert scales.shape == (E, N, K // GROUP)
    nb = packed_bytes(E, N, K, layout)
    if nb == 0:
        raise OracleError("unsupported shape for packing")
    out = np.empty(nb, np.uint8)
    _check(lib().orc_pack(_ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint16), E, N, K, layout,
                          _ptr(out, ctypes.c_uint8), nb), "pack")
    return out


def unpack(blob: np.ndarray, E: int, N: int, K: int, layout: int = 2):
    blob = _c(blob, np.uint8)
    codes = np.empty((E, N, K), np.uint8)
    scales = np.empty((E, N, K // GROUP), np.uint16)
    _check(lib().orc_unpack(_ptr(blob, ctypes.c_uint8), blob.size, E, N, K, layout,
                            _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint16)), "unpack")
    return codes, scales


def check_header(blob: np.ndarray, E: int, N: int, K: int, layout: int = 2) -> bool:
    blob = _c(blob, np.uint8)
    return lib().orc_check_header(_ptr(blob, ctypes.c_uint8), E, N, K, layout) == OK


# --- routing --------------------------------------------------------------

def align_capacity(T: int, topk: int, E: int, block_m: int) -> int:
    return int(lib().orc_align_capacity(T, topk, E, block_m))


def moe_align(topk_ids: np.ndarray, E: int, block_m: int):
    """Return (sorted_ids, expert_ids, num_tokens_padded) for the capacity layout."""
    ids = _c(topk_ids, np.int32)
    T, topk = ids.shape
    cap = align_capacity(T, topk, E, block_m)
    sorted_ids = np.empty(max(cap, 1), np.int32)[:cap]
    expert_ids = np.empty(max(cap // block_m, 1), np.int32)[:cap // block_m]
    ntp = np.zeros(1, np.int32)
    _check(lib().orc_moe_align(_ptr(ids, ctypes.c_int32), T, topk, E, block_m,
                               _ptr(sorted_ids, ctypes.c_int32), _ptr(expert_ids, ctypes.c_int32),
                               _ptr(ntp, ctypes.c_int32), cap), "moe_align")
    return sorted_ids, expert_ids, int(ntp[0])


# --- GEMM / activation / combine / layer -----------------------------------

def moe_gemm(A: np.ndarray, a_row_divisor: int, codes: np.ndarray, scales: np.ndarray,
             sorted_ids: np.ndarray, expert_ids: np.ndarray, num_tokens_padded: int,
             block_m: int, num_pairs: int, C: np.ndarray = None, nthreads=None) -> np.ndarray:
    """C[p, :] for every non-sentinel p named by the blocks; other rows of C untouched."""
    A = _c(A, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    E, N, K = codes.shape
    assert A.shape[1] == K
    sorted_ids = _c(sorted_ids, np.int32)
    expert_ids = _c(expert_ids, np.int32)
    if C is None:
        C = np.zeros((max(num_pairs, 1), N), np.uint16)[:num_pairs]
    C = _c(C, np.uint16)
    _check(lib().orc_moe_gemm(_ptr(A, ctypes.c_uint16), A.shape[0], a_row_divisor,
                              _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint16), E, N, K,
                              _ptr(sorted_ids, ctypes.c_int32), _ptr(expert_ids, ctypes.c_int32),
                              num_tokens_padded, block_m, num_pairs, _ptr(C, ctypes.c_uint16),
                              threads(nthreads)), "moe_gemm")
    return C


def grouped_contiguous(A: np.ndarray, m_indices: np.ndarray, codes: np.ndarray, scales: np.ndarray,
                       C: np.ndarray = None, nthreads=None) -> np.ndarray:
    """bf16 bits [M, N]: rows of A grouped per expert, m_indices[m] its expert (-1: padding, not written)."""
    A = _c(A, np.uint16)
    m_indices = _c(m_indices, np.int32)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    E, N, K = codes.shape
    M = A.shape[0]
    assert A.shape[1] == K and m_indices.shape == (M,)
    C = _c(np.zeros((M, N), np.uint16) if C is None else C, np.uint16)
    _check(lib().orc_grouped_contiguous(_ptr(A, ctypes.c_uint16), M, _ptr(m_indices, ctypes.c_int32),
                                        _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint16), E, N, K,
                                        _ptr(C, ctypes.c_uint16), threads(nthreads)), "orc_grouped_contiguous")
    return C


def grouped_masked(A: np.ndarray, masked_m: np.ndarray, codes: np.ndarray, scales: np.ndarray,
                   C: np.ndarray = None, nthreads=None) -> np.ndarray:
    """bf16 bits [G * max_m, N] from A [G, max_m, K]; rows past masked_m[g] are not written."""
    A = _c(A, np.uint16)
    masked_m = _c(masked_m, np.int32)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    G, max_m, K = A.shape
    E, N, K2 = codes.shape
    assert K2 == K and E == G and masked_m.shape == (G,)
    C = _c(np.zeros((G * max_m, N), np.uint16) if C is None else C, np.uint16)
    _check(lib().orc_grouped_masked(_ptr(A, ctypes.c_uint16), G, max_m, _ptr(masked_m, ctypes.c_int32),
                                    _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint16), N, K,
                                    _ptr(C, ctypes.c_uint16), threads(nthreads)), "orc_grouped_masked")
    return C


def moe_gemm_f32(A: np.ndarray, a_row_divisor: int, codes: np.ndarray, scales: np.ndarray,
                 sorted_ids: np.ndarray, expert_ids: np.ndarray, num_tokens_padded: int,
                 block_m: int, num_pairs: int, C: np.ndarray = None, nthreads=None) -> np.ndarray:
    """As moe_gemm, but C holds the FP32 sums unrounded (float32 [num_pairs, N])."""
    A = _c(A, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    E, N, K = codes.shape
    assert A.shape[1] == K
    sorted_ids = _c(sorted_ids, np.int32)
    expert_ids = _c(expert_ids, np.int32)
    if C is None:
        C = np.zeros((max(num_pairs, 1), N), np.float32)[:num_pairs]
    C = _c(C, np.float32)
    _check(lib().orc_moe_gemm_f32(_ptr(A, ctypes.c_uint16), A.shape[0], a_row_divisor,
                                  _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint16), E, N, K,
                                  _ptr(sorted_ids, ctypes.c_int32), _ptr(expert_ids, ctypes.c_int32),
                                  num_tokens_padded, block_m, num_pairs, _ptr(C, ctypes.c_float),
                                  threads(nthreads)), "moe_gemm_f32")
    return C


def silu_mul(C1: np.ndarray, topk_ids: np.ndarray, E: int, h: np.ndarray = None, nthreads=None):
    C1 = _c(C1, np.uint16)
    ids = _c(topk_ids, np.int32).ravel()
    P, I2 = C1.shape
    I = I2 // 2
    if h is None:
        h = np.zeros((P, I), np.uint16)
    _check(lib().orc_silu_mul(_ptr(C1, ctypes.c_uint16), _ptr(ids, ctypes.c_int32), P, E, I,
                              _ptr(h, ctypes.c_uint16), threads(nthreads)), "silu_mul")
    return h


def combine(C2: np.ndarray, topk_ids: np.ndarray, topk_w: np.ndarray, E: int, nthreads=None):
    """C2 as bf16 bits (uint16) or float32; returns bf16 bits [T, H]."""
    C2 = np.ascontiguousarray(C2)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    T, topk = ids.shape
    H = C2.shape[1]
    out = np.empty((T, H), np.uint16)
    if C2.dtype == np.float32:
        rc = lib().orc_combine_f32(_ptr(C2, ctypes.c_float), _ptr(ids, ctypes.c_int32),
                                   _ptr(w, ctypes.c_float), T, topk, E, H, _ptr(out, ctypes.c_uint16),
                                   threads(nthreads))
    else:
        C2 = _c(C2, np.uint16)
        rc = lib().orc_combine(_ptr(C2, ctypes.c_uint16), _ptr(ids, ctypes.c_int32),
                               _ptr(w, ctypes.c_float), T, topk, E, H, _ptr(out, ctypes.c_uint16),
                               threads(nthreads))
    _check(rc, "combine")
    return out


def moe_layer(x, topk_ids, topk_w, w13, w2, E: int, block_m: int = 16, nthreads=None):
    """bf16 bits [T, H] of one MoE layer; w13 = (codes, scales) of gate_up, w2 of down."""
    x = _c(x, np.uint16)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    c13, s13 = (_c(w13[0], np.uint8), _c(w13[1], np.uint16))
    c2, s2 = (_c(w2[0], np.uint8), _c(w2[1], np.uint16))
    T, H = x.shape
    topk = ids.shape[1]
    I = c2.shape[2]
    assert c13.shape == (E, 2 * I, H) and c2.shape == (E, H, I)
    out = np.empty((T, H), np.uint16)
    _check(lib().orc_moe_layer(_ptr(x, ctypes.c_uint16), _ptr(ids, ctypes.c_int32),
                               _ptr(w, ctypes.c_float), T, topk, E, H, I,
                               _ptr(c13, ctypes.c_uint8), _ptr(s13, ctypes.c_uint16),
                               _ptr(c2, ctypes.c_uint8), _ptr(s2, ctypes.c_uint16),
                               block_m, _ptr(out, ctypes.c_uint16), threads(nthreads)), "moe_layer")
    return out


# --- the binary64-sum variant (a second valid summation order) ----------------

def bf16_round_f64(d: float) -> int:
    """bf16 bits of a binary64 value, rounded once to nearest even."""
    return int(lib().orc_bf16_round_f64(float(d)))


def moe_gemm_f64sum(A, a_row_divisor, codes, scales, sorted_ids, expert_ids, num_tokens_padded, block_m,
                    num_pairs, C=None, nthreads=None):
    """As moe_gemm, with each dot product summed in binary64 and rounded to bf16 once
    (orc_moe_gemm_f64sum)."""
    return _gemm_variant("orc_moe_gemm_f64sum", np.uint16, ctypes.c_uint16, A, a_row_divisor, codes, scales,
                         sorted_ids, expert_ids, num_tokens_padded, block_m, num_pairs, C, nthreads)


def moe_gemm_f64(A, a_row_divisor, codes, scales, sorted_ids, expert_ids, num_tokens_padded, block_m,
                 num_pairs, C=None, nthreads=None):
    """The binary64 sums themselves, float64 [num_pairs, N] (orc_moe_gemm_f64)."""
    return _gemm_variant("orc_moe_gemm_f64", np.float64, ctypes.c_double, A, a_row_divisor, codes, scales,
                         sorted_ids, expert_ids, num_tokens_padded, block_m, num_pairs, C, nthreads)


def _gemm_variant(name, dtype, ctype, A, a_row_divisor, codes, scales, sorted_ids, expert_ids,
                  num_tokens_padded, block_m, num_pairs, C, nthreads):
    A = _c(A, np.uint16)
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint16)
    E, N, K = codes.shape
    assert A.shape[1] == K
    sorted_ids = _c(sorted_ids, np.int32)
    expert_ids = _c(expert_ids, np.int32)
    if C is None:
        C = np.zeros((max(num_pairs, 1), N), dtype)[:num_pairs]
    C = _c(C, dtype)
    _check(getattr(lib(), name)(_ptr(A, ctypes.c_uint16), A.shape[0], a_row_divisor,
                                _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint16), E, N, K,
                                _ptr(sorted_ids, ctypes.c_int32), _ptr(expert_ids, ctypes.c_int32),
                                num_tokens_padded, block_m, num_pairs, _ptr(C, ctype), threads(nthreads)), name)
    return C


def combine_f64(C2: np.ndarray, topk_ids: np.ndarray, topk_w: np.ndarray, E: int, nthreads=None):
    """Weighted sum of float64 C2 rows in binary64, rounded to bf16 once (orc_combine_f64)."""
    C2 = _c(C2, np.float64)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    T, topk = ids.shape
    H = C2.shape[1]
    out = np.empty((T, H), np.uint16)
    _check(lib().orc_combine_f64(_ptr(C2, ctypes.c_double), _ptr(ids, ctypes.c_int32), _ptr(w, ctypes.c_float),
                                 T, topk, E, H, _ptr(out, ctypes.c_uint16), threads(nthreads)), "combine_f64")
    return out


def moe_layer_f64sum(x, topk_ids, topk_w, w13, w2, E: int, block_m: int = 16, nthreads=None):
    """The layer with binary64 sums at the plain layer's rounding points (orc_moe_layer_f64sum)."""
    x = _c(x, np.uint16)
    ids = _c(topk_ids, np.int32)
    w = _c(topk_w, np.float32)
    c13, s13 = (_c(w13[0], np.uint8), _c(w13[1], np.uint16))
    c2, s2 = (_c(w2[0], np.uint8), _c(w2[1], np.uint16))
    T, H = x.shape
    topk = ids.shape[1]
    I = c2.shape[2]
    assert c13.shape == (E, 2 * I, H) and c2.shape == (E, H, I)
    out = np.empty((T, H), np.uint16)
    _check(lib().orc_moe_layer_f64sum(_ptr(x, ctypes.c_uint16), _ptr(ids, ctypes.c_int32),
                                      _ptr(w, ctypes.c_float), T, topk, E, H, I,
                                      _ptr(c13, ctypes.c_uint8), _ptr(s13, ctypes.c_uint16),
                                      _ptr(c2, ctypes.c_uint8), _ptr(s2, ctypes.c_uint16),
                                      block_m, _ptr(out, ctypes.c_uint16), threads(nthreads)), "moe_layer_f64sum")
    return out
