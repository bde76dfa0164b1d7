"""Python binding of libchord.so, the sm_103a W4A16 INT4 mixture-of-experts library.

Argument marshalling only: every function passes device pointers and sizes of
caller-allocated torch tensors to the C entry point of the same name declared
in ``include/chord.h`` and raises ``ChordError`` on a non-OK status.  All
compute runs in the library's CUDA kernels; there is no fallback of any kind.
If the library has not been built, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "ChordError", "ChordOpts", "load", "build",
    "chord_version", "chord_status_string", "chord_packed_weight_bytes", "chord_pack_weights",
    "chord_align_capacity", "chord_align_workspace_bytes", "chord_moe_align", "chord_select_block_m", "chord_select_kernel",
    "chord_gemm_workspace_bytes", "chord_gemm_launch_count", "chord_w4a16_moe_gemm", "chord_silu_mul", "chord_moe_combine",
    "chord_combine_plan", "chord_w4a16_moe_gemm_combine", "chord_combine_finish",
    "chord_layer_workspace_bytes", "chord_moe_layer", "chord_moe_layer_cached", "chord_moe_layer_cache_clear", "chord_get_device_error", "chord_selftest_wait_timeout",
    "chord_grouped_contiguous_workspace_bytes", "chord_grouped_contiguous_gemm",
    "chord_grouped_masked_workspace_bytes", "chord_grouped_masked_gemm",
    "KERNEL_AUTO", "KERNEL_TCGEN05", "KERNEL_WARP_MMA", "LAYOUT_WARP_MMA", "LAYOUT_TCGEN05",
    "DTYPE_BF16", "DTYPE_F32",
]

KERNEL_AUTO, KERNEL_TCGEN05, KERNEL_WARP_MMA = 0, 1, 2
LAYOUT_WARP_MMA, LAYOUT_TCGEN05, LAYOUT_GATE_UP_INTERLEAVED = 1, 2, 3
EPILOGUE_NONE, EPILOGUE_SILU_MUL = 0, 1
DTYPE_BF16, DTYPE_F32 = 0, 1
STATUS = {0: "CHORD_OK", 1: "CHORD_ERR_INVALID_ARG", 2: "CHORD_ERR_UNSUPPORTED", 3: "CHORD_ERR_LAYOUT_MISMATCH",
          4: "CHORD_ERR_BUFFER_TOO_SMALL", 5: "CHORD_ERR_CUDA", 6: "CHORD_ERR_DEVICE_VALIDATION",
          7: "CHORD_ERR_TIMEOUT"}


class ChordError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}")


class ChordOpts(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("validate", ctypes.c_int32), ("split_k", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("epilogue", ctypes.c_int32), ("mixed", ctypes.c_int32),
                ("fuse_combine", ctypes.c_int32), ("tc_pairs", ctypes.c_int32)]


_lock = threading.Lock()
_lib = None
_vp, _sz, _i32, _i64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64
_int = ctypes.c_int
_OPTS = ctypes.POINTER(ChordOpts)

_SIGS = {
    "chord_version": (_int, []),
    "chord_status_string": (ctypes.c_char_p, [_int]),
    "chord_packed_weight_bytes": (_sz, [_int, _int, _int, _int]),
    "chord_pack_weights": (_int, [_vp, _vp, _int, _int, _int, _int, _int, _vp, _sz, _vp]),
    "chord_align_capacity": (_i64, [_int, _int, _int, _int]),
    "chord_align_workspace_bytes": (_sz, [_int, _int, _int]),
    "chord_moe_align": (_int, [_vp, _int, _int, _int, _int, _vp, _vp, _vp, _i64, _vp, _sz, _OPTS, _vp]),
    "chord_moe_align_noalloc": (_int, [_vp, _int, _int, _int, _int, _vp, _vp, _vp, _i64, _OPTS, _vp]),
    "chord_select_block_m": (_int, [_int, _int, _int, _int, _int, _int]),
    "chord_select_kernel": (_int, [_int, _int, _int]),
    "chord_gemm_workspace_bytes": (_sz, [_i64, _int, _int, _int, _OPTS]),
    "chord_gemm_launch_count": (_int, [_i64, _int, _int, _int, _sz, _OPTS]),
    "chord_w4a16_moe_gemm": (_int, [_vp, _i64, _int, _vp, _sz, _int, _int, _int, _vp, _vp, _vp, _i64, _int, _i64,
                                    _vp, _vp, _sz, _OPTS, _vp]),
    "chord_silu_mul": (_int, [_vp, _vp, _i64, _int, _int, _vp, _vp]),
    "chord_combine_plan": (_int, [_vp, _vp, _int, _int, _int, _vp, _vp]),
    "chord_w4a16_moe_gemm_combine": (_int, [_vp, _vp, _sz, _int, _int, _int, _vp, _vp, _vp, _i64, _int, _int, _int,
                                            _vp, _vp, _vp, _vp, _sz, _OPTS, _vp]),
    "chord_combine_finish": (_int, [_vp, _vp, _vp, _int, _int, _int, _int, _vp, _vp]),
    "chord_moe_combine": (_int, [_vp, _int, _vp, _vp, _int, _int, _int, _int, _vp, _vp]),
    "chord_layer_workspace_bytes": (_sz, [_int, _int, _int, _int, _int, _int]),
    "chord_moe_layer": (_int, [_vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _vp, _sz, _vp, _sz, _int, _vp,
                               _sz, _vp, _OPTS, _vp]),
    "chord_moe_layer_cached": (_int, [_vp, _vp, _vp, _int, _int, _int, _int, _int, _int, _vp, _sz, _vp, _sz, _int,
                                      _vp, _sz, _vp, _OPTS, _vp]),
    "chord_moe_layer_cache_clear": (_int, []),
    "chord_get_device_error": (_int, [_vp, ctypes.POINTER(_i32)]),
    "chord_selftest_wait_timeout": (_int, [_vp]),
    "chord_grouped_contiguous_workspace_bytes": (_sz, [_i64, _int]),
    "chord_grouped_contiguous_gemm": (_int, [_vp, _i64, _vp, _vp, _sz, _int, _int, _int, _vp, _vp, _sz, _OPTS, _vp]),
    "chord_grouped_masked_workspace_bytes": (_sz, [_int, _int, _int]),
    "chord_grouped_masked_gemm": (_int, [_vp, _int, _int, _vp, _int, _vp, _sz, _int, _int, _vp, _vp, _sz, _OPTS,
                                         _vp]),
}


def build(force: bool = False) -> str:
    """Compile libchord.so for sm_103a (nvcc) if it is missing or stale."""
    return _build.build(force=force)


def load():
    """Load libchord.so (built in-tree); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libchord.so is not built ({path}); call build() first")
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                f = getattr(L, name)
                f.restype, f.argtypes = res, args
            _lib = L
    return _lib


def _check(st: int, what: str):
    if st != 0:
        raise ChordError(st, what)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream) or 0)


def _o(opts):
    return None if opts is None else ctypes.byref(opts)


def _nbytes(t):
    return t.numel() * t.element_size()


# --- entry points (same names as the C ABI) ---------------------------------

def chord_version() -> int:
    return load().chord_version()


def chord_status_string(status: int) -> str:
    return load().chord_status_string(status).decode()


def chord_packed_weight_bytes(E: int, N: int, K: int, layout: int = LAYOUT_TCGEN05) -> int:
    return load().chord_packed_weight_bytes(E, N, K, layout)


def chord_pack_weights(codes, scales, packed, layout: int = LAYOUT_TCGEN05, group_size: int = 32, stream=None):
    """codes uint8 [E, N, K] (0..15), scales bf16 [E, N, K/32], packed uint8 output (device tensors)."""
    E, N, K = codes.shape
    _check(load().chord_pack_weights(_p(codes), _p(scales), E, N, K, group_size, layout, _p(packed),
                                     _nbytes(packed), _s(stream)), "chord_pack_weights")


def chord_align_capacity(T: int, topk: int, E: int, block_m: int) -> int:
    return load().chord_align_capacity(T, topk, E, block_m)


def chord_align_workspace_bytes(T: int, topk: int, E: int) -> int:
    return load().chord_align_workspace_bytes(T, topk, E)


def chord_moe_align(topk_ids, E: int, block_m: int, sorted_ids, expert_ids, num_tokens_padded, workspace,
                    opts=None, stream=None):
    T, topk = topk_ids.shape
    _check(load().chord_moe_align(_p(topk_ids), T, topk, E, block_m, _p(sorted_ids), _p(expert_ids),
                                  _p(num_tokens_padded), sorted_ids.numel(), _p(workspace),
                                  _nbytes(workspace) if workspace is not None else 0, _o(opts), _s(stream)),
           "chord_moe_align")


def chord_moe_align_noalloc(topk_ids, E: int, block_m: int, sorted_ids, expert_ids, num_tokens_padded,
                            opts=None, stream=None):
    """chord_moe_align without a workspace, for callers that cannot allocate:
    its scratch is a fixed 256 KiB array inside the library (see chord.h for the
    size limit and for why overlapping calls must be serialised)."""
    T, topk = topk_ids.shape
    _check(load().chord_moe_align_noalloc(_p(topk_ids), T, topk, E, block_m, _p(sorted_ids), _p(expert_ids),
                                          _p(num_tokens_padded), sorted_ids.numel(), _o(opts), _s(stream)),
           "chord_moe_align_noalloc")


def chord_select_block_m(T: int, topk: int, E_local: int, E_global: int, N: int, K: int) -> int:
    return load().chord_select_block_m(T, topk, E_local, E_global, N, K)


def chord_select_kernel(block_m: int, N: int, K: int) -> int:
    return load().chord_select_kernel(block_m, N, K)


def chord_gemm_workspace_bytes(num_pairs: int, N: int, K: int, block_m: int, opts=None) -> int:
    return load().chord_gemm_workspace_bytes(num_pairs, N, K, block_m, _o(opts))


def chord_gemm_launch_count(num_pairs: int, N: int, K: int, block_m: int, workspace_bytes: int, opts=None) -> int:
    return int(load().chord_gemm_launch_count(num_pairs, N, K, block_m, workspace_bytes, _o(opts)))


def chord_w4a16_moe_gemm(A, a_row_divisor: int, packed, E: int, N: int, K: int, sorted_ids, expert_ids,
                         num_tokens_padded, block_m: int, num_pairs: int, C, workspace=None, opts=None,
                         stream=None):
    _check(load().chord_w4a16_moe_gemm(_p(A), A.shape[0], a_row_divisor, _p(packed), _nbytes(packed), E, N, K,
                                       _p(sorted_ids), _p(expert_ids), _p(num_tokens_padded), sorted_ids.numel(),
                                       block_m, num_pairs, _p(C), _p(workspace),
                                       _nbytes(workspace) if workspace is not None else 0, _o(opts), _s(stream)),
           "chord_w4a16_moe_gemm")


def chord_silu_mul(C1, topk_ids, E: int, h, stream=None):
    P, I2 = C1.shape
    _check(load().chord_silu_mul(_p(C1), _p(topk_ids), P, E, I2 // 2, _p(h), _s(stream)), "chord_silu_mul")


def chord_combine_plan(topk_ids, topk_w, E: int, pair_w, stream=None):
    T, topk = topk_ids.shape
    _check(load().chord_combine_plan(_p(topk_ids), _p(topk_w), T, topk, E, _p(pair_w), _s(stream)),
           "chord_combine_plan")


def chord_w4a16_moe_gemm_combine(A, packed, E: int, N: int, K: int, sorted_ids, expert_ids, num_tokens_padded,
                                 block_m: int, topk: int, pair_w, C2, out, workspace=None, opts=None, stream=None):
    T = out.shape[0]
    _check(load().chord_w4a16_moe_gemm_combine(
        _p(A), _p(packed), _nbytes(packed), E, N, K, _p(sorted_ids), _p(expert_ids), _p(num_tokens_padded),
        sorted_ids.numel(), block_m, T, topk, _p(pair_w), _p(C2), _p(out), _p(workspace),
        0 if workspace is None else _nbytes(workspace), _o(opts), _s(stream)), "chord_w4a16_moe_gemm_combine")


def chord_combine_finish(C2, topk_ids, topk_w, E: int, out, stream=None):
    T, topk = topk_ids.shape
    H = out.shape[1]
    _check(load().chord_combine_finish(_p(C2), _p(topk_ids), _p(topk_w), T, topk, E, H, _p(out), _s(stream)),
           "chord_combine_finish")


def chord_moe_combine(C2, topk_ids, topk_w, E: int, out, stream=None):
    """C2 bf16 or float32 [T * topk, H] (the dtype of the tensor selects c2_dtype)."""
    import torch
    T, topk = topk_ids.shape
    c2_dtype = DTYPE_F32 if C2.dtype == torch.float32 else DTYPE_BF16
    _check(load().chord_moe_combine(_p(C2), c2_dtype, _p(topk_ids), _p(topk_w), T, topk, E, C2.shape[1], _p(out),
                                    _s(stream)), "chord_moe_combine")


def chord_layer_workspace_bytes(T: int, topk: int, E: int, H: int, I: int, block_m: int = 0) -> int:
    return load().chord_layer_workspace_bytes(T, topk, E, H, I, block_m)


def chord_moe_layer(x, topk_ids, topk_w, E: int, E_global: int, I: int, packed_w13, packed_w2, workspace, out,
                    block_m: int = 0, opts=None, stream=None):
    T, H = x.shape
    topk = topk_ids.shape[1]
    _check(load().chord_moe_layer(_p(x), _p(topk_ids), _p(topk_w), T, topk, E, E_global, H, I, _p(packed_w13),
                                  _nbytes(packed_w13), _p(packed_w2), _nbytes(packed_w2), block_m, _p(workspace),
                                  _nbytes(workspace), _p(out), _o(opts), _s(stream)), "chord_moe_layer")


def chord_moe_layer_cached(x, topk_ids, topk_w, E: int, E_global: int, I: int, packed_w13, packed_w2, workspace,
                           out, block_m: int = 0, opts=None, stream=None):
    T, H = x.shape
    topk = topk_ids.shape[1]
    _check(load().chord_moe_layer_cached(_p(x), _p(topk_ids), _p(topk_w), T, topk, E, E_global, H, I,
                                         _p(packed_w13), _nbytes(packed_w13), _p(packed_w2), _nbytes(packed_w2),
                                         block_m, _p(workspace), _nbytes(workspace), _p(out), _o(opts), _s(stream)),
           "chord_moe_layer_cached")


def chord_moe_layer_cache_clear() -> int:
    return int(load().chord_moe_layer_cache_clear())


def chord_grouped_contiguous_workspace_bytes(M: int, E: int) -> int:
    return load().chord_grouped_contiguous_workspace_bytes(M, E)


def chord_grouped_contiguous_gemm(A, m_indices, packed, E: int, N: int, K: int, C, workspace, opts=None,
                                  stream=None):
    """A bf16 [M, K] grouped per expert (segments padded to 128 rows), m_indices int32 [M] (-1: padding)."""
    _check(load().chord_grouped_contiguous_gemm(_p(A), A.shape[0], _p(m_indices), _p(packed), _nbytes(packed), E, N,
                                                K, _p(C), _p(workspace), _nbytes(workspace), _o(opts), _s(stream)),
           "chord_grouped_contiguous_gemm")


def chord_grouped_masked_workspace_bytes(G: int, max_m: int, expected_m: int) -> int:
    return load().chord_grouped_masked_workspace_bytes(G, max_m, expected_m)


def chord_grouped_masked_gemm(A, masked_m, expected_m: int, packed, N: int, K: int, C, workspace, opts=None,
                              stream=None):
    """A bf16 [G, max_m, K], masked_m int32 [G]; C flat [G * max_m, N]."""
    G, max_m, _ = A.shape
    _check(load().chord_grouped_masked_gemm(_p(A), G, max_m, _p(masked_m), expected_m, _p(packed), _nbytes(packed),
                                            N, K, _p(C), _p(workspace), _nbytes(workspace), _o(opts), _s(stream)),
           "chord_grouped_masked_gemm")


def chord_selftest_wait_timeout(stream=None):
    _check(load().chord_selftest_wait_timeout(_s(stream)), "chord_selftest_wait_timeout")


def chord_get_device_error(stream=None) -> int:
    code = ctypes.c_int32(0)
    _check(load().chord_get_device_error(_s(stream), ctypes.byref(code)), "chord_get_device_error")
    return code.value
