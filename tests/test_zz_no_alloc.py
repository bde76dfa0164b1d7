"""chord_moe_align_noalloc: the routing alignment for callers that cannot
allocate device memory (for example code running during a CUDA graph capture
that forbids allocation, or an engine plugin limited to the engine's buffers).
Its scratch is a fixed array inside the library instead of a caller buffer.

It must give exactly what chord_moe_align gives (integer outputs: bit for
bit), call after call, even when a later call needs less scratch than an
earlier one left filled.  This file is collected last so a failure here
cannot hide the result of any other test."""
import numpy as np
import pytest
import torch

import oracle
import w4a16_int4_mixture_moe_gb300 as chord
import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    chord.build()
    chord.load()
    oracle.build()
    chord.chord_get_device_error()


def _buffers(T, topk, E, bm):
    cap = chord.chord_align_capacity(T, topk, E, bm)
    s = torch.full((max(cap, 1),), -7, dtype=torch.int32, device=DEV)[:cap]
    e = torch.full((max(cap // bm, 1),), -7, dtype=torch.int32, device=DEV)[:cap // bm]
    n = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    return s, e, n


def _with_workspace(ids_d, E, bm):
    T, topk = ids_d.shape
    s, e, n = _buffers(T, topk, E, bm)
    ws = torch.empty(chord.chord_align_workspace_bytes(T, topk, E), dtype=torch.uint8, device=DEV)
    chord.chord_moe_align(ids_d, E, bm, s, e, n, ws)
    return s.cpu().numpy(), e.cpu().numpy(), int(n.item())


def _no_alloc(ids_d, E, bm):
    T, topk = ids_d.shape
    s, e, n = _buffers(T, topk, E, bm)
    chord.chord_moe_align_noalloc(ids_d, E, bm, s, e, n)
    return s.cpu().numpy(), e.cpu().numpy(), int(n.item())


def _oracle(ids, E, bm):
    s, e, n = oracle.moe_align(ids, E, bm)
    return np.asarray(s), np.asarray(e), int(n)


def test_no_alloc_align_matches_workspace_align_on_two_calls():
    # first a large call (32 slices of 4096 pairs x 48 experts of scratch),
    # then smaller ones: one slice (EP8 decode: 4096 pairs) and two slices of
    # 64 experts, which read fewer scratch entries than the first left filled
    cases = [(wl.make_routing(wl.SKEWED)[0], wl.SKEWED.E, 256),
             (wl.make_routing(wl.EP8_DECODE)[0], wl.EP8_DECODE.E, 16),
             (wl.random_ids(5, 1024, 8, 64, p_nonlocal=0.1), 64, 32)]
    for ids, E, bm in cases:
        ids_d = torch.from_numpy(ids).to(DEV)
        got = _no_alloc(ids_d, E, bm)
        want = _with_workspace(ids_d, E, bm)
        orc = _oracle(ids, E, bm)
        assert got[2] == want[2] == orc[2]
        for i in (0, 1):
            np.testing.assert_array_equal(got[i], want[i])
            np.testing.assert_array_equal(got[i], orc[i])
    assert chord.chord_get_device_error() == 0


def test_no_alloc_align_repeat_and_limit():
    ids = wl.random_ids(3, 4096, 8, 384)
    ids_d = torch.from_numpy(ids).to(DEV)
    first = _no_alloc(ids_d, 384, 32)
    second = _no_alloc(ids_d, 384, 32)
    want = _with_workspace(ids_d, 384, 32)
    for a, b, c in zip(first, second, want):
        np.testing.assert_array_equal(np.asarray(a), np.asarray(c))
        np.testing.assert_array_equal(np.asarray(b), np.asarray(c))
    # above the fixed scratch (E = 1024 allows 262,144 pairs): refused, nothing enqueued
    T = 262144 // 8 + 1
    big = torch.zeros((T, 8), dtype=torch.int32, device=DEV)
    s, e, n = _buffers(T, 8, 1024, 8)
    with pytest.raises(chord.ChordError) as ei:
        chord.chord_moe_align_noalloc(big, 1024, 8, s, e, n)
    assert ei.value.status == 4  # CHORD_ERR_BUFFER_TOO_SMALL
    torch.cuda.synchronize()
    # no kernel ran: the outputs still hold their fill
    assert (s == -7).all() and (e == -7).all() and (n == -7).all()
    assert chord.chord_get_device_error() == 0
