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


def test_no_alloc_align_matches_workspace_align_on_two_calls():
    # first a large call (many slices, many experts), then a smaller one that
    # reads fewer scratch entries than the first left behind
    cases = [(wl.SKEWED, 256), (wl.EP8_DECODE, 16)]
    for w, bm in cases:
        ids, _ = wl.make_routing(w)
        ids_d = torch.from_numpy(ids).to(DEV)
        got = _no_alloc(ids_d, w.E, bm)
        want = _with_workspace(ids_d, w.E, bm)
        assert got[2] == want[2]
        np.testing.assert_array_equal(got[0], want[0])
        np.testing.assert_array_equal(got[1], want[1])
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
    assert chord.chord_get_device_error() == 0
