"""Seeded synthetic workloads for the W4A16 INT4 mixture-of-experts expert GEMM.

This module only draws inputs.  It holds none of the method's arithmetic (no
dequantisation, no GEMM, no activation, no combine): it is shared by the CPU
oracle's tests, the CUDA parity tests and ``bench.py`` so that both sides see
the same bits.

Shapes follow the Kimi-K2.x expert shapes the Chord article measures on
("vLLM x Novita AI: Chord", section "Measurement" and its gate_up + down table):
hidden H = 7168, intermediate I = 2048 (EP8, 48 of 384 experts local) or I = 256
(TP8, all 384 experts), top-8 routing.  The small case is sized for a CPU that
finishes in seconds.

Value distributions (all drawn with numpy PCG64; one independent child stream
per tensor, spawned from the workload seed, so a tensor does not depend on the
sizes of the others):

* activations x ~ N(0, 1) drawn in float32, rounded to bf16 (round to nearest
  even, by torch's dtype conversion);
* weight codes uniform in {0, ..., 15} (uint4 with offset 8);
* group-32 scales |N(0, 0.02)| + 1e-3 drawn and summed in float32, then rounded
  to bf16 once;
* routing: ``softmax`` (top-2 of a softmax over N(0,1) logits, weights
  renormalised), ``uniform`` (8 distinct experts uniformly at random, weights a
  softmax over 8 N(0,1) logits) or ``zipf`` (expert popularity proportional to
  rank^-s over a seeded permutation of the experts, 8 distinct experts drawn
  without replacement by Gumbel-top-k, weights as for ``uniform``).  Experts
  at or above ``E_local`` are routed to another rank and appear as -1.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

GROUP = 32

# tensor stream indices within a workload seed
_S_ROUTE_IDS, _S_ROUTE_W, _S_X, _S_W13_Q, _S_W13_S, _S_W2_Q, _S_W2_S = range(7)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One MoE layer shape plus its routing recipe."""
    name: str
    T: int            # tokens
    E: int            # local experts (the experts this GPU holds)
    E_global: int     # experts the router draws from
    topk: int
    H: int            # hidden size = K of gate_up = N of down
    I: int            # intermediate size; gate_up N = 2 * I
    routing: str      # "softmax" | "uniform" | "zipf"
    seed: int
    zipf_s: float = 1.2

    @property
    def P(self) -> int:
        """Number of routed (token, k) pairs, local or not."""
        return self.T * self.topk


def _bf16(a: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round to nearest even."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact widening)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _streams(seed: int):
    return [np.random.Generator(np.random.PCG64(s))
            for s in np.random.SeedSequence(seed).spawn(7)]


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z - z.max(axis=1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=1, keepdims=True)


def make_routing(w: Workload, rank: int = 0):
    """Return (topk_ids int32 [T, topk], topk_w float32 [T, topk]).

    Expert-parallel share ``rank`` holds global experts [rank*E, rank*E + E);
    ``topk_ids`` holds their local ids in [0, E) and -1 for pairs routed to
    experts outside this share.  Every share sees the same global routing.
    """
    st = _streams(w.seed)
    ri, rw = st[_S_ROUTE_IDS], st[_S_ROUTE_W]
    T, G, k = w.T, w.E_global, w.topk
    if w.routing == "softmax":
        logits = ri.standard_normal((T, G), dtype=np.float32).astype(np.float64)
        probs = _softmax_rows(logits)
        ids = np.argsort(-logits, axis=1, kind="stable")[:, :k]
        sel = np.take_along_axis(probs, ids, axis=1)
        wts = (sel / sel.sum(axis=1, keepdims=True)).astype(np.float32)
    elif w.routing in ("uniform", "zipf"):
        if w.routing == "uniform":
            keys = ri.random((T, G))
            ids = np.argsort(keys, axis=1, kind="stable")[:, :k]
        else:
            perm = ri.permutation(G)
            pop = np.empty(G, dtype=np.float64)
            pop[perm] = np.arange(1, G + 1, dtype=np.float64) ** (-w.zipf_s)
            gumbel = -np.log(-np.log(ri.random((T, G))))
            keys = np.log(pop)[None, :] + gumbel
            ids = np.argsort(-keys, axis=1, kind="stable")[:, :k]
        logits = rw.standard_normal((T, k), dtype=np.float32).astype(np.float64)
        wts = _softmax_rows(logits).astype(np.float32)
    else:
        raise ValueError(f"unknown routing {w.routing!r}")
    ids = ids.astype(np.int32)
    lo = rank * w.E
    ids = np.where((ids >= lo) & (ids < lo + w.E), ids - lo, -1).astype(np.int32)
    return np.ascontiguousarray(ids), np.ascontiguousarray(wts)


def make_x(w: Workload) -> np.ndarray:
    """bf16 bits [T, H], x ~ N(0, 1)."""
    st = _streams(w.seed)[_S_X]
    return _bf16(st.standard_normal((w.T, w.H), dtype=np.float32))


def _codes(rng, shape):
    return rng.integers(0, 16, size=shape, dtype=np.uint8)


def _scales(rng, shape):
    s = np.abs(rng.standard_normal(shape, dtype=np.float32) * np.float32(0.02))
    return _bf16(s + np.float32(1e-3))


def make_w13(w: Workload):
    """gate_up weights: codes uint8 [E, 2I, H] in 0..15, scales bf16 bits [E, 2I, H/32].

    Rows 0..I-1 are the gate projection, rows I..2I-1 the up projection.
    """
    st = _streams(w.seed)
    return (_codes(st[_S_W13_Q], (w.E, 2 * w.I, w.H)),
            _scales(st[_S_W13_S], (w.E, 2 * w.I, w.H // GROUP)))


def make_w2(w: Workload):
    """down weights: codes uint8 [E, H, I] in 0..15, scales bf16 bits [E, H, I/32]."""
    st = _streams(w.seed)
    return (_codes(st[_S_W2_Q], (w.E, w.H, w.I)),
            _scales(st[_S_W2_S], (w.E, w.H, w.I // GROUP)))


def random_codes(seed: int, shape) -> np.ndarray:
    """Stand-alone uint4 codes for unit tests."""
    return _codes(np.random.Generator(np.random.PCG64(seed)), shape)


def random_scales(seed: int, shape) -> np.ndarray:
    """Stand-alone bf16 group scales for unit tests."""
    return _scales(np.random.Generator(np.random.PCG64(seed)), shape)


def random_bf16(seed: int, shape, std: float = 1.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return _bf16(rng.standard_normal(shape, dtype=np.float32) * np.float32(std))


def random_ids(seed: int, T: int, topk: int, E: int, p_nonlocal: float = 0.0,
               distinct: bool = True) -> np.ndarray:
    """Arbitrary routing ids in [0, E) with a share of -1 entries (for edge tests)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    if distinct and topk <= E:
        ids = np.argsort(rng.random((T, E)), axis=1)[:, :topk]
    else:
        ids = rng.integers(0, E, size=(T, topk))
    if p_nonlocal > 0:
        ids = np.where(rng.random((T, topk)) < p_nonlocal, -1, ids)
    return np.ascontiguousarray(ids.astype(np.int32))


def random_weights(seed: int, T: int, topk: int) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed))
    return _softmax_rows(rng.standard_normal((T, topk))).astype(np.float32)


# --- the five measured workloads -------------------------------------------

TINY = Workload("tiny_T16_E8_top2_H256_I128", T=16, E=8, E_global=8, topk=2,
                H=256, I=128, routing="softmax", seed=0)
EP8_DECODE = Workload("ep8_decode_T512_E48of384_top8_H7168_I2048", T=512, E=48,
                      E_global=384, topk=8, H=7168, I=2048, routing="uniform", seed=1)
EP8_PREFILL = Workload("ep8_prefill_T8192_E48of384_top8_H7168_I2048", T=8192, E=48,
                       E_global=384, topk=8, H=7168, I=2048, routing="uniform", seed=2)
TP8_T = (1, 16, 128, 1024, 4096)


def tp8(T: int) -> Workload:
    return Workload(f"tp8_T{T}_E384_top8_H7168_I256", T=T, E=384, E_global=384,
                    topk=8, H=7168, I=256, routing="uniform", seed=3)


SKEWED = Workload("skewed_zipf1.2_T16384_E48of384_top8_H7168_I2048", T=16384, E=48,
                  E_global=384, topk=8, H=7168, I=2048, routing="zipf", seed=4)

# The skewed configuration's own description has cold experts with 0-2 rows,
# which Zipf(1.2) over 384 experts does not produce for the 48 local ones
# (their fewest rows are about 30).  A steeper Zipf(2.0) does: hot experts with
# thousands of rows, about twenty local experts with 0-8 rows and one with none
# (seed 5).  It is a parity case and a measurement of the per-block regime.
SKEWED_COLD = Workload("skewed_cold_zipf2.0_T16384_E48of384_top8_H7168_I2048", T=16384, E=48,
                       E_global=384, topk=8, H=7168, I=2048, routing="zipf", seed=5, zipf_s=2.0)

ALL = {w.name: w for w in (TINY, EP8_DECODE, EP8_PREFILL, *[tp8(t) for t in TP8_T], SKEWED, SKEWED_COLD)}


def by_name(name: str) -> Optional[Workload]:
    return ALL.get(name)
