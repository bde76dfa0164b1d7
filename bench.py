"""Benchmark of the W4A16 INT4 MoE expert layer on GB300 (one JSON line).

A step is one pass of the whole hot path over one batch: moe_align ->
gate_up GEMM -> SiLU*up -> down GEMM -> top-k combine, every step of it a
libchord.so kernel launched through the C ABI.  The default workload is the
Kimi-K2-shaped EP8 decode layer (48 local experts of 384, T = 512 tokens,
top-8, H = 7168, I = 2048); the same run also times the EP8 prefill layer
(T = 8192, the tensor-core regime) and reports it under ``regimes.prefill``.
``--workload`` picks another of the five configurations.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun (N > 1) rank r runs expert-parallel share r of the layer
(global experts [48r, 48r + 48) of the same tokens): the shares are
independent, nothing crosses ranks on the data path, and the reported time
is the max over ranks of the time per layer call (all ranks' shares run
concurrently).  ``--impl reference`` times the CPU oracle on the host cores
instead (rank 0 only); that arm loads no CUDA code.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "W4A16 MoE µs/call; achieved HBM GB/s (decode) & BF16 TFLOP/s (prefill)"
UNIT = "µs/call"
WORKLOADS = {
    "ep8_decode": wl.EP8_DECODE, "ep8_prefill": wl.EP8_PREFILL, "skewed": wl.SKEWED, "tiny": wl.TINY,
    "skewed_cold": wl.SKEWED_COLD,
    **{f"tp8_T{t}": wl.tp8(t) for t in wl.TP8_T},
}
L2_BYTES = 129 * 2 ** 20
KERNEL_SRC = {
    "tc": os.path.join(ROOT, "w4a16_int4_mixture_moe_gb300", "csrc", "chord_gemm_tc.cu"),
    "warp_mma": os.path.join(ROOT, "w4a16_int4_mixture_moe_gb300", "csrc", "chord_gemm_decode.cu"),
}

KERNEL_NAME = {"tc": "gemm_tc_kernel", "warp_mma": "gemm_decode_kernel"}

# ----------------------------------------------------------------- accounting

def routing_stats(ids, E):
    flat = ids.ravel()
    local = flat[(flat >= 0) & (flat < E)]
    rows_per_expert = np.bincount(local, minlength=E)
    return rows_per_expert


def gemm_algorithmic(rows_per_expert, N, K, out_cols=None):
    """Bytes and FLOPs one GEMM launch must move / do: packed INT4 + scales of
    every expert with at least one row, activations read, outputs written
    (out_cols bf16 columns per row: N, or N/2 with the fused SiLU * up), sorted
    ids read; FLOPs over real rows only."""
    rows = int(rows_per_expert.sum())
    used = int((rows_per_expert > 0).sum())
    wbytes = used * N * K * 9 // 16
    nbytes = wbytes + rows * K * 2 + rows * (N if out_cols is None else out_cols) * 2 + rows * 4
    flops = 2 * rows * N * K
    return nbytes, flops


def select_block_m(T, topk, E_local, E_global):
    """The library's tok_e block-size rule restated on the host (the reference
    arm names the block size in its config without loading the CUDA library;
    a CPU test checks this against chord_select_block_m over many shapes).
    A block holds the mean plus three standard deviations of a Poisson count
    of tok_e = T * topk / E_global rows, in steps of 16, at most 256; 8 when
    that fits 8; 32 when it exceeds 32 but the mean plus two standard
    deviations fits 32."""
    eg = E_global if E_global > 0 else (E_local if E_local > 0 else 1)
    tok_e = T * (topk if topk > 0 else 1) / eg
    need = tok_e + 3.0 * math.sqrt(tok_e) + 1.0
    if need <= 8.0:
        return 8
    if need > 32.0 and tok_e + 2.0 * math.sqrt(tok_e) + 1.0 <= 32.0:
        return 32
    return min(256, int(math.ceil(need / 16.0)) * 16)


def arm_config(w, bm, world):
    """The config object of the JSON line, identical in both arms: the
    workload, its routing statistics and the regime of its dominant GEMM."""
    ids, _ = wl.make_routing(w)
    rpe = routing_stats(ids, w.E)
    b1, f1_ = gemm_algorithmic(rpe, 2 * w.I, w.H)
    peaks = load_peaks()
    # The gate_up GEMM dominates.  It is HBM-bound when its algorithmic FLOP per
    # byte is below the machine's ridge (measured BF16 peak / measured HBM
    # bandwidth), tensor-bound above it.
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    regime = "decode" if f1_ / max(b1, 1) < ridge else "prefill"
    routed = int((rpe > 0).sum()) * (2 * w.I * w.H + w.H * w.I) * 9 // 16
    cfg = {"workload": w.name, "T": w.T, "E_local": w.E, "E_global": w.E_global, "topk": w.topk, "H": w.H,
           "I": w.I, "block_m": bm, "regime": regime, "local_pairs": int(rpe.sum()),
           "tok_e": round(float(rpe.sum()) / w.E, 2),
           "parallelism": f"expert-parallel shares x{world} (share r = global experts [{w.E}r, {w.E}r+{w.E}))",
           "l2": (f"inputs larger than L2: {routed / 1e6:.0f} MB of packed weights routed per step vs "
                  f"{L2_BYTES / 1e6:.0f} MB L2" if routed >= 2 * L2_BYTES else
                  f"L2 flushed before every timed step: {routed / 1e6:.1f} MB of packed weights routed per step "
                  f"fit in the {L2_BYTES / 1e6:.0f} MB L2")}
    return cfg, regime, peaks


def reduce_max(values, dist, device):
    """Element-wise maximum of per-rank float values over all ranks (the
    slowest rank sets the job's time); identity without a process group."""
    if dist is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def per_call_us(total_ms, steps):
    """Microseconds per layer call from the max-over-ranks time of `steps`
    calls.  Every rank runs its own expert-parallel share of the same call
    concurrently, so N ranks together complete one call per step: the time is
    not divided by the rank count."""
    return total_ms * 1e3 / max(steps, 1)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "src": "fallback"}


def kernel_sha(kind):
    h = hashlib.sha256()
    for p in (KERNEL_SRC[kind], os.path.join(os.path.dirname(KERNEL_SRC[kind]), "chord_common.cuh")):
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(kind, workload, which="gate_up"):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kind}_gemm_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m_sha = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", txt)
    m_b = re.search(rf"dram_bytes_per_launch_{which}:\s*([0-9.eE+]+)", txt)
    if not (m_sha and m_b) or m_sha.group(1) != kernel_sha(kind):
        return None
    return float(m_b.group(1))


def roofline(bound, nbytes, flops, us, peaks, kname, traffic):
    """Roofline object of one GEMM launch: achieved = algorithmic bytes (HBM
    bound) or FLOPs (tensor bound) / its event-timed duration.  A tensor-bound
    launch reports its fraction of the sustained cuBLAS rate (it runs inside a
    long step) as `frac` and of the burst rate as `frac_burst`."""
    if bound == "hbm":
        ach = nbytes / (us * 1e-6) / 1e9
        return {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic, "kernel": kname,
                "peak_src": peaks["src"]}
    ach = flops / (us * 1e-6) / 1e12
    pk, pb = peaks["bf16_tflops_sustained"], peaks["bf16_tflops"]
    return {"bound": "tensor", "achieved": round(ach, 1), "peak": pk, "unit": "TFLOP/s",
            "frac": round(ach / pk, 4), "peak_burst": pb, "frac_burst": round(ach / pb, 4),
            "traffic": traffic, "kernel": kname, "peak_src": peaks["src"]}


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons around a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", self.gpu_id], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()
        t0 = time.time()
        while not self.samples and time.time() - t0 < 5:
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t_lo, t_hi):
        win = [p for t, p in self.samples if t_lo - 0.25 <= t <= t_hi + 0.25]
        if not win and self.samples:  # region shorter than the sampling period: nearest samples
            win = [min(self.samples, key=lambda s: abs(s[0] - (t_lo + t_hi) / 2))[1]]
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(p[1]) for p in win if num(p[1]) is not None]
        mx = [num(p[2]) for p in win if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in win for n, v in zip(names, p[5:9]) if v.strip().lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(win)}


def gpu_id_for(torch, dev):
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        return vis.split(",")[dev] if vis else str(dev)


# ------------------------------------------------------------------ CPU oracle

def oracle_sample(w, target_s, nthreads=None, block_m=8):
    """Time the oracle layer on a token sample sized to about target_s seconds;
    return (us per full call, sample description, cores, seconds per sample,
    tokens in the sample)."""
    import oracle
    oracle.build()
    ids, wts = wl.make_routing(w)
    x = wl.make_x(w)
    w13, w2 = wl.make_w13(w), wl.make_w2(w)
    cores = oracle.threads(nthreads)
    local = (ids >= 0) & (ids < w.E)
    total_pairs = int(local.sum())

    def run(nt):
        t0 = time.perf_counter()
        oracle.moe_layer(x[:nt], ids[:nt], wts[:nt], w13, w2, w.E, block_m=block_m, nthreads=cores)
        return time.perf_counter() - t0

    nt = min(w.T, 4)
    dt = run(nt)
    while nt < w.T and dt < target_s / 4:
        nt = min(w.T, nt * 4)
        dt = run(nt)
    pairs = int(local[:nt].sum())
    us_full = dt * 1e6 * (total_pairs / max(pairs, 1))
    desc = (f"oracle layer on the first {nt} of {w.T} tokens ({pairs} of {total_pairs} local pairs), "
            f"{dt:.2f} s; scaled to the full call by local pairs")
    return us_full, desc, cores, dt, nt


def run_reference(args, w):
    """The reference arm: the CPU oracle as it stands, on the host cores, on a
    bounded token sample of the same workload.  It loads no CUDA code: the
    block size in its config comes from the host restatement of the rule."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    steps, warmup = args.steps, args.warmup
    bm = args.block_m or select_block_m(w.T, w.topk, w.E, w.E_global)
    cfg, _, _ = arm_config(w, bm, int(os.environ.get("WORLD_SIZE", "1")))
    budget = 150.0
    per_step = max(0.5, min(20.0, budget / max(1, steps + warmup)))
    _, desc, cores, _, nt = oracle_sample(w, per_step, block_m=bm)
    import oracle
    ids, wts = wl.make_routing(w)
    x = wl.make_x(w)
    w13, w2 = wl.make_w13(w), wl.make_w2(w)
    local = (ids >= 0) & (ids < w.E)
    scale = local.sum() / max(1, local[:nt].sum())
    for _ in range(warmup):
        oracle.moe_layer(x[:nt], ids[:nt], wts[:nt], w13, w2, w.E, block_m=bm, nthreads=cores)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.moe_layer(x[:nt], ids[:nt], wts[:nt], w13, w2, w.E, block_m=bm, nthreads=cores)
    el = time.perf_counter() - t0
    us = el / max(steps, 1) * 1e6 * scale
    line = {"impl": "reference", "metric": METRIC, "value": round(us, 1), "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "warmup": warmup, "ms_per_step": round(el / max(steps, 1) * 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": round(us, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(us, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU arm

GROUPED = {
    # the grouped contracts on the EP8 shapes: contiguous segments of the
    # prefill routing's per-expert row counts (padded to 128 rows), and masked
    # budgets of 32 rows holding the decode routing's counts
    "grouped_contiguous_ep8_prefill": ("contiguous", wl.EP8_PREFILL),
    "grouped_masked_ep8_decode": ("masked", wl.EP8_DECODE),
}


def run_grouped(args, name):
    """gate_up then down through one grouped contract; value = their µs sum
    (the pages' grouped rows time gate_up + down)."""
    import torch
    import w4a16_int4_mixture_moe_gb300 as chord
    contract, w = GROUPED[name]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    chord.build()
    chord.load()
    ids, _ = wl.make_routing(w)
    counts = routing_stats(ids, w.E)
    E, H, I = w.E, w.H, w.I
    rng = np.random.default_rng(w.seed + 100)
    if contract == "contiguous":
        m_idx = np.concatenate([np.concatenate([np.full(c, e), np.full(-(-c // 128) * 128 - c, -1)])
                                for e, c in enumerate(counts)]).astype(np.int32)
        rows_a = m_idx.size
        idx_h = torch.from_numpy(m_idx)
        ws1 = chord.chord_grouped_contiguous_workspace_bytes(rows_a, E)
        shape_a, max_m, expected_m = (rows_a,), 0, 0
    else:
        max_m = 32
        expected_m = max(1, int(round(counts.mean())))
        masked = np.minimum(counts, max_m).astype(np.int32)
        rows_a = E * max_m
        idx_h = torch.from_numpy(masked)
        ws1 = chord.chord_grouped_masked_workspace_bytes(E, max_m, expected_m)
        shape_a = (E, max_m)
    x = torch.from_numpy(wl._bf16(rng.standard_normal((rows_a, H), dtype=np.float32)).view(np.int16))
    x = x.view(torch.bfloat16).to(dev).reshape(*shape_a, H)
    hmid = torch.randn((rows_a, I), device=dev).to(torch.bfloat16).reshape(*shape_a, I)
    c13, s13 = wl.make_w13(w)
    p13 = torch.empty(chord.chord_packed_weight_bytes(E, 2 * I, H), dtype=torch.uint8, device=dev)
    chord.chord_pack_weights(torch.from_numpy(c13).to(dev), torch.from_numpy(s13.view(np.int16)).to(dev).view(torch.bfloat16), p13)
    del c13, s13
    c2, s2 = wl.make_w2(w)
    p2 = torch.empty(chord.chord_packed_weight_bytes(E, H, I), dtype=torch.uint8, device=dev)
    chord.chord_pack_weights(torch.from_numpy(c2).to(dev), torch.from_numpy(s2.view(np.int16)).to(dev).view(torch.bfloat16), p2)
    del c2, s2
    idx = idx_h.to(dev)
    ws = torch.empty(max(ws1, 16), dtype=torch.uint8, device=dev)
    C1 = torch.empty((rows_a, 2 * I), dtype=torch.bfloat16, device=dev)
    C2 = torch.empty((rows_a, H), dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream()

    def gemm(A, p, N, K, C):
        if contract == "contiguous":
            chord.chord_grouped_contiguous_gemm(A, idx, p, E, N, K, C, ws, stream=stream)
        else:
            chord.chord_grouped_masked_gemm(A, idx, expected_m, p, N, K, C, ws, stream=stream)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        gemm(x, p13, 2 * I, H, C1)
        if ev:
            ev[1].record(stream)
        gemm(hmid, p2, H, I, C2)
        if ev:
            ev[2].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_id_for(torch, 0))
    sampler.start()
    t_lo = time.time()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    g1 = g2 = 0.0
    for _ in range(args.steps):
        step(ev)
        torch.cuda.synchronize()
        g1 += ev[0].elapsed_time(ev[1])
        g2 += ev[1].elapsed_time(ev[2])
    t_hi = time.time()
    sampler.stop()
    g1, g2 = g1 / args.steps, g2 / args.steps
    # end to end: activations and indices from pinned host memory, outputs back
    x_h, idx_p = x.cpu().pin_memory(), idx_h.pin_memory()
    out_h = torch.empty_like(C2, device="cpu").pin_memory()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        x.copy_(x_h, non_blocking=True)
        idx.copy_(idx_p, non_blocking=True)
        step()
        out_h.copy_(C2, non_blocking=True)
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_us = f0.elapsed_time(f1) * 1e3 / args.steps
    peaks = load_peaks()
    b1, f1_ = gemm_algorithmic(counts, 2 * I, H)
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    bmg = (chord.chord_select_block_m(rows_a, 1, E, E, 2 * I, H) if contract == "contiguous" else
           chord.chord_select_block_m(expected_m, 1, 1, 1, 2 * I, H))
    kind = "warp_mma" if chord.chord_select_kernel(bmg, 2 * I, H) == chord.KERNEL_WARP_MMA else "tc"
    roof = roofline("hbm" if f1_ / b1 < ridge else "tensor", b1, f1_, g1 * 1e3, peaks,
                    KERNEL_NAME[kind] + " (gate_up)", None)
    cfg = {"workload": name, "contract": contract, "E": E, "H": H, "I": I, "rows": int(counts.sum()),
           "rows_with_padding": rows_a, "max_m": max_m or None, "expected_m": expected_m or None, "block_m": bmg,
           "parallelism": "one GPU",
           "l2": "inputs larger than L2: packed weights streamed per step exceed the 129 MB L2"}
    line = {"metric": "W4A16 MoE grouped gate_up + down µs/call", "value": round((g1 + g2) * 1e3, 2), "unit": UNIT,
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(g1 + g2, 4),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": cfg,
            "gemm_us": {"gate_up": round(g1 * 1e3, 2), "down": round(g2 * 1e3, 2)},
            "roofline": roof, "clocks": sampler.summary(t_lo, t_hi),
            "e2e": {"value": round(e2e_us, 2), "unit": UNIT, "h2d_bytes_per_step": x.numel() * 2 + idx.numel() * 4,
                    "d2h_bytes_per_step": C2.numel() * 2},
            "gpu_launches": 4 * args.steps}
    print(json.dumps(line), flush=True)


class LayerRig:
    """One workload's layer on the GPU: packed weights, routing and buffers
    resident in HBM, the step (align -> gate_up [+ SiLU * up] -> down ->
    combine, every kernel through the C ABI) captured as CUDA graphs, and the
    public chord_moe_layer call for the end-to-end and host-cost timings."""

    def __init__(self, chord, torch, w, dev, rank, args):
        self.chord, self.torch, self.w, self.dev = chord, torch, w, dev
        # Rank r runs expert-parallel share r (global experts [r*E, r*E + E)) of the
        # same tokens; shares past E_global / E repeat.
        shares = max(1, w.E_global // w.E)
        self.ids, self.wts = wl.make_routing(w, rank % shares)
        self.x = wl.make_x(w)
        T, topk, E, H, I = w.T, w.topk, w.E, w.H, w.I
        P = T * topk
        bm = args.block_m or chord.chord_select_block_m(T, topk, E, w.E_global, 2 * I, H)
        self.bm = bm
        # Decode regime (the warp-level kernel runs gate_up): w13 packed with its
        # gate and up rows interleaved and SiLU * up in the GEMM's epilogue.
        # tcgen05 kernel: the separate SiLU * up pass, measured faster there (the
        # accumulator drain is on the tensor pipe's critical path).  --unfused and
        # --fused force either.
        fused = chord.chord_select_kernel(bm, 2 * I, H) == chord.KERNEL_WARP_MMA
        fused = (fused or args.fused) and not args.unfused
        self.fused = fused
        c13, s13 = wl.make_w13(w)
        w13_layout = chord.LAYOUT_GATE_UP_INTERLEAVED if fused else chord.LAYOUT_TCGEN05
        self.p13 = torch.empty(chord.chord_packed_weight_bytes(E, 2 * I, H, w13_layout), dtype=torch.uint8,
                               device=dev)
        chord.chord_pack_weights(torch.from_numpy(c13).to(dev),
                                 torch.from_numpy(s13.view(np.int16)).to(dev).view(torch.bfloat16), self.p13,
                                 layout=w13_layout)
        del c13, s13
        c2, s2 = wl.make_w2(w)
        self.p2 = torch.empty(chord.chord_packed_weight_bytes(E, H, I), dtype=torch.uint8, device=dev)
        chord.chord_pack_weights(torch.from_numpy(c2).to(dev),
                                 torch.from_numpy(s2.view(np.int16)).to(dev).view(torch.bfloat16), self.p2)
        del c2, s2
        torch.cuda.synchronize()

        cap = chord.chord_align_capacity(T, topk, E, bm)
        self.xd = torch.from_numpy(self.x.view(np.int16)).to(dev).view(torch.bfloat16)
        self.idd = torch.from_numpy(self.ids).to(dev)
        self.wd = torch.from_numpy(self.wts).to(dev)
        self.sorted_ids = torch.empty(cap, dtype=torch.int32, device=dev)
        self.expert_ids = torch.empty(cap // bm, dtype=torch.int32, device=dev)
        self.ntp = torch.empty(1, dtype=torch.int32, device=dev)
        self.aws = torch.empty(max(4, chord.chord_align_workspace_bytes(T, topk, E)), dtype=torch.uint8, device=dev)
        self.C1 = None if fused else torch.empty((P, 2 * I), dtype=torch.bfloat16, device=dev)
        self.h = torch.empty((P, I), dtype=torch.bfloat16, device=dev)
        self.C2 = torch.empty((P, H), dtype=torch.float32, device=dev)
        # top-k combine fused into the down GEMM (as chord_moe_layer runs it), or the separate pass
        self.fuse_combine = getattr(args, "fused_combine", False) and topk <= 32
        self.pair_w = torch.empty(P, dtype=torch.float32, device=dev)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.stream = torch.cuda.current_stream()
        mixed = getattr(args, "mixed", 0)
        fc = 1 if self.fuse_combine else -1
        self.f32_out = chord.ChordOpts(out_dtype=chord.DTYPE_F32, mixed=mixed, fuse_combine=fc)
        self.silu_opts = chord.ChordOpts(epilogue=chord.EPILOGUE_SILU_MUL if fused else chord.EPILOGUE_NONE,
                                         mixed=mixed, fuse_combine=fc)
        # K-slice / split-tail partial sums (workspace of each GEMM)
        self.split = (chord.chord_gemm_workspace_bytes(P, 2 * I, H, bm, self.silu_opts),
                      chord.chord_gemm_workspace_bytes(P, H, I, bm, self.f32_out))
        self.gws = torch.empty(max(16, *self.split), dtype=torch.uint8, device=dev)
        # align: one launch up to 4096 pairs, three above; each GEMM's launches as the
        # library reports them (the GEMM, the mixed regime's warp-level launch, a
        # split reduction); the SiLU * up pass when unfused; combine
        # split reduction); the SiLU * up pass when unfused; the combine (plan and
        # finishing pass when fused into the down GEMM)
        self.launches_per_step = ((1 if P <= 4096 else 3) + (0 if fused else 1) + (2 if self.fuse_combine else 1) +
                                  chord.chord_gemm_launch_count(P, 2 * I, H, bm, self.split[0], self.silu_opts) +
                                  chord.chord_gemm_launch_count(P, H, I, bm, self.split[1], self.f32_out))
        # public layer call: its own workspace and copies of the inputs
        self.lws = torch.empty(chord.chord_layer_workspace_bytes(T, topk, E, H, I, bm), dtype=torch.uint8,
                               device=dev)
        self.x_e, self.ids_e, self.w_e = (torch.empty_like(self.xd), torch.empty_like(self.idd),
                                          torch.empty_like(self.wd))
        used = int((routing_stats(self.ids, E) > 0).sum())
        self.routed_bytes = used * (2 * I * H + H * I) * 9 // 16
        # When the weights one step routes to fit in L2 they would stay there from
        # step to step: a buffer twice the L2 size is written before every timed
        # replay (outside the timed events) so each step reads them from HBM.
        self.small = self.routed_bytes < 2 * L2_BYTES
        self.flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev) if self.small else None

    # ---- the step, launched on stream `st`
    def gemm1(self, st):
        c = self.chord
        w = self.w
        c.chord_w4a16_moe_gemm(self.xd, w.topk, self.p13, w.E, 2 * w.I, w.H, self.sorted_ids, self.expert_ids,
                               self.ntp, self.bm, w.P, self.h if self.fused else self.C1, workspace=self.gws,
                               opts=self.silu_opts, stream=st)

    def down(self, st):
        w = self.w
        if self.fuse_combine:
            self.chord.chord_w4a16_moe_gemm_combine(self.h, self.p2, w.E, w.H, w.I, self.sorted_ids, self.expert_ids,
                                                    self.ntp, self.bm, w.topk, self.pair_w, self.C2, self.out,
                                                    workspace=self.gws, opts=self.f32_out, stream=st)
            return
        self.chord.chord_w4a16_moe_gemm(self.h, 1, self.p2, w.E, w.H, w.I, self.sorted_ids, self.expert_ids,
                                        self.ntp, self.bm, w.P, self.C2, workspace=self.gws, opts=self.f32_out,
                                        stream=st)

    def step(self, st, marks=None):
        c, w = self.chord, self.w
        c.chord_moe_align(self.idd, w.E, self.bm, self.sorted_ids, self.expert_ids, self.ntp, self.aws, stream=st)
        if marks:
            marks[0].record(st)
        self.gemm1(st)
        if marks:
            marks[1].record(st)
        if not self.fused:
            c.chord_silu_mul(self.C1, self.idd, w.E, self.h, stream=st)
        if self.fuse_combine:
            c.chord_combine_plan(self.idd, self.wd, w.E, self.pair_w, stream=st)
        if marks:
            marks[2].record(st)
        self.down(st)
        if marks:
            marks[3].record(st)
        if self.fuse_combine:
            c.chord_combine_finish(self.C2, self.idd, self.wd, w.E, self.out, stream=st)
        else:
            c.chord_moe_combine(self.C2, self.idd, self.wd, w.E, self.out, stream=st)

    def capture(self, fn):
        torch = self.torch
        fn(self.stream)
        torch.cuda.synchronize()
        side = torch.cuda.Stream(device=self.dev)
        side.wait_stream(self.stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            fn(side)
        self.stream.wait_stream(side)
        torch.cuda.synchronize()
        return g

    def timed(self, graph, reps):
        """Device time of `reps` replays (ms, summed), CUDA events on the
        launching stream: back to back, or each after an L2 flush when the
        step's weights fit in L2."""
        torch = self.torch
        if not self.small:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(self.stream)
            for _ in range(reps):
                graph.replay()
            b.record(self.stream)
            b.synchronize()
            return a.elapsed_time(b)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        for a, b in evs:
            self.flush.zero_()
            a.record(self.stream)
            graph.replay()
            b.record(self.stream)
        evs[-1][1].synchronize()
        return sum(a.elapsed_time(b) for a, b in evs)

    def gemm_times(self, nrep):
        """Per-GEMM device durations (ms): event record nodes around gate_up and
        down inside a second capture of the step, replayed nrep times."""
        torch = self.torch
        try:
            marks = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
            g_marked = self.capture(lambda st: self.step(st, marks))
        except (TypeError, RuntimeError):
            g1 = self.timed(self.capture(self.gemm1), nrep) / nrep
            g2 = self.timed(self.capture(self.down), nrep) / nrep
            return g1, g2, "each GEMM's graph replayed alone"
        g1 = g2 = 0.0
        for _ in range(nrep):
            if self.small:
                self.flush.zero_()
            g_marked.replay()
            marks[3].synchronize()
            g1 += marks[0].elapsed_time(marks[1])
            g2 += marks[2].elapsed_time(marks[3])
        return g1 / nrep, g2 / nrep, "events inside the step's graph"

    def layer_call(self, cached=True):
        """The public layer call: chord_moe_layer_cached (the layer's launches
        recorded once into a CUDA graph, replayed), or the eager chord_moe_layer."""
        w = self.w
        fn = self.chord.chord_moe_layer_cached if cached else self.chord.chord_moe_layer
        fn(self.x_e, self.ids_e, self.w_e, w.E, w.E_global, w.I, self.p13, self.p2, self.lws, self.out,
           block_m=self.bm, opts=self.silu_opts, stream=self.stream)

    def e2e(self, steps, warmup, barrier, cached=True):
        """The public layer call end to end (chord_moe_layer_cached, or the eager
        chord_moe_layer): x, ids and weights copied from pinned host memory, the
        output copied back, all inside the timed region (CUDA events on the
        launching stream).  Returns (ms summed over steps, h2d bytes per step,
        d2h bytes per step)."""
        torch = self.torch
        x_h = torch.from_numpy(self.x.view(np.int16)).view(torch.bfloat16).pin_memory()
        ids_h = torch.from_numpy(self.ids).pin_memory()
        w_h = torch.from_numpy(self.wts).pin_memory()
        out_h = torch.empty(tuple(self.out.shape), dtype=torch.bfloat16).pin_memory()

        def one():
            self.x_e.copy_(x_h, non_blocking=True)
            self.ids_e.copy_(ids_h, non_blocking=True)
            self.w_e.copy_(w_h, non_blocking=True)
            self.layer_call(cached)
            out_h.copy_(self.out, non_blocking=True)

        for _ in range(warmup):
            one()
        barrier()
        f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        f0.record(self.stream)
        for _ in range(steps):
            one()
        f1.record(self.stream)
        barrier()
        return f0.elapsed_time(f1), self.x.nbytes + self.ids.nbytes + self.wts.nbytes, self.w.T * self.w.H * 2

    def host_us_per_call(self, calls=200, cached=True):
        """Host (CPU) time of one layer enqueue through the public binding
        (cached: a graph replay after the first call; else the eager call): the
        median over `calls` calls, each issued after the stream has drained, so
        no call waits on a full launch queue."""
        torch = self.torch
        self.layer_call(cached)
        torch.cuda.synchronize()
        ts = []
        for _ in range(calls):
            t0 = time.perf_counter()
            self.layer_call(cached)
            ts.append(time.perf_counter() - t0)
            torch.cuda.synchronize()
        return float(np.median(ts)) * 1e6

    def kernel_kind(self, N, K):
        return "warp_mma" if self.chord.chord_select_kernel(self.bm, N, K) == self.chord.KERNEL_WARP_MMA else "tc"

    def split_desc(self):
        w, P = self.w, self.w.P

        def one(nbytes, N, K):
            if nbytes == 0:
                return "none"
            if self.kernel_kind(N, K) == "tc":
                return "tcgen05 split tail (last partial wave in K slices, decided on the device)"
            return f"{nbytes // (P * N * 4)} K slices"
        return {"gate_up": one(self.split[0], 2 * w.I, w.H), "down": one(self.split[1], w.H, w.I)}

    def release(self):
        for k in list(vars(self)):
            if k not in ("chord", "torch", "w", "dev"):
                setattr(self, k, None)
        self.torch.cuda.empty_cache()


def regime_summary(rig, g1, g2, peaks):
    """Both GEMMs of one workload with their algorithmic work and roofline
    fractions (the bound of each GEMM from its own FLOP per byte)."""
    w = rig.w
    rpe = routing_stats(rig.ids, w.E)
    b1, f1_ = gemm_algorithmic(rpe, 2 * w.I, w.H, out_cols=w.I if rig.fused else 2 * w.I)
    b2, f2_ = gemm_algorithmic(rpe, w.H, w.I)
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    k1, k2 = rig.kernel_kind(2 * w.I, w.H), rig.kernel_kind(w.H, w.I)
    r1 = roofline("hbm" if f1_ / b1 < ridge else "tensor", b1, f1_, g1 * 1e3, peaks, KERNEL_NAME[k1] + " (gate_up)",
                  profiled_traffic(k1, w.name, "gate_up"))
    r2 = roofline("hbm" if f2_ / b2 < ridge else "tensor", b2, f2_, g2 * 1e3, peaks, KERNEL_NAME[k2] + " (down)",
                  profiled_traffic(k2, w.name, "down"))
    ach = {"gate_up_GBps": round(b1 / (g1 * 1e-3) / 1e9, 1), "down_GBps": round(b2 / (g2 * 1e-3) / 1e9, 1),
           "gate_up_TFLOPs": round(f1_ / (g1 * 1e-3) / 1e12, 2), "down_TFLOPs": round(f2_ / (g2 * 1e-3) / 1e12, 2),
           "gate_up_bytes": b1, "down_bytes": b2, "gate_up_flops": f1_, "down_flops": f2_}
    return r1, r2, ach


def measure_prefill_regime(chord, torch, dev, rank, world, args, pg):
    """The EP8 prefill layer (T = 8192, tensor-core regime) in the same run as
    the decode line: whole-step µs per call, both GEMMs with their TFLOP/s and
    fractions of the burst and sustained BF16 rates, end to end through the
    public call."""
    w = wl.EP8_PREFILL
    sub = argparse.Namespace(**{**vars(args), "block_m": 0, "fused": False, "unfused": False, "mixed": 0})
    rig = LayerRig(chord, torch, w, dev, rank, sub)
    peaks = load_peaks()

    def barrier():
        if pg:
            pg.barrier()
        torch.cuda.synchronize()

    steps = max(1, min(args.steps, 300))
    g_step = rig.capture(rig.step)
    for _ in range(max(3, min(args.warmup, 10))):
        g_step.replay()
    sampler = ClockSampler(gpu_id_for(torch, dev.index or 0))
    sampler.start()
    barrier()
    t_lo = time.time()
    total_ms = rig.timed(g_step, steps)
    barrier()
    t_hi = time.time()
    sampler.stop()
    g1, g2, how = rig.gemm_times(max(1, min(steps, 100)))
    e2e_steps = max(1, min(steps, 20))
    e2e_ms, hb, db = rig.e2e(e2e_steps, 3, barrier)
    assert chord.chord_get_device_error(rig.stream) == 0
    total_ms, e2e_ms, g1, g2 = reduce_max([total_ms, e2e_ms, g1, g2], pg, dev)
    r1, r2, ach = regime_summary(rig, g1, g2, peaks)
    cfg, regime, _ = arm_config(w, rig.bm, world)
    out = {"config": cfg, "value": round(per_call_us(total_ms, steps), 2), "unit": UNIT, "steps": steps,
           "gemm_us": {"gate_up": round(g1 * 1e3, 2), "down": round(g2 * 1e3, 2)}, "gemm_achieved": ach,
           "roofline": r1, "roofline_down": r2, "clocks": sampler.summary(t_lo, t_hi),
           "e2e": {"value": round(per_call_us(e2e_ms, e2e_steps), 2), "unit": UNIT, "h2d_bytes_per_step": hb,
                   "d2h_bytes_per_step": db},
           "details": {"timing": f"CUDA graph replay per step, device events; GEMMs: {how}",
                       "silu_mul": "fused into gate_up" if rig.fused else "separate pass",
                       "combine": "fused into the down GEMM" if rig.fuse_combine else "separate pass",
                       "split_k": rig.split_desc()},
           "gpu_launches": rig.launches_per_step * steps}
    rig.release()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="ep8_decode", choices=sorted(WORKLOADS) + sorted(GROUPED))
    ap.add_argument("--impl", default="chord", choices=["chord", "reference"])
    ap.add_argument("--block-m", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill-regime", action="store_true",
                    help="skip the EP8 prefill measurement that the default decode line carries")
    ap.add_argument("--unfused", action="store_true", help="separate SiLU * up pass instead of the fused epilogue")
    ap.add_argument("--fused", action="store_true", help="SiLU * up in the gate_up epilogue on either kernel")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--fused-combine", action="store_true",
                    help="the top-k combine fused into the down GEMM (chord_moe_layer opts.fuse_combine = 1) "
                         "instead of the separate pass")
    ap.add_argument("--mixed", type=int, default=None, choices=[-1, 0, 1],
                    help="per-block regime of tcgen05-regime GEMMs (opts.mixed): 1 on, -1 off, 0 the library's "
                         "choice; default: on for the cold-tail skewed workload, the library's choice otherwise")
    args = ap.parse_args()
    if args.workload in GROUPED:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the grouped workloads have no oracle arm"}))
            return
        return run_grouped(args, args.workload)
    w = WORKLOADS[args.workload]
    if args.mixed is None:
        # the caller that knows its routing has a cold tail asks for the split
        args.mixed = 1 if w.name == wl.SKEWED_COLD.name else 0
    if args.impl == "reference":
        return run_reference(args, w)
    args.warmup = max(args.warmup, 3)

    import torch
    import w4a16_int4_mixture_moe_gb300 as chord

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    chord.build()
    chord.load()

    def barrier():
        if pg:
            pg.barrier()
        torch.cuda.synchronize()

    rig = LayerRig(chord, torch, w, dev, rank, args)
    # The step replays as a CUDA graph: one host launch per replay, so a small
    # step is not timed at the host's enqueue rate.
    g_step = rig.capture(rig.step)

    # ---- device-resident timing of the whole step
    for _ in range(args.warmup):
        g_step.replay()
    assert chord.chord_get_device_error(rig.stream) == 0
    sampler = ClockSampler(gpu_id_for(torch, local_rank))
    sampler.start()
    barrier()
    t_lo = time.time()
    total_ms = rig.timed(g_step, args.steps)
    barrier()
    t_hi = time.time()
    sampler.stop()

    # ---- per-GEMM durations, measured live with events on the launching stream
    g1, g2, gemm_timing = rig.gemm_times(max(1, min(args.steps, 200)))

    # ---- end to end through the public layer call, host buffers, copies timed
    e2e_ms, h2d, d2h = rig.e2e(args.steps, args.warmup, barrier)
    e2e_eager_steps = max(1, min(args.steps, 200))
    e2e_eager_ms, _, _ = rig.e2e(e2e_eager_steps, args.warmup, barrier, cached=False)
    host_us = rig.host_us_per_call()
    host_eager_us = rig.host_us_per_call(cached=False)
    assert chord.chord_get_device_error(rig.stream) == 0

    total_ms, e2e_ms, e2e_eager_ms, g1, g2, host_us, host_eager_us = reduce_max(
        [total_ms, e2e_ms, e2e_eager_ms, g1, g2, host_us, host_eager_us], pg, dev)
    us_per_call = per_call_us(total_ms, args.steps)
    e2e_us = per_call_us(e2e_ms, args.steps)

    cfg, regime, peaks = arm_config(w, rig.bm, world)
    r1, r2, ach = regime_summary(rig, g1, g2, peaks)
    clk = sampler.summary(t_lo, t_hi)
    details = {"timing": f"CUDA graph replay per step (align, GEMMs, combine), device events; GEMMs: {gemm_timing}",
               "silu_mul": "fused into gate_up" if rig.fused else "separate pass", "split_k": rig.split_desc(),
               "combine": "fused into the down GEMM" if rig.fuse_combine else "separate pass",
               "e2e": "chord_moe_layer_cached (the layer's launches recorded once into a CUDA graph, replayed) with "
                      "pinned host buffers, the copies in and out inside the timed region",
               "host_us_per_call": "median CPU time of one chord_moe_layer_cached enqueue through the Python binding "
                                   "(a graph replay); host_us_per_call_eager: the same for the eager chord_moe_layer"}
    line = {
        "metric": METRIC, "value": round(us_per_call, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": cfg,
        "gemm_us": {"gate_up": round(g1 * 1e3, 2), "down": round(g2 * 1e3, 2)},
        "gemm_achieved": ach,
        "roofline": r1,
        "roofline_down": r2,
        "clocks": clk,
        "e2e": {"value": round(e2e_us, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "e2e_eager": {"value": round(per_call_us(e2e_eager_ms, e2e_eager_steps), 2), "unit": UNIT},
        "host_us_per_call": round(host_us, 2),
        "host_us_per_call_eager": round(host_eager_us, 2),
        "gpu_launches": rig.launches_per_step * args.steps,
        "details": details,
    }
    rig.release()
    del g_step
    if args.workload == "ep8_decode" and not args.no_prefill_regime:
        line["regimes"] = {"decode": {"workload": w.name, "value": line["value"], "gemm_us": line["gemm_us"],
                                      "roofline": r1, "roofline_down": r2},
                           "prefill": measure_prefill_regime(chord, torch, dev, rank, world, args, pg)}
    if rank == 0 and not args.no_cpu_baseline:
        us_cpu, desc, cores, _, _ = oracle_sample(w, args.cpu_seconds, block_m=rig_bm(cfg))
        line["cpu_baseline"] = {"value": round(us_cpu, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
                                "sample": desc}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


def rig_bm(cfg):
    return int(cfg.get("block_m") or 8)


if __name__ == "__main__":
    main()
