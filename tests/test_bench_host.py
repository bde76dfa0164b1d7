"""Host-side arithmetic of bench.py, checked on the CPU: the algorithmic bytes
and FLOPs a GEMM launch is credited with (the numerator of the roofline
fraction), the regime each workload's line reports, and the max-over-ranks
time without a process group."""
import numpy as np

import bench
import workloads as wl


def test_gemm_algorithmic_hand_example():
    """Experts with 3, 0 and 2 rows of a 256 x 128 weight: two experts' packed
    codes and scales (N*K/2 + N*K/16 bytes each), 5 activation rows of K bf16, 5
    output rows of N bf16 (N/2 with the fused SiLU * up), 5 int32 ids; FLOPs
    2 * rows * N * K, padding and the empty expert not counted."""
    rpe = np.array([3, 0, 2])
    b, f = bench.gemm_algorithmic(rpe, 256, 128)
    assert b == 2 * (256 * 128 // 2 + 256 * 128 // 16) + 5 * 128 * 2 + 5 * 256 * 2 + 5 * 4 == 40724
    assert f == 2 * 5 * 256 * 128
    b2, _ = bench.gemm_algorithmic(rpe, 256, 128, out_cols=128)
    assert b2 == b - 5 * 128 * 2


def test_ep8_decode_gate_up_credit():
    """EP8 decode (T = 512, 48 of 384 experts, top-8): every local expert gets
    rows, 525 local pairs.  gate_up with the fused SiLU * up: 48 * 4096 * 7168
    * 9/16 weight bytes, 525 rows of 7168 bf16 in, 525 rows of 2048 bf16 out,
    525 ids."""
    w = wl.EP8_DECODE
    ids, _ = wl.make_routing(w)
    rpe = bench.routing_stats(ids, w.E)
    assert int(rpe.sum()) == 525 and int((rpe > 0).sum()) == 48
    b, f = bench.gemm_algorithmic(rpe, 2 * w.I, w.H, out_cols=w.I)
    assert b == 48 * 4096 * 7168 * 9 // 16 + 525 * 7168 * 2 + 525 * 2048 * 2 + 525 * 4 == 802402356
    assert f == 2 * 525 * 4096 * 7168 == 30828134400


def test_regime_follows_the_measured_ridge():
    """The line's regime: HBM-bound (decode) when the gate_up GEMM's FLOP per
    byte is below the sustained BF16 peak over the copy bandwidth, tensor-bound
    (prefill) above it."""
    expect = {"ep8_decode": "decode", "ep8_prefill": "prefill", "skewed": "prefill", "tiny": "decode",
              "tp8_T1": "decode", "tp8_T128": "decode", "tp8_T1024": "decode", "tp8_T4096": "decode"}
    for name, regime in expect.items():
        w = bench.WORKLOADS[name]
        cfg, got, peaks = bench.arm_config(w, 16, 1)
        ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        ids, _ = wl.make_routing(w)
        b, f = bench.gemm_algorithmic(bench.routing_stats(ids, w.E), 2 * w.I, w.H)
        assert (f / b < ridge) == (regime == "decode"), name
        assert got == regime, name
        assert cfg["local_pairs"] == int(((ids >= 0) & (ids < w.E)).sum())


def test_reduce_max_without_a_process_group():
    assert bench.reduce_max([1.5, 2.0], None, None) == [1.5, 2.0]


def test_host_block_size_rule_matches_the_library():
    """bench.select_block_m (the reference arm's config label, computed without
    loading the CUDA library) equals chord_select_block_m over a grid of
    token counts, top-k and expert counts, including the five workloads."""
    import w4a16_int4_mixture_moe_gb300 as chord
    chord.build()
    chord.load()
    shapes = [(w.T, w.topk, w.E, w.E_global) for w in bench.WORKLOADS.values()]
    for T in (0, 1, 2, 5, 16, 100, 128, 512, 1000, 1024, 3000, 4096, 8192, 16384, 65536):
        for topk in (1, 2, 6, 8):
            for E_local, E_global in ((8, 8), (48, 384), (384, 384), (64, 256), (1, 1)):
                shapes.append((T, topk, E_local, E_global))
    for T, topk, el, eg in shapes:
        assert bench.select_block_m(T, topk, el, eg) == chord.chord_select_block_m(T, topk, el, eg, 0, 0), \
            (T, topk, el, eg)


def test_time_per_call_is_not_divided_by_ranks():
    """N ranks run N expert-parallel shares of one call concurrently: the time
    per call is the max-over-ranks time over the steps, whatever N is."""
    assert bench.per_call_us(318.5, 1000) == 318.5
    assert bench.per_call_us(0.0, 0) == 0.0


def test_reference_arm_loads_no_cuda_library():
    """The reference arm (the oracle on the host cores) runs without importing
    the CUDA package, so only the oracle's library is loaded in it; its config
    equals the one the GPU arm builds for the same workload and block size."""
    import subprocess
    import sys
    code = ("import sys, json, io, contextlib; sys.argv = ['bench.py', '--impl', 'reference', '--workload', 'tiny', "
            "'--steps', '1', '--warmup', '0']; import bench; buf = io.StringIO()\n"
            "with contextlib.redirect_stdout(buf): bench.main()\n"
            "line = json.loads(buf.getvalue().strip().splitlines()[-1])\n"
            "assert 'w4a16_int4_mixture_moe_gb300' not in sys.modules, 'CUDA package imported'\n"
            "maps = open('/proc/self/maps').read()\n"
            "assert 'libchord' not in maps, 'libchord.so mapped'\n"
            "cfg, _, _ = bench.arm_config(bench.WORKLOADS['tiny'], line['config']['block_m'], 1)\n"
            "assert cfg == line['config'], (cfg, line['config'])\n"
            "print('ok', line['value'])")
    r = subprocess.run([sys.executable, "-c", code], cwd=bench.ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout + r.stderr
