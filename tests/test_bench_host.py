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
