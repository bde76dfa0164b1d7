"""The warp-level GEMM's one-FMA dequantisation, checked on the CPU for every
input it can see.

When a packed weight's header says every group scale s lies in [2^-126, 0.5),
the kernel forms each weight as fma(a, b, c) in bf16 with
  a = the half-word (q << 4), read as a bf16 number,
  b = the bits of s plus 0x4080 (129 added to the exponent field),
  c = s * -8,
and relies on three facts: a is q * 2^-129, b is s * 2^129, and the single
rounding of a*b + c equals the subtract-then-scale value bf16((q - 8) * s) that
the oracle computes.  Here those facts are checked exhaustively (all 16 codes
times all 15,999 scale bit patterns of the range) in exact float64 arithmetic:
a*b + c has at most 12 significant bits, so float64 holds it exactly and the
one rounding to bf16 is the only rounding, as in the FMA.  The patterns just
outside the range show why the header excludes them.
"""
import numpy as np
import pytest

import oracle
import workloads as wl


def bf16_value(bits):
    """bf16 bit patterns -> their exact values (float64), subnormals included."""
    return (np.asarray(bits, np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_round(x):
    """float64 values that float32 holds exactly -> bf16 bits, round to nearest even."""
    x32 = np.asarray(x, np.float64).astype(np.float32)
    assert np.array_equal(x32.astype(np.float64), x), "value not exact in float32"
    return wl._bf16(x32)


@pytest.fixture(scope="module")
def orc():
    oracle.build()
    return oracle


def test_embedded_nibble_is_q_times_2_pow_minus_129():
    """A nibble in bits 4..7 of an otherwise zero half-word: exponent field 0
    (q < 8, subnormal) or 1 (q >= 8); both have the spacing 2^-133."""
    q = np.arange(16, dtype=np.uint32)
    np.testing.assert_array_equal(bf16_value(q << 4), q.astype(np.float64) * 2.0 ** -129)


def test_exponent_add_is_times_2_pow_129_on_the_range():
    s = np.arange(0x0080, 0x3F00, dtype=np.uint32)
    b = bf16_value(s + 0x4080)
    np.testing.assert_array_equal(b, bf16_value(s) * 2.0 ** 129)
    assert np.isfinite(b).all()
    # at 0.5 the sum is the pattern of +inf; a subnormal scale has no exponent to add to
    assert np.isinf(bf16_value(0x3F00 + 0x4080))
    assert bf16_value(0x0040 + 0x4080) != bf16_value(0x0040) * 2.0 ** 129


def test_fma_form_equals_subtract_then_scale_on_the_whole_range(orc):
    s_bits = np.arange(0x0080, 0x3F00, dtype=np.uint16)          # every scale of the range
    q = np.arange(16, dtype=np.uint8)
    S, Q = np.meshgrid(s_bits, q, indexing="ij")
    a = bf16_value(Q.astype(np.uint32) << 4)
    b = bf16_value(S.astype(np.uint32) + 0x4080)
    c = bf16_value(bf16_round(bf16_value(S) * -8.0))            # the kernel's s * -8, itself exact
    np.testing.assert_array_equal(c, bf16_value(S) * -8.0)
    got = bf16_round(a * b + c)                                  # exact in float64, one rounding
    want = orc.dequant_pairs(Q.ravel(), S.ravel()).reshape(Q.shape)
    np.testing.assert_array_equal(got, want)
    # q = 8 gives +0 on both sides (s > 0)
    assert (got[:, 8] == 0).all()


def test_negative_scale_would_flip_the_sign_of_zero(orc):
    """Why the range excludes s <= 0: for q = 8 the FMA gives q*s - 8s = +0
    while subtract-then-scale gives (+0) * s = -0 for a negative s."""
    s = np.array([0xBC00], np.uint16)                           # -2^-7
    a = bf16_value(np.array([8 << 4], np.uint32))
    fma = a * (bf16_value(s) * 2.0 ** 129) + bf16_value(s) * -8.0
    assert bf16_round(fma)[0] == 0x0000
    assert orc.dequant_pairs(np.array([8], np.uint8), s)[0] == 0x8000
