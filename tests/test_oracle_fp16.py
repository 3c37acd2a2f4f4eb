"""Pins for the oracle's hand-written IEEE-754 binary16 conversion.

The pages store up_logits and out as fp16 after fp32 arithmetic ("Fused MoE
GEMM 提交说明", §完整算子代码: dtype float16, accum_dtype float32) but do not
say how fp32 is rounded; the oracle reads it as round-to-nearest-even.  numpy's
float16 casts implement exactly that, so they pin the oracle independently.
"""
import numpy as np

import oracle


def test_decode_all_bit_patterns():
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = oracle.half_bits_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_encode_random_doubles_and_floats():
    rng = np.random.default_rng(1234)
    n = 1_000_000
    mag = np.exp(rng.uniform(np.log(2.0 ** -30), np.log(2.0 ** 17), n))
    v = mag * rng.choice([-1.0, 1.0], n)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.double_to_half_bits(v), ref)
    f = v.astype(np.float32)
    with np.errstate(over="ignore"):
        ref32 = f.astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.double_to_half_bits(f.astype(np.float64)), ref32)


def test_encode_round_trip_every_finite_half():
    bits = np.arange(1 << 16, dtype=np.uint16)
    vals = bits.view(np.float16)
    finite = np.isfinite(vals)
    back = oracle.double_to_half_bits(vals[finite].astype(np.float64))
    assert np.array_equal(back, bits[finite])


def test_encode_ties_and_boundaries():
    ulp1 = 2.0 ** -10                     # spacing of halves in [1, 2)
    # (value, expected bits); a list, since 0.0 and -0.0 are equal dict keys
    cases = [
        (1.0 + ulp1 / 2, 0x3C00),           # tie -> even (1.0)
        (1.0 + 3 * ulp1 / 2, 0x3C02),       # tie -> even (1 + 2 ulp)
        (1.0 + ulp1 / 2 + 2.0 ** -40, 0x3C01),
        (65504.0, 0x7BFF),
        (65519.99, 0x7BFF),
        (65520.0, 0x7C00),                  # tie above max rounds to inf
        (-70000.0, 0xFC00),
        (2.0 ** -24, 0x0001),               # smallest subnormal
        (2.0 ** -25, 0x0000),               # tie -> even (0)
        (3 * 2.0 ** -25, 0x0002),           # tie -> even (2 quanta)
        (2.0 ** -14 - 2.0 ** -25, 0x0400),  # tie: largest subnormal vs smallest normal
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (float("inf"), 0x7C00),
        (float("-inf"), 0xFC00),
    ]
    got = oracle.double_to_half_bits(np.array([v for v, _ in cases]))
    assert [int(g) for g in got] == [b for _, b in cases]
    assert (int(oracle.double_to_half_bits(np.array([np.nan]))[0]) & 0x7C00) == 0x7C00
    assert (int(oracle.double_to_half_bits(np.array([np.nan]))[0]) & 0x03FF) != 0
