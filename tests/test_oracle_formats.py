"""Pins for the oracle's number-format helpers against independent library routines.

fp16 decode/encode is checked against numpy's IEEE binary16; float->bf16 against
torch's round-to-nearest-even conversion; the single-rounding double->bf16
against exact rational arithmetic (fractions).
"""
from fractions import Fraction

import numpy as np
import torch


def test_half_to_double_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.signbit(orc.half_to_double(0x8000))


def test_double_to_half_matches_numpy(orc):
    rng = np.random.default_rng(7)
    xs = np.concatenate([
        rng.standard_normal(4000) * 3,
        rng.standard_normal(500) * 1e-5,            # subnormal range
        np.array([65504.0, 65519.0, 65520.0, 1e6, -0.0, 0.0, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26]),
        # exact ties between two fp16 neighbours
        (np.arange(1024, 1100) + 0.5) * 2.0 ** -10,
    ])
    for x in xs:
        ref = np.array([x]).astype(np.float16).view(np.uint16)[0]
        assert orc.double_to_half(float(x)) == ref, x


def test_float_to_bf16_matches_torch(orc):
    rng = np.random.default_rng(3)
    xs = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * 10,
        (rng.standard_normal(500) * 1e-39).astype(np.float32),          # fp32 subnormals
        np.array([3.3961514e38, 3.4e38, -3.4e38, 0.0, -0.0, np.inf, -np.inf], np.float32),
        # ties: low 16 bits exactly 0x8000
        (np.arange(0x3F800000, 0x3F800000 + 64 * 0x10000, 0x10000, dtype=np.uint32)
         | 0x8000).view(np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.float_to_bf16(float(x)) for x in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)
    assert orc.float_to_bf16(float("nan")) == 0x7FFF


def _exact_bf16(x: float) -> float:
    """Round x to bf16 by exact rational arithmetic (normal range only)."""
    f = Fraction(x)
    if f == 0:
        return 0.0
    sign = -1 if f < 0 else 1
    f = abs(f)
    e = f.numerator.bit_length() - f.denominator.bit_length()
    while Fraction(2) ** e > f:
        e -= 1
    while Fraction(2) ** (e + 1) <= f:
        e += 1
    q = Fraction(2) ** (e - 7)
    m = f / q
    lo = m.numerator // m.denominator
    rem = m - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return sign * float(lo * q)


def test_double_to_bf16_single_rounding(orc):
    rng = np.random.default_rng(11)
    xs = list(rng.lognormal(0, 3, 2000))
    # a double just above a bf16 tie that float() would first round onto the tie
    xs.append(1.0 + 2.0 ** -8 + 2.0 ** -40)
    xs.append(1.0 + 2.0 ** -8)            # exact tie -> even (1.0)
    xs.append(1.0 + 3 * 2.0 ** -8)        # exact tie -> even (1 + 2^-6)
    for x in xs:
        got = orc.bf16_to_float(orc.double_to_bf16(float(x)))
        assert got == _exact_bf16(float(x)), x
    assert orc.bf16_to_float(orc.double_to_bf16(1.0 + 2.0 ** -8 + 2.0 ** -40)) == 1.0 + 2.0 ** -7
