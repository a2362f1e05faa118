"""CPU checks of the binary32 identities the KV-append kernel's quantiser
relies on (the kernel itself is checked bit for bit on the GPU against the
oracle, tests/test_kv_append.py); exact rational arithmetic, no GPU.

* The scale absmax / 127 without a division: q0 = RN(a r), r = RN(1/127);
  the remainder a - 127 q0 is a binary32 number (so one FMA gives it
  exactly); q1 = RN(q0 + rem r) equals RN(a / 127).  Markstein's division by
  a constant, checked for every positive finite bf16 value a (subnormals
  included), which is every absmax a row of bf16 values can have.
* Codes by a rounding add: for |q| < 127.5 (the kernel's quotients are within
  127 (1 + 2^-23) plus the reciprocal's error), RN(q + 1.5 * 2^23) - 1.5 * 2^23
  is rint(q) (ties to even) and the low byte of the sum's bit pattern is that
  integer's two's complement byte.
"""
import math
import struct
from fractions import Fraction

import numpy as np


def _f32(bits):
    return struct.unpack("<f", struct.pack("<I", bits))[0]


def _rn32(x: Fraction) -> Fraction:
    """Round a rational to the nearest binary32 value, ties to even (normal or subnormal; no overflow here)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = math.floor(math.log2(x.numerator) - math.log2(x.denominator))
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    m = x / quantum
    n = m.numerator // m.denominator
    frac = m - n
    if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return sign * n * quantum


def test_rn32_agrees_with_binary32_division():
    # the rounding helper itself, against numpy's IEEE binary32 division
    rng = np.random.default_rng(0)
    for a, b in zip(rng.standard_normal(200).astype(np.float32), rng.uniform(0.5, 300, 200).astype(np.float32)):
        want = np.float32(a) / np.float32(b)
        assert _rn32(Fraction(float(a)) / Fraction(float(b))) == Fraction(float(want))


def test_division_by_127_without_a_divide_is_exact_for_every_bf16_magnitude():
    r = _rn32(Fraction(1, 127))
    for hi in range(0x0001, 0x7F80):  # positive finite bf16 bit patterns
        a = Fraction(_f32(hi << 16))
        q0 = _rn32(a * r)
        rem = a - 127 * q0
        assert rem == 0 or _rn32(rem) == rem, hex(hi)  # the FMA's remainder is exact
        assert _rn32(q0 + rem * r) == _rn32(a / 127), hex(hi)


def test_rounding_add_gives_the_even_rounded_code_in_the_low_byte():
    magic = np.float32(12582912.0)  # 1.5 * 2^23
    rng = np.random.default_rng(1)
    k = np.arange(-128, 128, dtype=np.float32)
    ties = k + np.float32(0.5)
    near = np.concatenate([np.nextafter(ties, np.float32(-np.inf)), ties, np.nextafter(ties, np.float32(np.inf))])
    q = np.concatenate([near, k, rng.uniform(-127.5, 127.5, 200000).astype(np.float32)])
    q = q[np.abs(q) < 127.5]
    s = (q + magic).astype(np.float32)  # one binary32 rounding
    assert np.array_equal(s - magic, np.rint(q))  # rint: half to even
    low = (s.view(np.uint32) & 0xFF).astype(np.uint8).view(np.int8)
    assert np.array_equal(low.astype(np.int32), np.rint(q).astype(np.int32))
