"""The quantize-write kernel computes each scale s = RN(a / q_max) without a
division: s0 = RN(a * RN(1/q)), rho = fma(-s0, q, a), s = fma(rho, RN(1/q), s0).
The absmax a of BF16 inputs is itself a BF16 value, so the claim that this is
the correctly rounded quotient can be checked exhaustively: every positive
finite BF16 a (subnormals included), for q = 127, 7 and 448, in exact rational
arithmetic with round-to-nearest-even to binary32 (an FMA rounds once).

This checks the kernel's arithmetic method on the CPU; it shares no code with
the kernel or the oracle."""
import math
from fractions import Fraction as Fr

import numpy as np
import pytest


def rn32(x: Fr) -> Fr:
    """Round an exact rational to the nearest binary32 value, ties to even."""
    if x == 0:
        return Fr(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = math.floor(math.log2(x.numerator) - math.log2(x.denominator))
    while Fr(2) ** e > x:
        e -= 1
    while Fr(2) ** (e + 1) <= x:
        e += 1
    e = max(e, -126)                      # below 2^-126: fixed quantum 2^-149
    quantum = Fr(2) ** (e - 23)
    n = x / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fr(1, 2) or (rem == Fr(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * quantum


def test_rn32_matches_numpy_float32_division():
    rng = np.random.default_rng(0)
    a = rng.standard_normal(2000).astype(np.float32)
    b = rng.standard_normal(2000).astype(np.float32)
    for x, y in zip(a, b):
        assert rn32(Fr(float(x)) / Fr(float(y))) == Fr(float(np.float32(x) / np.float32(y)))


@pytest.mark.parametrize("q", [127, 7, 448])
def test_scale_sequence_is_exact_for_every_bf16_absmax(q):
    inv = rn32(Fr(1, q))
    # the kernel's constants are RN(1/q)
    assert float(inv) == {127: float.fromhex("0x1.020408p-7"), 7: float.fromhex("0x1.24924ap-3"),
                          448: float.fromhex("0x1.24924ap-9")}[q]
    bits = np.arange(1, 0x7F80, dtype=np.uint32)          # every positive finite BF16
    vals = (bits << 16).view(np.float32)
    for v in vals:
        a = Fr(float(v))
        s0 = rn32(a * inv)
        rho = rn32(a - s0 * q)
        s = rn32(rho * inv + s0)
        assert s == rn32(a / q), float(v)
