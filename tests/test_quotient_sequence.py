"""The quantizers compute every quotient x / s without a division: with
n = -RN(1/s) (an IEEE reciprocal, once per scale group), q0' = RN(x n),
r = fma(q0', s, x) and q1' = fma(r, n, q0'), where Markstein's theorem gives
q1' = -RN(x / s) (the kernels take IEEE division for s below 2^-82, where a
residual could fall below the binary32 subnormal quantum).  (The theorem asks RN(x n) to be within
one ulp of the quotient; with a correctly rounded reciprocal it can be up to
~1.13 ulp away, and for tiny x the residual can be inexact: the test shows
that every quotient of magnitude 2^-20 or more is still exact over the whole
domain, and smaller ones, which every code maps to 0 or a signed 0, stay
below 2^-19 with the right sign.)  The sign of a zero quotient is kept: x = -0
gives q1' = +0 and x = +0 gives q1' = -0.

This checks the sequence against IEEE binary32 division on the CPU, in float64
emulation that is exact: q0' s has at most 48 significant bits and cancels
against x, so q0' s + x is exact in float64 before its one rounding to
binary32 (that is what the FMA computes); the second FMA's sum can exceed 53
bits, so a float64 result that lands exactly on a binary32 midpoint is redone
in exact rational arithmetic.

Domain: every scale the kernels produce, s = RN(a / q_max) for a BF16 absmax a
and q_max in {127, 7, 448, 1}, against every BF16 x with |x| <= a.  Scaling a
and x by the same power of two scales s, RN(1/s), q0', r and q1' exactly while
none of them leaves the normal range, so a in [1, 2) (all 128 BF16 mantissas)
with every BF16 x in [-a, a] covers the interior; a sample of a at the
exponent extremes (down to the smallest a whose scale is at least 2^-125, up
to the largest finite BF16) covers the edges, where x and the quotients may
be subnormal.  It checks the kernels' arithmetic method; it shares no code
with the kernels or the oracle."""
from fractions import Fraction as Fr

import numpy as np
import pytest

QMAX = [127, 7, 448, 1]


def bf16_values(lo_bits: int, hi_bits: int) -> np.ndarray:
    return (np.arange(lo_bits, hi_bits, dtype=np.uint32) << 16).view(np.float32)


def rn32_scale(a: np.ndarray, q: int) -> np.ndarray:
    # IEEE binary32 division (numpy rounds float32 division to nearest even)
    return (a.astype(np.float32) / np.float32(q)).astype(np.float32)


def _f32_from_f64_exact(v: np.ndarray, exact) -> np.ndarray:
    """Round float64 values to binary32; entries that sit exactly on a binary32
    midpoint (where rounding twice could differ from rounding once) are taken
    from exact(index) instead."""
    out = v.astype(np.float32)
    bits = v.view(np.uint64)
    mid = ((bits & np.uint64(0x1FFFFFFF)) == np.uint64(0x10000000)) & (np.abs(v) >= 2.0 ** -126)
    for i in np.flatnonzero(mid):
        out[i] = exact(i)
    return out


def markstein_neg_quotient(x: np.ndarray, s: np.ndarray):
    """The kernels' sequence, emulated exactly; returns q1' = -RN(x / s)."""
    y = (np.float32(1.0) / s).astype(np.float32)          # IEEE rcp.rn
    n = -y
    q0 = (x * n).astype(np.float32)                       # RN(x n)
    r64 = q0.astype(np.float64) * s.astype(np.float64) + x.astype(np.float64)  # exact
    r = r64.astype(np.float32)                            # one rounding: the FMA
    v64 = r.astype(np.float64) * n.astype(np.float64) + q0.astype(np.float64)

    def exact(i):
        return np.float32(float(_rn32(Fr(float(r[i])) * Fr(float(n[i])) + Fr(float(q0[i])))))
    q1 = _f32_from_f64_exact(v64, exact)
    # the sign of an exact zero sum: RN(+0 + -0) = +0 in round to nearest
    z = (v64 == 0)
    both_neg = np.signbit(r.astype(np.float64) * n.astype(np.float64)) & np.signbit(q0) & z
    q1[z] = np.where(both_neg[z], np.float32(-0.0), np.float32(0.0))
    return q1


def _rn32(x: Fr) -> Fr:
    import math
    if x == 0:
        return Fr(0)
    sign = -1 if x < 0 else 1
    x = abs(x)
    e = math.floor(math.log2(x.numerator) - math.log2(x.denominator))
    while Fr(2) ** e > x:
        e -= 1
    while Fr(2) ** (e + 1) <= x:
        e += 1
    e = max(e, -126)
    quantum = Fr(2) ** (e - 23)
    m = x / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fr(1, 2) or (rem == Fr(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * quantum


TINY = 2.0 ** -20   # far below the smallest quotient any code distinguishes from 0 (INT: 1/2, FP8: 2^-10)


def check_pairs(x: np.ndarray, s: np.ndarray):
    """Quotients the codes depend on are bit-exact; tiny ones (|x / s| < 2^-20,
    all coded 0 or signed 0) stay tiny with the quotient's sign."""
    q1 = markstein_neg_quotient(x, s)
    want = -(x / s).astype(np.float32)
    big = np.abs(want) >= TINY
    bad = np.flatnonzero(big & (q1.view(np.uint32) != want.view(np.uint32)))
    assert bad.size == 0, [(float(x[i]), float(s[i]), float(q1[i]), float(want[i])) for i in bad[:5]]
    small = ~big
    assert np.all(np.abs(q1[small]) < 2 * TINY)
    assert np.all(np.signbit(q1[small]) == np.signbit(want[small]))


def test_emulation_catches_a_plain_product():
    # a planted mistake: RN(x RN(1/s)) alone is not the quotient everywhere
    a = bf16_values(0x3F80, 0x4000)
    s = rn32_scale(a, 127)
    x = np.repeat(a[:, None], 64, 1).ravel() * np.tile(np.linspace(-1, 1, 64, dtype=np.float32), a.size)
    x = (x.astype(np.float32).view(np.uint32) & 0xFFFF0000).view(np.float32)
    ss = np.repeat(s, 64)
    plain = -(x * (np.float32(1.0) / ss).astype(np.float32)).astype(np.float32)
    assert np.any(plain != -(x / ss).astype(np.float32))


@pytest.mark.parametrize("q", QMAX)
def test_every_bf16_pair_with_absmax_in_one_binade(q):
    a_all = bf16_values(0x3F80, 0x4000)                   # [1, 2): 128 mantissas
    x_pos = bf16_values(0, 0x4000)                        # every BF16 in [0, 2), subnormals and zero included
    for a in a_all:
        x = x_pos[x_pos <= a]
        x = np.concatenate([x, -x])                       # -0 included
        s = np.full(x.shape, rn32_scale(np.array([a]), q)[0], np.float32)
        check_pairs(x, s)


@pytest.mark.parametrize("q", QMAX)
def test_absmax_at_the_exponent_edges(q):
    rng = np.random.default_rng(q)
    x_all = bf16_values(0, 0x7F80)                        # every positive finite BF16
    # smallest a with RN(a / q) >= 2^-82, the binades above it, and the largest finite BF16s
    s_min = 2.0 ** -82
    lo_a = [v for v in bf16_values(0x1600, 0x1C00) if float(rn32_scale(np.array([v]), q)[0]) >= s_min][:160]
    hi_a = list(bf16_values(0x7E00, 0x7F80)[::3])
    for a in lo_a[::4] + hi_a[::4]:
        x = x_all[x_all <= a]
        if x.size > 20000:                                # every x near a, a sample below
            x = np.concatenate([x[-12000:], rng.choice(x[:-12000], 8000, replace=False)])
        x = np.concatenate([x, -x])
        s = np.full(x.shape, rn32_scale(np.array([a]), q)[0], np.float32)
        assert s[0] >= s_min
        check_pairs(x, s)


def test_signed_zero_quotients():
    s = np.array([0.5, 3.0], np.float32)
    q1 = markstein_neg_quotient(np.array([0.0, -0.0], np.float32), s)
    assert not np.signbit(q1[1]) and np.signbit(q1[0])     # -RN(x / s): -0 for +0, +0 for -0
