"""Pins of the oracle's quantizer against what the pages and mathematics fix.

* The INT8 worked example ("Use Less Memory: Quantization and Offloading",
  §5 Exercise 1), typed in as tests/golden/worked_example_int8.json.
* The symmetric-quantization error bound |x - x_hat| <= s/2 (plus FP32
  rounding of the quotient) and the code range [-q_max, q_max] (§2.1).
* Exact round trip of values the format represents with s = 1.
* The E4M3FN encoder against torch's CPU float8_e4m3fn conversion (a library
  routine) and against a brute-force nearest-value search.
* INT4 nibble order by a hand case.
* Per-channel K: a constant channel saturates at ±127; scales equal the block
  absmax (computed with torch.amax) / 127; blocks do not interact.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import quantize as oq

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# q_max as the pages print it ("Use Less Memory", §2.1 format table: signed
# INT8 127, signed INT4 7) and OCP E4M3FN's largest finite value
PAGE_QMAX = {oq.INT8: 127, oq.INT4: 7, oq.FP8: 448}


class Fmt:
    def __init__(self, dtype, gran=oq.PER_TOKEN_HEAD, group=0):
        self.dtype, self.gran, self.group = dtype, gran, group


def bf16_bits(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# worked example
# ---------------------------------------------------------------------------

def test_worked_example_int8():
    with open(os.path.join(GOLDEN, "worked_example_int8.json")) as f:
        g = json.load(f)
    x = np.asarray(g["input"], dtype=np.float32)
    codes, s = oq.quantize_symmetric(x, oq.INT8)
    assert codes.tolist() == g["codes"]
    # the page prints s to ten digits, computed from the decimal inputs
    assert abs(float(s) - g["scale_printed"]) <= 1e-7 * g["scale_printed"]
    assert abs(float(np.max(np.abs(x))) - g["absmax"]) < 1e-6
    # quotients before rounding: the page prints three decimals computed with
    # its rounded s (1.20 / 0.029921 = 40.1056, printed 40.104); they agree
    # with the exact quotients to 1.5e-3, far inside the rounding decision
    r = x / s
    np.testing.assert_allclose(r, g["quotients_printed"], atol=1.5e-3)
    # reconstructions: the page multiplies by its 6-digit s = 0.029921 and
    # prints 5 decimals; with the exact s the difference is |q| * 2.6e-7
    x_hat = oq.dequantize_rows(codes, s, oq.INT8)
    tol = np.abs(codes) * abs(float(s) - g["scale_used_in_steps_3_4"]) + 5.1e-6
    assert np.all(np.abs(x_hat - g["reconstructed_printed"]) <= tol)
    err = np.abs(x.astype(np.float64) - x_hat)
    assert abs(err.max() - g["max_abs_error_printed"]) < 2e-5
    rel = err / np.abs(x.astype(np.float64))
    assert abs(100 * rel.max() - g["max_rel_error_percent_printed"]) < 0.005


@pytest.mark.parametrize("precision", ["fp16", "bf16"])
def test_worked_example_codes_independent_of_input_precision(precision):
    with open(os.path.join(GOLDEN, "worked_example_int8.json")) as f:
        g = json.load(f)
    dt = torch.float16 if precision == "fp16" else torch.bfloat16
    x = torch.tensor(g["input"], dtype=torch.float32).to(dt).to(torch.float32).numpy()
    codes, s = oq.quantize_symmetric(x, oq.INT8)
    assert codes.tolist() == g["codes"]


# ---------------------------------------------------------------------------
# invariants of the symmetric quantizer
# ---------------------------------------------------------------------------

def _random_groups(rng, n, g, scale_spread=True):
    x = rng.standard_normal((n, g)).astype(np.float32)
    if scale_spread:
        x *= np.exp2(rng.integers(-20, 20, size=(n, 1))).astype(np.float32)
    return torch.as_tensor(x).to(torch.bfloat16).to(torch.float32).numpy()


@pytest.mark.parametrize("dtype", [oq.INT8, oq.INT4])
def test_int_error_bound_and_range(dtype):
    rng = np.random.default_rng(1)
    x = _random_groups(rng, 4000, 32)
    codes, s = oq.quantize_symmetric(x, dtype)
    q_max = PAGE_QMAX[dtype]
    assert codes.min() >= -q_max and codes.max() <= q_max
    x_hat = codes.astype(np.float64) * s.astype(np.float64)[:, None]
    err = np.abs(x.astype(np.float64) - x_hat)
    # |x/s - RN(x/s)| <= 2^-24 |x/s| <= 2^-24 q_max (1 + 2^-23)
    bound = s.astype(np.float64)[:, None] * (0.5 + 2.0 * q_max * 2.0 ** -24)
    assert np.all(err <= bound)
    # the absmax element lands on +-q_max
    i = np.argmax(np.abs(x), axis=1)
    top = codes[np.arange(len(x)), i]
    assert np.all(np.abs(top) == q_max)
    assert np.all(np.sign(top) == np.sign(x[np.arange(len(x)), i]))
    # the scale is the FP32 quotient absmax / q_max
    a = np.abs(x).max(axis=1)
    assert np.array_equal(s, (a / np.float32(q_max)).astype(np.float32))


def test_int_ties_round_to_even():
    # absmax 127 gives s = 1 exactly, so x / s = x; halves are ties
    x = np.array([[127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5]], dtype=np.float32)
    codes, s = oq.quantize_symmetric(x, oq.INT8)
    assert s[0] == 1.0
    assert codes[0].tolist() == [127, 0, 2, 2, 0, -2, -2, 4]


def test_fp8_error_bound():
    rng = np.random.default_rng(2)
    x = _random_groups(rng, 3000, 128)
    codes, s = oq.quantize_symmetric(x, oq.FP8)
    x_hat = oq.e4m3fn_decode(codes) * s.astype(np.float64)[:, None]
    r = np.abs(x.astype(np.float64)) / s.astype(np.float64)[:, None]
    # RNE to 3 mantissa bits: half a quantum, quantum 2^(e-3) (>= 2^-9)
    e = np.floor(np.log2(np.maximum(r, 2.0 ** -6)))
    half_q = np.exp2(e - 4)
    bound = (half_q + r * 2.0 ** -23) * s.astype(np.float64)[:, None]
    assert np.all(np.abs(x - x_hat) <= bound * (1 + 1e-12))
    i = np.argmax(np.abs(x), axis=1)
    top = codes[np.arange(len(x)), i]
    assert np.all((top & 0x7F) == 0x7E)


@pytest.mark.parametrize("dtype", [oq.INT8, oq.INT4])
def test_int_exact_round_trip(dtype):
    q_max = PAGE_QMAX[dtype]
    rng = np.random.default_rng(3)
    x = rng.integers(-q_max, q_max + 1, size=(500, 32)).astype(np.float32)
    x[:, 5] = q_max * np.where(rng.random(500) < 0.5, -1, 1)
    codes, s = oq.quantize_symmetric(x, dtype)
    assert np.all(s == 1.0)
    assert np.array_equal(codes.astype(np.float32), x)


def test_fp8_exact_round_trip():
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = oq.e4m3fn_decode(finite).astype(np.float32)
    rng = np.random.default_rng(4)
    for _ in range(50):
        pick = rng.choice(finite, size=64)
        pick[0] = 0x7E if rng.random() < 0.5 else 0xFE  # absmax 448 -> s = 1
        x = oq.e4m3fn_decode(pick).astype(np.float32)
        codes, s = oq.quantize_symmetric(x, oq.FP8)
        assert s == 1.0
        # +0 / -0 both decode to 0; compare values, then bits away from zero
        assert np.array_equal(oq.e4m3fn_decode(codes), oq.e4m3fn_decode(pick))
        nz = (pick & 0x7F) != 0
        assert np.array_equal(codes[nz], pick[nz])
    assert np.all(np.isfinite(vals))


def test_zero_group():
    for dtype in (oq.INT8, oq.INT4, oq.FP8):
        x = np.zeros((3, 16), dtype=np.float32)
        x[1, 3] = -0.0
        codes, s = oq.quantize_symmetric(x, dtype)
        assert np.all(s == 0) and not np.any(np.signbit(s))
        assert np.all(codes.view(np.uint8) == 0)


def test_fp8_sign_of_zero_quotient():
    # -tiny / s rounds to zero: the sign bit is kept (0x80)
    x = np.array([448.0, -1e-6, -0.0, 1e-6], dtype=np.float32)
    codes, s = oq.quantize_symmetric(x, oq.FP8)
    assert s == 1.0
    assert codes.tolist() == [0x7E, 0x80, 0x80, 0x00]


# ---------------------------------------------------------------------------
# E4M3FN codec
# ---------------------------------------------------------------------------

def test_e4m3fn_decode_table():
    # spec points: 0x08 = 2^-6 (min normal), 0x01 = 2^-9 (min subnormal),
    # 0x7E = 448 (max), 0x38 = 1.0, 0x7F NaN, sign bit
    d = oq.e4m3fn_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x3C, 0x7E, 0xFE, 0x80], np.uint8))
    assert d.tolist() == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.5, 448.0, -448.0, -0.0]
    assert np.isnan(oq.e4m3fn_decode(np.array([0x7F, 0xFF], np.uint8))).all()
    # against torch's float8_e4m3fn for every finite code
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oq.e4m3fn_decode(codes), ref)


def test_e4m3fn_encode_decode_round_trip_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oq.e4m3fn_decode(codes).astype(np.float32)
    assert np.array_equal(oq.e4m3fn_encode(vals), codes)


def _e4m3fn_points():
    codes = np.arange(0, 0x7F, dtype=np.uint8)          # 0 .. 0x7E, nonnegative
    return codes, oq.e4m3fn_decode(codes)


def _torch_e4m3fn(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3fn_encode_vs_torch_strided_sweep():
    # every 61st float32 bit pattern in [0, 448], both signs
    bits = np.arange(0, 0x43E00001, 61, dtype=np.uint32)
    x = bits.view(np.float32)
    for sgn in (1.0, -1.0):
        xs = (sgn * x).astype(np.float32)
        assert np.array_equal(oq.e4m3fn_encode(xs), _torch_e4m3fn(xs))


def test_e4m3fn_encode_vs_torch_at_ties():
    # midpoints between neighbouring representable values and their float32
    # neighbours: where rounding decisions happen
    _, pts = _e4m3fn_points()
    mids = ((pts[:-1] + pts[1:]) / 2).astype(np.float32)
    cand = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(np.inf)), pts.astype(np.float32)])
    cand = cand[cand <= 448]
    for sgn in (1.0, -1.0):
        xs = (sgn * cand).astype(np.float32)
        assert np.array_equal(oq.e4m3fn_encode(xs), _torch_e4m3fn(xs))


def test_e4m3fn_encode_vs_brute_force_nearest():
    codes, pts = _e4m3fn_points()
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.uniform(0, 448, 20000), np.exp2(rng.uniform(-12, 8.8, 20000)),
        ((pts[:-1] + pts[1:]) / 2)]).astype(np.float32)
    x = x[x <= 448]
    enc = oq.e4m3fn_encode(x)
    xd = x.astype(np.float64)
    for xi, ci in zip(xd, enc):
        dist = np.abs(pts - xi)
        best = np.flatnonzero(dist == dist.min())
        want = best[0] if len(best) == 1 else best[np.flatnonzero(codes[best] % 2 == 0)[0]]
        assert ci == codes[want], (xi, ci, codes[want])


def test_e4m3fn_saturates():
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3e38, -500.0, -1e30], np.float32)
    assert oq.e4m3fn_encode(x).tolist() == [0x7E] * 7 + [0xFE] * 2


# ---------------------------------------------------------------------------
# INT4 packing
# ---------------------------------------------------------------------------

def test_int4_nibble_order_hand_case():
    # element 0 (= 1) in the low nibble, element 1 (= -1 = 0xF) in the high
    assert oq.pack_int4(np.array([1, -1], np.int8)).tolist() == [0xF1]
    assert oq.pack_int4(np.array([-7, 7, 0, -1], np.int8)).tolist() == [0x79, 0xF0]


def test_int4_pack_unpack_all_pairs():
    a, b = np.meshgrid(np.arange(-7, 8), np.arange(-7, 8))
    codes = np.stack([a.ravel(), b.ravel()], axis=1).astype(np.int8)
    packed = oq.pack_int4(codes)
    assert packed.shape == (225, 1)
    assert np.array_equal(oq.unpack_int4(packed), codes)
    # 128 channels pack into 64 bytes per head vector
    assert oq.pack_int4(np.zeros(128, np.int8)).shape == (64,)


# ---------------------------------------------------------------------------
# the paged write
# ---------------------------------------------------------------------------

def test_paged_write_locations_and_skip():
    h, d, bs = 2, 32, 4
    cache = oq.OracleCache(6, bs, h, d, Fmt(oq.INT8), Fmt(oq.INT8))
    rng = np.random.default_rng(6)
    k = bf16_bits(rng.standard_normal((3, h, d)))
    v = bf16_bits(rng.standard_normal((3, h, d)))
    slots = np.array([5 * bs + 3, -1, 2 * bs + 0])
    oq.quantize_write(cache, k, v, slots)
    ck, sk = oq.quantize_symmetric(oq.bf16_bits_to_f32(k), oq.INT8)
    assert np.array_equal(cache.codes["k"][5, 3], ck[0].view(np.uint8))
    assert np.array_equal(cache.codes["k"][2, 0], ck[2].view(np.uint8))
    assert np.array_equal(cache.scales["k"][5, 3], sk[0])
    # the skipped token wrote nothing: only two rows are nonzero
    assert np.count_nonzero(cache.scales["k"]) == 2 * h
    assert np.count_nonzero(cache.scales["v"]) == 2 * h


def test_grouped_int4_write():
    h, d, bs, g = 2, 128, 16, 32
    cache = oq.OracleCache(4, bs, h, d, Fmt(oq.INT8), Fmt(oq.INT4, oq.PER_TOKEN_GROUP, g))
    rng = np.random.default_rng(7)
    v = rng.standard_normal((5, h, d)).astype(np.float32)
    v[:, :, 32:64] *= 100.0  # one loud group must not change the others' scales
    vb = bf16_bits(v)
    oq.quantize_write(cache, vb, vb, np.arange(5) + 16)
    vf = oq.bf16_bits_to_f32(vb)
    s = cache.scales["v"][1, :5]                                   # [5, H, 4]
    want = (np.abs(vf.reshape(5, h, 4, g)).max(axis=-1) / np.float32(7)).astype(np.float32)
    assert np.array_equal(s, want)
    codes = oq.unpack_int4(cache.codes["v"][1, :5])
    x_hat = codes.reshape(5, h, 4, g) * s[..., None].astype(np.float64)
    err = np.abs(vf.reshape(5, h, 4, g) - x_hat)
    assert np.all(err <= s[..., None] * (0.5 + 2 * 7 * 2.0 ** -24))


def test_per_channel_k():
    h, d, bs = 2, 64, 16
    cache = oq.OracleCache(5, bs, h, d, Fmt(oq.INT8, oq.PER_BLOCK_CHANNEL), Fmt(oq.INT8))
    rng = np.random.default_rng(8)
    n = 21                       # block 3 gets 16 rows, block 1 gets 5 rows
    x = rng.standard_normal((n, h, d)).astype(np.float32)
    x[:16, 1, 7] = -2.5          # constant channel in block 3
    x[16:, 0, 9] = 1e4           # loud channel in block 1 only
    xb = bf16_bits(x)
    slots = np.concatenate([3 * bs + rng.permutation(16), 1 * bs + np.arange(5)])
    oq.quantize_write(cache, xb, xb, slots)
    xf = torch.from_numpy(oq.bf16_bits_to_f32(xb))
    # scales = block absmax over the rows written into the block / 127
    want3 = (torch.amax(xf[:16].abs(), dim=0) / 127.0).numpy()
    want1 = (torch.amax(xf[16:].abs(), dim=0) / 127.0).numpy()
    assert np.array_equal(cache.scales["k"][3], want3)
    assert np.array_equal(cache.scales["k"][1], want1)
    assert np.all(cache.scales["k"][[0, 2, 4]] == 0)
    # the constant channel saturates on every row of its block
    codes3 = cache.codes["k"][3].view(np.int8)
    assert np.all(codes3[:, 1, 7] == -127)
    # every code is within half a step of its own channel's scale
    x_hat = oq.dequantize_cache_rows(cache, "k", slots // bs, slots % bs)
    err = np.abs(xf.numpy().astype(np.float64) - x_hat)
    s_rows = cache.scales["k"][slots // bs].astype(np.float64)
    assert np.all(err <= s_rows * (0.5 + 2 * 127 * 2.0 ** -24))
    # the loud channel of block 1 does not leak into block 3
    assert cache.scales["k"][3, 0, 9] < 1.0


# ---- INT2 (KIVI's 2-bit codes; q_max by the format table's rule 2^(b-1) - 1)
def test_int2_q_max_follows_the_table_rule():
    for bits, dt in ((8, oq.INT8), (4, oq.INT4), (2, oq.INT2)):
        assert oq.Q_MAX[dt] == 2 ** (bits - 1) - 1
    assert oq.Q_MAX[oq.INT8] == PAGE_QMAX[oq.INT8] and oq.Q_MAX[oq.INT4] == PAGE_QMAX[oq.INT4]


def test_int2_packing_hand_case():
    codes = np.array([[1, -1, 0, 1, -1, -1, 0, 0]], np.int8)
    packed = oq.pack_int2(codes)
    # byte 0: 01 | 11 << 2 | 00 << 4 | 01 << 6 = 0x4D; byte 1: 11 | 11 << 2 = 0x0F
    assert packed.tolist() == [[0x4D, 0x0F]]
    assert np.array_equal(oq.unpack_int2(packed), codes)


def test_int2_round_trip_ties_and_bound():
    rng = np.random.default_rng(12)
    exact = rng.integers(-1, 2, size=(50, 32)).astype(np.float32)
    exact[:, 0] = 1.0                                   # absmax 1 -> s = 1
    codes, s = oq.quantize_symmetric(exact, oq.INT2)
    assert np.all(s == 1.0) and np.array_equal(codes.astype(np.float32), exact)
    ties = np.array([[1.0, 0.5, -0.5, 0.49, 0.51]], np.float32)
    codes, s = oq.quantize_symmetric(ties, oq.INT2)
    assert codes.tolist() == [[1, 0, 0, 0, 1]]        # halves go to the even code 0
    x = rng.standard_normal((200, 32)).astype(np.float32)
    codes, s = oq.quantize_symmetric(x, oq.INT2)
    assert codes.min() >= -1 and codes.max() <= 1
    err = np.abs(oq.dequantize_rows(codes, s[:, None], oq.INT2) - x)
    assert np.all(err <= s[:, None] * (0.5 + 2.0 ** -23))
