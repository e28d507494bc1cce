"""Pins of the oracle's randomized Walsh-Hadamard rotation (oracle/rotation.py)
against a library routine, exact integer arithmetic, algebraic identities and
the pages' claim that the rotation spreads outlier peaks over all channels
("Quantized KV caches in production", Numerical Formats)."""
import numpy as np
import pytest

import oracle
from oracle import rotation as R

D_ALL = [1, 2, 4, 8, 16, 32, 64, 128]


@pytest.mark.parametrize("d", D_ALL)
def test_hadamard_is_the_library_sylvester_matrix(d):
    scipy_linalg = pytest.importorskip("scipy.linalg")
    assert np.array_equal(R.hadamard(d), scipy_linalg.hadamard(d))


@pytest.mark.parametrize("d", [64, 128])
def test_hadamard_rows_are_orthogonal(d):
    h = R.hadamard(d)
    assert np.array_equal(h @ h.T, d * np.eye(d, dtype=np.int64))


@pytest.mark.parametrize("d", [8, 64, 128])
def test_butterfly_equals_the_matrix_on_exact_inputs(d):
    # small integers: every butterfly sum is exact in float32, so the result
    # must equal H x exactly; a swapped (a - b) / (b - a) or a skipped stage
    # gives a different matrix
    rng = np.random.default_rng(d)
    x = rng.integers(-1000, 1000, size=(5, d)).astype(np.int64)
    got = R.fwht_float32(x.astype(np.float32))
    assert np.array_equal(got.astype(np.int64), x @ R.hadamard(d).T)


@pytest.mark.parametrize("d", [64, 128])
def test_butterfly_float32_rounding_only(d):
    rng = np.random.default_rng(7)
    x = rng.standard_normal((20, d)).astype(np.float32)
    exact = x.astype(np.float64) @ R.hadamard(d).T
    got = R.fwht_float32(x).astype(np.float64)
    # log2(d) rounded additions of values bounded by the row's l1 norm
    bound = np.log2(d) * 2.0 ** -23 * np.abs(x).astype(np.float64).sum(axis=1, keepdims=True)
    assert np.all(np.abs(got - exact) <= bound)


def test_sign_words():
    words = np.array([1 | (1 << 31), 1 << 1, 0, 1 << 31], dtype=np.uint32)
    s = R.signs_from_words(words, 128)
    neg = np.flatnonzero(s < 0).tolist()
    assert neg == [0, 31, 33, 127]
    assert set(np.unique(s).tolist()) <= {-1.0, 1.0}


@pytest.mark.parametrize("d", [64, 128])
def test_signs_go_before_the_transform(d):
    rng = np.random.default_rng(11)
    sigma = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0)
    x = rng.integers(-50, 50, size=(3, d)).astype(np.float32)
    got = R.rotate_rows_float32(x, sigma).astype(np.float64)
    want = (x.astype(np.float64) * sigma) @ R.hadamard(d).T
    assert np.array_equal(got, want)


@pytest.mark.parametrize("d", [64, 128])
def test_query_rotation_preserves_dot_products_and_output_round_trips(d):
    rng = np.random.default_rng(3)
    sigma = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0)
    q = rng.standard_normal(d)
    k = rng.standard_normal((9, d))
    yk = (k * sigma) @ R.hadamard(d).T             # rotated keys, float64
    qr = R.rotate_query_fp64(q, sigma)
    assert np.allclose(yk @ qr, k @ q, rtol=1e-12, atol=1e-12)
    o = rng.standard_normal(d)
    yo = (o * sigma) @ R.hadamard(d).T
    assert np.allclose(R.unrotate_output_fp64(yo, sigma), o, rtol=1e-12, atol=1e-12)


def test_a_spike_is_spread_evenly():
    # one outlier channel becomes a +-1 pattern of equal magnitude on all channels
    d = 128
    sigma = R.signs_from_words(np.array([0x12345678, 0x9ABCDEF0, 0x0F0F0F0F, 0x33333333], np.uint32), d)
    x = np.zeros(d, dtype=np.float32)
    x[17] = 20.0
    y = R.rotate_rows_float32(x, sigma)
    assert np.all(np.abs(y) == 20.0)


def test_rotation_lowers_int4_error_on_an_outlier_channel():
    # the pages' point: with one channel x20 (the long-context K recipe), the
    # per-(token, head) INT4 step is set by the outlier; after the rotation the
    # energy is spread and the reconstruction error of the row drops
    d = 128
    rng = np.random.default_rng(5)
    sigma = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0)
    x = rng.standard_normal((64, d)).astype(np.float32)
    x[:, 3] *= 20.0
    codes, s = oracle.quantize_symmetric(x, oracle.INT4)
    err_plain = np.abs(oracle.dequantize_rows(codes, s[:, None], oracle.INT4) - x).mean()
    y = R.rotate_rows_float32(x, sigma)
    codes_r, s_r = oracle.quantize_symmetric(y, oracle.INT4)
    y_hat = oracle.dequantize_rows(codes_r, s_r[:, None], oracle.INT4)
    x_back = (y_hat @ R.hadamard(d).T) * sigma / d
    err_rot = np.abs(x_back - x).mean()
    assert err_rot < 0.5 * err_plain


def test_rotated_decode_equals_attention_over_back_rotated_rows():
    # composition pin: the oracle's rotated decode (q rotated, output rotated
    # back) must equal plain float64 attention with the original q over the
    # dequantized rows rotated back, row by row
    import workloads as wl
    d, hkv, hq = 64, 2, 4
    rng = np.random.default_rng(9)
    sigma = np.where(rng.integers(0, 2, d) == 1, -1.0, 1.0)
    kf = wl.CacheFormat(wl.INT4, wl.PER_TOKEN_HEAD)
    vf = wl.CacheFormat(wl.INT4, wl.PER_TOKEN_GROUP, 32)
    n, nb, bs = 40, 4, 16
    oc = oracle.OracleCache(nb, bs, hkv, d, kf, vf, rotation_signs=sigma)
    kx = rng.standard_normal((n, hkv, d)).astype(np.float32)
    vx = rng.standard_normal((n, hkv, d)).astype(np.float32)
    to_bits = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    table = np.array([[2, 0, 3]], dtype=np.int64)
    slots = np.array([table[0, t // bs] * bs + t % bs for t in range(n)])
    oracle.quantize_write(oc, to_bits(kx), to_bits(vx), slots)
    q_bits = to_bits(rng.standard_normal((1, hq, d)))
    got = oracle.paged_decode_fp64(oc, q_bits, table, np.array([n]))
    blocks, offs = slots // bs, slots % bs
    k_back = (oracle.dequantize_cache_rows(oc, "k", blocks, offs) @ R.hadamard(d).T) * sigma / d
    v_back = (oracle.dequantize_cache_rows(oc, "v", blocks, offs) @ R.hadamard(d).T) * sigma / d
    q = oracle.bf16_bits_to_f32(q_bits[0]).astype(np.float64)
    for h in range(hq):
        want = oracle.attention_fp64(q[h], k_back[:, h // 2], v_back[:, h // 2])
        assert np.allclose(got[0, h], want, rtol=1e-10, atol=1e-12)


def test_rotation_rejects_per_channel_k():
    import workloads as wl
    kf = wl.CacheFormat(wl.INT8, wl.PER_BLOCK_CHANNEL)
    vf = wl.CacheFormat(wl.INT8, wl.PER_TOKEN_HEAD)
    oc = oracle.OracleCache(1, 16, 1, 64, kf, vf, rotation_signs=np.ones(64))
    z = np.zeros((1, 1, 64), np.uint16)
    with pytest.raises(ValueError):
        oracle.quantize_write(oc, z, z, np.array([0]))
