"""Oracle: symmetric quantization of K/V and the paged write (test
infrastructure; see the package docstring).

Every step follows "Use Less Memory: Quantization and Offloading", §2.1
Symmetric Quantization Formula and §5 Exercise 1, in the page's order:

  1. absmax a = max |x| over the scale group,
  2. s = a / q_max,
  3. x_q = clip(round(x / s), -q_max, q_max),
  4. x_hat = x_q * s (dequantization, done by the attention reader).

Precision: x is BF16 widened to FP32 (exact); a, s and x / s are FP32 with
correctly rounded IEEE division (numpy float32 arithmetic); round is
round-half-to-even (np.rint).  FP8 replaces step 3's integer rounding by the
OCP E4M3FN encoding of the FP32 quotient with round-to-nearest-even and
saturation to ±448 ("Quantized KV caches in production", Numerical Formats;
"Use Less Memory", §2.3).  A group whose absmax is 0 gets s = +0 and all
codes +0 (the pages leave 0/0 undefined).
"""
from __future__ import annotations

import numpy as np

INT8 = "int8"
INT4 = "int4"
INT2 = "int2"
FP8 = "fp8_e4m3fn"
PER_TOKEN_HEAD = "token_head"
PER_TOKEN_GROUP = "token_group"
PER_BLOCK_CHANNEL = "block_channel"

# q_max per target format: "Use Less Memory", §2.1 format table (INT8 127,
# INT4 7); FP8 E4M3FN's largest finite value 448 (OCP 8-bit FP spec, named in
# "Quantized KV caches in production", Numerical Formats).  INT2 (the 2-bit
# codes of KIVI, same page): the table's rule q_max = 2^(b-1) - 1 gives 1.
Q_MAX = {INT8: 127, INT4: 7, INT2: 1, FP8: 448}


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Widen BF16 (given as uint16 bit patterns) to float32; exact."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


# ---------------------------------------------------------------------------
# FP8 E4M3FN (OCP): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
# no infinities, exponent 15 with mantissa 7 is NaN, largest finite 448,
# subnormals m * 2^-9.
# ---------------------------------------------------------------------------

def e4m3fn_decode(code) -> np.ndarray:
    """E4M3FN bit patterns (uint8) to their exact values (float64)."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3fn_encode(r) -> np.ndarray:
    """Encode finite float32 values as E4M3FN with round-to-nearest-even and
    saturation of magnitudes >= 448 to ±448.  The sign bit of the input is
    kept, so -0.0 and negatives that round to zero give 0x80."""
    r = np.asarray(r, dtype=np.float32)
    sign = (np.signbit(r).astype(np.uint8) << 7).astype(np.uint8)
    mag = np.abs(r).astype(np.float64)
    sat = mag >= 448.0
    mag = np.where(sat, 448.0, mag)            # saturating: |r| >= 448 -> 448
    # subnormal binade [0, 2^-6): representable points k * 2^-9; k = 8 is the
    # smallest normal 2^-6, whose bit pattern 0x08 continues the count.
    k_sub = np.rint(mag * 2.0 ** 9)
    # normal binades [2^e, 2^(e+1)): points 2^e * (1 + j/8), j = 0..7
    _, ex = np.frexp(np.where(mag > 0, mag, 1.0))
    e = ex.astype(np.int64) - 1
    k = np.rint(mag * np.exp2(3.0 - e))          # in [8, 16]
    carry = k == 16
    e = np.where(carry, e + 1, e)
    k = np.where(carry, 8, k)
    normal = ((e + 7) << 3) | (k.astype(np.int64) - 8)
    code = np.where(mag < 2.0 ** -6, k_sub.astype(np.int64), normal)
    return (code.astype(np.uint8) | sign).astype(np.uint8)


# ---------------------------------------------------------------------------
# the symmetric quantizer over scale groups
# ---------------------------------------------------------------------------

def quantize_symmetric(x, dtype: str):
    """Quantize float32 ``x`` [..., n]; the last axis is one scale group.

    Returns (codes, s): codes int8 [..., n] in [-q_max, q_max] for INT8/INT4,
    uint8 E4M3FN bit patterns for FP8; s float32 [...]."""
    x = np.asarray(x, dtype=np.float32)
    q_max = np.float32(Q_MAX[dtype])
    a = np.max(np.abs(x), axis=-1)                      # step 1
    s = (a / q_max).astype(np.float32)                  # step 2
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (x / s[..., None]).astype(np.float32)       # step 3: x / s
    zero = s == 0
    r = np.where(zero[..., None], np.float32(0.0), r)
    if dtype == FP8:
        codes = e4m3fn_encode(r)
    else:
        codes = np.clip(np.rint(r), -q_max, q_max).astype(np.int8)
    codes = np.where(zero[..., None], np.zeros((), codes.dtype), codes)
    return codes, s


def dequantize_rows(codes, s, dtype: str) -> np.ndarray:
    """x_hat = x_q * s in float64 (exact: both factors have <= 24 bits)."""
    if dtype == FP8:
        qv = e4m3fn_decode(codes)
    else:
        qv = np.asarray(codes, dtype=np.int8).astype(np.float64)
    return qv * np.asarray(s, dtype=np.float64)


def pack_int4(codes) -> np.ndarray:
    """Two's-complement 4-bit codes [..., n] (n even) to bytes [..., n/2];
    element 2j goes to the low nibble of byte j, element 2j+1 to the high."""
    c = np.asarray(codes, dtype=np.int8).astype(np.int64) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def pack_int2(codes) -> np.ndarray:
    """Two's-complement 2-bit codes [..., n] (n % 4 == 0) to bytes
    [..., n/4]; element 4j + m goes to bits 2m .. 2m + 1 of byte j."""
    c = np.asarray(codes, dtype=np.int8).astype(np.int64) & 0x3
    return (c[..., 0::4] | (c[..., 1::4] << 2) | (c[..., 2::4] << 4) | (c[..., 3::4] << 6)).astype(np.uint8)


def unpack_int2(packed) -> np.ndarray:
    """Inverse of pack_int2: bytes [..., m] to int8 codes [..., 4m]."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    out = np.empty(p.shape[:-1] + (4 * p.shape[-1],), dtype=np.int64)
    for m in range(4):
        c = (p >> (2 * m)) & 0x3
        out[..., m::4] = np.where(c >= 2, c - 4, c)
    return out.astype(np.int8)


def unpack_int4(packed) -> np.ndarray:
    """Inverse of pack_int4: bytes [..., m] to int8 codes [..., 2m]."""
    p = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    lo = p & 0xF
    hi = (p >> 4) & 0xF
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    out = np.where(out >= 8, out - 16, out)
    return out.astype(np.int8)


# ---------------------------------------------------------------------------
# the paged cache ("PidokuInfra 12 KV Cache Quantization", §5 Where the scales
# live): codes (num_blocks, block_size, n_kv_heads, head_dim) and one scale per
# (block, slot, kv_head); grouped scales add a trailing group axis; per-channel
# K scales are (num_blocks, n_kv_heads, head_dim).  Scales are FP32.
# ---------------------------------------------------------------------------

class OracleCache:
    """Host-side paged cache for one layer: K and V codes and scales."""

    def __init__(self, num_blocks, block_size, num_kv_heads, head_dim, k_fmt, v_fmt, rotation_signs=None):
        # rotation_signs: None, or sigma (+1 / -1, [head_dim]) of the
        # randomized Walsh-Hadamard rotation applied to every K and V row
        # before quantization (oracle/rotation.py)
        self.rotation = None if rotation_signs is None else np.asarray(rotation_signs, dtype=np.float64)
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.num_kv_heads = int(num_kv_heads)
        self.head_dim = int(head_dim)
        self.fmt = {"k": k_fmt, "v": v_fmt}
        self.codes = {}
        self.scales = {}
        for which, fmt in self.fmt.items():
            row = head_dim // 2 if fmt.dtype == INT4 else (head_dim // 4 if fmt.dtype == INT2 else head_dim)
            self.codes[which] = np.zeros(
                (num_blocks, block_size, num_kv_heads, row), dtype=np.uint8)
            self.scales[which] = np.zeros(self.scale_shape(fmt), dtype=np.float32)

    def scale_shape(self, fmt):
        nb, bs, h, d = self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim
        if fmt.gran == PER_TOKEN_HEAD:
            return (nb, bs, h)
        if fmt.gran == PER_TOKEN_GROUP:
            return (nb, bs, h, d // fmt.group)
        if fmt.gran == PER_BLOCK_CHANNEL:
            return (nb, h, d)
        raise ValueError(fmt.gran)


def _codes_to_bytes(codes, dtype):
    if dtype == INT4:
        return pack_int4(codes)
    if dtype == INT2:
        return pack_int2(codes)
    return np.asarray(codes).view(np.uint8) if codes.dtype == np.int8 else codes


def _quantize_tokens(x, fmt):
    """Per-token formats: x float32 [N, H, d] -> (code bytes [N, H, row],
    scales [N, H] or [N, H, d/group])."""
    n, h, d = x.shape
    if fmt.gran == PER_TOKEN_HEAD:
        codes, s = quantize_symmetric(x, fmt.dtype)
    elif fmt.gran == PER_TOKEN_GROUP:
        g = fmt.group
        codes, s = quantize_symmetric(x.reshape(n, h, d // g, g), fmt.dtype)
        codes = codes.reshape(n, h, d)
    else:
        raise ValueError(fmt.gran)
    return _codes_to_bytes(codes, fmt.dtype), s


def quantize_write(cache: OracleCache, k_bits, v_bits, slot_mapping):
    """Quantize BF16 K and V rows (uint16 bits [N, H, d]) and store them at
    their slots: slot = physical_block * block_size + offset; slots < 0 are
    skipped.  Per-channel K takes, for each physical block touched and each
    (kv_head, channel), the absmax over the tokens this call writes into that
    block ("PidokuInfra 12", K is more sensitive than V: per-channel K; KIVI
    in "Quantized KV caches in production", Numerical Formats)."""
    slots = np.asarray(slot_mapping, dtype=np.int64)
    keep = slots >= 0
    bs = cache.block_size
    blk = slots[keep] // bs
    off = slots[keep] % bs
    for which, bits in (("k", k_bits), ("v", v_bits)):
        fmt = cache.fmt[which]
        x = bf16_bits_to_f32(np.asarray(bits)[keep])
        if cache.rotation is not None:
            if fmt.gran == PER_BLOCK_CHANNEL:
                raise ValueError("the rotation applies to per-token formats only")
            from .rotation import rotate_rows_float32
            x = rotate_rows_float32(x, cache.rotation)
        if fmt.gran == PER_BLOCK_CHANNEL:
            for b in np.unique(blk):
                rows = np.flatnonzero(blk == b)
                # the group of one (kv_head, channel) is the block's new rows
                xb = np.transpose(x[rows], (1, 2, 0))          # [H, d, rows]
                codes, s = quantize_symmetric(xb, fmt.dtype)   # s: [H, d]
                codes = np.transpose(codes, (2, 0, 1))         # [rows, H, d]
                cache.codes[which][b, off[rows]] = _codes_to_bytes(codes, fmt.dtype)
                cache.scales[which][b] = s
        else:
            code_bytes, s = _quantize_tokens(x, fmt)
            cache.codes[which][blk, off] = code_bytes
            cache.scales[which][blk, off] = s
    return cache


def dequantize_cache_rows(cache: OracleCache, which: str, blocks, offsets) -> np.ndarray:
    """x_hat (float64 [n, H, d]) of the cache rows at (blocks[i], offsets[i])."""
    fmt = cache.fmt[which]
    blocks = np.asarray(blocks, dtype=np.int64)
    offsets = np.asarray(offsets, dtype=np.int64)
    raw = cache.codes[which][blocks, offsets]            # [n, H, row]
    h, d = cache.num_kv_heads, cache.head_dim
    if fmt.dtype == INT4:
        codes = unpack_int4(raw)
    elif fmt.dtype == INT2:
        codes = unpack_int2(raw)
    elif fmt.dtype == INT8:
        codes = raw.view(np.int8)
    else:
        codes = raw
    if fmt.gran == PER_TOKEN_HEAD:
        s = cache.scales[which][blocks, offsets][..., None]           # [n, H, 1]
        return dequantize_rows(codes, s, fmt.dtype)
    if fmt.gran == PER_TOKEN_GROUP:
        g = fmt.group
        s = cache.scales[which][blocks, offsets]                       # [n, H, d/g]
        c = codes.reshape(codes.shape[0], h, d // g, g)
        return dequantize_rows(c, s[..., None], fmt.dtype).reshape(-1, h, d)
    if fmt.gran == PER_BLOCK_CHANNEL:
        s = cache.scales[which][blocks]                                # [n, H, d]
        return dequantize_rows(codes, s, fmt.dtype)
    raise ValueError(fmt.gran)
