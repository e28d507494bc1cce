"""Pins of the oracle's float64 paged decode attention.

* Against torch.nn.functional.scaled_dot_product_attention in float64 (a
  library routine, with GQA by repeating each kv head over its consecutive
  query heads) on dense un-paged tensors.  The inputs are chosen exactly
  representable by the quantizer (integer values with absmax 127 per token,
  so s = 1 and x_hat = x), which makes the expected value independent of the
  oracle's own dequantization.
* Closed forms: context 1 gives v_hat_0; identical keys or q = 0 give the
  mean of v_hat; context 0 gives 0.
* Paging invariance: permuting physical blocks together with the block table
  leaves the output unchanged (bit for bit).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import quantize as oq
from oracle import attention as oa


class Fmt:
    def __init__(self, dtype, gran=oq.PER_TOKEN_HEAD, group=0):
        self.dtype, self.gran, self.group = dtype, gran, group


def bf16_bits(x):
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _build(rng, ctx, hkv, d, bs, k_fmt, v_fmt, kv_values=None, spare=3):
    """Write every position of every sequence through the oracle's
    quantize_write into a cache with a shuffled block table."""
    ctx = np.asarray(ctx)
    nblk = (ctx + bs - 1) // bs
    num_blocks = int(nblk.sum()) + spare
    perm = rng.permutation(num_blocks)
    table = np.full((len(ctx), max(int(nblk.max()), 1)), -1, np.int64)
    o = 0
    for b, n in enumerate(nblk):
        table[b, :n] = perm[o:o + n]
        o += n
    cache = oq.OracleCache(num_blocks, bs, hkv, d, k_fmt, v_fmt)
    seqs = np.concatenate([np.full(c, b) for b, c in enumerate(ctx)])
    pos = np.concatenate([np.arange(c) for c in ctx])
    if kv_values is None:
        k = rng.standard_normal((len(seqs), hkv, d))
        v = rng.standard_normal((len(seqs), hkv, d))
    else:
        k, v = kv_values(len(seqs))
    slots = table[seqs, pos // bs] * bs + pos % bs
    oq.quantize_write(cache, bf16_bits(k), bf16_bits(v), slots)
    return cache, table, k, v, seqs, pos


def _sdpa_dense(q, k, v, hq, hkv):
    """torch SDPA in float64: q [Hq, d], k, v [n, Hkv, d]."""
    g = hq // hkv
    kk = torch.as_tensor(k, dtype=torch.float64).permute(1, 0, 2).repeat_interleave(g, 0)
    vv = torch.as_tensor(v, dtype=torch.float64).permute(1, 0, 2).repeat_interleave(g, 0)
    qq = torch.as_tensor(q, dtype=torch.float64)[:, None, :]
    return F.scaled_dot_product_attention(qq[None], kk[None], vv[None])[0, :, 0, :].numpy()


@pytest.mark.parametrize("hq,hkv", [(4, 2), (8, 8), (8, 1), (16, 2)])
def test_decode_vs_sdpa_exact_inputs(hq, hkv):
    rng = np.random.default_rng(hq * 10 + hkv)
    d, bs = 32, 16
    ctx = [1, 17, 40, 16]

    def exact_values(n):
        # integers in [-127, 127] with |x| = 127 somewhere in each (token,
        # head) row, times a per-row power of two 2^e: s = 2^e exactly and
        # the INT8 codes equal the integers, so x_hat = x with no rounding
        # and every row has its own scale
        k = rng.integers(-127, 128, size=(n, hkv, d)).astype(np.float64)
        v = rng.integers(-127, 128, size=(n, hkv, d)).astype(np.float64)
        k[:, :, 0] = 127
        v[:, :, 1] = -127
        k *= np.exp2(rng.integers(-7, -2, size=(n, hkv, 1)))  # keeps logits moderate
        v *= np.exp2(rng.integers(-3, 4, size=(n, hkv, 1)))
        return k, v

    cache, table, k, v, seqs, pos = _build(
        rng, ctx, hkv, d, bs, Fmt(oq.INT8), Fmt(oq.INT8), kv_values=exact_values)
    q = rng.standard_normal((len(ctx), hq, d))
    qb = bf16_bits(q)
    out = oa.paged_decode_fp64(cache, qb, table, np.array(ctx))
    qf = oq.bf16_bits_to_f32(qb).astype(np.float64)
    for b, n in enumerate(ctx):
        rows = np.flatnonzero(seqs == b)
        ref = _sdpa_dense(qf[b], k[rows], v[rows], hq, hkv)
        np.testing.assert_allclose(out[b], ref, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("kfmt,vfmt", [
    (Fmt(oq.FP8), Fmt(oq.FP8)),
    (Fmt(oq.INT8, oq.PER_BLOCK_CHANNEL), Fmt(oq.INT4, oq.PER_TOKEN_GROUP, 32)),
    (Fmt(oq.FP8), Fmt(oq.INT4, oq.PER_TOKEN_GROUP, 32)),
])
def test_decode_vs_sdpa_on_dequantized(kfmt, vfmt):
    # general formats: the dense reference uses the oracle's dequantized rows
    # read back in position order (paging and attention are what is checked)
    rng = np.random.default_rng(9)
    hq, hkv, d, bs = 8, 2, 64, 16
    ctx = [33, 64, 5]
    cache, table, k, v, seqs, pos = _build(rng, ctx, hkv, d, bs, kfmt, vfmt)
    q = bf16_bits(rng.standard_normal((len(ctx), hq, d)))
    out = oa.paged_decode_fp64(cache, q, table, np.array(ctx))
    qf = oq.bf16_bits_to_f32(q).astype(np.float64)
    for b, n in enumerate(ctx):
        t = np.arange(n)
        blocks = table[b, t // bs]
        kh = oq.dequantize_cache_rows(cache, "k", blocks, t % bs)
        vh = oq.dequantize_cache_rows(cache, "v", blocks, t % bs)
        np.testing.assert_allclose(out[b], _sdpa_dense(qf[b], kh, vh, hq, hkv),
                                   rtol=1e-12, atol=1e-12)
        # and the single-pair entry point agrees
        for h in (0, hq - 1):
            one = oa.paged_decode_one_fp64(cache, q[b, h], table[b], n, h, hq)
            assert np.array_equal(one, out[b, h])


def test_closed_forms():
    rng = np.random.default_rng(10)
    hq, hkv, d, bs = 2, 1, 16, 16
    # context 1: the output is v_hat_0
    cache, table, k, v, seqs, pos = _build(rng, [1], hkv, d, bs, Fmt(oq.INT8), Fmt(oq.INT8))
    q = bf16_bits(rng.standard_normal((1, hq, d)))
    out = oa.paged_decode_fp64(cache, q, table, np.array([1]))
    v0 = oq.dequantize_cache_rows(cache, "v", table[0, :1], [0])[0, 0]
    assert np.array_equal(out[0, 0], v0) and np.array_equal(out[0, 1], v0)
    # identical keys: uniform attention, the output is the mean of v_hat
    n = 50
    same_k = lambda m: (np.tile(rng.standard_normal((1, hkv, d)), (m, 1, 1)),
                        rng.standard_normal((m, hkv, d)))
    cache, table, k, v, seqs, pos = _build(rng, [n], hkv, d, bs, Fmt(oq.INT8), Fmt(oq.INT8),
                                           kv_values=same_k)
    out = oa.paged_decode_fp64(cache, q, table, np.array([n]))
    t = np.arange(n)
    vh = oq.dequantize_cache_rows(cache, "v", table[0, t // bs], t % bs)[:, 0]
    np.testing.assert_allclose(out[0, 0], vh.mean(axis=0), rtol=1e-13, atol=1e-13)
    # q = 0: uniform attention as well
    qz = bf16_bits(np.zeros((1, hq, d)))
    cache, table, k, v, seqs, pos = _build(rng, [n], hkv, d, bs, Fmt(oq.FP8), Fmt(oq.FP8))
    out = oa.paged_decode_fp64(cache, qz, table, np.array([n]))
    vh = oq.dequantize_cache_rows(cache, "v", table[0, t // bs], t % bs)[:, 0]
    np.testing.assert_allclose(out[0, 1], vh.mean(axis=0), rtol=1e-13, atol=1e-13)
    # context 0: zeros
    out = oa.paged_decode_fp64(cache, q, table, np.array([0]))
    assert np.all(out == 0)


def test_softmax_scale_is_inverse_sqrt_head_dim():
    # keys 127 e_0 and 0, values 127 e_0 and 127 e_1 (all exact: s = 1), q =
    # 2^-5 e_0: the weights are softmax([127 * 2^-5 / sqrt(d), 0])
    d, bs = 64, 16
    cache = oq.OracleCache(1, bs, 1, d, Fmt(oq.INT8), Fmt(oq.INT8))
    k = np.zeros((2, 1, d)); k[0, 0, 0] = 127.0
    v = np.zeros((2, 1, d)); v[0, 0, 0] = 127.0; v[1, 0, 1] = 127.0
    oq.quantize_write(cache, bf16_bits(k), bf16_bits(v), np.array([0, 1]))
    q = np.zeros((1, 1, d)); q[0, 0, 0] = 2.0 ** -5
    out = oa.paged_decode_fp64(cache, bf16_bits(q), np.array([[0]]), np.array([2]))
    z = 127.0 * 2.0 ** -5 / math.sqrt(d)
    w0 = math.exp(z) / (math.exp(z) + 1.0)
    assert abs(out[0, 0, 0] - 127 * w0) < 1e-12 and abs(out[0, 0, 1] - 127 * (1 - w0)) < 1e-12


def test_paging_invariance():
    rng = np.random.default_rng(11)
    hq, hkv, d, bs = 4, 2, 32, 16
    ctx = [70, 3, 48]
    cache, table, k, v, seqs, pos = _build(rng, ctx, hkv, d, bs, Fmt(oq.FP8),
                                           Fmt(oq.INT4, oq.PER_TOKEN_GROUP, 32))
    q = bf16_bits(rng.standard_normal((len(ctx), hq, d)))
    out = oa.paged_decode_fp64(cache, q, table, np.array(ctx))
    # move every physical block to a new index and rewrite the table
    perm = rng.permutation(cache.num_blocks)
    moved = oq.OracleCache(cache.num_blocks, bs, hkv, d, cache.fmt["k"], cache.fmt["v"])
    for w in ("k", "v"):
        moved.codes[w][perm] = cache.codes[w]
        moved.scales[w][perm] = cache.scales[w]
    table2 = np.where(table >= 0, perm[np.maximum(table, 0)], -1)
    out2 = oa.paged_decode_fp64(moved, q, table2, np.array(ctx))
    assert np.array_equal(out, out2)
