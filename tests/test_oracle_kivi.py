"""Pins of the oracle's per-channel K cache with a full-precision tail
(oracle/kivi.py): appends reproduce whole-block writes, a tail-only sequence
is plain attention over the BF16 rows, a block-aligned sequence is the plain
paged decode, and the mixed case equals torch's float64 attention over the
concatenation of the dequantized blocks and the tail."""
import numpy as np
import torch

import oracle
import workloads as wl

KF = wl.CacheFormat(wl.INT8, wl.PER_BLOCK_CHANNEL)
VF = wl.CacheFormat(wl.INT4, wl.PER_TOKEN_GROUP, 32)
BS, H, D, HQ = 16, 2, 64, 4


def _bits(a):
    return (np.asarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _setup(ctx, seed=0):
    rng = np.random.default_rng(seed)
    b = len(ctx)
    nblk = [(n + BS - 1) // BS for n in ctx]
    table = np.full((b, max(max(nblk), 1)), -1, np.int64)
    perm = rng.permutation(sum(nblk) + 1)
    off = 0
    for i, m in enumerate(nblk):
        table[i, :m] = perm[off:off + m]
        off += m
    cache = oracle.OracleCache(sum(nblk) + 1, BS, H, D, KF, VF)
    k = [_bits(rng.standard_normal((n, H, D))) for n in ctx]
    v = [_bits(rng.standard_normal((n, H, D))) for n in ctx]
    res_k = np.zeros((b, BS, H, D), np.uint16)
    res_v = np.zeros((b, BS, H, D), np.uint16)
    return table, cache, k, v, res_k, res_v, rng


def _append_all(cache, res_k, res_v, k, v, table, ctx):
    for step in range(max(ctx)):
        lens = np.array([step + 1 if step < n else 0 for n in ctx])
        kn = np.stack([k[i][min(step, n - 1)] if n else np.zeros((H, D), np.uint16) for i, n in enumerate(ctx)])
        vn = np.stack([v[i][min(step, n - 1)] if n else np.zeros((H, D), np.uint16) for i, n in enumerate(ctx)])
        oracle.kivi_append(cache, res_k, res_v, kn, vn, table, lens)


def test_appends_reproduce_whole_block_writes():
    ctx = [40, 16, 7]
    table, cache, k, v, res_k, res_v, _ = _setup(ctx)
    _append_all(cache, res_k, res_v, k, v, table, ctx)
    ref = oracle.OracleCache(cache.num_blocks, BS, H, D, KF, VF)
    for i, n in enumerate(ctx):
        for blk in range(n // BS):
            slots = table[i, blk] * BS + np.arange(BS)
            oracle.quantize_write(ref, k[i][blk * BS:(blk + 1) * BS], v[i][blk * BS:(blk + 1) * BS], slots)
        tail = np.arange((n // BS) * BS, n)
        assert np.array_equal(res_k[i][tail % BS], k[i][tail])
        assert np.array_equal(res_v[i][tail % BS], v[i][tail])
    for x in ("k", "v"):
        assert np.array_equal(cache.codes[x], ref.codes[x])
        assert np.array_equal(cache.scales[x].view(np.uint32), ref.scales[x].view(np.uint32))


def test_tail_only_is_attention_over_the_bf16_rows():
    ctx = [9]
    table, cache, k, v, res_k, res_v, rng = _setup(ctx)
    _append_all(cache, res_k, res_v, k, v, table, ctx)
    q = _bits(rng.standard_normal((1, HQ, D)))
    got = oracle.kivi_decode_fp64(cache, res_k, res_v, q, table, np.array(ctx))
    kf = oracle.bf16_bits_to_f32(k[0]).astype(np.float64)
    vf = oracle.bf16_bits_to_f32(v[0]).astype(np.float64)
    qf = oracle.bf16_bits_to_f32(q[0]).astype(np.float64)
    for h in range(HQ):
        assert np.allclose(got[0, h], oracle.attention_fp64(qf[h], kf[:, h // 2], vf[:, h // 2]), rtol=1e-12)


def test_block_aligned_sequence_is_the_plain_paged_decode():
    ctx = [48]
    table, cache, k, v, res_k, res_v, rng = _setup(ctx)
    _append_all(cache, res_k, res_v, k, v, table, ctx)
    q = _bits(rng.standard_normal((1, HQ, D)))
    got = oracle.kivi_decode_fp64(cache, res_k, res_v, q, table, np.array(ctx))
    want = oracle.paged_decode_fp64(cache, q, table, np.array(ctx))
    assert np.array_equal(got, want)


def test_mixed_case_against_torch_sdpa():
    ctx = [37, 50]
    table, cache, k, v, res_k, res_v, rng = _setup(ctx, seed=3)
    _append_all(cache, res_k, res_v, k, v, table, ctx)
    q = _bits(rng.standard_normal((2, HQ, D)))
    got = oracle.kivi_decode_fp64(cache, res_k, res_v, q, table, np.array(ctx))
    for i, n in enumerate(ctx):
        nq = (n // BS) * BS
        t = np.arange(nq)
        kh = oracle.dequantize_cache_rows(cache, "k", table[i][t // BS], t % BS)
        vh = oracle.dequantize_cache_rows(cache, "v", table[i][t // BS], t % BS)
        kt = oracle.bf16_bits_to_f32(k[i][nq:n]).astype(np.float64)
        vt = oracle.bf16_bits_to_f32(v[i][nq:n]).astype(np.float64)
        ka, va = np.concatenate([kh, kt]), np.concatenate([vh, vt])
        qf = oracle.bf16_bits_to_f32(q[i]).astype(np.float64)
        for h in range(HQ):
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.tensor(qf[h][None, None]), torch.tensor(ka[None, :, h // 2]),
                torch.tensor(va[None, :, h // 2]))[0, 0].numpy()
            assert np.allclose(got[i, h], ref, rtol=1e-10, atol=1e-12)
