"""Oracle: per-channel K caches that take appends (test infrastructure; see
the package docstring).

"Quantized KV caches in production: FP8 vs INT8 vs INT4", Numerical Formats:
KIVI quantizes K per channel and V per token.  A per-channel K scale spans
the tokens of a block ("PidokuInfra 12 KV Cache Quantization", K is more
sensitive than V), so a block can only be quantized once all of its tokens
are known.

Reading (the pages give no rule for appends): a sequence keeps the tokens of
its last, incomplete block in full precision -- the BF16 K and V rows sit in
a residual buffer, row p % block_size for position p -- and when the block's
last token arrives, the block is quantized as quantize_write would quantize
its block_size tokens written in one call (per-channel K over exactly those
tokens, V per its own format).  The decode attends over the quantized
complete blocks followed by the full-precision tail.
"""
from __future__ import annotations

import numpy as np

from .attention import _sequence_rows, attention_fp64
from .quantize import OracleCache, bf16_bits_to_f32, dequantize_cache_rows, quantize_write


def kivi_append(cache: OracleCache, res_k, res_v, k_bits_new, v_bits_new, block_tables, context_lens):
    """One appended token per sequence (context_lens: lengths after it, 0 =
    no token).  res_k, res_v: uint16 BF16 bits [B, block_size, H, d], updated
    in place; k_bits_new, v_bits_new: [B, H, d].  A block completed by its
    token is quantized into the cache."""
    bs = cache.block_size
    for b, n in enumerate(np.asarray(context_lens, dtype=np.int64)):
        if n < 1:
            continue
        r = (n - 1) % bs
        res_k[b, r] = k_bits_new[b]
        res_v[b, r] = v_bits_new[b]
        if n % bs == 0:
            blk = int(block_tables[b][(n - 1) // bs])
            slots = blk * bs + np.arange(bs)
            quantize_write(cache, res_k[b], res_v[b], slots)


def kivi_decode_fp64(cache: OracleCache, res_k, res_v, q_bits, block_tables, context_lens) -> np.ndarray:
    """float64 [B, H_q, d]: attention over the quantized complete blocks
    [0, 16 floor(n / 16)) and the residual's full-precision tail."""
    q_bits = np.asarray(q_bits, dtype=np.uint16)
    bsz, hq, d = q_bits.shape
    bs = cache.block_size
    g = hq // cache.num_kv_heads
    out = np.zeros((bsz, hq, d), dtype=np.float64)
    for b in range(bsz):
        n = int(context_lens[b])
        if n == 0:
            continue
        nq = (n // bs) * bs
        blocks, offs = _sequence_rows(cache, block_tables[b], nq)
        k_hat = dequantize_cache_rows(cache, "k", blocks, offs)
        v_hat = dequantize_cache_rows(cache, "v", blocks, offs)
        tail = np.arange(nq, n) % bs
        k_t = bf16_bits_to_f32(np.asarray(res_k[b])[tail]).astype(np.float64)
        v_t = bf16_bits_to_f32(np.asarray(res_v[b])[tail]).astype(np.float64)
        k_all = np.concatenate([k_hat, k_t])
        v_all = np.concatenate([v_hat, v_t])
        q = bf16_bits_to_f32(q_bits[b]).astype(np.float64)
        for h in range(hq):
            kv = h // g
            out[b, h] = attention_fp64(q[h], k_all[:, kv, :], v_all[:, kv, :])
    return out
