"""Oracle: paged decode attention over the quantized cache, in float64 (test
infrastructure; see the package docstring).

"PidokuInfra 12 KV Cache Quantization", §5 The kernel side: for every cached
token the reader loads the codes and their scales, dequantizes
(x_hat = x_q * s, "Use Less Memory", §2.1) and forms q·kᵀ; the output is
softmax(q·kᵀ / sqrt(d)) · V (§5, K is more sensitive than V).  Blocks are
found through the sequence's block table (PagedAttention, "Quantized KV caches
in production" and the "KV Cache Quantization" glossary).  Query head h reads
kv head h // (H_q / H_kv) (GQA groups of consecutive query heads, glossary).

Everything is float64: q is BF16 widened exactly, x_hat = code * s is exact,
the softmax subtracts the row maximum before exp.  A sequence with context 0
produces zeros.
"""
from __future__ import annotations

import math

import numpy as np

from .quantize import OracleCache, bf16_bits_to_f32, dequantize_cache_rows


def attention_fp64(q, k_hat, v_hat) -> np.ndarray:
    """softmax(q · k_hatᵀ / sqrt(d)) · v_hat for one query row.

    q: float64 [d]; k_hat, v_hat: float64 [n, d].  Returns float64 [d]."""
    n, d = k_hat.shape
    if n == 0:
        return np.zeros(d, dtype=np.float64)
    z = (k_hat @ q) / math.sqrt(d)
    p = np.exp(z - np.max(z))
    return (p @ v_hat) / np.sum(p)


def _sequence_rows(cache: OracleCache, block_table_row, n):
    bs = cache.block_size
    t = np.arange(n, dtype=np.int64)
    blocks = np.asarray(block_table_row, dtype=np.int64)[t // bs]
    return blocks, t % bs


def paged_decode_one_fp64(cache: OracleCache, q_bits_row, block_table_row,
                          context_len: int, q_head: int, num_q_heads: int) -> np.ndarray:
    """Output (float64 [d]) of one (sequence, query head) pair."""
    g = num_q_heads // cache.num_kv_heads
    kv = q_head // g
    blocks, offs = _sequence_rows(cache, block_table_row, int(context_len))
    k_hat = dequantize_cache_rows(cache, "k", blocks, offs)[:, kv, :]
    v_hat = dequantize_cache_rows(cache, "v", blocks, offs)[:, kv, :]
    q = bf16_bits_to_f32(q_bits_row).astype(np.float64)
    if cache.rotation is None:
        return attention_fp64(q, k_hat, v_hat)
    from .rotation import rotate_query_fp64, unrotate_output_fp64
    o = attention_fp64(rotate_query_fp64(q, cache.rotation), k_hat, v_hat)
    return unrotate_output_fp64(o, cache.rotation)


def paged_decode_fp64(cache: OracleCache, q_bits, block_tables, context_lens) -> np.ndarray:
    """Decode attention for every sequence and query head.

    q_bits: BF16 bits uint16 [B, H_q, d]; block_tables: int [B, max_blocks];
    context_lens: int [B].  Returns float64 [B, H_q, d]."""
    q_bits = np.asarray(q_bits, dtype=np.uint16)
    bsz, hq, d = q_bits.shape
    g = hq // cache.num_kv_heads
    out = np.zeros((bsz, hq, d), dtype=np.float64)
    for b in range(bsz):
        n = int(context_lens[b])
        if n == 0:
            continue
        blocks, offs = _sequence_rows(cache, block_tables[b], n)
        k_hat = dequantize_cache_rows(cache, "k", blocks, offs)
        v_hat = dequantize_cache_rows(cache, "v", blocks, offs)
        q = bf16_bits_to_f32(q_bits[b]).astype(np.float64)
        if cache.rotation is not None:
            # rotated cache: q' = H (sigma q) / d, output sigma (H o') / d
            from .rotation import rotate_query_fp64, unrotate_output_fp64
            q = rotate_query_fp64(q, cache.rotation)
        for h in range(hq):
            kv = h // g
            out[b, h] = attention_fp64(q[h], k_hat[:, kv, :], v_hat[:, kv, :])
        if cache.rotation is not None:
            out[b] = unrotate_output_fp64(out[b], cache.rotation)
    return out
