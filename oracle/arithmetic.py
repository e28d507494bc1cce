"""Oracle: the pages' byte and step-time arithmetic (test infrastructure).

* Bytes per token: 2 · L · H_kv · d · b ("Use Less Memory", §5 Exercise 3;
  "Quantized KV caches in production", The Mathematics of KV Cache Growth).
* Scale overhead of a per-(token, head) scale and of INT4 with group scales
  ("PidokuInfra 12", §5 Where the scales live).
* Decode step time = (KV bytes read + weight bytes) / bandwidth, maximum
  concurrency under a KV budget ("PidokuInfra 12", §4 Tiny example) and the
  speedup model (W + KV) / (W + KV / 2) (§6-9 Under the hood).

Units follow the pages: decimal GB (1e9) where they print "GB", binary KiB /
GiB where they print those.
"""
from __future__ import annotations

import math


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, bytes_per_elem: float) -> float:
    """K and V bytes one token occupies across all layers."""
    return 2 * layers * kv_heads * head_dim * bytes_per_elem


def kv_bytes_per_sequence(layers, kv_heads, head_dim, bytes_per_elem, tokens) -> float:
    return kv_bytes_per_token(layers, kv_heads, head_dim, bytes_per_elem) * tokens


def per_token_scale_overhead(head_dim: int, code_bytes_per_elem: float, scale_bytes: int) -> float:
    """Scale bytes over code bytes for one (token, head) vector."""
    return scale_bytes / (head_dim * code_bytes_per_elem)


def int4_grouped_vector_bytes(head_dim: int, group: int, scale_bytes: int) -> float:
    """Packed INT4 codes plus one scale per group, for one head vector."""
    return head_dim / 2 + (head_dim // group) * scale_bytes


def max_sequences(budget_bytes: float, bytes_per_sequence: float) -> int:
    return int(math.floor(budget_bytes / bytes_per_sequence))


def decode_step_seconds(kv_bytes: float, weight_bytes: float, bandwidth_bytes_per_s: float) -> float:
    return (kv_bytes + weight_bytes) / bandwidth_bytes_per_s


def kv_quantization_speedup(weight_bytes: float, kv16_bytes: float) -> float:
    """(W + KV_fp16) / (W + KV_fp16 / 2)."""
    return (weight_bytes + kv16_bytes) / (weight_bytes + kv16_bytes / 2)
