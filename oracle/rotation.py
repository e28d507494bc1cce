"""Oracle: randomized Walsh-Hadamard rotation of K, V and q (test
infrastructure; see the package docstring).

"Quantized KV caches in production: FP8 vs INT8 vs INT4", Numerical Formats
(INT4 and sub-4-bit): rotation techniques (QuaRot) apply randomized
orthogonal Walsh-Hadamard transforms to the activations, spreading outlier
peaks over all channels before uniform 4-bit quantization; the same page's
accuracy section names INT4 with Hadamard rotations among the schemes that
keep baseline quality.

Readings (the pages give no formula):

* the transform of a row x (d channels) is y = H_d (sigma * x): H_d is the
  Sylvester Hadamard matrix (H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]],
  entry (i, j) = (-1)^popcount(i & j)), sigma in {+1, -1}^d are random signs
  drawn once per cache (the "randomized" part), shared by K, V and all
  heads.  H_d is left unnormalized (H_d H_d^T = d I): the scale of each
  quantization group absorbs the factor, and the decode divides by d, a
  power of two;
* the cache stores the quantized y of every K and V row; y is computed in
  FP32 by the radix-2 butterfly with stages h = 1, 2, 4, ..., d/2, each
  replacing (a, b) = (y[j], y[j + h]) by (a + b, a - b), rounded to nearest
  (the bits that the quantizer sees, so both sides agree on every code);
* the decode uses q' = H_d (sigma * q) / d, so q' . y_k = q . k, and returns
  sigma * (H_d o') / d for o' = softmax(...) . y_v (the rotated output).
"""
from __future__ import annotations

import numpy as np


def hadamard(d: int) -> np.ndarray:
    """The d x d Sylvester Hadamard matrix (int64), d a power of two."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1), dtype=np.int64)
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def signs_from_words(words, d: int) -> np.ndarray:
    """sigma (float64 [d], entries +1 / -1) from 32-bit words: bit c % 32 of
    word c // 32 set means sigma_c = -1."""
    w = np.asarray(words, dtype=np.uint64)
    bits = np.array([(int(w[c // 32]) >> (c % 32)) & 1 for c in range(d)])
    return np.where(bits == 1, -1.0, 1.0)


def fwht_float32(x) -> np.ndarray:
    """H_d applied along the last axis by the radix-2 butterfly in float32,
    stages h = 1, 2, ..., d/2 in that order."""
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    h = 1
    while h < d:
        idx = np.arange(d).reshape(-1, 2 * h)
        lo, hi = idx[:, :h].ravel(), idx[:, h:].ravel()
        a, b = y[..., lo], y[..., hi]
        y[..., lo] = a + b
        y[..., hi] = a - b
        h *= 2
    return y


def rotate_rows_float32(x, sigma) -> np.ndarray:
    """y = H_d (sigma * x) in float32 for float32 rows x [..., d] (the sign
    flips are exact)."""
    s32 = np.asarray(sigma, dtype=np.float32)
    return fwht_float32(np.asarray(x, dtype=np.float32) * s32)


def rotate_query_fp64(q, sigma) -> np.ndarray:
    """q' = H_d (sigma * q) / d in float64 (q [..., d])."""
    q = np.asarray(q, dtype=np.float64)
    d = q.shape[-1]
    return (q * sigma) @ hadamard(d).T.astype(np.float64) / d


def unrotate_output_fp64(o, sigma) -> np.ndarray:
    """sigma * (H_d o') / d in float64 (o' [..., d])."""
    o = np.asarray(o, dtype=np.float64)
    d = o.shape[-1]
    return (o @ hadamard(d).T.astype(np.float64)) * sigma / d
