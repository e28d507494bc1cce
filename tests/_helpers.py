"""Shared test glue: build one workload's caches through the CUDA path (the
C-ABI binding) and through the CPU oracle from the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import workloads as wl

RTOL = 1e-2   # attention tolerance: |o - ref| <= max(ATOL, RTOL * |ref|)
ATOL = 2e-3


def oracle_signs(w):
    """The oracle's sigma (+1 / -1 per channel) of a rotated workload, else None."""
    words = wl.rotation_words(w)
    if words is None:
        return None
    import oracle
    return oracle.signs_from_words(words, w.head_dim)


def bits(t: torch.Tensor) -> np.ndarray:
    """BF16 tensor -> uint16 numpy bit patterns (host copy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def all_positions(w):
    """(seq, pos) for every cached position, sequence-major, in two calls:
    positions written before the call under test, then the call under test."""
    s0, p0 = wl.prewritten_positions(w)
    s1, p1 = wl.write_positions(w)
    return (s0, p0), (s1, p1)


def gpu_write(kvq, w, fmt, cache, table, seqs, pos, device="cuda", k=None, v=None):
    if k is None:
        k, v = wl.gather_tokens(w, seqs, pos, device=device)
    slots = torch.as_tensor(wl.slot_mapping(table, seqs, pos, w.block_size), device=device)
    kvq.kvq_quantize_write(k, v, slots, fmt, cache)
    return k, v, slots


def oracle_write(oracle_cache, k, v, slots):
    import oracle
    oracle.quantize_write(oracle_cache, bits(k), bits(v), slots.detach().cpu().numpy())


def compare_cache(cache, oc):
    """Byte-exact comparison of codes and scales (scales as bit patterns)."""
    for w_ in ("k", "v"):
        got_c = cache[w_ + "_cache"].cpu().numpy()
        assert got_c.shape == oc.codes[w_].shape
        bad = np.argwhere(got_c != oc.codes[w_])
        assert bad.size == 0, f"{w_} codes differ at {bad[:5].tolist()} (of {len(bad)})"
        got_s = cache[w_ + "_scale"].cpu().numpy().view(np.uint32)
        want_s = oc.scales[w_].view(np.uint32)
        bad = np.argwhere(got_s != want_s)
        assert bad.size == 0, f"{w_} scales differ at {bad[:5].tolist()} (of {len(bad)})"


def check_attention(out, ref, what=""):
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(out - ref)
    tol = np.maximum(ATOL, RTOL * np.abs(ref))
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (
        f"{what}: {len(bad)} elements out of tolerance; first {bad[:4].tolist()}: "
        f"got {out[tuple(bad[0])]}, want {ref[tuple(bad[0])]}; max abs err {err.max():.3g}")
    big = np.abs(ref) >= 0.2
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    return float(err.max()), max_rel
