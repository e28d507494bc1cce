"""Shared test glue: build one workload's caches through the CUDA path (the
C-ABI binding) and through the CPU oracle from the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import workloads as wl

# Attention tolerance, as stated for the decode output against the oracle's
# fp64 attention over the same dequantized values: max abs error <= ATOL over
# every element AND max rel error <= RTOL over the elements whose reference
# magnitude is at least REL_FLOOR (a relative error near a zero reference
# says nothing; with the floor the relative bound follows from the absolute
# one, and both are asserted).
ATOL = 2e-3
RTOL = 1e-2
REL_FLOOR = 0.2


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


def attention_errors(out, ref):
    """(max abs error over all elements, max rel error over |ref| >= REL_FLOOR)."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(out - ref)
    big = np.abs(ref) >= REL_FLOOR
    max_abs = float(err.max()) if err.size else 0.0
    max_rel = float((err[big] / np.abs(ref[big])).max()) if big.any() else 0.0
    if not np.all(np.isfinite(out)):
        max_abs = max_rel = float("inf")
    return max_abs, max_rel


def check_attention(out, ref, what=""):
    """Assert the stated tolerance (both bounds) and print both maxima."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    max_abs, max_rel = attention_errors(out, ref)
    print(f"[attention] {what}: max abs err {max_abs:.3e}, max rel err {max_rel:.3e} "
          f"(|ref| max {np.abs(ref).max() if ref.size else 0.0:.3g})")
    if not (max_abs <= ATOL and max_rel <= RTOL):
        err = np.abs(out - ref)
        bad = np.argwhere(~(err <= ATOL))
        first = tuple(bad[0]) if bad.size else ()
        raise AssertionError(
            f"{what}: max abs err {max_abs:.3e} (bound {ATOL}), max rel err {max_rel:.3e} (bound {RTOL}); "
            f"{len(bad)} elements above the absolute bound; first {bad[:4].tolist()}"
            + (f": got {out[first]}, want {ref[first]}" if first else ""))
    return max_abs, max_rel
