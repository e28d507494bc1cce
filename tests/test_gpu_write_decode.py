"""kvq_write_decode (the step's new token written inside the decode launch)
against the two-call path and against the oracle, through the C ABI.

Every sequence's positions [0, n - 1) are written first with
kvq_quantize_write; the step then writes position n - 1 and decodes over
[0, n).  The fused call must leave the cache byte-identical to
kvq_quantize_write + kvq_paged_decode and give the identical output (same
kernels, same work split), and both must match the oracle: codes and scales
byte for byte, attention within the stated tolerance (max abs error <= 2e-3
everywhere, max rel error <= 1e-2 where |ref| >= 0.2).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import _helpers as H

pytestmark = pytest.mark.gpu

kvq = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global kvq
    from quantized_paged_kv_write_gb300 import build
    build.build()
    import quantized_paged_kv_write_gb300 as m
    m.load_library()
    kvq = m
    yield


def _fmt(dtype, gran=wl.PER_TOKEN_HEAD, group=0):
    return wl.CacheFormat(dtype, gran, group) if group else wl.CacheFormat(dtype, gran)


FP8 = _fmt(wl.FP8)
INT8 = _fmt(wl.INT8)
INT4G = _fmt(wl.INT4, wl.PER_TOKEN_GROUP, 32)
INT4T = _fmt(wl.INT4)

CASES = {
    # name: (k format, v format, q heads, kv heads, head dim, contexts)
    "fp8_fp8": (FP8, FP8, 32, 8, 128, [300, 17, 1, 0, 64, 33]),
    "int8_int8": (INT8, INT8, 32, 8, 128, [129, 16, 48, 2]),
    "fp8_int4": (FP8, INT4G, 32, 8, 128, [257, 31, 200]),
    "int8_int4_wide": (INT8, INT4G, 64, 8, 128, [97, 1, 160]),
    "int8_fp8_d64": (INT8, FP8, 12, 4, 64, [70, 33, 17]),
    "many_short": (FP8, INT4G, 16, 4, 128, [17 + (i * 7) % 30 for i in range(40)]),
    "int4_int4_wide": (INT4T, INT4G, 64, 8, 128, [150, 17, 1]),
    "int4_fp8_d64": (INT4T, FP8, 8, 2, 64, [90, 40]),
    "fp8_int2": (FP8, _fmt(wl.INT2, wl.PER_TOKEN_GROUP, 32), 32, 8, 128, [100, 17, 48]),
}


def _workload(name):
    rotate = name.endswith("_rot")
    kf, vf, hq, hkv, d, ctx = CASES[name[:-4] if rotate else name]
    base = wl.WORKLOADS["long_mixed"]
    return wl.scaled(base, batch=len(ctx), contexts=ctx, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                     name="wd_" + name, k_fmt=kf, v_fmt=vf, decode_steps=0, rotate=rotate)


def _setup(w, ctx):
    """Cache with positions [0, n_b - 1) of every sequence written through
    both sides."""
    table, nb = wl.block_tables(w, spare_blocks=3)
    fmt = kvq.cache_format(w.k_fmt, w.v_fmt, w.num_kv_heads, w.head_dim, nb, w.block_size,
                           rotation_signs=wl.rotation_words(w))
    cache = kvq.allocate_cache(fmt)
    oc = oracle.OracleCache(nb, w.block_size, w.num_kv_heads, w.head_dim, w.k_fmt, w.v_fmt,
                            rotation_signs=H.oracle_signs(w))
    seqs = np.concatenate([np.full(max(n - 1, 0), b, np.int64) for b, n in enumerate(ctx)])
    pos = np.concatenate([np.arange(max(n - 1, 0), dtype=np.int64) for n in ctx])
    if len(seqs):
        k, v, slots = H.gpu_write(kvq, w, fmt, cache, table, seqs, pos)
        H.oracle_write(oc, k, v, slots)
    torch.cuda.synchronize()
    return fmt, cache, oc, table


def _new_tokens(w, ctx):
    live = np.array([b for b, n in enumerate(ctx) if n >= 1], np.int64)
    pos = np.array([ctx[b] - 1 for b in live], np.int64)
    k1, v1 = wl.gather_tokens(w, live, pos, device="cuda")
    k_new = torch.zeros((len(ctx), w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    v_new = torch.zeros_like(k_new)
    if len(live):
        k_new[torch.as_tensor(live, device="cuda")] = k1
        v_new[torch.as_tensor(live, device="cuda")] = v1
    return k_new, v_new, live, pos, k1, v1


def _clone(cache):
    return {k: t.clone() for k, t in cache.items()}


def _step(w, fmt, cache, oc, table, ctx, q):
    """One step both ways; returns the fused cache and output after checking
    them against the two-call path and the oracle."""
    ctx = np.asarray(ctx, np.int32)
    k_new, v_new, live, pos, k1, v1 = _new_tokens(w, ctx)
    bt = torch.as_tensor(table, device="cuda")
    cl = torch.as_tensor(ctx, device="cuda")
    mc = int(ctx.max())

    two = _clone(cache)
    if len(live):
        slots = torch.as_tensor(wl.slot_mapping(table, live, pos, w.block_size), device="cuda")
        kvq.kvq_quantize_write(k1, v1, slots, fmt, two)
    out_two = kvq.kvq_paged_decode(q, fmt, two, bt, cl, mc)

    fused = _clone(cache)
    out_f = kvq.kvq_write_decode(q, k_new, v_new, fmt, fused, bt, cl, mc)
    torch.cuda.synchronize()
    assert kvq.kvq_device_errors() == 0

    for key in fused:
        assert torch.equal(fused[key], two[key]), f"{key} differs from the two-call path"
    assert torch.equal(out_f, out_two), "output differs from the two-call path"

    if len(live):
        H.oracle_write(oc, k1, v1, torch.as_tensor(wl.slot_mapping(table, live, pos, w.block_size)))
    H.compare_cache(fused, oc)
    ref = oracle.paged_decode_fp64(oc, H.bits(q), table, ctx)
    H.check_attention(out_f.cpu().numpy(), ref, w.name)
    return fused, out_f


@pytest.mark.parametrize("name", list(CASES) + ["int4_int4_wide_rot", "fp8_int4_rot", "int4_fp8_d64_rot"])
def test_write_decode_matches_two_calls_and_oracle(name):
    w = _workload(name)
    ctx = wl.context_lens(w)
    fmt, cache, oc, table = _setup(w, ctx)
    q = wl.queries(w, device="cuda")
    _step(w, fmt, cache, oc, table, ctx, q)


def test_three_steps_in_a_row():
    # contexts grow by one per step; the new tokens cross a block boundary
    # (16 -> 17 and 32 -> 33) inside the run
    w = wl.scaled(_workload("fp8_int4"), decode_steps=3)  # the block tables cover the growth
    ctx0 = np.array([30, 15, 200], np.int32)
    fmt, cache, oc, table = _setup(w, ctx0)
    for s in range(3):
        ctx = ctx0 + s
        q = wl.queries(w, step=s, device="cuda")
        cache, _ = _step(w, fmt, cache, oc, table, ctx, q)


def test_per_channel_k_is_rejected():
    kivi = wl.scaled(wl.WORKLOADS["llama3_70b_kivi"], batch=2, contexts=[20, 5], name="wd_kivi")
    table, nb = wl.block_tables(kivi, spare_blocks=1)
    fmt = kvq.cache_format(kivi.k_fmt, kivi.v_fmt, kivi.num_kv_heads, kivi.head_dim, nb, kivi.block_size)
    cache = kvq.allocate_cache(fmt)
    q = wl.queries(kivi, device="cuda")
    k_new = torch.zeros((2, kivi.num_kv_heads, kivi.head_dim), dtype=torch.bfloat16, device="cuda")
    bt = torch.as_tensor(table, device="cuda")
    cl = torch.as_tensor(np.array([20, 5], np.int32), device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_write_decode(q, k_new, k_new.clone(), fmt, cache, bt, cl, 20)
    assert e.value.status == kvq.KVQ_ERR_UNSUPPORTED
