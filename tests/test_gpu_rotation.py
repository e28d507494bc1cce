"""Walsh-Hadamard-rotated caches through the C ABI against the oracle.

With the rotation on, every K and V row is rotated in FP32 before it is
quantized ("Quantized KV caches in production", Numerical Formats: randomized
orthogonal Walsh-Hadamard transforms before 4-bit quantization); the codes
and scales must equal the oracle's byte for byte, and the decode (query
rotated, output rotated back) must match the oracle's float64 attention
within the stated tolerance (max abs error <= 2e-3 everywhere, max rel
error <= 1e-2 where |ref| >= 0.2).
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


INT4T = wl.CacheFormat(wl.INT4, wl.PER_TOKEN_HEAD)
INT4G = wl.CacheFormat(wl.INT4, wl.PER_TOKEN_GROUP, 32)
INT8 = wl.CacheFormat(wl.INT8, wl.PER_TOKEN_HEAD)
FP8 = wl.CacheFormat(wl.FP8, wl.PER_TOKEN_HEAD)

CASES = {
    # name: (k, v, q heads, kv heads, head dim, contexts)
    "int4_int4g": (INT4T, INT4G, 32, 8, 128, [300, 37, 16]),
    "int4_int4g_wide": (INT4T, INT4G, 64, 8, 128, [129, 64]),
    "int4_fp8_d64": (INT4T, FP8, 8, 2, 64, [90, 17, 45]),
    "int8_int4g": (INT8, INT4G, 16, 4, 128, [70, 200]),
    "fp8_fp8": (FP8, FP8, 32, 8, 128, [150, 33]),
    "int8_int8_d64": (INT8, INT8, 12, 4, 64, [65, 31]),
    "int4_int4g_g3": (INT4T, INT4G, 6, 2, 128, [77, 20]),    # packed, one inactive row slot
    "int4_int4g_mha": (INT4T, INT4G, 4, 4, 64, [50, 18]),    # G = 1
}


def _workload(name, rotate=True, outliers=True):
    kf, vf, hq, hkv, d, ctx = CASES[name]
    base = wl.WORKLOADS["llama3_8b_int4_rot"]
    return wl.scaled(base, batch=len(ctx), contexts=ctx, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                     name="rot_" + name, k_fmt=kf, v_fmt=vf, rotate=rotate, outliers=outliers)


def _setup(w):
    table, nb = wl.block_tables(w, spare_blocks=2)
    fmt = kvq.cache_format(w.k_fmt, w.v_fmt, w.num_kv_heads, w.head_dim, nb, w.block_size,
                           rotation_signs=wl.rotation_words(w))
    cache = kvq.allocate_cache(fmt)
    oc = oracle.OracleCache(nb, w.block_size, w.num_kv_heads, w.head_dim, w.k_fmt, w.v_fmt,
                            rotation_signs=H.oracle_signs(w))
    for seqs, pos in H.all_positions(w):
        if len(seqs):
            k, v, slots = H.gpu_write(kvq, w, fmt, cache, table, seqs, pos)
            H.oracle_write(oc, k, v, slots)
    torch.cuda.synchronize()
    return fmt, cache, oc, table


def _decode(w, fmt, cache, table):
    ctx = wl.context_lens(w)
    q = wl.queries(w, device="cuda")
    out = kvq.kvq_paged_decode(q, fmt, cache, torch.as_tensor(table, device="cuda"),
                               torch.as_tensor(ctx, device="cuda"), int(ctx.max()))
    torch.cuda.synchronize()
    return q, ctx, out.cpu().numpy()


@pytest.mark.parametrize("name", list(CASES))
def test_rotated_write_bit_exact_and_decode(name):
    w = _workload(name)
    fmt, cache, oc, table = _setup(w)
    H.compare_cache(cache, oc)
    q, ctx, out = _decode(w, fmt, cache, table)
    assert kvq.kvq_device_errors() == 0
    ref = oracle.paged_decode_fp64(oc, H.bits(q), table, ctx)
    H.check_attention(out, ref, w.name)


def test_rotation_lowers_the_int4_reconstruction_error_of_k():
    # the K outlier channels (x20) set each per-(token, head) INT4 step; the
    # rotation spreads them over all channels, so the rows read back from the
    # device cache (dequantized, rotated back) are closer to the BF16 inputs
    errs = {}
    for rotate in (False, True):
        w = _workload("int4_int4g", rotate=rotate)
        fmt, cache, oc, table = _setup(w)
        back = oracle.OracleCache(oc.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.k_fmt, w.v_fmt,
                                  rotation_signs=oc.rotation)
        for x in ("k", "v"):
            back.codes[x] = cache[x + "_cache"].cpu().numpy()
            back.scales[x] = cache[x + "_scale"].cpu().numpy()
        n = int(wl.context_lens(w)[0])
        pos = np.arange(n)
        slots = wl.slot_mapping(table, np.zeros(n, np.int64), pos, w.block_size)
        k_hat = oracle.dequantize_cache_rows(back, "k", slots // w.block_size, slots % w.block_size)
        if rotate:
            k_hat = (k_hat @ oracle.hadamard(w.head_dim).T) * oc.rotation / w.head_dim
        # the rows the device wrote (the generator draws per device)
        k = wl.sequence_kv(w, "k", 0, "cuda", n).float().cpu().numpy().astype(np.float64)
        errs[rotate] = float(np.abs(k_hat - k).mean())
    assert errs[True] < 0.7 * errs[False], errs


def test_rotation_needs_per_token_k():
    w = wl.scaled(wl.WORKLOADS["llama3_70b_kivi"], batch=1, contexts=[20], name="rot_kivi", rotate=True)
    table, nb = wl.block_tables(w)
    fmt = kvq.cache_format(w.k_fmt, w.v_fmt, w.num_kv_heads, w.head_dim, nb, w.block_size,
                           rotation_signs=wl.rotation_words(w))
    cache = kvq.allocate_cache(fmt)
    k, v = wl.gather_tokens(w, np.zeros(4, np.int64), np.arange(4), device="cuda")
    slots = torch.as_tensor(wl.slot_mapping(table, np.zeros(4, np.int64), np.arange(4), 16), device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_quantize_write(k, v, slots, fmt, cache)
    assert e.value.status == kvq.KVQ_ERR_UNSUPPORTED
