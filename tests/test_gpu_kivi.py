"""Per-channel K caches that take appends (kvq_kivi_append / kvq_kivi_decode)
through the C ABI against the oracle (oracle/kivi.py).

Sequences are prefilled (complete blocks through kvq_quantize_write, the
incomplete block's rows copied into the residual), then take one token per
step.  After every step the cache codes, scales and residual rows must equal
the oracle's byte for byte, and the decode over the quantized blocks plus the
full-precision tail must be within the stated tolerance (max abs error <= 2e-3 everywhere, max rel
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


KCHAN = wl.CacheFormat(wl.INT8, wl.PER_BLOCK_CHANNEL)
KCHAN2 = wl.CacheFormat(wl.INT2, wl.PER_BLOCK_CHANNEL)
CASES = {
    # name: (K format, V format, q heads, kv heads, head dim, contexts)
    "int4g_v": (KCHAN, wl.CacheFormat(wl.INT4, wl.PER_TOKEN_GROUP, 32), 64, 8, 128, [33, 16, 5, 70]),
    "int8_v_d64": (KCHAN, wl.CacheFormat(wl.INT8, wl.PER_TOKEN_HEAD), 8, 2, 64, [47, 1, 15]),
    "int2_kv": (KCHAN2, wl.CacheFormat(wl.INT2, wl.PER_TOKEN_GROUP, 32), 32, 8, 128, [40, 16, 9]),
}
STEPS = 20


@pytest.mark.parametrize("name", list(CASES))
def test_appends_and_decode_match_the_oracle(name):
    kf, vf, hq, hkv, d, ctx0 = CASES[name]
    w = wl.scaled(wl.WORKLOADS["llama3_70b_kivi"], batch=len(ctx0), contexts=ctx0, num_q_heads=hq,
                  num_kv_heads=hkv, head_dim=d, k_fmt=kf, v_fmt=vf, decode_steps=STEPS, name="kivi_" + name)
    table, nb = wl.block_tables(w, spare_blocks=1)
    fmt = kvq.cache_format(w.k_fmt, w.v_fmt, hkv, d, nb, w.block_size)
    cache = kvq.allocate_cache(fmt)
    res = kvq.allocate_residual(fmt, w.batch)
    oc = oracle.OracleCache(nb, w.block_size, hkv, d, w.k_fmt, w.v_fmt)
    res_k = np.zeros((w.batch, 16, hkv, d), np.uint16)
    res_v = np.zeros((w.batch, 16, hkv, d), np.uint16)
    ctx0 = np.array(ctx0)
    # prefill: complete blocks through the quantize-write, the rest into the residual
    full = (ctx0 // 16) * 16
    seqs = np.concatenate([np.full(f, b, np.int64) for b, f in enumerate(full)])
    pos = np.concatenate([np.arange(f, dtype=np.int64) for f in full])
    if len(seqs):
        k, v, slots = H.gpu_write(kvq, w, fmt, cache, table, seqs, pos)
        H.oracle_write(oc, k, v, slots)
    for b, n in enumerate(ctx0):
        p = np.arange(full[b], n)
        if len(p):
            kt, vt = wl.gather_tokens(w, np.full(len(p), b), p, device="cuda")
            res["k"][b, p % 16] = kt
            res["v"][b, p % 16] = vt
            res_k[b, p % 16] = H.bits(kt)
            res_v[b, p % 16] = H.bits(vt)
    bt = torch.as_tensor(table, device="cuda")
    for s in range(STEPS):
        n = ctx0 + s + 1                         # lengths after this step's token
        kn, vn = wl.gather_tokens(w, np.arange(w.batch), n - 1, device="cuda")
        cl = torch.as_tensor(n.astype(np.int32), device="cuda")
        kvq.kvq_kivi_append(kn, vn, fmt, cache, bt, cl, res)
        q = wl.queries(w, step=s, device="cuda")
        out = kvq.kvq_kivi_decode(q, fmt, cache, bt, cl, int(n.max()), res)
        torch.cuda.synchronize()
        assert kvq.kvq_device_errors() == 0
        oracle.kivi_append(oc, res_k, res_v, H.bits(kn), H.bits(vn), table, n)
        H.compare_cache(cache, oc)
        assert np.array_equal(H.bits(res["k"]), res_k) and np.array_equal(H.bits(res["v"]), res_v)
        ref = oracle.kivi_decode_fp64(oc, res_k, res_v, H.bits(q), table, n)
        H.check_attention(out.cpu().numpy(), ref, f"{name} step {s}")


def test_per_token_k_is_rejected():
    f = wl.CacheFormat(wl.INT8, wl.PER_TOKEN_HEAD)
    fmt = kvq.cache_format(f, f, 2, 64, 4)
    cache = kvq.allocate_cache(fmt)
    res = kvq.allocate_residual(fmt, 1)
    bt = torch.zeros((1, 4), dtype=torch.int32, device="cuda")
    cl = torch.ones(1, dtype=torch.int32, device="cuda")
    kn = torch.zeros((1, 2, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_kivi_append(kn, kn, fmt, cache, bt, cl, res)
    assert e.value.status == kvq.KVQ_ERR_UNSUPPORTED
    q = torch.zeros((1, 4, 64), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_kivi_decode(q, fmt, cache, bt, cl, 1, res)
    assert e.value.status == kvq.KVQ_ERR_UNSUPPORTED


def test_tail_needs_no_block_table_entry():
    # a context of 16 m + r with a block table of exactly m entries: the tail
    # lives in the residual only
    kf, vf = KCHAN, wl.CacheFormat(wl.INT8, wl.PER_TOKEN_HEAD)
    w = wl.scaled(wl.WORKLOADS["llama3_70b_kivi"], batch=2, contexts=[32, 48], num_q_heads=8, num_kv_heads=2,
                  head_dim=64, v_fmt=vf, name="kivi_edge")
    table, nb = wl.block_tables(w)          # 2 and 3 blocks: no room past the contexts
    fmt = kvq.cache_format(kf, vf, 2, 64, nb, w.block_size)
    cache = kvq.allocate_cache(fmt)
    res = kvq.allocate_residual(fmt, 2)
    oc = oracle.OracleCache(nb, 16, 2, 64, kf, vf)
    res_k = np.zeros((2, 16, 2, 64), np.uint16)
    res_v = np.zeros((2, 16, 2, 64), np.uint16)
    seqs, pos = H.all_positions(w)[1]
    k, v, slots = H.gpu_write(kvq, w, fmt, cache, table, seqs, pos)
    H.oracle_write(oc, k, v, slots)
    bt = torch.as_tensor(table, device="cuda")
    n = np.array([33, 49])
    kn, vn = wl.gather_tokens(w, np.arange(2), n - 1, device="cuda")
    cl = torch.as_tensor(n.astype(np.int32), device="cuda")
    kvq.kvq_kivi_append(kn, vn, fmt, cache, bt, cl, res)
    q = wl.queries(w, device="cuda")
    out = kvq.kvq_kivi_decode(q, fmt, cache, bt, cl, 49, res)
    torch.cuda.synchronize()
    assert kvq.kvq_device_errors() == 0
    oracle.kivi_append(oc, res_k, res_v, H.bits(kn), H.bits(vn), np.pad(table, ((0, 0), (0, 1)), constant_values=-1), n)
    ref = oracle.kivi_decode_fp64(oc, res_k, res_v, H.bits(q), table, n)
    H.check_attention(out.cpu().numpy(), ref, "kivi edge")
