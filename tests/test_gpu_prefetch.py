"""kvq_prefetch_blocks (offloaded blocks from pinned host memory into device
block slots) through the C ABI: byte-exact copies against the oracle's block
copy, skipped out-of-range pairs, rejection of unpinned host memory, and the
double-buffered pattern of "Use Less Memory", §4 (prefetch into a second set
of buffers on another stream while a decode runs) giving the same attention
as the resident cache."""
import ctypes

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


FORMATS = {
    "fp8_fp8": (wl.CacheFormat(wl.FP8, wl.PER_TOKEN_HEAD), wl.CacheFormat(wl.FP8, wl.PER_TOKEN_HEAD), 8, 128),
    "kivi": (wl.CacheFormat(wl.INT8, wl.PER_BLOCK_CHANNEL), wl.CacheFormat(wl.INT4, wl.PER_TOKEN_GROUP, 32), 8, 128),
    "int4_int8_d64": (wl.CacheFormat(wl.INT4, wl.PER_TOKEN_HEAD), wl.CacheFormat(wl.INT8, wl.PER_TOKEN_HEAD), 2, 64),
}


def _fill_random(t: dict, seed: int):
    g = torch.Generator().manual_seed(seed)
    for key, x in t.items():
        if x.dtype == torch.uint8:
            x.copy_(torch.randint(0, 256, x.shape, generator=g, dtype=torch.uint8))
        else:
            x.copy_(torch.randn(x.shape, generator=g))


def _np(t: dict) -> dict:
    return {k: v.cpu().numpy().copy() for k, v in t.items()}


@pytest.mark.parametrize("name", list(FORMATS))
def test_prefetch_copies_blocks_byte_for_byte(name):
    kf, vf, hkv, d = FORMATS[name]
    fmt = kvq.cache_format(kf, vf, hkv, d, 40)
    host = kvq.allocate_host_pool(fmt, 57)
    _fill_random(host, 1)
    dev = kvq.allocate_cache(fmt)
    for key, x in dev.items():   # a known non-zero start, to see untouched slots
        x.copy_(torch.full(x.shape, 3, dtype=x.dtype, device=x.device))
    rng = np.random.default_rng(3)
    src = rng.choice(57, size=25, replace=False).astype(np.int32)
    dst = rng.choice(40, size=25, replace=False).astype(np.int32)
    want = _np(dev)
    oracle.prefetch_blocks(_np(host), want, src, dst)
    kvq.kvq_prefetch_blocks(host, torch.as_tensor(src, device="cuda"), torch.as_tensor(dst, device="cuda"), fmt, dev)
    torch.cuda.synchronize()
    assert kvq.kvq_device_errors() == 0
    got = _np(dev)
    for key in got:
        assert np.array_equal(got[key].view(np.uint8), want[key].view(np.uint8)), key


def test_out_of_range_pairs_set_the_error_bit_and_are_skipped():
    kf, vf, hkv, d = FORMATS["fp8_fp8"]
    fmt = kvq.cache_format(kf, vf, hkv, d, 6)
    host = kvq.allocate_host_pool(fmt, 5)
    _fill_random(host, 4)
    dev = kvq.allocate_cache(fmt)
    src = np.array([0, 5, -1, 2, 4], np.int32)   # 5 and -1: outside the host pool
    dst = np.array([1, 2, 3, 6, 0], np.int32)    # 6: outside the device cache
    want = _np(dev)
    assert oracle.prefetch_blocks(_np(host), want, src, dst) == 3
    kvq.kvq_prefetch_blocks(host, torch.as_tensor(src, device="cuda"), torch.as_tensor(dst, device="cuda"), fmt, dev)
    bits = kvq.kvq_device_errors()
    assert bits == kvq.DEVERR_BLOCK_RANGE
    got = _np(dev)
    for key in got:
        assert np.array_equal(got[key].view(np.uint8), want[key].view(np.uint8)), key


def test_unpinned_host_memory_is_rejected():
    kf, vf, hkv, d = FORMATS["fp8_fp8"]
    fmt = kvq.cache_format(kf, vf, hkv, d, 4)
    plain = {k: torch.zeros_like(v) for k, v in kvq.allocate_host_pool(fmt, 4).items()}  # pageable copies
    dev = kvq.allocate_cache(fmt)
    lib = kvq.load_library()
    idx = torch.zeros(1, dtype=torch.int32, device="cuda")
    hc = kvq._Caches(plain["k_cache"].data_ptr(), plain["v_cache"].data_ptr())
    hs = kvq._Scales(plain["k_scale"].data_ptr(), plain["v_scale"].data_ptr())
    caches, scales = kvq._caches(dev)
    cf = fmt.as_c()
    st = lib.kvq_prefetch_blocks(ctypes.byref(cf), hc, hs, 4, idx.data_ptr(), idx.data_ptr(), 1, caches, scales,
                                 torch.cuda.current_stream().cuda_stream)
    assert st == kvq.KVQ_ERR_INVALID_ARG
    with pytest.raises(ValueError):
        kvq.kvq_prefetch_blocks(plain, idx, idx, fmt, dev)


def test_double_buffered_prefetch_gives_the_resident_attention():
    # resident cache A (written through the quantize-write), offloaded to a
    # pinned host pool, prefetched on a side stream into buffer B under a
    # permuted block layout while a decode over A runs; decoding B through the
    # permuted block table gives exactly A's output
    w = wl.scaled(wl.WORKLOADS["long_mixed"], batch=3, contexts=[300, 45, 129], decode_steps=0, name="pf")
    table, nb = wl.block_tables(w)
    fmt = kvq.cache_format(w.k_fmt, w.v_fmt, w.num_kv_heads, w.head_dim, nb, w.block_size)
    cache_a = kvq.allocate_cache(fmt)
    for seqs, pos in H.all_positions(w):
        if len(seqs):
            H.gpu_write(kvq, w, fmt, cache_a, table, seqs, pos)
    host = kvq.allocate_host_pool(fmt, nb)
    for key in host:
        host[key].copy_(cache_a[key].cpu())
    perm = np.random.default_rng(5).permutation(nb).astype(np.int32)   # block b -> slot perm[b]
    table_b = np.where(table >= 0, perm[np.maximum(table, 0)], -1).astype(np.int32)
    cache_b = kvq.allocate_cache(fmt)
    q = wl.queries(w, device="cuda")
    ctx = wl.context_lens(w)
    cl = torch.as_tensor(ctx, device="cuda")
    side = torch.cuda.Stream()
    src = torch.as_tensor(np.arange(nb, dtype=np.int32), device="cuda")
    dst = torch.as_tensor(perm, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(side):
        kvq.kvq_prefetch_blocks(host, src, dst, fmt, cache_b, stream=side)
    out_a = kvq.kvq_paged_decode(q, fmt, cache_a, torch.as_tensor(table, device="cuda"), cl, int(ctx.max()))
    torch.cuda.current_stream().wait_stream(side)
    out_b = kvq.kvq_paged_decode(q, fmt, cache_b, torch.as_tensor(table_b, device="cuda"), cl, int(ctx.max()))
    torch.cuda.synchronize()
    assert kvq.kvq_device_errors() == 0
    assert torch.equal(out_a, out_b)
