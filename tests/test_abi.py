"""The C-ABI library builds for sm_103a, loads, and exports every function
include/kvq.h declares; host-side argument checks that need no GPU."""
import ctypes
import os
import re

import pytest

import quantized_paged_kv_write_gb300 as kvq
from quantized_paged_kv_write_gb300 import build as kbuild

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "kvq.h")


@pytest.fixture(scope="module")
def lib():
    kbuild.build()
    return kvq.load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(kvq.EXPORTED_SYMBOLS)
    for n in names:
        assert hasattr(lib, n), n


def test_build_id_matches_the_sources(lib):
    # the library that loaded was built from the sources in this tree
    assert kvq.kvq_build_id() == kbuild.source_hash()


def test_version_and_status_strings(lib):
    assert kvq.kvq_version() == 110
    assert kvq.kvq_status_string(0) == "ok"
    assert kvq.kvq_status_string(kvq.KVQ_ERR_WORKSPACE) == "workspace too small"
    assert kvq.kvq_status_string(-99) == "unknown status"


def _fmt(**kw):
    base = dict(k_dtype=0, v_dtype=0, k_gran=0, v_gran=0, k_group=0, v_group=0, num_kv_heads=8,
                head_dim=128, block_size=16, rotation=0, num_blocks=10)
    base.update(kw)
    return kvq._Format(**base)


def test_quantize_write_host_checks(lib):
    cz, sz = kvq._Caches(None, None), kvq._Scales(None, None)
    f = _fmt()
    # zero tokens: a no-op that touches nothing
    assert lib.kvq_quantize_write(None, None, None, 0, ctypes.byref(f), cz, sz, None) == kvq.KVQ_OK
    assert lib.kvq_quantize_write(None, None, None, 5, ctypes.byref(f), cz, sz, None) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_quantize_write(None, None, None, -1, ctypes.byref(f), cz, sz, None) == kvq.KVQ_ERR_INVALID_ARG
    for bad in (dict(block_size=32), dict(head_dim=96), dict(k_dtype=1, k_gran=1, k_group=32),
                dict(k_dtype=1, k_gran=2), dict(v_dtype=1, v_gran=1, v_group=64), dict(v_gran=2),
                dict(k_dtype=3, k_gran=2, head_dim=64), dict(v_dtype=3, v_gran=1, v_group=32, head_dim=64),
                dict(k_dtype=3), dict(v_dtype=3, v_gran=1, v_group=16),
                dict(num_kv_heads=16)):
        g = _fmt(**bad)
        assert lib.kvq_quantize_write(None, None, None, 0, ctypes.byref(g), cz, sz, None) == \
            kvq.KVQ_ERR_UNSUPPORTED, bad
    g = _fmt(rotation=2)  # no such rotation
    assert lib.kvq_quantize_write(None, None, None, 0, ctypes.byref(g), cz, sz, None) == kvq.KVQ_ERR_INVALID_ARG
    g = _fmt(rotation=1, k_gran=2)  # the rotation needs per-token K
    assert lib.kvq_quantize_write(None, None, None, 0, ctypes.byref(g), cz, sz, None) == kvq.KVQ_ERR_UNSUPPORTED
    g = _fmt(rotation=1, k_dtype=1, v_dtype=1, v_gran=1, v_group=32)
    assert lib.kvq_quantize_write(None, None, None, 0, ctypes.byref(g), cz, sz, None) == kvq.KVQ_OK


def test_write_decode_host_checks(lib):
    cz, sz = kvq._Caches(None, None), kvq._Scales(None, None)
    f = _fmt()
    chan = _fmt(k_gran=2)
    args = lambda fm, kn, vn, bsz: (None, kn, vn, bsz, 32, ctypes.byref(fm), cz, sz, None, 1, None, 0, None,
                                    None, 0, None)
    dummy = ctypes.c_void_p(256)  # never dereferenced: every call below returns before any device work
    assert lib.kvq_write_decode(*args(f, dummy, dummy, 0)) == kvq.KVQ_OK                 # empty batch
    assert lib.kvq_write_decode(*args(f, None, None, 2)) == kvq.KVQ_ERR_INVALID_ARG      # no new K / V
    assert lib.kvq_write_decode(*args(f, dummy, dummy, 2)) == kvq.KVQ_ERR_INVALID_ARG    # null q, caches
    assert lib.kvq_write_decode(*args(chan, dummy, dummy, 2)) == kvq.KVQ_ERR_UNSUPPORTED  # per-channel K


def test_prefetch_host_checks(lib):
    cz, sz = kvq._Caches(None, None), kvq._Scales(None, None)
    f = _fmt()
    assert lib.kvq_prefetch_blocks(ctypes.byref(f), cz, sz, 0, None, None, 0, cz, sz, None) == kvq.KVQ_OK
    assert lib.kvq_prefetch_blocks(ctypes.byref(f), cz, sz, 4, None, None, 2, cz, sz, None) == \
        kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_prefetch_blocks(ctypes.byref(f), cz, sz, 4, None, None, -1, cz, sz, None) == \
        kvq.KVQ_ERR_INVALID_ARG
    g = _fmt(head_dim=96)
    assert lib.kvq_prefetch_blocks(ctypes.byref(g), cz, sz, 0, None, None, 0, cz, sz, None) == \
        kvq.KVQ_ERR_UNSUPPORTED


def test_kivi_host_checks(lib):
    cz, sz = kvq._Caches(None, None), kvq._Scales(None, None)
    tok = _fmt()                        # per-token K: no full-precision tail
    chan = _fmt(k_gran=2)
    assert lib.kvq_kivi_append(None, None, 0, ctypes.byref(tok), cz, sz, None, 1, None, None, None, None) == \
        kvq.KVQ_ERR_UNSUPPORTED
    assert lib.kvq_kivi_append(None, None, 0, ctypes.byref(chan), cz, sz, None, 1, None, None, None, None) == \
        kvq.KVQ_OK
    assert lib.kvq_kivi_append(None, None, 2, ctypes.byref(chan), cz, sz, None, 1, None, None, None, None) == \
        kvq.KVQ_ERR_INVALID_ARG
    dec = lambda fm, r: (None, 2, 32, ctypes.byref(fm), cz, sz, None, 1, None, 0, r, r, None, None, 0, None)
    assert lib.kvq_kivi_decode(*dec(chan, None)) == kvq.KVQ_ERR_INVALID_ARG
    assert lib.kvq_kivi_decode(*dec(tok, ctypes.c_void_p(256))) == kvq.KVQ_ERR_UNSUPPORTED


def test_decode_host_checks(lib):
    cz, sz = kvq._Caches(None, None), kvq._Scales(None, None)
    f = _fmt()
    args = lambda bsz, hq: (None, bsz, hq, ctypes.byref(f), cz, sz, None, 1, None, 0, None, None, 0, None)
    assert lib.kvq_paged_decode(*args(0, 32)) == kvq.KVQ_OK                       # empty batch
    assert lib.kvq_paged_decode(*args(2, 32)) == kvq.KVQ_ERR_INVALID_ARG          # null pointers
    assert lib.kvq_paged_decode(*args(2, 12)) == kvq.KVQ_ERR_INVALID_ARG          # 12 % 8 != 0
    assert lib.kvq_paged_decode(*args(2, 128)) == kvq.KVQ_ERR_UNSUPPORTED         # G = 16
    assert lib.kvq_paged_decode(*args(-1, 32)) == kvq.KVQ_ERR_INVALID_ARG
