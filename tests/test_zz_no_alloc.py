"""kvq_paged_decode_noalloc -- the decode entry point for callers that cannot
allocate device memory at the call (engine or plugin hosts that own all
device memory, serving loops that must not enter the allocator).  It keeps
its split-K scratch in one static device array instead of a caller-provided
workspace.

The test calls it through the C ABI (ctypes on libkvq.so) twice in a row and
checks each result against kvq_paged_decode with a workspace.  Both calls run
the same kernels with the same split count on the same inputs, so the outputs
must be identical bit for bit: a tolerance could hide a stale or partly
overwritten read of the shared scratch.  The second call of each case runs on
the scratch the first one left behind.  It also checks that a shape whose
scratch would not fit the static array is refused before any work.  The file
is named to be collected last."""
import ctypes

import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kvq():
    from quantized_paged_kv_write_gb300 import build
    build.build()
    import quantized_paged_kv_write_gb300 as m
    m.load_library()
    return m


def _setup(kvq, name, **small):
    w = wl.scaled(wl.WORKLOADS[name], name=name + "_noalloc", decode_steps=0, **small)
    table, nb = wl.block_tables(w, spare_blocks=2)
    fmt = kvq.cache_format(w.k_fmt, w.v_fmt, w.num_kv_heads, w.head_dim, nb, w.block_size)
    cache = kvq.allocate_cache(fmt)
    seqs, pos = wl.write_positions(w)
    k, v = wl.gather_tokens(w, seqs, pos, device="cuda")
    slots = torch.as_tensor(wl.slot_mapping(table, seqs, pos, w.block_size), device="cuda")
    kvq.kvq_quantize_write(k, v, slots, fmt, cache)
    return w, fmt, cache, torch.as_tensor(table, device="cuda"), torch.as_tensor(wl.context_lens(w), device="cuda")


def _call_c_abi(kvq, q, fmt, cache, bt, cl, max_ctx, out):
    lib = kvq.load_library()
    cf = fmt.as_c()
    caches = kvq._Caches(cache["k_cache"].data_ptr(), cache["v_cache"].data_ptr())
    scales = kvq._Scales(cache["k_scale"].data_ptr(), cache["v_scale"].data_ptr())
    stream = torch.cuda.current_stream().cuda_stream
    return lib.kvq_paged_decode_noalloc(q.data_ptr(), q.shape[0], q.shape[1], ctypes.byref(cf), caches, scales,
                                        bt.data_ptr(), bt.shape[1], cl.data_ptr(), int(max_ctx),
                                        out.data_ptr(), stream)


@pytest.mark.parametrize("name,small", [
    ("llama3_8b_fp8", dict(batch=5, contexts=[300, 37, 16, 1, 999])),
    ("long_mixed", dict(batch=3, contexts=[129, 31, 200])),
    ("llama3_70b_kivi", dict(batch=2, contexts=[257, 40])),
])
def test_noalloc_matches_workspace_decode_twice(kvq, name, small):
    w, fmt, cache, bt, cl = _setup(kvq, name, **small)
    max_ctx = int(cl.max())
    for step in range(2):
        q = wl.queries(w, step=step, device="cuda")
        ref = kvq.kvq_paged_decode(q, fmt, cache, bt, cl, max_ctx)
        out = torch.full_like(ref, float("nan"))
        st = _call_c_abi(kvq, q, fmt, cache, bt, cl, max_ctx, out)
        assert st == kvq.KVQ_OK, kvq.kvq_status_string(st)
        torch.cuda.synchronize()
        # bit patterns, so that NaN in both would not pass unnoticed either
        assert torch.equal(out.view(torch.int32), ref.view(torch.int32)), (name, step)
        assert torch.isfinite(out).all(), (name, step)
    assert kvq.kvq_device_errors() == 0


def test_noalloc_rejects_shapes_beyond_the_static_scratch(kvq):
    w, fmt, cache, _, _ = _setup(kvq, "tiny_int8", batch=1, contexts=[20])
    big = 8192                                   # workspace far above 32 MiB
    need = kvq.kvq_decode_workspace_size(fmt, big, w.num_q_heads, 16)
    assert need > kvq.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((big, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((big, 1), dtype=torch.int32, device="cuda")
    cl = torch.zeros(big, dtype=torch.int32, device="cuda")
    out = torch.zeros((big, w.num_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    assert _call_c_abi(kvq, q, fmt, cache, bt, cl, 16, out) == kvq.KVQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
