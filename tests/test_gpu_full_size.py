"""Parity at the workloads' full sizes, in the launch configuration the bench
times (whole batch, one quantize-write call per prefill, one decode call).

The oracle cannot redo a whole 32k-65k-context batch, so it checks samples
it can compute one by one from the same BF16 inputs:
  * quantize-write: random tokens (per-token formats) or random whole blocks
    (per-channel K) are quantized by the oracle and compared byte for byte
    with the device cache;
  * decode: for sampled sequences the oracle quantizes the sequence's whole
    context itself and computes float64 attention for sampled query heads.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from tests import _helpers as H

pytestmark = pytest.mark.gpu

FULL = ["llama3_8b_fp8", "llama3_70b_kivi", "cb_mix_int8", "long_mixed", "llama3_8b_int4_rot", "llama3_70b_kivi2"]
STEPS_CHECKED = 3   # decode steps of the long-context workload run here


@pytest.fixture(scope="module")
def kvq():
    from quantized_paged_kv_write_gb300 import build
    build.build()
    import quantized_paged_kv_write_gb300 as m
    m.load_library()
    return m


class Built:
    """Full-size cache written through the C ABI, BF16 inputs kept."""

    def __init__(self, kvq, w):
        self.w = w
        self.ctx = wl.context_lens(w)
        self.table, self.nb = wl.block_tables(w)
        self.fmt = kvq.cache_format(w.k_fmt, w.v_fmt, w.num_kv_heads, w.head_dim, self.nb, w.block_size,
                                    rotation_signs=wl.rotation_words(w))
        self.cache = kvq.allocate_cache(self.fmt, "cuda")
        npos = wl.total_positions(w)
        self.k = [wl.sequence_kv(w, "k", b, "cuda", int(npos[b])) for b in range(w.batch)]
        self.v = [wl.sequence_kv(w, "v", b, "cuda", int(npos[b])) for b in range(w.batch)]
        self.calls = []
        for seqs, pos in H.all_positions(w):
            if len(seqs):
                self._write(kvq, seqs, pos)
        torch.cuda.synchronize()

    def _write(self, kvq, seqs, pos):
        kk = torch.cat([self.k[b][pos[seqs == b]] for b in np.unique(seqs)])
        vv = torch.cat([self.v[b][pos[seqs == b]] for b in np.unique(seqs)])
        order = np.concatenate([np.flatnonzero(seqs == b) for b in np.unique(seqs)])
        seqs, pos = seqs[order], pos[order]
        slots = torch.as_tensor(wl.slot_mapping(self.table, seqs, pos, self.w.block_size), device="cuda")
        kvq.kvq_quantize_write(kk, vv, slots, self.fmt, self.cache)
        self.calls.append((seqs, pos))

    def oracle_sequence(self, b, upto):
        """Oracle cache holding sequence b's positions [0, upto), written in
        the same calls the device saw."""
        oc = oracle.OracleCache(self.nb, self.w.block_size, self.w.num_kv_heads, self.w.head_dim,
                                self.w.k_fmt, self.w.v_fmt, rotation_signs=H.oracle_signs(self.w))
        kb = H.bits(self.k[b][:upto])
        vb = H.bits(self.v[b][:upto])
        for seqs, pos in self.calls:
            sel = (seqs == b) & (pos < upto)
            if not sel.any():
                continue
            p = pos[sel]
            slots = wl.slot_mapping(self.table, np.full(len(p), b), p, self.w.block_size)
            oracle.quantize_write(oc, kb[p], vb[p], slots)
        return oc


_built = {}


def built(kvq, name):
    if name not in _built:
        _built.clear()
        torch.cuda.empty_cache()
        _built[name] = Built(kvq, wl.WORKLOADS[name])
    return _built[name]


@pytest.mark.parametrize("name", FULL)
def test_full_size_quantize_write_samples(kvq, name):
    bl = built(kvq, name)
    w = bl.w
    rng = np.random.default_rng(100)
    assert kvq.kvq_device_errors() == 0
    seqs_all = np.concatenate([c[0] for c in bl.calls])
    pos_all = np.concatenate([c[1] for c in bl.calls])
    codes = {x: bl.cache[x + "_cache"] for x in ("k", "v")}
    scales = {x: bl.cache[x + "_scale"] for x in ("k", "v")}
    if w.k_fmt.gran == wl.PER_BLOCK_CHANNEL:
        # whole blocks: every row of the block and its channel scales
        picks = rng.choice(len(seqs_all) // w.block_size, size=64, replace=False) * w.block_size
        rows = np.concatenate([np.arange(p, p + w.block_size) for p in picks])
    else:
        rows = rng.choice(len(seqs_all), size=2048, replace=False)
    seqs, pos = seqs_all[rows], pos_all[rows]
    slots = wl.slot_mapping(bl.table, seqs, pos, w.block_size)
    kb = np.stack([H.bits(bl.k[s][p]) for s, p in zip(seqs, pos)])
    vb = np.stack([H.bits(bl.v[s][p]) for s, p in zip(seqs, pos)])
    oc = oracle.OracleCache(bl.nb, w.block_size, w.num_kv_heads, w.head_dim, w.k_fmt, w.v_fmt,
                            rotation_signs=H.oracle_signs(w))
    oracle.quantize_write(oc, kb, vb, slots)
    blk, off = slots // w.block_size, slots % w.block_size
    for x in ("k", "v"):
        got = codes[x][torch.as_tensor(blk, device="cuda"), torch.as_tensor(off, device="cuda")].cpu().numpy()
        assert np.array_equal(got, oc.codes[x][blk, off]), f"{x} codes differ"
        fmt = w.k_fmt if x == "k" else w.v_fmt
        if fmt.gran == wl.PER_BLOCK_CHANNEL:
            ub = np.unique(blk)
            got_s = scales[x][torch.as_tensor(ub, device="cuda")].cpu().numpy()
            assert np.array_equal(got_s.view(np.uint32), oc.scales[x][ub].view(np.uint32)), f"{x} scales differ"
        else:
            got_s = scales[x][torch.as_tensor(blk, device="cuda"), torch.as_tensor(off, device="cuda")]
            assert np.array_equal(got_s.cpu().numpy().view(np.uint32),
                                  oc.scales[x][blk, off].view(np.uint32)), f"{x} scales differ"


@pytest.mark.parametrize("name", FULL)
def test_full_size_decode_samples(kvq, name):
    bl = built(kvq, name)
    w = bl.w
    rng = np.random.default_rng(200)
    ctx = bl.ctx.copy()
    bt = torch.as_tensor(bl.table, device="cuda")
    steps = STEPS_CHECKED if w.decode_steps else 0
    for s in range(steps + 1):
        if s > 0:
            # the serving step: write position ctx of every sequence, attend ctx + 1
            seqs = np.arange(w.batch)
            pos = ctx.astype(np.int64)
            bl._write(kvq, seqs, pos)
            ctx = ctx + 1
        q = wl.queries(w, step=s, device="cuda")
        cl = torch.as_tensor(ctx, device="cuda")
        out = kvq.kvq_paged_decode(q, bl.fmt, bl.cache, bt, cl, int(ctx.max())).cpu().numpy()
        assert kvq.kvq_device_errors() == 0
    qb = H.bits(q)
    for b in rng.choice(w.batch, size=2, replace=False):
        oc = bl.oracle_sequence(int(b), int(ctx[b]))
        for h in rng.choice(w.num_q_heads, size=4, replace=False):
            ref = oracle.paged_decode_one_fp64(oc, qb[b, h], bl.table[b], int(ctx[b]), int(h), w.num_q_heads)
            H.check_attention(out[b, h], ref, f"{name} seq {b} head {h}")
