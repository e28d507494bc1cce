"""Seeded synthetic inputs for the quantized paged KV-cache path.

This module only *generates inputs*: layer shapes, cache formats (by name),
context lengths, block tables, slot mappings and seeded BF16 K/V/Q values with
the outlier pattern of the workloads.  It holds none of the quantization or
attention arithmetic.  Both the CUDA path (through the binding) and the CPU
oracle consume what it returns; neither side is imported here.

Value recipe (all workloads): values are drawn FP32 ~ N(0, 1) from a seeded
generator, the outlier factors are applied in FP32, and the result is rounded
to BF16 with round-to-nearest-even (``torch.Tensor.to(torch.bfloat16)``).
Each sequence's K, V and Q come from their own generator stream, keyed by
(workload seed, tensor, sequence, [decode step]), so any sequence can be
regenerated on its own.  The stream is torch's generator for the device the
values are made on: CPU and CUDA streams differ, each is deterministic.

Integer structure (context lengths, block-table permutation) comes from numpy
PCG64 and is identical on every machine.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

# Names of cache element formats and scale granularities.  The binding and the
# oracle each map these names to their own representation.
INT8 = "int8"
INT4 = "int4"
INT2 = "int2"
FP8 = "fp8_e4m3fn"
PER_TOKEN_HEAD = "token_head"       # one FP32 scale per (token, kv_head)
PER_TOKEN_GROUP = "token_group"     # one FP32 scale per (token, kv_head, channel group)
PER_BLOCK_CHANNEL = "block_channel"  # one FP32 scale per (block, kv_head, channel)

# Outlier pattern of the long-context workloads: four K channels are scaled
# x20 on every kv head, and the first four positions of every sequence
# ("sink" tokens) are scaled x10 in both K and V.
OUTLIER_K_CHANNELS = (3, 17, 64, 100)
OUTLIER_K_FACTOR = 20.0
SINK_TOKENS = 4
SINK_FACTOR = 10.0

_TENSOR_IDS = {"k": 1, "v": 2, "q": 3}


@dataclasses.dataclass(frozen=True)
class CacheFormat:
    """Element format and scale granularity of one cache tensor (K or V)."""
    dtype: str
    gran: str
    group: int = 0  # channels per scale group for PER_TOKEN_GROUP

    def code_bytes_per_row(self, head_dim: int) -> int:
        return {INT4: head_dim // 2, INT2: head_dim // 4}.get(self.dtype, head_dim)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    k_fmt: CacheFormat
    v_fmt: CacheFormat
    contexts: tuple            # ("fixed", (c0, c1, ...)) or ("uniform", lo, hi)
    outliers: bool
    seed: int
    # Positions written by the quantize-write under test, per sequence, given
    # relative to the sequence's final decode context: "all" or ("last", n).
    write: object = "all"
    decode_steps: int = 0      # >0: steps each append one token per sequence
    rotate: bool = False       # randomized Walsh-Hadamard rotation of K and V rows
    description: str = ""

    @property
    def group_size(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _fmt(dtype, gran=PER_TOKEN_HEAD, group=0):
    return CacheFormat(dtype, gran, group)


# The five workloads.  Shapes are those of a Llama-3-8B / Llama-3-70B layer
# (32/64 query heads, 8 kv heads, head_dim 128) with a 16-token block.
WORKLOADS = {
    "tiny_int8": Workload(
        name="tiny_int8", batch=2, num_q_heads=4, num_kv_heads=2, head_dim=64,
        block_size=16, k_fmt=_fmt(INT8), v_fmt=_fmt(INT8),
        contexts=("fixed", (37, 100)), outliers=False, seed=0,
        description="tiny INT8 check: batch 2, contexts {37, 100}, GQA 2, d 64"),
    "llama3_8b_fp8": Workload(
        name="llama3_8b_fp8", batch=27, num_q_heads=32, num_kv_heads=8,
        head_dim=128, block_size=16, k_fmt=_fmt(FP8), v_fmt=_fmt(FP8),
        contexts=("fixed", (32768,) * 27), outliers=True, seed=2,
        description="Llama-3-8B layer, FP8 E4M3FN per-(token, kv_head), "
                    "batch 27 x context 32768"),
    "llama3_70b_kivi": Workload(
        name="llama3_70b_kivi", batch=8, num_q_heads=64, num_kv_heads=8,
        head_dim=128, block_size=16,
        k_fmt=_fmt(INT8, PER_BLOCK_CHANNEL), v_fmt=_fmt(INT4, PER_TOKEN_GROUP, 32),
        contexts=("fixed", (65536,) * 8), outliers=True, seed=3,
        description="Llama-3-70B layer, K INT8 per-(block, kv_head, channel), "
                    "V INT4 group 32, batch 8 x context 65536"),
    "cb_mix_int8": Workload(
        name="cb_mix_int8", batch=256, num_q_heads=32, num_kv_heads=8,
        head_dim=128, block_size=16, k_fmt=_fmt(INT8), v_fmt=_fmt(INT8),
        contexts=("uniform", 512, 16384), outliers=False, seed=4,
        write=("last", 32),
        description="continuous-batching mix, INT8 per-(token, kv_head), "
                    "batch 256, contexts U[512, 16384], 8192-token chunk write"),
    "long_mixed": Workload(
        name="long_mixed", batch=64, num_q_heads=32, num_kv_heads=8,
        head_dim=128, block_size=16, k_fmt=_fmt(FP8), v_fmt=_fmt(INT4, PER_TOKEN_GROUP, 32),
        contexts=("fixed", (32768,) * 64), outliers=True, seed=5, decode_steps=100,
        description="mixed precision long context: K FP8 per-(token, kv_head), "
                    "V INT4 group 32, batch 64, context 32768 + 100 steps"),
    "llama3_70b_kivi2": Workload(
        name="llama3_70b_kivi2", batch=8, num_q_heads=64, num_kv_heads=8,
        head_dim=128, block_size=16,
        k_fmt=_fmt(INT2, PER_BLOCK_CHANNEL), v_fmt=_fmt(INT2, PER_TOKEN_GROUP, 32),
        contexts=("fixed", (65536,) * 8), outliers=True, seed=7,
        description="Llama-3-70B layer, KIVI 2-bit: K INT2 per-(block, kv_head, channel), "
                    "V INT2 group 32, batch 8 x context 65536"),
    "llama3_8b_int4_rot": Workload(
        name="llama3_8b_int4_rot", batch=27, num_q_heads=32, num_kv_heads=8,
        head_dim=128, block_size=16, k_fmt=_fmt(INT4), v_fmt=_fmt(INT4, PER_TOKEN_GROUP, 32),
        contexts=("fixed", (32768,) * 27), outliers=True, seed=6, rotate=True,
        description="Llama-3-8B layer, Walsh-Hadamard-rotated INT4: K per-(token, kv_head), "
                    "V group 32, batch 27 x context 32768"),
}


def scaled(w: Workload, batch: Optional[int] = None, contexts=None,
           name: Optional[str] = None, **changes) -> Workload:
    """A copy of workload ``w`` with a different batch and/or contexts (used
    for oracle-sized parity cases with the same formats and head shapes)."""
    kw = {}
    if batch is not None:
        kw["batch"] = batch
    if contexts is not None:
        kw["contexts"] = ("fixed", tuple(int(c) for c in contexts))
    kw.update(changes)
    return dataclasses.replace(w, name=name or (w.name + "_small"), **kw)


# ---------------------------------------------------------------------------
# integer structure
# ---------------------------------------------------------------------------

def _rng(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *key])))


def context_lens(w: Workload) -> np.ndarray:
    """Final decode context of each sequence (int32[batch])."""
    kind = w.contexts[0]
    if kind == "fixed":
        ctx = np.asarray(w.contexts[1], dtype=np.int64)
        assert ctx.shape == (w.batch,), (w.name, ctx.shape)
    elif kind == "uniform":
        lo, hi = w.contexts[1], w.contexts[2]
        ctx = _rng(w.seed, 11).integers(lo, hi + 1, size=w.batch)
    else:
        raise ValueError(kind)
    return ctx.astype(np.int32)


def total_positions(w: Workload) -> np.ndarray:
    """Positions each sequence holds by the end of all decode steps."""
    return context_lens(w).astype(np.int64) + w.decode_steps


def block_tables(w: Workload, spare_blocks: int = 0):
    """Seeded random permutation of all physical blocks, dealt to sequences in
    order.  Returns (int32[batch, max_blocks_per_seq], num_blocks); unused
    table entries are -1."""
    pos = total_positions(w)
    nblk = (pos + w.block_size - 1) // w.block_size
    num_blocks = int(nblk.sum()) + spare_blocks
    perm = _rng(w.seed, 12).permutation(num_blocks).astype(np.int32)
    max_blocks = int(nblk.max()) if w.batch else 0
    table = np.full((w.batch, max(max_blocks, 1)), -1, dtype=np.int32)
    off = 0
    for b in range(w.batch):
        table[b, : nblk[b]] = perm[off: off + nblk[b]]
        off += nblk[b]
    return table, num_blocks


def slot_mapping(table: np.ndarray, seq_ids: np.ndarray, positions: np.ndarray,
                 block_size: int) -> np.ndarray:
    """slot = physical_block * block_size + offset for each (seq, position)."""
    seq_ids = np.asarray(seq_ids, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    blk = table[seq_ids, positions // block_size].astype(np.int64)
    return blk * block_size + positions % block_size


def write_positions(w: Workload):
    """(seq_ids, positions) of the tokens written by the quantize-write under
    test (before any decode step), in sequence-major order."""
    ctx = context_lens(w).astype(np.int64)
    seqs, poss = [], []
    for b in range(w.batch):
        if w.write == "all":
            p = np.arange(ctx[b])
        else:
            n = min(int(w.write[1]), int(ctx[b]))
            p = np.arange(ctx[b] - n, ctx[b])
        seqs.append(np.full(p.shape, b, dtype=np.int64))
        poss.append(p)
    if not seqs:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    return np.concatenate(seqs), np.concatenate(poss)


def prewritten_positions(w: Workload):
    """(seq_ids, positions) that a chunked-prefill workload holds before the
    write under test (empty unless ``write`` is ("last", n))."""
    ctx = context_lens(w).astype(np.int64)
    seqs, poss = [], []
    if w.write == "all":
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    for b in range(w.batch):
        n = min(int(w.write[1]), int(ctx[b]))
        p = np.arange(0, ctx[b] - n)
        seqs.append(np.full(p.shape, b, dtype=np.int64))
        poss.append(p)
    return np.concatenate(seqs), np.concatenate(poss)


# ---------------------------------------------------------------------------
# BF16 values
# ---------------------------------------------------------------------------

def rotation_words(w: Workload):
    """Sign bits of the rotation (4 uint32 words; bit c set: sigma_c = -1),
    drawn from the workload's seeded generator, or None without rotation."""
    if not w.rotate:
        return None
    bits = _rng(w.seed, 13).integers(0, 2, size=128)
    return tuple(int(sum(int(bits[32 * k + j]) << j for j in range(32))) for k in range(4))


def _torch_gen(device, seed: int, *key: int) -> torch.Generator:
    g = torch.Generator(device=device)
    # fold the key into a 63-bit seed deterministically
    h = seed & 0xFFFFFFFF
    for k in key:
        h = (h * 1000003 + (int(k) & 0xFFFFFFFF) + 0x9E3779B9) & 0x7FFFFFFFFFFFFFFF
    g.manual_seed(h)
    return g


def sequence_kv(w: Workload, which: str, b: int, device="cpu",
                n_positions: Optional[int] = None) -> torch.Tensor:
    """BF16 K or V of sequence ``b`` for positions [0, n_positions):
    shape [n_positions, num_kv_heads, head_dim]."""
    if n_positions is None:
        n_positions = int(total_positions(w)[b])
    g = _torch_gen(device, w.seed, _TENSOR_IDS[which], b)
    x = torch.randn((n_positions, w.num_kv_heads, w.head_dim), generator=g,
                    device=device, dtype=torch.float32)
    if w.outliers:
        if which == "k":
            ch = [c for c in OUTLIER_K_CHANNELS if c < w.head_dim]
            x[:, :, ch] *= OUTLIER_K_FACTOR
        x[:SINK_TOKENS] *= SINK_FACTOR
    return x.to(torch.bfloat16)


def query(w: Workload, b: int, step: int = 0, device="cpu") -> torch.Tensor:
    """BF16 decode query of sequence ``b`` at decode step ``step``:
    shape [num_q_heads, head_dim]."""
    g = _torch_gen(device, w.seed, _TENSOR_IDS["q"], b, step)
    x = torch.randn((w.num_q_heads, w.head_dim), generator=g, device=device,
                    dtype=torch.float32)
    return x.to(torch.bfloat16)


def queries(w: Workload, step: int = 0, device="cpu") -> torch.Tensor:
    if w.batch == 0:
        return torch.zeros((0, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=device)
    return torch.stack([query(w, b, step, device) for b in range(w.batch)])


def gather_tokens(w: Workload, seq_ids: np.ndarray, positions: np.ndarray,
                  device="cpu"):
    """BF16 K and V rows for the listed (seq, position) pairs, in that order:
    two tensors [n, num_kv_heads, head_dim].  Sequences are generated one at a
    time, so peak memory is one sequence plus the result."""
    seq_ids = np.asarray(seq_ids, dtype=np.int64)
    positions = np.asarray(positions, dtype=np.int64)
    n = seq_ids.shape[0]
    k = torch.empty((n, w.num_kv_heads, w.head_dim), dtype=torch.bfloat16, device=device)
    v = torch.empty_like(k)
    if n == 0:
        return k, v
    order = np.argsort(seq_ids, kind="stable")
    s_sorted = seq_ids[order]
    bounds = np.flatnonzero(np.diff(s_sorted)) + 1
    starts = np.concatenate([[0], bounds])
    ends = np.concatenate([bounds, [n]])
    for st, en in zip(starts, ends):
        b = int(s_sorted[st])
        rows = order[st:en]
        need = int(positions[rows].max()) + 1
        ks = sequence_kv(w, "k", b, device, need)
        vs = sequence_kv(w, "v", b, device, need)
        ridx = torch.as_tensor(rows, device=device)
        pidx = torch.as_tensor(positions[rows], device=device)
        k[ridx] = ks[pidx]
        v[ridx] = vs[pidx]
        del ks, vs
    return k, v


# ---------------------------------------------------------------------------
# byte counts of the workload (used to express times as bandwidth)
# ---------------------------------------------------------------------------

def scale_floats_per_token_head(fmt: CacheFormat, head_dim: int, block_size: int) -> float:
    if fmt.gran == PER_TOKEN_HEAD:
        return 1.0
    if fmt.gran == PER_TOKEN_GROUP:
        return head_dim / fmt.group
    if fmt.gran == PER_BLOCK_CHANNEL:
        return head_dim / block_size
    raise ValueError(fmt.gran)


def kv_read_bytes_per_token(w: Workload) -> float:
    """Codes plus FP32 scales one decode reads per cached token (all kv
    heads).  Per-block scales are spread over the block's tokens."""
    per_head = 0.0
    for fmt in (w.k_fmt, w.v_fmt):
        per_head += fmt.code_bytes_per_row(w.head_dim)
        per_head += 4.0 * scale_floats_per_token_head(fmt, w.head_dim, w.block_size)
    return per_head * w.num_kv_heads


def write_bytes_per_token(w: Workload) -> float:
    """HBM bytes one quantize-write moves per token: BF16 K and V read, codes
    and scales written, the int64 slot read."""
    rd = 2 * w.num_kv_heads * w.head_dim * 2
    wr = 0.0
    for fmt in (w.k_fmt, w.v_fmt):
        wr += w.num_kv_heads * fmt.code_bytes_per_row(w.head_dim)
        wr += 4.0 * w.num_kv_heads * scale_floats_per_token_head(fmt, w.head_dim, w.block_size)
    return rd + wr + 8


def decode_bytes(w: Workload, ctx: np.ndarray, max_blocks_per_seq: int) -> float:
    """Algorithmic HBM bytes of one decode step: every cached token's codes
    and scales, Q (BF16), out (FP32), the block tables and context lengths."""
    ntok = float(np.asarray(ctx, dtype=np.int64).sum())
    nblk = float(((np.asarray(ctx, dtype=np.int64) + w.block_size - 1) // w.block_size).sum())
    kv = 0.0
    for fmt in (w.k_fmt, w.v_fmt):
        code = fmt.code_bytes_per_row(w.head_dim) * w.num_kv_heads
        if fmt.gran == PER_BLOCK_CHANNEL:
            kv += ntok * code + nblk * 4.0 * w.num_kv_heads * w.head_dim
        else:
            kv += ntok * (code + 4.0 * w.num_kv_heads *
                          scale_floats_per_token_head(fmt, w.head_dim, w.block_size))
    q = w.batch * w.num_q_heads * w.head_dim * 2
    out = w.batch * w.num_q_heads * w.head_dim * 4
    tables = nblk * 4 + w.batch * 4
    return kv + q + out + tables


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


__all__ = [n for n in dir() if not n.startswith("_")]
