"""Host logic of the seeded input generator: determinism, block-table and
slot-mapping structure of the five workloads."""
import numpy as np
import torch

import workloads as wl


def test_contexts_and_tables():
    for w in wl.WORKLOADS.values():
        ctx = wl.context_lens(w)
        assert ctx.shape == (w.batch,) and ctx.dtype == np.int32
        table, nb = wl.block_tables(w)
        used = table[table >= 0]
        # every physical block is dealt exactly once
        assert np.array_equal(np.sort(used), np.arange(nb))
        need = (wl.total_positions(w) + w.block_size - 1) // w.block_size
        assert np.array_equal((table >= 0).sum(axis=1), need)
    w4 = wl.WORKLOADS["cb_mix_int8"]
    c4 = wl.context_lens(w4)
    assert c4.min() >= 512 and c4.max() <= 16384
    assert np.array_equal(c4, wl.context_lens(w4))          # seeded
    seqs, pos = wl.write_positions(w4)
    assert len(seqs) == 8192                                  # 32 per sequence


def test_slot_mapping_unique_and_in_range():
    w = wl.scaled(wl.WORKLOADS["cb_mix_int8"], batch=6, contexts=[17, 1, 40, 16, 33, 5])
    table, nb = wl.block_tables(w)
    s0, p0 = wl.prewritten_positions(w)
    s1, p1 = wl.write_positions(w)
    slots = wl.slot_mapping(table, np.concatenate([s0, s1]), np.concatenate([p0, p1]), w.block_size)
    assert len(np.unique(slots)) == len(slots)
    assert slots.min() >= 0 and slots.max() < nb * w.block_size
    assert len(slots) == int(wl.context_lens(w).sum())


def test_values_seeded_and_outliers():
    w = wl.scaled(wl.WORKLOADS["llama3_8b_fp8"], batch=2, contexts=[40, 20])
    k0 = wl.sequence_kv(w, "k", 0)
    assert k0.dtype == torch.bfloat16 and k0.shape == (40, 8, 128)
    assert torch.equal(k0, wl.sequence_kv(w, "k", 0))
    assert not torch.equal(k0, wl.sequence_kv(w, "k", 1)[:20].repeat(2, 1, 1))
    k = k0.float()
    # outlier channels are ~20x louder, sink tokens ~10x
    loud = k[4:, :, list(wl.OUTLIER_K_CHANNELS)].abs().mean()
    quiet = k[4:, :, :3].abs().mean()
    assert 10 < loud / quiet < 40
    assert 5 < k[:4, :, :3].abs().mean() / quiet < 20
    kk, vv = wl.gather_tokens(w, np.array([1, 0, 0]), np.array([3, 39, 0]))
    assert torch.equal(kk[1], k0[39]) and torch.equal(kk[2], k0[0])
    assert torch.equal(vv[0], wl.sequence_kv(w, "v", 1)[3])
