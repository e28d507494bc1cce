"""Pins of the oracle's block prefetch (oracle/offload.py): a hand case, the
untouched slots, skipped out-of-range pairs, and a round trip through an
offload (device -> host) and back."""
import numpy as np

import oracle


def _pool(nb, seed, bs=16, h=2, row=8, ks=(16, 2), vs=(16, 2, 4)):
    rng = np.random.default_rng(seed)
    return {"k_cache": rng.integers(0, 256, (nb, bs, h, row), dtype=np.uint8),
            "v_cache": rng.integers(0, 256, (nb, bs, h, row // 2), dtype=np.uint8),
            "k_scale": rng.standard_normal((nb,) + ks).astype(np.float32),
            "v_scale": rng.standard_normal((nb,) + vs).astype(np.float32)}


def test_hand_case_and_untouched_slots():
    host, dev = _pool(5, 1), _pool(3, 2)
    before = {k: v.copy() for k, v in dev.items()}
    assert oracle.prefetch_blocks(host, dev, [4, 0], [0, 2]) == 0
    for key in dev:
        assert np.array_equal(dev[key][0], host[key][4])
        assert np.array_equal(dev[key][2], host[key][0])
        assert np.array_equal(dev[key][1], before[key][1])   # slot 1 not named


def test_out_of_range_pairs_are_skipped():
    host, dev = _pool(4, 3), _pool(4, 4)
    before = {k: v.copy() for k, v in dev.items()}
    assert oracle.prefetch_blocks(host, dev, [4, -1, 1, 2], [0, 1, 9, 3]) == 3
    for key in dev:
        assert np.array_equal(dev[key][3], host[key][2])
        assert np.array_equal(dev[key][:3], before[key][:3])


def test_offload_and_prefetch_round_trip():
    dev = _pool(6, 5)
    host = _pool(6, 6)
    perm = np.random.default_rng(7).permutation(6)
    oracle.prefetch_blocks(dev, host, np.arange(6), perm)        # offload: device block b -> host perm[b]
    back = _pool(6, 8)
    oracle.prefetch_blocks(host, back, perm, np.arange(6))       # prefetch it back
    for key in dev:
        assert np.array_equal(back[key], dev[key])
