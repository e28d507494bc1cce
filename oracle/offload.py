"""Oracle: prefetch of offloaded cache blocks from host memory into device
block slots (test infrastructure; see the package docstring).

"Use Less Memory: Quantization and Offloading", §3 (the CPU RAM tier holds
KV blocks that do not fit in HBM) and §4 Pipelining and Latency Overlap
(while step t computes, the blocks step t + 1 needs are copied from CPU RAM
into a second set of GPU buffers).  The copy moves whole cache blocks in the
cache's own layout: the codes of every (token, kv head) row of the block and
the block's scales, unchanged.

Reading: a block is the unit (its codes [block_size, H, row] and its scales,
whatever the granularity); src[i] is a block of the host pool, dst[i] a block
slot of the device cache; entries outside either pool are skipped.
"""
from __future__ import annotations

import numpy as np


def prefetch_blocks(host, dev, src, dst):
    """host, dev: dicts with "k_cache", "v_cache" (uint8 [nb, bs, H, row]) and
    "k_scale", "v_scale" (float32, leading axis = block); copies block src[i]
    of host into block dst[i] of dev in place.  Returns the number of pairs
    skipped as out of range."""
    src = np.asarray(src, dtype=np.int64)
    dst = np.asarray(dst, dtype=np.int64)
    nh = host["k_cache"].shape[0]
    nd = dev["k_cache"].shape[0]
    ok = (src >= 0) & (src < nh) & (dst >= 0) & (dst < nd)
    for key in ("k_cache", "v_cache", "k_scale", "v_scale"):
        dev[key][dst[ok]] = host[key][src[ok]]
    return int((~ok).sum())
