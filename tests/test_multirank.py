"""The multi-process path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The decode shards by sequence: every rank owns a batch of its own sequences
(same shapes and context lengths, its own seeded data) and nothing crosses
ranks on the data path; the only collectives are the timing barrier and the
max over ranks of the step time, from which rank 0 reports the whole job's
throughput.  The reference arm runs on rank 0 alone; other ranks exit 0
without work."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as wl


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    got_world, got_rank, _ = bench.dist_setup()
    assert (got_world, got_rank) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(world)
    # per-rank step times: the job's time is the slowest rank's
    t = bench.max_over_ranks(0.25 + rank, world, torch.device("cpu"))
    w = bench.rank_shard(wl.WORKLOADS["cb_mix_int8"], rank)
    results[rank] = (t, w.seed, tuple(int(c) for c in wl.context_lens(w)[:8]),
                     float(wl.decode_bytes(w, wl.context_lens(w), wl.block_tables(w)[0].shape[1])))
    bench.barrier(world)
    dist.destroy_process_group()


def test_two_gloo_ranks_share_timing_and_own_their_sequences():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        r = dict(results)
    assert set(r) == {0, 1}
    # max over ranks seen by both
    assert r[0][0] == r[1][0] == 1.25
    # distinct data, identical shapes and bytes: rank 0 reports world x bytes
    assert r[0][1] != r[1][1]
    assert r[0][2] == r[1][2]
    assert r[0][3] == r[1][3]


def test_rank_shard_keeps_shapes_and_changes_data():
    w = wl.WORKLOADS["llama3_8b_fp8"]
    w1 = bench.rank_shard(w, 1)
    assert bench.rank_shard(w, 0) is w
    assert np.array_equal(wl.context_lens(w), wl.context_lens(w1))
    assert (w1.batch, w1.num_q_heads, w1.num_kv_heads, w1.head_dim, w1.k_fmt, w1.v_fmt) == \
           (w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.k_fmt, w.v_fmt)
    a = wl.sequence_kv(w, "k", 0, "cpu", 16)
    b = wl.sequence_kv(w1, "k", 0, "cpu", 16)
    assert not torch.equal(a, b)


def test_reference_arm_runs_on_rank_zero_only():
    class Args:
        steps, warmup, gpus = 5, 3, 2
    # a non-zero rank returns at once: no oracle work, no output line
    assert bench.run_reference(Args(), wl.WORKLOADS["llama3_8b_fp8"], 2, 1) == 0
