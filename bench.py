"""Benchmark: quantize-on-write + paged quantized decode attention on GB300.

By default one step is one serving decode step of the Llama-3-8B-shaped FP8
workload (batch 27, 32 query heads, 8 kv heads, head_dim 128, block 16, every
sequence at context 32768, FP8 E4M3FN per-(token, kv_head) scales):
quantize-write the step's new token of every sequence into the paged cache,
then paged decode attention over the 32768 cached tokens.  ``--workload``
selects another workload for the headline (see Step for what their step
writes).  Inputs are seeded synthetic BF16 with the workload's outlier
pattern, generated on the device; the cache is resident in HBM before timing.

value     = algorithmic HBM bytes of a step (codes + scales read, Q, out,
            block tables, the write's BF16 in / codes out) / step time, GB/s:
            the median of --repeats timed windows of --steps steps each
            (min and max in ``spread``)
e2e       = the same through the public API with the step's inputs copied
            from pinned host memory and the output copied back, every step
roofline  = the decode call (split + reduce kernels) against the measured
            HBM copy bandwidth; `traffic` is the DRAM bytes per launch of the
            committed ncu capture (profiles/decode_traffic.json) when the
            decode sources are unchanged since it was taken, else null
quant_write = the prefill write (every position before the step's) timed
            separately (at least 10 launches)
configs   = every one of the five workloads measured the same way (decode,
            prefill quantize-write, the workload's serving step), one after
            the other on the same GPU (single-GPU runs only)
cpu_baseline = the CPU oracle on a bounded sample of the same step, one
            worker process per host core

``--impl reference`` times the CPU oracle as the reference arm (there is no
runnable reference implementation; the oracle is the plain restatement of
the method), on all host cores.  Under torchrun every rank runs its own
replica (weak scaling).
"""
from __future__ import annotations

import os

import argparse
import ctypes
import json
import multiprocessing
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

import workloads as wl

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "paged quantized decode attn HBM GB/s (% of GB300 peak), tokens/s; quant-write GB/s"
REF_BUDGET_S = 90.0   # timed oracle work of one --impl reference run (wall seconds)
CONFIG_WORKLOADS = ("tiny_int8", "llama3_8b_fp8", "llama3_70b_kivi", "cb_mix_int8", "long_mixed")
NOMINAL_HBM_GBS = 8000.0   # the GB300 nominal "~8 TB/s" the targets are quoted against
FALLBACK_HBM_GBS = 6800.0


DECODE_SOURCES = ("common.cuh", "quantize_rows.cuh", "paged_decode_impl.cuh", "decode_launch.cuh", "decode_k0.cu",
                  "decode_k1.cu", "decode_k2.cu", "decode_k3.cu", "decode_k4.cu", "kvq_internal.h")


def decode_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "quantized_paged_kv_write_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu capture of this
    workload, or None if there is none or the decode sources changed since."""
    try:
        with open(os.path.join(ROOT, "profiles", "decode_traffic.json")) as f:
            rec = json.load(f).get(workload)
        if rec and rec["source_hash"] == decode_source_hash():
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def measured_hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s)"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.proc = None
        self.path = None
        sel = []
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        self.cmd = ["nvidia-smi", f"--query-gpu=timestamp,{self.FIELDS}", "--format=csv,noheader,nounits",
                    "-lms", "100"] + sel

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            self.out = os.fdopen(fd, "w")
            self.proc = subprocess.Popen(self.cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.t0 = time.time()

    def mark(self):
        return time.time()

    def stop(self, t_begin, t_end):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                rows.append((ts, float(parts[1]), float(parts[2]), parts[4:9]))
            except Exception:
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t_begin - 1 <= r[0] <= t_end + 1]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in use for k, v in enumerate(r[3][1:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "in_timed_region": bool(inside)}


# ---------------------------------------------------------------------------
# the workload on the device
# ---------------------------------------------------------------------------
class Step:
    """Resident cache + the inputs of the serving step.

    The step writes, for every sequence, the workload's new tokens and then
    decodes over the whole context:
      * decode workloads: the last position (one token per sequence);
      * the chunked-prefill workload: its chunk (the last 32 positions);
      * per-channel K: the last block (a block's K scales cover the tokens
        written into it together);
      * the long-context workload with decode steps: step s writes position
        ctx + s and decodes over ctx + s + 1 (its 100 steps repeat in turn).
    Everything before the step's positions is written once, untimed, by one
    quantize-write of all prefill tokens (also the quant-write measurement).
    """

    def __init__(self, kvq, w: wl.Workload, device):
        self.kvq, self.w, self.dev = kvq, w, device
        ctx = wl.context_lens(w).astype(np.int64)
        table, nb = wl.block_tables(w)
        self.table_np = table
        self.fmt = kvq.cache_format(w.k_fmt, w.v_fmt, w.num_kv_heads, w.head_dim, nb, w.block_size,
                                    rotation_signs=wl.rotation_words(w))
        self.cache = kvq.allocate_cache(self.fmt, device)
        self.tables = torch.as_tensor(table, device=device)
        bs = w.block_size
        if w.decode_steps:
            nsteps = w.decode_steps
            pre_end = ctx
            step_pos = [ctx + s for s in range(nsteps)]             # one token per sequence
        else:
            nsteps = 1
            if w.k_fmt.gran == wl.PER_BLOCK_CHANNEL:
                n = (ctx - 1) % bs + 1
            elif w.write != "all":
                n = np.minimum(int(w.write[1]), ctx)
            else:
                n = np.ones_like(ctx)
            pre_end = ctx - n
            step_pos = None
        pk, pv, ps = [], [], []
        sk = [[] for _ in range(nsteps)]
        sv = [[] for _ in range(nsteps)]
        ss = [[] for _ in range(nsteps)]
        npos = wl.total_positions(w)
        for b in range(w.batch):
            k = wl.sequence_kv(w, "k", b, device, int(npos[b]))
            v = wl.sequence_kv(w, "v", b, device, int(npos[b]))
            pre = np.arange(pre_end[b])
            pk.append(k[: pre_end[b]])
            pv.append(v[: pre_end[b]])
            ps.append(torch.as_tensor(wl.slot_mapping(table, np.full(len(pre), b), pre, bs), device=device))
            for s in range(nsteps):
                pos = (np.array([step_pos[s][b]]) if step_pos is not None
                       else np.arange(pre_end[b], ctx[b]))
                sk[s].append(k[torch.as_tensor(pos, device=device)])
                sv[s].append(v[torch.as_tensor(pos, device=device)])
                ss[s].append(torch.as_tensor(wl.slot_mapping(table, np.full(len(pos), b), pos, bs), device=device))
            del k, v
        self.pk, self.pv, self.pslots = torch.cat(pk), torch.cat(pv), torch.cat(ps)
        self.steps_in = [(torch.cat(sk[s]).contiguous(), torch.cat(sv[s]).contiguous(), torch.cat(ss[s]))
                         for s in range(nsteps)]
        self.step_ctx = [ctx + s + 1 if w.decode_steps else ctx for s in range(nsteps)]
        self.ctx_t = [torch.as_tensor(c.astype(np.int32), device=device) for c in self.step_ctx]
        self.max_ctx = int(max(c.max() for c in self.step_ctx))
        self.q = [wl.queries(w, step=s, device=device) for s in range(nsteps)]
        self.nsteps = nsteps
        self.k_i = 0
        self.out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device=device)
        nbytes = kvq.kvq_decode_workspace_size(self.fmt, w.batch, w.num_q_heads, self.max_ctx)
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        kvq.kvq_quantize_write(self.pk, self.pv, self.pslots, self.fmt, self.cache)
        torch.cuda.synchronize()

    # the step's inputs (step s of a growing workload, else the single step)
    def inputs(self, s=None):
        s = self.k_i if s is None else s
        k, v, slots = self.steps_in[s]
        return k, v, slots, self.q[s], self.ctx_t[s]

    def write(self):
        k, v, slots, _, _ = self.inputs()
        self.kvq.kvq_quantize_write(k, v, slots, self.fmt, self.cache)

    def decode(self):
        _, _, _, q, ctx_t = self.inputs()
        self.kvq.kvq_paged_decode(q, self.fmt, self.cache, self.tables, ctx_t, self.max_ctx,
                                  out=self.out, workspace=self.ws)
        self.k_i = (self.k_i + 1) % self.nsteps

    def step(self):
        self.write()
        self.decode()

    # one token per sequence with per-token K: the write can ride in the
    # decode launch (kvq_write_decode)
    def fused_ok(self):
        return self.w.k_fmt.gran != wl.PER_BLOCK_CHANNEL and self.step_tokens_written() == self.w.batch

    def fused(self):
        k, v, _, q, ctx_t = self.inputs()
        self.kvq.kvq_write_decode(q, k, v, self.fmt, self.cache, self.tables, ctx_t, self.max_ctx,
                                  out=self.out, workspace=self.ws)
        self.k_i = (self.k_i + 1) % self.nsteps

    # algorithmic bytes, averaged over the step cycle
    def decode_bytes(self):
        return float(np.mean([wl.decode_bytes(self.w, c, self.table_np.shape[1]) for c in self.step_ctx]))

    def write_bytes(self, ntok):
        return wl.write_bytes_per_token(self.w) * ntok

    def step_tokens_written(self):
        return int(self.steps_in[0][2].numel())

    def step_bytes(self):
        return self.decode_bytes() + self.write_bytes(self.step_tokens_written())

    def kv_tokens(self):
        return float(np.mean([c.sum() for c in self.step_ctx]))


def timed(fn, steps, stream):
    """CUDA-event time of `steps` calls of fn, synchronized on both sides."""
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


# ---------------------------------------------------------------------------
# CPU oracle on a bounded sample of the step
# ---------------------------------------------------------------------------
class OracleSample:
    """The oracle's quantize-write + decode step on one sequence of the
    workload (all query heads), the CPU baseline's unit of work.  ``index``
    picks sequence index % batch, with its own seeded data for index > 0.
    The cache state (every cached token but the sequence's last) is written
    once, untimed; each step then quantizes the last token and decodes a
    context prefix of `ctx_len` tokens (the whole context by default)."""

    def __init__(self, w: wl.Workload, index: int = 0):
        import oracle
        self.oracle = oracle
        b = index % max(w.batch, 1)
        ctx = wl.context_lens(w)[b:b + 1]
        seed = w.seed if index == 0 else w.seed + 7919 * index
        self.sub = sub = wl.scaled(w, batch=1, contexts=ctx, seed=seed, name=w.name + "_cpu_sample")
        self.ctx = int(ctx[0])
        self.table, nb = wl.block_tables(sub)
        pos = np.arange(self.ctx)
        k, v = wl.gather_tokens(sub, np.zeros(self.ctx, np.int64), pos)
        slots = wl.slot_mapping(self.table, np.zeros(self.ctx, np.int64), pos, sub.block_size)
        kb = k.view(torch.int16).numpy().view(np.uint16)
        vb = v.view(torch.int16).numpy().view(np.uint16)
        self.q = wl.queries(sub).view(torch.int16).numpy().view(np.uint16)
        words = wl.rotation_words(sub)
        self.oc = oracle.OracleCache(nb, sub.block_size, sub.num_kv_heads, sub.head_dim, sub.k_fmt, sub.v_fmt,
                                     rotation_signs=None if words is None else
                                     oracle.signs_from_words(words, sub.head_dim))
        oracle.quantize_write(self.oc, kb[:-1], vb[:-1], slots[:-1])     # cache state (untimed)
        self.last = (kb[-1:], vb[-1:], slots[-1:])

    def step(self, ctx_len=None):
        """One timed step; returns (algorithmic bytes, wall s, process CPU s)."""
        n = self.ctx if ctx_len is None else int(ctx_len)
        t0, c0 = time.perf_counter(), time.process_time()
        self.oracle.quantize_write(self.oc, *self.last)                           # the step's write
        self.oracle.paged_decode_fp64(self.oc, self.q, self.table, np.array([n]))  # the step's decode
        dt, dc = time.perf_counter() - t0, time.process_time() - c0
        nbytes = wl.decode_bytes(self.sub, np.array([n]), self.table.shape[1]) + wl.write_bytes_per_token(self.sub)
        return nbytes, dt, dc

    def describe(self, ctx_len=None):
        w = self.sub
        n = self.ctx if ctx_len is None else int(ctx_len)
        return ("quantize-write of 1 new token + fp64 decode of 1 sequence (%d query heads, %d of its %d "
                "context tokens)" % (w.num_q_heads, n, self.ctx))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


# one OracleSample per worker process of the pool (set by _pool_init)
_POOL_SAMPLE = None
_POOL_BARRIER = None


def _pool_init(w, counter, lock, barrier):
    global _POOL_SAMPLE, _POOL_BARRIER
    torch.set_num_threads(1)
    with lock:
        idx = counter.value
        counter.value += 1
    _POOL_SAMPLE = OracleSample(w, idx)
    _POOL_BARRIER = barrier


def _pool_step(ctx_len):
    # every worker holds one task at the barrier, so the round's steps run
    # side by side, one per process; the wall clock is shared by the host's
    # processes
    _POOL_BARRIER.wait(timeout=900)
    t0 = time.time()
    nbytes, _, dc = _POOL_SAMPLE.step(ctx_len)
    return nbytes, t0, time.time(), dc


class OraclePool:
    """The oracle on every host core: `workers` processes (spawned, one
    thread each), each holding one sequence of the workload; a round is one
    step of every worker at the same time."""

    def __init__(self, w: wl.Workload, workers=None):
        self.n = int(workers or host_cores())
        ctx = multiprocessing.get_context("spawn")
        self.counter = ctx.Value("i", 0)
        self.lock = ctx.Lock()
        self.barrier = ctx.Barrier(self.n)
        saved = {v: os.environ.get(v) for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")}
        os.environ.update({v: "1" for v in saved})   # inherited by the spawned workers
        try:
            self.pool = ctx.Pool(self.n, initializer=_pool_init,
                                 initargs=(w, self.counter, self.lock, self.barrier))
        finally:
            for v, old in saved.items():
                if old is None:
                    os.environ.pop(v, None)
                else:
                    os.environ[v] = old

    def round(self, ctx_len=None):
        """(bytes, wall seconds, CPU seconds) of one round of all workers."""
        rs = [self.pool.apply_async(_pool_step, (ctx_len,)) for _ in range(self.n)]
        out = [r.get(timeout=1800) for r in rs]
        return (sum(o[0] for o in out), max(o[2] for o in out) - min(o[1] for o in out), sum(o[3] for o in out))

    def close(self):
        self.pool.terminate()
        self.pool.join()


def cpu_baseline(w: wl.Workload, min_seconds: float = 10.0, workers=None):
    """The oracle timed on the host's cores: every worker process steps its
    own sequence (write of the new token + fp64 decode over the whole
    context) at the same time, rounds repeated until at least `min_seconds`
    of wall time; value = all workers' bytes / wall time."""
    pool = OraclePool(w, workers)
    try:
        pool.round()                      # untimed: the workers' set-up and a first step
        tb = tt = tc = 0.0
        reps = 0
        while reps == 0 or tt < min_seconds:
            b, t, c = pool.round()
            tb, tt, tc, reps = tb + b, tt + t, tc + c, reps + 1
    finally:
        pool.close()
    ctx = int(wl.context_lens(w)[0])
    smp_desc = ("%d worker processes (one per host core, one thread each), each: quantize-write of 1 new token "
                "+ fp64 decode of its own sequence (%d query heads, %d context tokens)" % (pool.n, w.num_q_heads, ctx))
    return {"value": tb / tt / 1e9, "unit": "GB/s", "cores": pool.n, "kind": "oracle",
            "sample": "%s; %d round(s), %.1f s" % (smp_desc, reps, tt),
            "cpu_seconds_per_wall_second": round(tc / tt, 2)}


def workload_config(w, extra=None):
    cfg = {
        "workload": w.name + ": " + w.description,
        "batch": w.batch, "context": int(wl.context_lens(w).max()), "q_heads": w.num_q_heads,
        "kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "block_size": w.block_size,
        "k_format": f"{w.k_fmt.dtype}/{w.k_fmt.gran}", "v_format": f"{w.v_fmt.dtype}/{w.v_fmt.gran}"
        + (f"{w.v_fmt.group}" if w.v_fmt.group else ""),
        "step": "quantize-write one new token per sequence + paged decode over the full context",
        "l2": "inputs larger than L2: each step reads the whole %.2f GB cache (L2 129 MB)"
              % (wl.decode_bytes(w, wl.context_lens(w), 1) / 1e9),
    }
    if extra:
        cfg.update(extra)
    return cfg


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def rank_shard(w: wl.Workload, rank: int) -> wl.Workload:
    """Rank r's share of a multi-GPU run: a batch of its own sequences with
    the workload's shapes, formats and context lengths, its data drawn with a
    rank-specific seed.  The ranks share no data and exchange nothing on the
    data path (weak scaling: the job's units are world x batch sequences)."""
    if rank == 0:
        return w
    return wl.scaled(w, contexts=wl.context_lens(w), seed=w.seed + 7919 * rank, name=f"{w.name}_rank{rank}")


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def run_reference(args, w, world, rank, workers=None):
    """The reference arm: the CPU oracle, timed as it stands, on every host
    core (one worker process per core, each on its own sequence).  Each step
    is one round of all workers over a context prefix sized so that the
    whole run's timed work stays near REF_BUDGET_S seconds."""
    if rank != 0:
        return 0
    pool = OraclePool(w, workers)
    try:
        _, t_full, _ = pool.round()              # calibration: one whole-sequence round (untimed)
        per_step = REF_BUDGET_S / max(1, args.steps + args.warmup)
        bs = w.block_size
        ctx = int(wl.context_lens(w)[0])
        n = ctx if t_full <= per_step else max(bs, int(ctx * per_step / t_full) // bs * bs)
        for _ in range(args.warmup):
            pool.round(n)
        tot_b = tot_t = tot_c = 0.0
        for _ in range(args.steps):
            b, t, c = pool.round(n)
            tot_b, tot_t, tot_c = tot_b + b, tot_t + t, tot_c + c
    finally:
        pool.close()
    value = tot_b / tot_t / 1e9
    desc = ("%d worker processes (one per host core), each: quantize-write of 1 new token + fp64 decode of its own "
            "sequence (%d query heads, %d of its %d context tokens)" % (pool.n, w.num_q_heads, n, ctx))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 quantize / f64 attention",
        "data": "synthetic", "config": workload_config(w, {"sample": desc + " per step"}),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": pool.n, "kind": "oracle",
                         "sample": desc + " per step, %d steps, %.1f s" % (args.steps, tot_t),
                         "cpu_seconds_per_wall_second": round(tot_c / tot_t, 2)},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def host_call_us(fn, calls=20):
    """Host wall-clock microseconds per call of fn (the GPU queue stays far
    from full: a few dozen launches)."""
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(calls):
        fn()
    t1 = time.perf_counter()
    torch.cuda.synchronize()
    return 1e6 * (t1 - t0) / calls


def raw_step_call(kvq, st):
    """The workload's step as one C-ABI call through ctypes with every
    argument marshalled once (no binding checks): host cost of the library
    call itself plus the ctypes transition.  None for two-call steps."""
    if not st.fused_ok():
        return None
    lib = kvq.load_library()
    k, v, _, q, ctx_t = st.inputs(0)
    cf = st.fmt.as_c()
    caches, scales = kvq._caches(st.cache)
    handle = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), q.shape[0], q.shape[1], ctypes.byref(cf), caches, scales,
            st.tables.data_ptr(), st.tables.shape[1], ctx_t.data_ptr(), st.max_ctx, st.out.data_ptr(),
            st.ws.data_ptr(), st.ws.numel(), handle)

    def call():
        if lib.kvq_write_decode(*args) != 0:
            raise RuntimeError("kvq_write_decode failed")
    return call


def measure_workload(kvq, w, dev, stream, steps, peak, st=None):
    """One workload's decode, prefill quantize-write and serving step on this
    GPU (each timed with CUDA events on the launching stream)."""
    own = st is None
    if own:
        st = Step(kvq, w, dev)
    fused = st.fused_ok()
    step_fn = st.fused if fused else st.step
    n = st.nsteps if st.nsteps > 1 else max(steps, 20)
    for _ in range(3):
        step_fn()
    step_s = timed(step_fn, n, stream) / n
    dec_s = timed(st.decode, n, stream) / n
    for _ in range(2):
        kvq.kvq_quantize_write(st.pk, st.pv, st.pslots, st.fmt, st.cache)
    qw_iters = 10
    qw_s = timed(lambda: kvq.kvq_quantize_write(st.pk, st.pv, st.pslots, st.fmt, st.cache), qw_iters,
                 stream) / qw_iters
    sw_s = timed(st.write, n, stream) / n
    host_us = host_call_us(step_fn)
    errs = kvq.kvq_device_errors(clear=True)
    ntok = int(st.pslots.numel())
    dec_b, qw_b = st.decode_bytes(), st.write_bytes(ntok)
    traffic = recorded_traffic(w.name)
    out = {
        "workload": w.name + ": " + w.description,
        "step_call": "kvq_write_decode" if fused else "kvq_quantize_write + kvq_paged_decode",
        "ms_per_step": step_s * 1e3, "steps_timed": n,
        "step_gbs": st.step_bytes() / step_s / 1e9, "tokens_per_s": w.batch / step_s,
        "decode": {"gbs": dec_b / dec_s / 1e9, "ms": dec_s * 1e3, "bytes": dec_b,
                   "frac_of_measured_hbm": dec_b / dec_s / 1e9 / peak,
                   "frac_of_nominal_hbm": dec_b / dec_s / 1e9 / NOMINAL_HBM_GBS,
                   "kv_tokens_per_s": st.kv_tokens() / dec_s,
                   "dram_bytes_over_algorithmic": (traffic / dec_b) if traffic else None},
        "quant_write": {"gbs": qw_b / qw_s / 1e9, "ms": qw_s * 1e3, "tokens": ntok, "bytes": qw_b,
                        "iterations": qw_iters,
                        "frac_of_measured_hbm": qw_b / qw_s / 1e9 / peak,
                        "frac_of_nominal_hbm": qw_b / qw_s / 1e9 / NOMINAL_HBM_GBS},
        "step_write": {"tokens": st.step_tokens_written(), "us": sw_s * 1e6,
                       "gbs": st.write_bytes(st.step_tokens_written()) / sw_s / 1e9},
        "host_us_per_step_call": host_us,
        "device_errors": errs,
    }
    if own:
        del st
        torch.cuda.empty_cache()
    return out


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--repeats", type=int, default=10, help="timed windows of --steps steps (median reported)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b_fp8", choices=list(wl.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefetch", action="store_true", help="skip the host-tier prefetch measurement")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload table")
    ap.add_argument("--batch", type=int, default=None,
                    help="fewer sequences of the same shape (profiling captures only)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    args.repeats = max(args.repeats, 1)
    w = wl.WORKLOADS[args.workload]
    if args.batch is not None and args.batch != w.batch:
        w = wl.scaled(w, batch=args.batch, contexts=wl.context_lens(w)[: args.batch],
                      name=f"{w.name}_batch{args.batch}")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, w, world, rank)
    w = rank_shard(w, rank)

    import quantized_paged_kv_write_gb300 as kvq
    from quantized_paged_kv_write_gb300 import build
    build.build()
    kvq.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peak, peak_src = measured_hbm_peak()

    st = Step(kvq, w, dev)
    fused = st.fused_ok()
    kvq.kvq_device_errors(clear=True)
    for _ in range(args.warmup):
        st.step()
        if fused:
            st.fused()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)

    # ---- two-call steps (write, then decode), per-call events for the decode
    def two_call_loop():
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for k in range(args.steps):
            st.write()
            ev[k][0].record(stream)
            st.decode()
            ev[k][1].record(stream)
        e1.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        return (max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.steps, world, dev),
                statistics.mean(a.elapsed_time(b) for a, b in ev) / 1e3, t0, t1)

    # ---- fused steps (kvq_write_decode): the headline when the format allows
    def fused_loop():
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            st.fused()
        e1.record(stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
        return max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.steps, world, dev), t0, t1

    # --repeats timed windows of exactly --steps steps each
    step_list, two_list, dec_list = [], [], []
    t_begin = t_end = None
    for _ in range(args.repeats):
        two_s, dec_s, t0, t1 = two_call_loop()
        t_begin = t0 if t_begin is None else t_begin
        if fused:
            step_s, _, t1 = fused_loop()
        else:
            step_s = two_s
        t_end = t1
        step_list.append(step_s)
        two_list.append(two_s)
        dec_list.append(dec_s)
    clk = clocks.stop(t_begin, t_end)
    errs = kvq.kvq_device_errors(clear=True)

    step_bytes = st.step_bytes()
    step_s = statistics.median(step_list)
    two_s = statistics.median(two_list)
    dec_s = statistics.median(dec_list)
    value = world * step_bytes / step_s / 1e9
    dec_bytes = st.decode_bytes()
    dec_gbs = dec_bytes / dec_s / 1e9
    spread = {"repeats": args.repeats, "steps_per_repeat": args.steps,
              "value_min": world * step_bytes / max(step_list) / 1e9,
              "value_max": world * step_bytes / min(step_list) / 1e9,
              "decode_gbs_min": dec_bytes / max(dec_list) / 1e9, "decode_gbs_max": dec_bytes / min(dec_list) / 1e9,
              "timed_region_s": float(sum(two_list) + (sum(step_list) if fused else 0.0)) * args.steps}

    # ---- quantize-write of the whole prefill (884,736 tokens), separately
    qw_iters = max(10, min(50, args.steps // 20))
    for _ in range(2):
        kvq.kvq_quantize_write(st.pk, st.pv, st.pslots, st.fmt, st.cache)
    qw_s = timed(lambda: kvq.kvq_quantize_write(st.pk, st.pv, st.pslots, st.fmt, st.cache), qw_iters, stream)
    qw_s /= qw_iters
    ntok = int(st.pslots.numel())
    qw_gbs = st.write_bytes(ntok) / qw_s / 1e9

    # ---- host latency of one step call: through the binding, and as a bare
    # C-ABI call through ctypes
    host = {"binding_us": host_call_us(st.fused if fused else st.step)}
    raw = raw_step_call(kvq, st)
    if raw is not None:
        host["c_abi_us"] = host_call_us(raw)
    host["gpu_us"] = step_s * 1e6
    kvq.kvq_device_errors(clear=True)

    # ---- per-channel K with a full-precision tail: the serving step appends
    # one token per sequence (position ctx, residual row ctx % 16) and decodes
    # over the quantized blocks plus the tail (the step of 15 in 16 that does
    # not complete a block)
    kivi = None
    if rank == 0 and w.k_fmt.gran == wl.PER_BLOCK_CHANNEL:
        res = kvq.allocate_residual(st.fmt, w.batch, dev)
        ctx_now = wl.context_lens(w).astype(np.int64)
        # a block-aligned context starts a new block; otherwise the tail holds
        # the rows of the incomplete block (none here: the workload is aligned)
        n1 = torch.as_tensor((ctx_now + 1).astype(np.int32), device=dev)
        kn, vn = wl.gather_tokens(w, np.arange(w.batch), ctx_now, device=dev)
        qk = wl.queries(w, device=dev)
        mc = int(ctx_now.max()) + 1
        ws_k = torch.empty(max(kvq.kvq_decode_workspace_size(st.fmt, w.batch, w.num_q_heads, mc), 256),
                           dtype=torch.uint8, device=dev)

        def kivi_step():
            kvq.kvq_kivi_append(kn, vn, st.fmt, st.cache, st.tables, n1, res)
            kvq.kvq_kivi_decode(qk, st.fmt, st.cache, st.tables, n1, mc, res, out=st.out, workspace=ws_k)

        for _ in range(3):
            kivi_step()
        k_iters = max(20, min(500, args.steps // 4))
        kivi_s = timed(kivi_step, k_iters, stream) / k_iters
        kb = float(wl.decode_bytes(w, ctx_now, st.table_np.shape[1]))
        kivi = {"value": kb / kivi_s / 1e9, "unit": "GB/s", "ms_per_step": kivi_s * 1e3,
                "step": "kvq_kivi_append (one token per sequence into the full-precision tail) + kvq_kivi_decode "
                        "(quantized blocks + tail)", "gpu_launches_per_step": 3}
        del res, ws_k
        kvq.kvq_device_errors(clear=True)

    # ---- offload tier: blocks prefetched from pinned host memory into a
    # second device buffer (double buffering), alone and beside the decode
    pf = None
    if rank == 0 and not args.no_prefetch:
        nbk = st.fmt.num_blocks
        host_pool = kvq.allocate_host_pool(st.fmt, nbk)
        for key in host_pool:
            host_pool[key].copy_(st.cache[key].cpu())
        buf_b = kvq.allocate_cache(st.fmt, dev)
        all_idx = torch.arange(nbk, dtype=torch.int32, device=dev)
        pf_bytes = float(sum(t.numel() * t.element_size() for t in host_pool.values()))
        side = torch.cuda.Stream()
        for _ in range(2):
            kvq.kvq_prefetch_blocks(host_pool, all_idx, all_idx, st.fmt, buf_b)
        pf_iters = 5
        pf_s = timed(lambda: kvq.kvq_prefetch_blocks(host_pool, all_idx, all_idx, st.fmt, buf_b), pf_iters,
                     stream) / pf_iters
        # a transfer of about half a decode step (the pages' "hidden" case)
        n_ov = max(1, min(nbk, int(nbk * 0.5 * dec_s / pf_s)))
        ov_idx = all_idx[:n_ov].contiguous()
        ov_iters = 50
        pf_part_s = timed(lambda: kvq.kvq_prefetch_blocks(host_pool, ov_idx, ov_idx, st.fmt, buf_b), ov_iters,
                          stream) / ov_iters
        dec_only_s = timed(st.decode, ov_iters, stream) / ov_iters

        def both():
            # step t's decode, then the blocks of step t + 1 on the side stream
            side.wait_stream(stream)
            st.decode()
            with torch.cuda.stream(side):
                kvq.kvq_prefetch_blocks(host_pool, ov_idx, ov_idx, st.fmt, buf_b, stream=side)
            stream.wait_stream(side)

        both()
        both_s = timed(both, ov_iters, stream) / ov_iters
        pf = {"gbs": pf_bytes / pf_s / 1e9, "bytes": pf_bytes, "ms": pf_s * 1e3, "blocks": int(nbk),
              "source": "pinned host memory (CPU-GPU link) -> HBM, one gather kernel",
              "overlap": {"prefetch_blocks": n_ov, "prefetch_ms": pf_part_s * 1e3, "decode_ms": dec_only_s * 1e3,
                          "both_ms": both_s * 1e3,
                          "hidden_fraction": (dec_only_s + pf_part_s - both_s) / pf_part_s}}
        del host_pool, buf_b
        kvq.kvq_device_errors(clear=True)

    # ---- end to end through the public API with host buffers
    e2e_steps = max(20, min(200, args.steps))
    # every step's inputs (new K / V rows, slot mapping, queries, context
    # lengths, block tables) packed into one pinned host buffer, copied to
    # the device as one transfer per step; the cache stays resident
    names = ["k", "v", "slots", "q", "ctx", "tables"]
    if fused:  # the fused call takes no slot mapping
        names.remove("slots")
    proto = dict(zip(["k", "v", "slots", "q", "ctx"], st.inputs(0)), tables=st.tables)
    layout, off = {}, 0
    for nm in names:
        t = proto[nm]
        layout[nm] = (off, t.shape, t.dtype)
        off += (t.numel() * t.element_size() + 255) // 256 * 256
    h_steps = []
    for s_ in range(st.nsteps):
        src = dict(zip(["k", "v", "slots", "q", "ctx"], st.inputs(s_)), tables=st.tables)
        hb = torch.empty(off, dtype=torch.uint8).pin_memory()
        for nm in names:
            o, shape, dt = layout[nm]
            n = src[nm].numel() * src[nm].element_size()
            hb[o:o + n].copy_(src[nm].contiguous().view(-1).view(torch.uint8).cpu())
        h_steps.append(hb)
    # Two device input buffers and two outputs: step t's inputs go to the
    # device on a copy stream while step t - 1 computes, and step t's output
    # comes back while step t + 1 computes (every copy is still made, every
    # step, inside the timed region).
    d_bufs = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]

    def dview(buf, nm):
        o, shape, dt = layout[nm]
        n = int(np.prod(shape)) * torch.empty((), dtype=dt).element_size()
        return buf[o:o + n].view(dt).view(shape)

    d_ins = [{nm: dview(buf, nm) for nm in names} for buf in d_bufs]
    d_outs = [torch.empty_like(st.out) for _ in range(2)]
    h_outs = [torch.empty(st.out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = off
    d2h = h_outs[0].numel() * 4
    copy_stream = torch.cuda.Stream(device=dev)
    ev = {key: [torch.cuda.Event() for _ in range(2)] for key in ("in_ready", "done", "copied")}

    def e2e_run(nsteps):
        """nsteps pipelined end-to-end steps; returns seconds per step."""
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)

        def upload(t):
            b = t % 2
            copy_stream.wait_stream(stream) if t < 2 else copy_stream.wait_event(ev["done"][b])
            with torch.cuda.stream(copy_stream):
                d_bufs[b].copy_(h_steps[t % st.nsteps], non_blocking=True)
                ev["in_ready"][b].record(copy_stream)

        upload(0)
        for t in range(nsteps):
            b = t % 2
            if t + 1 < nsteps:
                upload(t + 1)
            stream.wait_event(ev["in_ready"][b])
            if t >= 2:
                stream.wait_event(ev["copied"][b])   # out[b] of step t - 2 is on the host
            d = d_ins[b]
            if fused:
                kvq.kvq_write_decode(d["q"], d["k"], d["v"], st.fmt, st.cache, d["tables"], d["ctx"], st.max_ctx,
                                     out=d_outs[b], workspace=st.ws)
            else:
                kvq.kvq_quantize_write(d["k"], d["v"], d["slots"], st.fmt, st.cache)
                kvq.kvq_paged_decode(d["q"], st.fmt, st.cache, d["tables"], d["ctx"], st.max_ctx, out=d_outs[b],
                                     workspace=st.ws)
            ev["done"][b].record(stream)
            copy_stream.wait_event(ev["done"][b])
            with torch.cuda.stream(copy_stream):
                h_outs[b].copy_(d_outs[b], non_blocking=True)
                ev["copied"][b].record(copy_stream)
        stream.wait_stream(copy_stream)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / nsteps

    e2e_run(3)
    e2e_runs = [e2e_run(e2e_steps) for _ in range(3)]
    e2e_s = max_over_ranks(statistics.median(e2e_runs), world, dev)
    e2e_val = world * step_bytes / e2e_s / 1e9
    # the same step with no overlap (copy in, step, copy out, in order)
    d_in0 = d_ins[0]

    def e2e_serial_step(i=[0]):
        d_bufs[0].copy_(h_steps[i[0] % st.nsteps], non_blocking=True)
        i[0] += 1
        if fused:
            kvq.kvq_write_decode(d_in0["q"], d_in0["k"], d_in0["v"], st.fmt, st.cache, d_in0["tables"], d_in0["ctx"],
                                 st.max_ctx, out=d_outs[0], workspace=st.ws)
        else:
            kvq.kvq_quantize_write(d_in0["k"], d_in0["v"], d_in0["slots"], st.fmt, st.cache)
            kvq.kvq_paged_decode(d_in0["q"], st.fmt, st.cache, d_in0["tables"], d_in0["ctx"], st.max_ctx,
                                 out=d_outs[0], workspace=st.ws)
        h_outs[0].copy_(d_outs[0], non_blocking=True)

    e2e_serial_s = timed(e2e_serial_step, e2e_steps, stream) / e2e_steps

    # ---- the five workloads, one after the other (single-GPU runs only)
    configs = None
    if world == 1 and not args.no_configs and args.batch is None:
        configs = {}
        configs[w.name] = measure_workload(kvq, w, dev, stream, args.steps, peak, st=st)
    del st, d_bufs, d_ins, d_outs, h_steps
    torch.cuda.empty_cache()
    if configs is not None:
        for name in CONFIG_WORKLOADS:
            if name not in configs:
                configs[name] = measure_workload(kvq, wl.WORKLOADS[name], dev, stream, args.steps, peak)
        configs = {name: configs[name] for name in CONFIG_WORKLOADS if name in configs}

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "%s cache, f16 MMA operands, f32 accumulate" % w.k_fmt.dtype,
            "data": "synthetic (seeded BF16 N(0,1), K channels x20, sink tokens x10)",
            "config": workload_config(w),
            "spread": spread,
            "tokens_per_s": world * w.batch / step_s,
            "step_tokens_written": int(proto["k"].shape[0]),
            "step_call": ("kvq_write_decode (write fused into the decode launch)" if fused
                          else "kvq_quantize_write + kvq_paged_decode"),
            "two_call_step": {"value": world * step_bytes / two_s / 1e9, "ms_per_step": two_s * 1e3},
            "frac_of_measured_hbm": value / peak, "frac_of_nominal_hbm": value / NOMINAL_HBM_GBS,
            "decode": {"gbs": dec_gbs, "ms": dec_s * 1e3, "bytes": dec_bytes,
                       "frac_of_nominal_hbm": dec_gbs / NOMINAL_HBM_GBS},
            "quant_write": {"gbs": qw_gbs, "ms": qw_s * 1e3, "tokens": ntok,
                            "bytes": float(wl.write_bytes_per_token(w) * ntok), "iterations": qw_iters,
                            "frac_of_measured_hbm": qw_gbs / peak, "frac_of_nominal_hbm": qw_gbs / NOMINAL_HBM_GBS},
            "roofline": {"bound": "hbm", "kernel": "kvq_paged_decode (split + reduce kernels)",
                         "achieved": dec_gbs, "peak": peak, "unit": "GB/s", "frac": dec_gbs / peak,
                         "traffic": recorded_traffic(w.name), "peak_source": peak_src,
                         "algorithmic_bytes": dec_bytes},
            "host_us_per_step_call": host,
            "configs": configs,
            "cpu_baseline": cpu,
            "prefetch": pf,
            "kivi_tail_step": kivi,
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_s * 1e3,
                    "copies": "every step: its inputs host -> device on a copy stream while the previous step "
                              "computes, its output device -> host while the next computes",
                    "serial": {"value": world * step_bytes / e2e_serial_s / 1e9, "ms_per_step": e2e_serial_s * 1e3}},
            # per repeat: the two-call loop (one write launch for the step's
            # few tokens + split + reduce) and, when fused, the fused loop
            # (split + reduce)
            "gpu_launches": (3 + (2 if fused else 0)) * args.steps * args.repeats,
            "clocks": clk,
            "device_errors": errs,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
