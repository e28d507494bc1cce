"""Benchmark: quantize-on-write + paged quantized decode attention on GB300.

One step is one serving decode step of the Llama-3-8B-shaped FP8 workload
(batch 27, 32 query heads, 8 kv heads, head_dim 128, block 16, every sequence
at context 32768, FP8 E4M3FN per-(token, kv_head) scales): quantize-write the
step's new token of every sequence into the paged cache, then paged decode
attention over the 32768 cached tokens.  Inputs are seeded synthetic BF16 with
the outlier pattern of the workload (four K channels x20, four sink tokens
x10), generated on the device; the cache is resident in HBM before timing.

value     = algorithmic HBM bytes of a step (codes + scales read, Q, out,
            block tables, the write's BF16 in / codes out) / step time, GB/s
e2e       = the same through the public API with the step's inputs copied
            from pinned host memory and the output copied back, every step
roofline  = the decode call (split + reduce kernels) against the measured
            HBM copy bandwidth
quant_write = the full prefill write (884,736 tokens) timed separately
cpu_baseline = the CPU oracle on a bounded sample of the same step

``--impl reference`` times the CPU oracle as the reference arm (there is no
runnable reference implementation; the oracle is the plain restatement of
the method).  Under torchrun every rank runs its own replica (weak scaling).
"""
from __future__ import annotations

import os

# the CPU oracle legs run single-threaded so that "cores" is what was used
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
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
NOMINAL_HBM_GBS = 7900.0
FALLBACK_HBM_GBS = 6800.0


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
    """Resident cache + the per-step inputs of the serving step."""

    def __init__(self, kvq, w: wl.Workload, device):
        self.kvq, self.w, self.dev = kvq, w, device
        ctx = wl.context_lens(w)
        self.ctx = ctx
        table, nb = wl.block_tables(w)
        self.table_np = table
        self.fmt = kvq.cache_format(w.k_fmt, w.v_fmt, w.num_kv_heads, w.head_dim, nb, w.block_size)
        self.cache = kvq.allocate_cache(self.fmt, device)
        self.tables = torch.as_tensor(table, device=device)
        self.ctx_t = torch.as_tensor(ctx, device=device)
        self.max_ctx = int(ctx.max())
        # prefill: every position but the last of each sequence, one call per
        # sequence; the prefill write is also the quant-write measurement
        self.prefill = []
        for b in range(w.batch):
            k = wl.sequence_kv(w, "k", b, device, int(ctx[b]))
            v = wl.sequence_kv(w, "v", b, device, int(ctx[b]))
            pos = np.arange(ctx[b])
            slots = torch.as_tensor(wl.slot_mapping(table, np.full(ctx[b], b), pos, w.block_size), device=device)
            self.prefill.append((k, v, slots))
        self.pk = torch.cat([p[0] for p in self.prefill])
        self.pv = torch.cat([p[1] for p in self.prefill])
        self.pslots = torch.cat([p[2] for p in self.prefill])
        del self.prefill
        last = self.pslots.new_tensor(np.cumsum(ctx) - 1)
        # the step writes the last position of every sequence
        self.new_k = self.pk[last].contiguous()
        self.new_v = self.pv[last].contiguous()
        self.new_slots = self.pslots[last].contiguous()
        self.q = wl.queries(w, device=device)
        self.out = torch.empty((w.batch, w.num_q_heads, w.head_dim), dtype=torch.float32, device=device)
        nbytes = kvq.kvq_decode_workspace_size(self.fmt, w.batch, w.num_q_heads, self.max_ctx)
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        kvq.kvq_quantize_write(self.pk, self.pv, self.pslots, self.fmt, self.cache)
        torch.cuda.synchronize()

    def write(self):
        self.kvq.kvq_quantize_write(self.new_k, self.new_v, self.new_slots, self.fmt, self.cache)

    def decode(self):
        self.kvq.kvq_paged_decode(self.q, self.fmt, self.cache, self.tables, self.ctx_t, self.max_ctx,
                                  out=self.out, workspace=self.ws)

    def step(self):
        self.write()
        self.decode()

    # algorithmic bytes
    def decode_bytes(self):
        return wl.decode_bytes(self.w, self.ctx, self.table_np.shape[1])

    def write_bytes(self, ntok):
        return wl.write_bytes_per_token(self.w) * ntok

    def step_bytes(self):
        return self.decode_bytes() + self.write_bytes(self.w.batch)


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
def cpu_oracle_step(w: wl.Workload, nseq: int = 2):
    """Run the oracle's quantize-write + decode for `nseq` sequences of the
    workload (all their cached tokens, all query heads).  Returns (bytes,
    seconds) where bytes are the same algorithmic bytes the GPU step counts
    for that many sequences."""
    import oracle
    ctx = wl.context_lens(w)[:nseq]
    sub = wl.scaled(w, batch=nseq, contexts=ctx, name=w.name + "_cpu_sample")
    table, nb = wl.block_tables(sub)
    seqs = np.concatenate([np.full(c, b) for b, c in enumerate(ctx)])
    pos = np.concatenate([np.arange(c) for c in ctx])
    k, v = wl.gather_tokens(sub, seqs, pos)
    slots = wl.slot_mapping(table, seqs, pos, sub.block_size)
    kb = k.view(torch.int16).numpy().view(np.uint16)
    vb = v.view(torch.int16).numpy().view(np.uint16)
    q = wl.queries(sub).view(torch.int16).numpy().view(np.uint16)
    oc = oracle.OracleCache(nb, sub.block_size, sub.num_kv_heads, sub.head_dim, sub.k_fmt, sub.v_fmt)
    last = np.cumsum(ctx) - 1
    rest = np.setdiff1d(np.arange(len(slots)), last)
    oracle.quantize_write(oc, kb[rest], vb[rest], slots[rest])      # cache state (untimed)
    t0 = time.perf_counter()
    oracle.quantize_write(oc, kb[last], vb[last], slots[last])      # the step's write
    oracle.paged_decode_fp64(oc, q, table, ctx)                     # the step's decode
    dt = time.perf_counter() - t0
    nbytes = wl.decode_bytes(sub, ctx, table.shape[1]) + wl.write_bytes_per_token(sub) * nseq
    return nbytes, dt


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


def run_reference(args, w, world, rank):
    """The reference arm: the CPU oracle, timed as it stands."""
    if rank != 0:
        return 0
    for _ in range(args.warmup):
        cpu_oracle_step(w, nseq=1)
    tot_b = tot_t = 0.0
    for _ in range(args.steps):
        b, t = cpu_oracle_step(w, nseq=1)
        tot_b += b
        tot_t += t
    value = tot_b / tot_t / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / max(args.steps, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 quantize / f64 attention",
        "data": "synthetic", "config": workload_config(w, {"sample": "1 of %d sequences per step" % w.batch}),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "quantize-write of 1 token + fp64 decode of 1 sequence (32 q heads, "
                                   "full context) per step"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama3_8b_fp8", choices=list(wl.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=None,
                    help="fewer sequences of the same shape (profiling captures only)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    w = wl.WORKLOADS[args.workload]
    if args.batch is not None and args.batch != w.batch:
        w = wl.scaled(w, batch=args.batch, contexts=wl.context_lens(w)[: args.batch],
                      name=f"{w.name}_batch{args.batch}")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, w, world, rank)

    import quantized_paged_kv_write_gb300 as kvq
    from quantized_paged_kv_write_gb300 import build
    build.build()
    kvq.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    peak, peak_src = measured_hbm_peak()

    st = Step(kvq, w, dev)
    kvq.kvq_device_errors(clear=True)
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()

    # ---- timed region: K steps, per-call events for the decode
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_begin = time.time()
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
    t_end = time.time()
    barrier(world)
    step_s = max_over_ranks(e0.elapsed_time(e1) / 1e3 / args.steps, world, dev)
    dec_s = statistics.mean(a.elapsed_time(b) for a, b in ev) / 1e3
    clk = clocks.stop(t_begin, t_end)
    errs = kvq.kvq_device_errors(clear=True)

    step_bytes = st.step_bytes()
    value = world * step_bytes / step_s / 1e9
    dec_bytes = st.decode_bytes()
    dec_gbs = dec_bytes / dec_s / 1e9

    # ---- quantize-write of the whole prefill (884,736 tokens), separately
    qw_iters = max(3, min(20, args.steps // 50))
    for _ in range(2):
        kvq.kvq_quantize_write(st.pk, st.pv, st.pslots, st.fmt, st.cache)
    qw_s = timed(lambda: kvq.kvq_quantize_write(st.pk, st.pv, st.pslots, st.fmt, st.cache), qw_iters, stream)
    qw_s /= qw_iters
    ntok = int(st.pslots.numel())
    qw_gbs = st.write_bytes(ntok) / qw_s / 1e9

    # ---- end to end through the public API with host buffers
    e2e_steps = max(3, min(200, args.steps // 10))
    h_in = {n: getattr(st, n).cpu().pin_memory() for n in ("new_k", "new_v", "new_slots", "q")}
    h_tables = st.tables.cpu().pin_memory()
    h_ctx = st.ctx_t.cpu().pin_memory()
    h_out = torch.empty(st.out.shape, dtype=torch.float32).pin_memory()
    d_in = {n: torch.empty_like(getattr(st, n)) for n in h_in}
    d_tables = torch.empty_like(st.tables)
    d_ctx = torch.empty_like(st.ctx_t)
    h2d = sum(t.numel() * t.element_size() for t in h_in.values()) + h_tables.numel() * 4 + h_ctx.numel() * 4
    d2h = h_out.numel() * 4

    def e2e_step():
        for n in h_in:
            d_in[n].copy_(h_in[n], non_blocking=True)
        d_tables.copy_(h_tables, non_blocking=True)
        d_ctx.copy_(h_ctx, non_blocking=True)
        kvq.kvq_quantize_write(d_in["new_k"], d_in["new_v"], d_in["new_slots"], st.fmt, st.cache)
        kvq.kvq_paged_decode(d_in["q"], st.fmt, st.cache, d_tables, d_ctx, st.max_ctx, out=st.out,
                             workspace=st.ws)
        h_out.copy_(st.out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    e2e_s = max_over_ranks(timed(e2e_step, e2e_steps, stream) / e2e_steps, world, dev)
    e2e_val = world * step_bytes / e2e_s / 1e9

    # ---- CPU oracle baseline (rank 0, N = 1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b_, t_ = cpu_oracle_step(w, nseq=1)
        cpu = {"value": b_ / t_ / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": "quantize-write of 1 new token + fp64 decode of 1 of the 27 sequences "
                         "(32 query heads, 32768 tokens), %.1f s" % t_}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": step_s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "%s cache, f16 MMA operands, f32 accumulate" % w.k_fmt.dtype,
            "data": "synthetic (seeded BF16 N(0,1), K channels x20, sink tokens x10)",
            "config": workload_config(w),
            "tokens_per_s": world * w.batch / step_s,
            "frac_of_measured_hbm": value / peak, "frac_of_nominal_hbm": value / NOMINAL_HBM_GBS,
            "decode": {"gbs": dec_gbs, "ms": dec_s * 1e3, "bytes": dec_bytes,
                       "kv_tokens_per_s": float(st.ctx.sum()) / dec_s},
            "quant_write": {"gbs": qw_gbs, "ms": qw_s * 1e3, "tokens": ntok, "bytes": st.write_bytes(ntok),
                            "frac_of_measured_hbm": qw_gbs / peak, "frac_of_nominal_hbm": qw_gbs / NOMINAL_HBM_GBS},
            "roofline": {"bound": "hbm", "kernel": "kvq_paged_decode (split + reduce kernels)",
                         "achieved": dec_gbs, "peak": peak, "unit": "GB/s", "frac": dec_gbs / peak,
                         "traffic": None, "peak_source": peak_src},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_s * 1e3},
            "gpu_launches": 3 * args.steps,
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
