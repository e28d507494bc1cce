"""Host-side legs of bench.py on CPU: the oracle timing helpers and the
reference arm's JSON line (the CUDA arm needs a GPU and is exercised by the
GPU runs)."""
import io
import json
from contextlib import redirect_stdout

import workloads as wl
import bench


def test_cpu_baseline_runs_one_worker_per_core_until_the_time_floor():
    w = wl.WORKLOADS["tiny_int8"]
    cb = bench.cpu_baseline(w, min_seconds=0.05, workers=2)
    assert cb["kind"] == "oracle" and cb["unit"] == "GB/s"
    assert cb["value"] > 0 and cb["cores"] == 2
    assert "round(s)" in cb["sample"] and "2 worker processes" in cb["sample"]


def test_oracle_pool_workers_hold_distinct_sequences():
    w = wl.WORKLOADS["tiny_int8"]
    pool = bench.OraclePool(w, workers=2)
    try:
        b1, t1, _ = pool.round()
        b2, t2, _ = pool.round(16)
    finally:
        pool.close()
    # tiny_int8 has contexts {37, 100}: the two workers hold one each
    one = [bench.OracleSample(w, i) for i in range(2)]
    assert b1 == sum(s.step()[0] for s in one)
    assert b2 == sum(s.step(16)[0] for s in one)
    assert t1 > 0 and t2 > 0


def test_host_cores_is_the_affinity_count():
    import os
    assert bench.host_cores() == len(os.sched_getaffinity(0))


def test_oracle_sample_counts_the_prefix_bytes():
    w = wl.WORKLOADS["tiny_int8"]
    smp = bench.OracleSample(w)
    b_full, t_full, _ = smp.step()
    b_pref, t_pref, _ = smp.step(16)
    assert t_full > 0 and t_pref > 0
    assert b_pref < b_full
    assert "16 of its" in smp.describe(16)


def test_reference_arm_prints_one_contract_line():
    class Args:
        steps, warmup, gpus = 3, 1, 1
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.run_reference(Args(), wl.WORKLOADS["tiny_int8"], 1, 0, workers=2)
    assert rc == 0
    lines = [ln for ln in buf.getvalue().splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["kind"] == "oracle"
    assert d["cpu_baseline"]["cores"] == 2
    assert d["metric"] == bench.METRIC
