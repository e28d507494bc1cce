"""Pins of the oracle's byte and step-time arithmetic against the numbers the
pages print (tests/golden/page_arithmetic.json, each entry with its source),
and of the bench's byte accounting against the oracle's."""
import json
import os

import numpy as np
import pytest

from oracle import arithmetic as ar
import workloads as wl

with open(os.path.join(os.path.dirname(__file__), "golden", "page_arithmetic.json")) as _f:
    GOLDEN = json.load(_f)
GiB = 1024 ** 3


def test_llama3_8b_bytes_per_token():
    g = GOLDEN["llama3_8b"]
    L, H, d = g["layers"], g["kv_heads"], g["head_dim"]
    assert ar.kv_bytes_per_token(L, H, d, 2) == g["bytes_per_token"]["fp16"]
    assert ar.kv_bytes_per_token(L, H, d, 1) == g["bytes_per_token"]["fp8_int8"]
    assert ar.kv_bytes_per_token(L, H, d, 0.5) == g["bytes_per_token"]["int4"]
    assert ar.kv_bytes_per_token(1, H, d, 1) == g["bytes_per_token_per_layer_fp8"]
    for key, b in (("fp16", 2), ("fp8_int8", 1), ("int4", 0.5)):
        per_req = ar.kv_bytes_per_sequence(L, H, d, b, 16384) / GiB
        assert per_req == g["per_request_16k_gib"][key]
        assert 16 * per_req == g["sixteen_requests_gib"][key]
    assert 4 * GiB / ar.kv_bytes_per_token(L, H, d, 1) == g["active_window_tokens_in_4gib_fp8"]


def test_h100_step_model():
    g = GOLDEN["h100_step_model"]
    L, H, d, n = 32, 8, 128, g["context"]
    per = {k: ar.kv_bytes_per_sequence(L, H, d, b, n) for k, b in
           (("fp16", 2), ("fp8", 1), ("int4", 0.5))}
    for k in per:
        assert abs(per[k] / 1e9 - g["per_sequence_gb"][k]) < 0.006
        assert ar.max_sequences(g["budget_gb"] * 1e9, per[k]) == g["max_sequences"][k]
    seqs = g["max_sequences"]
    for k in ("fp8", "int4"):
        assert abs(seqs[k] / seqs["fp16"] - g["concurrency_gain_printed"][k]) < 0.05
    read = {k: seqs[k] * per[k] for k in ("fp16", "fp8")}
    for k in read:
        assert abs(read[k] / 1e9 - g["step_kv_read_gb"][k]) < 0.05
    # both printed step times imply the same bandwidth, ~3.35 TB/s
    bw = [(read[k] + g["weights_gb"] * 1e9) / (g["step_ms"][k] * 1e-3) for k in ("fp16", "fp8")]
    assert abs(bw[0] - bw[1]) / bw[0] < 0.005 and abs(bw[0] / 1e12 - 3.35) < 0.01
    for k in ("fp16", "fp8"):
        t = ar.decode_step_seconds(read[k], g["weights_gb"] * 1e9, 3.35e12)
        assert abs(t * 1e3 - g["step_ms"][k]) < 0.05
    # throughput gain: (27 / 22.1 ms) / (13 / 21.4 ms) = 2.01; the page prints
    # 2.05 (its text calls the step times "about the same")
    gain = (seqs["fp8"] / g["step_ms"]["fp8"]) / (seqs["fp16"] / g["step_ms"]["fp16"])
    assert abs(gain - g["throughput_gain_printed"]) < 0.05


def test_speedup_model():
    g = GOLDEN["speedup_model"]
    for ctx, want in zip(g["contexts"], g["speedup_printed"]):
        kv16 = g["batch"] * ar.kv_bytes_per_sequence(32, 8, 128, 2, ctx)
        s = ar.kv_quantization_speedup(g["weights_gb"] * 1e9, kv16)
        assert abs(s - want) < 0.015, (ctx, s, want)


def test_scale_overhead():
    g = GOLDEN["scale_overhead"]
    assert abs(100 * ar.per_token_scale_overhead(128, 1, 2) - g["int8_head_dim_128_overhead_percent_printed"]) < 0.05
    assert ar.int4_grouped_vector_bytes(128, 32, 2) == g["int4_group32_vector_bytes"]
    assert abs(256 / ar.int4_grouped_vector_bytes(128, 32, 2) - g["int4_group32_compression_printed"]) < 0.07
    # with the FP32 scales this build stores: 3.125% and 80 B
    assert ar.per_token_scale_overhead(128, 1, 4) == 0.03125
    assert ar.int4_grouped_vector_bytes(128, 32, 4) == 80


def test_llama3_70b_bytes_per_token():
    g = GOLDEN["llama3_70b"]
    # the page labels 160 KB "16-bit"; the formula gives 160 KiB at 1 byte per
    # element and twice that at 2 bytes (the page's later 64k / 8-request
    # figures follow from its own 160 KB)
    one_byte = ar.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], 1)
    assert one_byte == g["bytes_per_token_printed_kb"] * 1024
    assert ar.kv_bytes_per_token(g["layers"], g["kv_heads"], g["head_dim"], 2) == 327680
    per_req = one_byte * 65536 / 1e9
    assert abs(per_req - g["single_64k_request_gb_printed"]) < 1.0
    assert abs(8 * g["single_64k_request_gb_printed"] - g["eight_requests_gb_printed"]) == 0


def test_bench_byte_accounting_matches_page_formula():
    # the decode bytes the bench divides by follow the pages' per-token
    # formula, one layer, plus scales
    w = wl.WORKLOADS["llama3_8b_fp8"]
    per_tok_codes = ar.kv_bytes_per_token(1, w.num_kv_heads, w.head_dim, 1)
    assert wl.kv_read_bytes_per_token(w) == per_tok_codes + 2 * 4 * w.num_kv_heads
    w3 = wl.WORKLOADS["llama3_70b_kivi"]
    assert wl.kv_read_bytes_per_token(w3) == (
        ar.kv_bytes_per_token(1, 8, 128, 1) / 2 + ar.kv_bytes_per_token(1, 8, 128, 0.5) / 2
        + 8 * 128 * 4 / 16 + 8 * 4 * 4)
    assert wl.kv_read_bytes_per_token(wl.WORKLOADS["long_mixed"]) == 1696
    assert wl.kv_read_bytes_per_token(w3) == 1920
