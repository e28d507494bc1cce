"""Planted mistakes: each test swaps one oracle function for a copy with one
plausible error (on the CPU, in the oracle only) and checks that at least one
of the oracle's pins fails.  A pin set that let any of these through would
not be pinning the oracle."""
import numpy as np
import pytest

from oracle import attention as oa
from oracle import quantize as oq
from tests import test_oracle_attention as TA
from tests import test_oracle_quantize as TQ


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def _quantize_round_half_away(x, dtype):
    x = np.asarray(x, dtype=np.float32)
    q_max = np.float32(oq.Q_MAX[dtype])
    a = np.max(np.abs(x), axis=-1)
    s = (a / q_max).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (x / s[..., None]).astype(np.float32)
    zero = s == 0
    r = np.where(zero[..., None], np.float32(0.0), r)
    if dtype == oq.FP8:
        codes = oq.e4m3fn_encode(r)
    else:
        codes = np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -q_max, q_max).astype(np.int8)  # mistake
    return np.where(zero[..., None], np.zeros((), codes.dtype), codes), s


def _quantize_reciprocal(x, dtype):
    x = np.asarray(x, dtype=np.float32)
    q_max = np.float32(oq.Q_MAX[dtype])
    a = np.max(np.abs(x), axis=-1)
    s = (a * (np.float32(1) / q_max)).astype(np.float32)   # mistake: a * (1/q_max)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (x / s[..., None]).astype(np.float32)
    zero = s == 0
    r = np.where(zero[..., None], np.float32(0.0), r)
    codes = oq.e4m3fn_encode(r) if dtype == oq.FP8 else np.clip(np.rint(r), -q_max, q_max).astype(np.int8)
    return np.where(zero[..., None], np.zeros((), codes.dtype), codes), s


def test_rounding_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(oq, "quantize_symmetric", _quantize_round_half_away)
    assert _fails(TQ.test_int_ties_round_to_even)


def test_reciprocal_scale_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(oq, "quantize_symmetric", _quantize_reciprocal)
    assert _fails(TQ.test_int_error_bound_and_range, oq.INT8)


def test_qmax_mistake_is_caught(monkeypatch):
    monkeypatch.setitem(oq.Q_MAX, oq.INT8, 128)
    assert _fails(TQ.test_worked_example_int8)
    monkeypatch.setitem(oq.Q_MAX, oq.INT8, 127)
    monkeypatch.setitem(oq.Q_MAX, oq.INT4, 8)
    assert _fails(TQ.test_int_exact_round_trip, oq.INT4)


def test_nibble_order_mistake_is_caught(monkeypatch):
    def swapped(codes):
        c = np.asarray(codes, dtype=np.int8).astype(np.int64) & 0xF
        return (c[..., 1::2] | (c[..., 0::2] << 4)).astype(np.uint8)
    monkeypatch.setattr(oq, "pack_int4", swapped)
    assert _fails(TQ.test_int4_nibble_order_hand_case)


def test_fp8_fnuz_maximum_mistake_is_caught(monkeypatch):
    real = oq.e4m3fn_encode

    def sat240(r):
        r = np.asarray(r, dtype=np.float32)
        return real(np.clip(r, -240, 240))
    monkeypatch.setattr(oq, "e4m3fn_encode", sat240)
    assert _fails(TQ.test_e4m3fn_saturates)
    assert _fails(TQ.test_e4m3fn_encode_decode_round_trip_all_codes)


def test_fp8_truncation_mistake_is_caught(monkeypatch):
    real = oq.e4m3fn_encode

    def toward_zero(r):
        r = np.asarray(r, dtype=np.float32)
        c = real(r)
        back = oq.e4m3fn_decode(c)
        # step one code toward zero wherever rounding went up in magnitude
        up = np.abs(back) > np.abs(r.astype(np.float64))
        return np.where(up & ((c & 0x7F) > 0), c - 1, c).astype(np.uint8)
    monkeypatch.setattr(oq, "e4m3fn_encode", toward_zero)
    assert _fails(TQ.test_e4m3fn_encode_vs_torch_at_ties)


def test_softmax_scale_mistake_is_caught(monkeypatch):
    def by_d(q, k_hat, v_hat):
        n, d = k_hat.shape
        if n == 0:
            return np.zeros(d)
        z = (k_hat @ q) / d                       # mistake: 1/d
        p = np.exp(z - z.max())
        return (p @ v_hat) / p.sum()
    monkeypatch.setattr(oa, "attention_fp64", by_d)
    assert _fails(TA.test_softmax_scale_is_inverse_sqrt_head_dim)
    assert _fails(TA.test_decode_vs_sdpa_exact_inputs, 4, 2)


def test_gqa_mapping_mistake_is_caught(monkeypatch):
    def interleaved(cache, q_bits, block_tables, context_lens):
        q_bits = np.asarray(q_bits, dtype=np.uint16)
        bsz, hq, d = q_bits.shape
        out = np.zeros((bsz, hq, d))
        for b in range(bsz):
            n = int(context_lens[b])
            if n == 0:
                continue
            t = np.arange(n)
            blocks = np.asarray(block_tables[b])[t // cache.block_size]
            kh = oq.dequantize_cache_rows(cache, "k", blocks, t % cache.block_size)
            vh = oq.dequantize_cache_rows(cache, "v", blocks, t % cache.block_size)
            q = oq.bf16_bits_to_f32(q_bits[b]).astype(np.float64)
            for h in range(hq):
                kv = h % cache.num_kv_heads             # mistake: interleaved groups
                out[b, h] = oa.attention_fp64(q[h], kh[:, kv], vh[:, kv])
        return out
    monkeypatch.setattr(oa, "paged_decode_fp64", interleaved)
    assert _fails(TA.test_decode_vs_sdpa_exact_inputs, 16, 2)


def test_scale_row_mistake_is_caught(monkeypatch):
    real = oq.dequantize_cache_rows

    def first_row_scale(cache, which, blocks, offsets):
        # mistake: per-token scales read from the block's row 0
        out = real(cache, which, blocks, offsets)
        if cache.fmt[which].gran != oq.PER_TOKEN_HEAD:
            return out
        blocks = np.asarray(blocks)
        offsets = np.asarray(offsets)
        right = cache.scales[which][blocks, offsets][..., None].astype(np.float64)
        wrong = cache.scales[which][blocks, 0][..., None].astype(np.float64)
        with np.errstate(divide="ignore", invalid="ignore"):
            return np.where(right != 0, out / right * wrong, out)
    monkeypatch.setattr(oa, "dequantize_cache_rows", first_row_scale)
    assert _fails(TA.test_decode_vs_sdpa_exact_inputs, 4, 2)


def test_per_channel_scope_mistake_is_caught(monkeypatch):
    real_write = oq.quantize_write

    def global_channel_scale(cache, k_bits, v_bits, slot_mapping):
        # mistake: one per-channel scale over every token of the call instead
        # of per block
        real_write(cache, k_bits, v_bits, slot_mapping)
        if cache.fmt["k"].gran != oq.PER_BLOCK_CHANNEL:
            return cache
        slots = np.asarray(slot_mapping)
        keep = slots >= 0
        x = oq.bf16_bits_to_f32(np.asarray(k_bits)[keep])
        blk, off = slots[keep] // cache.block_size, slots[keep] % cache.block_size
        xt = np.transpose(x, (1, 2, 0))
        codes, s = oq.quantize_symmetric(xt, oq.INT8)
        cache.codes["k"][blk, off] = np.transpose(codes, (2, 0, 1)).view(np.uint8)
        for b in np.unique(blk):
            cache.scales["k"][b] = s
        return cache
    monkeypatch.setattr(oq, "quantize_write", global_channel_scale)
    assert _fails(TQ.test_per_channel_k)


# ---- the rotation (oracle/rotation.py)
from oracle import rotation as orot  # noqa: E402
from tests import test_oracle_rotation as TR  # noqa: E402


def _fwht_swapped_difference(x):
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    h = 1
    while h < d:
        idx = np.arange(d).reshape(-1, 2 * h)
        lo, hi = idx[:, :h].ravel(), idx[:, h:].ravel()
        a, b = y[..., lo], y[..., hi]
        y[..., lo] = a + b
        y[..., hi] = b - a          # mistake: b - a
        h *= 2
    return y


def _rotate_signs_after(x, sigma):
    return orot.fwht_float32(np.asarray(x, dtype=np.float32)) * np.asarray(sigma, np.float32)  # mistake


def _query_without_division(q, sigma):
    q = np.asarray(q, dtype=np.float64)
    return (q * sigma) @ orot.hadamard(q.shape[-1]).T.astype(np.float64)       # mistake: no / d


def test_butterfly_sign_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(orot, "fwht_float32", _fwht_swapped_difference)
    assert _fails(TR.test_butterfly_equals_the_matrix_on_exact_inputs, 64)


def test_sign_placement_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(orot, "rotate_rows_float32", _rotate_signs_after)
    assert _fails(TR.test_signs_go_before_the_transform, 64)


def test_query_scale_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(orot, "rotate_query_fp64", _query_without_division)
    assert _fails(TR.test_query_rotation_preserves_dot_products_and_output_round_trips, 64)


# ---- INT2 codes and the KIVI full-precision tail
import oracle  # noqa: E402
from oracle import kivi as ok  # noqa: E402
from oracle.attention import _sequence_rows, attention_fp64  # noqa: E402
from tests import test_oracle_kivi as TK  # noqa: E402


def test_int2_crumb_order_mistake_is_caught(monkeypatch):
    def reversed_crumbs(codes):
        c = np.asarray(codes, dtype=np.int8).astype(np.int64) & 0x3
        return (c[..., 3::4] | (c[..., 2::4] << 2) | (c[..., 1::4] << 4) | (c[..., 0::4] << 6)).astype(np.uint8)
    monkeypatch.setattr(oq, "pack_int2", reversed_crumbs)
    assert _fails(TQ.test_int2_packing_hand_case)


def test_int2_qmax_mistake_is_caught(monkeypatch):
    monkeypatch.setitem(oq.Q_MAX, oq.INT2, 2)    # 2^(b-1) instead of 2^(b-1) - 1
    assert _fails(TQ.test_int2_q_max_follows_the_table_rule)
    assert _fails(TQ.test_int2_round_trip_ties_and_bound)


def test_kivi_block_completion_off_by_one_is_caught(monkeypatch):
    def early(cache, res_k, res_v, k_new, v_new, block_tables, context_lens):
        bs = cache.block_size
        for b, n in enumerate(np.asarray(context_lens, dtype=np.int64)):
            if n < 1:
                continue
            res_k[b, (n - 1) % bs] = k_new[b]
            res_v[b, (n - 1) % bs] = v_new[b]
            if n % bs == bs - 1:                      # mistake: one token early
                blk = int(block_tables[b][(n - 1) // bs])
                oq.quantize_write(cache, res_k[b], res_v[b], blk * bs + np.arange(bs))
    monkeypatch.setattr(oracle, "kivi_append", early)
    assert _fails(TK.test_appends_reproduce_whole_block_writes)


def _decode_with(tail_shift=0, ceil_blocks=False):
    def decode(cache, res_k, res_v, q_bits, block_tables, context_lens):
        q_bits = np.asarray(q_bits, dtype=np.uint16)
        bsz, hq, d = q_bits.shape
        bs = cache.block_size
        g = hq // cache.num_kv_heads
        out = np.zeros((bsz, hq, d), dtype=np.float64)
        for b in range(bsz):
            n = int(context_lens[b])
            nq = -(-n // bs) * bs if ceil_blocks else (n // bs) * bs
            nq = min(nq, n) if not ceil_blocks else nq
            blocks, offs = _sequence_rows(cache, block_tables[b], min(nq, n))
            k_hat = oq.dequantize_cache_rows(cache, "k", blocks, offs)
            v_hat = oq.dequantize_cache_rows(cache, "v", blocks, offs)
            tail = (np.arange(min(nq, n), n) + tail_shift) % bs
            k_t = oq.bf16_bits_to_f32(np.asarray(res_k[b])[tail]).astype(np.float64)
            v_t = oq.bf16_bits_to_f32(np.asarray(res_v[b])[tail]).astype(np.float64)
            k_all, v_all = np.concatenate([k_hat, k_t]), np.concatenate([v_hat, v_t])
            q = oq.bf16_bits_to_f32(q_bits[b]).astype(np.float64)
            for h in range(hq):
                out[b, h] = attention_fp64(q[h], k_all[:, h // g, :], v_all[:, h // g, :])
        return out
    return decode


def test_kivi_tail_row_mistake_is_caught(monkeypatch):
    monkeypatch.setattr(oracle, "kivi_decode_fp64", _decode_with(tail_shift=1))   # rows shifted by one
    assert _fails(TK.test_tail_only_is_attention_over_the_bf16_rows)
    assert _fails(TK.test_mixed_case_against_torch_sdpa)


def test_kivi_incomplete_block_read_from_the_cache_is_caught(monkeypatch):
    # mistake: the incomplete block is read from the (never written) cache
    monkeypatch.setattr(oracle, "kivi_decode_fp64", _decode_with(ceil_blocks=True))
    assert _fails(TK.test_mixed_case_against_torch_sdpa)


def test_unmutated_kivi_decode_passes_the_pins(monkeypatch):
    # the restatement above, without a planted mistake, passes: the mutants
    # fail because of their mistakes, not because of the restatement
    assert ok.kivi_decode_fp64 is oracle.kivi_decode_fp64
    monkeypatch.setattr(oracle, "kivi_decode_fp64", _decode_with())
    TK.test_tail_only_is_attention_over_the_bf16_rows()
    TK.test_mixed_case_against_torch_sdpa()


# ---- host-tier block copy
from tests import test_oracle_offload as TO  # noqa: E402


def test_prefetch_index_swap_is_caught(monkeypatch):
    real = oracle.prefetch_blocks

    def swapped(host, dev, src, dst):
        return real(host, dev, dst, src)            # mistake: source and destination ids swapped
    monkeypatch.setattr(oracle, "prefetch_blocks", swapped)
    assert _fails(TO.test_hand_case_and_untouched_slots)


def test_prefetch_scales_left_behind_is_caught(monkeypatch):
    def codes_only(host, dev, src, dst):
        src, dst = np.asarray(src, np.int64), np.asarray(dst, np.int64)
        ok = (src >= 0) & (src < host["k_cache"].shape[0]) & (dst >= 0) & (dst < dev["k_cache"].shape[0])
        for key in ("k_cache", "v_cache"):          # mistake: the scales are not copied
            dev[key][dst[ok]] = host[key][src[ok]]
        return int((~ok).sum())
    monkeypatch.setattr(oracle, "prefetch_blocks", codes_only)
    assert _fails(TO.test_hand_case_and_untouched_slots)
