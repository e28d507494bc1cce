"""CPU oracle for quantize-on-write into a paged KV cache and paged decode
attention over the quantized cache.

THIS PACKAGE IS TEST INFRASTRUCTURE.  It is a plain, slow restatement of what
the pages define, used only by ``tests/``, by ``__graft_entry__.smoke()`` and
by the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py``.  The
product path (``quantized_paged_kv_write_gb300``) never imports it, and it
imports nothing from the product path: the two share no code, tables or
constants.  Only the seeded input generator (``workloads``) feeds both.

Sources, cited by page title and section:

* "Use Less Memory: Quantization and Offloading" (int8ai.com), §2.1 Symmetric
  Quantization Formula and its format table (q_max 127 for INT8, 7 for INT4),
  §2.3 FP8 formats, §5 Exercise 1 (the INT8 worked example) and Exercise 3
  (bytes per token).
* "PidokuInfra 12 KV Cache Quantization", §4 Tiny example (step-time
  arithmetic), §5 "Where the scales live" (cache and scale layout, INT4
  group-32 overhead), "K is more sensitive than V" (per-channel K, per-token
  V), "The kernel side" (dequantize while reading, softmax(q·kᵀ/√d)·V),
  §6-9 (speedup model).
* "Quantized KV caches in production: FP8 vs INT8 vs INT4" (llms.blog),
  "The Mathematics of KV Cache Growth" and "Numerical Formats" (OCP E4M3,
  KIVI per-channel K / per-token V), "PagedAttention and Memory Layouts".
* "KV Cache Quantization" glossary (inferensys.com): symmetric quantization,
  GQA query-head groups sharing one kv head.

Readings where the pages are silent or garbled (each also listed in the
design notes): round = round-half-to-even; scale and quotient in FP32 with
correctly rounded division; E4M3 is the OCP E4M3FN format (max 448, the
pages' "±240" is the E4M3FNUZ maximum); a zero group gets scale +0 and codes
+0; FP8 keeps the sign of a quotient that rounds to zero; INT4 packs element
2j in the low nibble; per-channel K scales cover the tokens written into a
block by one call; GQA maps query head h to kv head h // (H_q / H_kv); the
decode attends to positions [0, context_len) with scale 1/sqrt(head_dim).

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(page values, closed forms, invariants, library routines, brute force).  The
composed decode over a whole paged cache has no worked example on the pages;
its pieces are pinned and the composition is checked against
``torch.nn.functional.scaled_dot_product_attention`` in float64.
"""

from .quantize import (  # noqa: F401
    INT8, INT4, INT2, FP8, PER_TOKEN_HEAD, PER_TOKEN_GROUP, PER_BLOCK_CHANNEL, Q_MAX,
    bf16_bits_to_f32, quantize_symmetric, e4m3fn_encode, e4m3fn_decode,
    pack_int4, unpack_int4, pack_int2, unpack_int2, OracleCache, quantize_write, dequantize_rows,
    dequantize_cache_rows,
)
from .attention import paged_decode_fp64, paged_decode_one_fp64, attention_fp64  # noqa: F401
from . import arithmetic  # noqa: F401
from .offload import prefetch_blocks  # noqa: F401
from .kivi import kivi_append, kivi_decode_fp64  # noqa: F401
from .rotation import (  # noqa: F401
    hadamard, signs_from_words, fwht_float32, rotate_rows_float32, rotate_query_fp64, unrotate_output_fp64,
)
