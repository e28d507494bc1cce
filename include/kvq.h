/*
 * kvq.h -- C ABI of libkvq: quantize-on-write into a paged KV cache and paged
 * decode attention that dequantizes while reading, for NVIDIA GB300 (sm_103a).
 *
 * What is computed (cited by page title and section):
 *
 *   Quantize-on-write.  "Use Less Memory: Quantization and Offloading", §2.1
 *   Symmetric Quantization Formula and §5 Exercise 1: for each scale group
 *   s = max|x| / q_max and x_q = clip(round(x / s), -q_max, q_max), with
 *   q_max = 127 (INT8), 7 (INT4), 1 (INT2, the same rule 2^(b-1) - 1 for the
 *   2-bit codes of KIVI, "Quantized KV caches in production", Numerical
 *   Formats); FP8 stores x / s as OCP E4M3FN (largest
 *   finite 448, so s = max|x| / 448), rounded to nearest even and saturated.
 *   The cache and scale layout is the one of "PidokuInfra 12 KV Cache
 *   Quantization", §5 Where the scales live:
 *       codes  [num_blocks, block_size, num_kv_heads, head_dim]  (INT4: head_dim/2, INT2: head_dim/4 bytes)
 *       scales [num_blocks, block_size, num_kv_heads]            FP32, one per (token, kv_head)
 *   with two further granularities from the same page ("K is more sensitive
 *   than V": per-channel K, per-token V; group-32 INT4 scales):
 *       grouped scales     [num_blocks, block_size, num_kv_heads, head_dim/group]
 *       per-channel scales [num_blocks, num_kv_heads, head_dim]  (K only)
 *
 *   Paged decode.  "PidokuInfra 12", §5 The kernel side: for every KV block
 *   the reader loads codes and scales, dequantizes (x_hat = x_q * s) and forms
 *   q·kᵀ; the output is softmax(q·kᵀ / sqrt(head_dim)) · V over positions
 *   [0, context_len) of the sequence, blocks found through its block table
 *   (PagedAttention, "Quantized KV caches in production").  Query head h
 *   reads kv head h / (num_q_heads / num_kv_heads) (GQA, "KV Cache
 *   Quantization" glossary).
 *
 * Numerical contract.  Quantization: BF16 input widened to FP32 exactly,
 * absmax in FP32; s and every x / s are equal, bit for bit, to the IEEE
 * correctly rounded FP32 quotients (the kernels reach those bits without a
 * division per element: the scale by one FMA residual correction of
 * RN(absmax * RN(1 / q_max)), proven for every BF16 absmax; each quotient
 * by Markstein's correction step from RN(1 / s) and two FMAs, with IEEE
 * division for scales below 2^-82), then round-half-to-even and clip
 * (INT) or saturating RNE to E4M3FN.  A group with absmax 0 stores s = +0
 * and codes 0.  FP8 keeps the sign of a quotient that rounds to zero (0x80).
 * INT4 codes are two's complement nibbles, element 2j in the low nibble of
 * byte j; INT2 codes are two's complement 2-bit fields, element 4j + m in
 * bits 2m .. 2m + 1 of byte j.  Decode: q is BF16, codes are dequantized
 * exactly, products accumulate in FP32; out is FP32.  Inputs must be finite.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, contiguous
 *     row-major in the shapes given; BF16 tensors are passed as raw 16-bit
 *     words.  Pointers must be 16-byte aligned.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without waiting for it.
 *   - The library allocates no device memory.  It keeps one 32-bit sticky
 *     error word per device (a __device__ variable) that kernels set when
 *     they meet invalid device-side data; read it with kvq_device_errors().
 *   - Return value: KVQ_OK or a negative kvq_status found on the host before
 *     anything is enqueued (nothing is written on error).
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kvq_stream_t; /* same type as cudaStream_t */

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = -1, /* null pointer, negative size, misaligned pointer */
  KVQ_ERR_UNSUPPORTED = -2, /* format, head_dim, block_size or GQA ratio not built */
  KVQ_ERR_WORKSPACE = -3,   /* workspace smaller than kvq_decode_workspace_size() */
  KVQ_ERR_CUDA = -4         /* a CUDA runtime/driver call failed (launch, attribute) */
} kvq_status;

typedef enum { KVQ_INT8 = 0, KVQ_INT4 = 1, KVQ_FP8_E4M3FN = 2, KVQ_INT2 = 3 } kvq_dtype;

typedef enum {
  KVQ_PER_TOKEN_HEAD = 0,   /* scale [num_blocks, block_size, H_kv]                 */
  KVQ_PER_TOKEN_GROUP = 1,  /* scale [num_blocks, block_size, H_kv, head_dim/group] */
  KVQ_PER_BLOCK_CHANNEL = 2 /* scale [num_blocks, H_kv, head_dim] (K only)          */
} kvq_gran;

/* Rotation of the cached rows ("Quantized KV caches in production: FP8 vs
 * INT8 vs INT4", Numerical Formats: randomized orthogonal Walsh-Hadamard
 * transforms spread outlier peaks over all channels before 4-bit
 * quantization).  With KVQ_ROT_HADAMARD every K and V row x is stored as the
 * quantization of y = H (sigma * x): H the Sylvester Hadamard matrix of order
 * head_dim (entry (i, j) = (-1)^popcount(i & j), unnormalized), sigma the
 * format's random signs, y computed in FP32 by the radix-2 butterfly with
 * stages 1, 2, 4, ... (each (a, b) -> (a + b, a - b), rounded to nearest).
 * Scales are then RN(max|y| / q_max).  The decode returns the same attention
 * as for the unrotated rows: it uses H (sigma * q) / head_dim as the query
 * and rotates the output back, sigma * (H o) / head_dim. */
typedef enum { KVQ_ROT_NONE = 0, KVQ_ROT_HADAMARD = 1 } kvq_rotation;

/* Sticky device error bits (kvq_device_errors). */
enum {
  KVQ_DEVERR_SLOT_RANGE = 1u << 0,    /* slot_mapping[t] >= num_blocks * block_size      */
  KVQ_DEVERR_BLOCK_RANGE = 1u << 1,   /* block table entry outside [0, num_blocks)       */
  KVQ_DEVERR_CONTEXT_RANGE = 1u << 2, /* context_len < 0 or > max_blocks_per_seq * bs
                                         or > max_context_len                             */
  KVQ_DEVERR_TIMEOUT = 1u << 3,       /* a bounded wait on an mbarrier ran out           */
  KVQ_DEVERR_CHANNEL_RUN = 1u << 4    /* per-channel K: a run of tokens into a block does
                                         not fill the block's rows from row 0 in order
                                         (see kvq_quantize_write)                         */
};

/* Layout of one layer's paged cache.  Supported combinations:
 *   K: INT8, FP8 or INT4 with PER_TOKEN_HEAD, or INT8 or INT2 with
 *      PER_BLOCK_CHANNEL;
 *   V: INT8 or FP8 with PER_TOKEN_HEAD, or INT4 or INT2 with PER_TOKEN_GROUP,
 *      group 32;
 *   head_dim 64 or 128 (128 with an INT2 tensor); block_size 16;
 *   1 <= num_kv_heads <= 8.
 * INT2 codes (KIVI's 2-bit codes, "Quantized KV caches in production",
 * Numerical Formats; q_max 1 by the rule of the format table, 2^(b-1) - 1)
 * are two's complement, channel 4j + m in bits 2m .. 2m + 1 of byte j.
 * INT4 codes (q_max 7, half a byte each: "Use Less Memory: Quantization and
 * Offloading", §2.1 format table) are two's complement nibbles, channel 2j in
 * the low nibble of byte j of the row (the pages fix no nibble order). */
typedef struct {
  int32_t k_dtype, v_dtype; /* kvq_dtype */
  int32_t k_gran, v_gran;   /* kvq_gran */
  int32_t k_group, v_group; /* channels per scale for PER_TOKEN_GROUP, else ignored */
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t rotation; /* kvq_rotation; KVQ_ROT_HADAMARD needs per-token K */
  int64_t num_blocks;
  uint32_t rotation_signs[4]; /* KVQ_ROT_HADAMARD: bit c % 32 of word c / 32
                                 set means sigma_c = -1 (c < head_dim) */
} kvq_format;

typedef struct {
  void *k_cache; /* uint8 codes, layout above */
  void *v_cache;
} kvq_caches;

typedef struct {
  float *k_scale; /* FP32 scales, layout by granularity above */
  float *v_scale;
} kvq_scales;

/*
 * kvq_quantize_write -- quantize num_tokens new K and V vectors and store the
 * codes and scales at their paged slots.
 *
 *   k_bf16, v_bf16  [num_tokens, num_kv_heads, head_dim] BF16 (read only)
 *   slot_mapping    [num_tokens] int64: slot = physical_block * block_size +
 *                   offset; a negative slot skips the token (padding)
 *   fmt, caches, scales  the cache (written in place)
 *
 * Per-(token, head) and grouped scales depend only on the token.  With
 * PER_BLOCK_CHANNEL K, the scale of (block, head, channel) is the absmax
 * over the tokens THIS CALL writes into that block, divided by q_max (127 for
 * INT8, 1 for INT2); the call overwrites the block's K scales, so a block
 * must receive all its tokens in one call, as one run of adjacent entries of
 * slot_mapping (a prefill or a chunk of it that starts on a block boundary).
 * The kernel checks this run by run: a run (a maximal sequence of adjacent
 * tokens whose slots fall in one block) must write the block's rows 0, 1,
 * 2, ... in order.  A run that starts past row 0 (the block's earlier rows
 * came from another run or another call) or skips a row sets
 * KVQ_DEVERR_CHANNEL_RUN; its codes and scales are still written, scaled
 * over the run's own tokens, so the block's other rows no longer match its
 * scales.  (Two runs that both start at row 0 of one block are duplicate
 * slots, below.)  Rows of a block that the call does not write are left
 * untouched (one token per step into a per-channel K cache goes through
 * kvq_kivi_append instead).
 * Duplicate slots within one call race (unspecified winner).
 * Out-of-range slots set KVQ_DEVERR_SLOT_RANGE and are skipped.
 * num_tokens == 0 is a no-op.
 */
int kvq_quantize_write(const void *k_bf16, const void *v_bf16, const int64_t *slot_mapping,
                       int64_t num_tokens, const kvq_format *fmt, kvq_caches caches,
                       kvq_scales scales, kvq_stream_t stream);

/*
 * kvq_decode_workspace_size -- bytes of device workspace kvq_paged_decode
 * needs for this shape on the CURRENT device (it depends on the SM count).
 * The workspace holds split-K partial softmax states; the caller allocates
 * it (any 256-byte aligned device buffer) and may reuse it across calls on
 * one stream.  Returns KVQ_OK and writes *bytes, or an error status.
 */
int kvq_decode_workspace_size(const kvq_format *fmt, int32_t batch, int32_t num_q_heads,
                              int32_t max_context_len, size_t *bytes);

/*
 * kvq_paged_decode -- one decode step of attention for `batch` sequences.
 *
 *   q_bf16        [batch, num_q_heads, head_dim] BF16
 *   block_tables  [batch, max_blocks_per_seq] int32 physical block ids
 *   context_lens  [batch] int32, tokens attended per sequence (0 -> out = 0)
 *   max_context_len  host-side upper bound of context_lens (sizes the work
 *                 split; a larger device value sets KVQ_DEVERR_CONTEXT_RANGE
 *                 and that sequence's output is left 0)
 *   out           [batch, num_q_heads, head_dim] FP32 (written)
 *   workspace     device buffer of at least kvq_decode_workspace_size() bytes
 *
 * num_q_heads must be a multiple of num_kv_heads with ratio 1..8.
 * Block ids outside [0, num_blocks) set KVQ_DEVERR_BLOCK_RANGE; the
 * offending block is skipped.  batch == 0 is a no-op.
 */
int kvq_paged_decode(const void *q_bf16, int32_t batch, int32_t num_q_heads,
                     const kvq_format *fmt, kvq_caches caches, kvq_scales scales,
                     const int32_t *block_tables, int32_t max_blocks_per_seq,
                     const int32_t *context_lens, int32_t max_context_len, float *out,
                     void *workspace, size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_write_decode -- one decode step with the step's new tokens written in
 * the same launch: for every sequence b with context_lens[b] = n >= 1, the
 * token at position n - 1 (K and V rows k_new_bf16[b], v_new_bf16[b]) is
 * quantized into its slot table[b][(n - 1) / 16] * 16 + (n - 1) % 16
 * exactly as kvq_quantize_write would, and the decode then attends over
 * [0, n) including it.  Results (cache bytes, scales and out) equal those of
 * kvq_quantize_write on those slots followed by kvq_paged_decode.  Passages:
 * "Use Less Memory: Quantization and Offloading", §2.1 (quantize on write)
 * and "PidokuInfra 12 KV Cache Quantization", §5 The kernel side (dequantize
 * on read); the fusion itself is this library's.
 *
 *   k_new_bf16, v_new_bf16  [batch, num_kv_heads, head_dim] BF16, 16-byte
 *                 aligned, caller-owned device memory (read only)
 *   other arguments as kvq_paged_decode (same workspace size)
 *
 * K must be per-(token, head) (INT8, FP8 or INT4): per-channel K blocks take
 * no appends here (KVQ_ERR_UNSUPPORTED; see kvq_kivi_append).  The block holding the new token must not be
 * referenced by another sequence of the same call (it is written while the
 * call reads the cache).  A block id outside [0, num_blocks) sets
 * KVQ_DEVERR_BLOCK_RANGE and that token is not written.
 */
int kvq_write_decode(const void *q_bf16, const void *k_new_bf16, const void *v_new_bf16,
                     int32_t batch, int32_t num_q_heads, const kvq_format *fmt,
                     kvq_caches caches, kvq_scales scales, const int32_t *block_tables,
                     int32_t max_blocks_per_seq, const int32_t *context_lens,
                     int32_t max_context_len, float *out, void *workspace,
                     size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_kivi_append / kvq_kivi_decode -- a per-channel K cache that takes one
 * token per sequence and step ("Quantized KV caches in production", Numerical
 * Formats: KIVI, K per channel and V per token; a per-channel scale spans a
 * block's tokens, "PidokuInfra 12 KV Cache Quantization", K is more
 * sensitive than V).  The tokens of a sequence's last, incomplete block stay
 * in full precision in a caller-owned residual: res_k_bf16, res_v_bf16 BF16
 * [batch, 16, num_kv_heads, head_dim], row p % 16 for position p.
 *
 * kvq_kivi_append: context_lens[b] = n >= 1 is the length after this step's
 * token (k_new_bf16 / v_new_bf16 [batch, num_kv_heads, head_dim] BF16), which
 * goes to residual row (n - 1) % 16; when n % 16 == 0 the block's 16 rows are
 * quantized into block table[b][(n - 1) / 16] exactly as kvq_quantize_write
 * would write those 16 tokens in one call (per-channel K over them, V per its
 * format).  n == 0 skips the sequence.  Errors as kvq_quantize_write (block
 * ids) and kvq_paged_decode (context lengths).
 *
 * kvq_kivi_decode: as kvq_paged_decode over the complete blocks
 * [0, 16 floor(n / 16)) of the cache, plus the residual rows of the tail
 * [16 floor(n / 16), n) in full precision (merged by the split-reduce in
 * FP32).  Same workspace as kvq_paged_decode.
 *
 * Both need K INT8 or INT2 with KVQ_PER_BLOCK_CHANNEL (else
 * KVQ_ERR_UNSUPPORTED).
 * A prefill writes its complete blocks with kvq_quantize_write and copies
 * the rows of its incomplete block into the residual.
 */
int kvq_kivi_append(const void *k_new_bf16, const void *v_new_bf16, int32_t batch,
                    const kvq_format *fmt, kvq_caches caches, kvq_scales scales,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, void *res_k_bf16, void *res_v_bf16,
                    kvq_stream_t stream);
int kvq_kivi_decode(const void *q_bf16, int32_t batch, int32_t num_q_heads,
                    const kvq_format *fmt, kvq_caches caches, kvq_scales scales,
                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                    const int32_t *context_lens, int32_t max_context_len,
                    const void *res_k_bf16, const void *res_v_bf16, float *out, void *workspace,
                    size_t workspace_bytes, kvq_stream_t stream);

/*
 * kvq_prefetch_blocks -- copy offloaded cache blocks from a pool in pinned
 * host memory into device block slots ("Use Less Memory: Quantization and
 * Offloading", §3 The Three-Tier Memory Hierarchy and §4 Pipelining and
 * Latency Overlap: while one step computes, the blocks the next step needs
 * move into a second set of GPU buffers).
 *
 *   fmt          the device cache's format; the host pool has the same
 *                per-block layout with host_num_blocks blocks
 *   host_caches, host_scales  the host pool: pinned (page-locked) host
 *                memory, 16-byte aligned, read only
 *   src_blocks, dst_blocks  [num_pairs] int32 device arrays: host block
 *                src_blocks[i] goes to device block slot dst_blocks[i]
 *                (codes and scales, byte for byte)
 *   caches, scales  the device cache (written)
 *
 * One kernel on `stream` gathers all pairs over the CPU-GPU link; run it on
 * its own stream to overlap a decode on another (the caller orders the two
 * with events, double-buffering the slots).  Pairs with an index outside
 * either pool set KVQ_DEVERR_BLOCK_RANGE and are skipped.  Host memory that
 * is not pinned is rejected with KVQ_ERR_INVALID_ARG.  num_pairs == 0 is a
 * no-op.
 */
int kvq_prefetch_blocks(const kvq_format *fmt, kvq_caches host_caches, kvq_scales host_scales,
                        int64_t host_num_blocks, const int32_t *src_blocks,
                        const int32_t *dst_blocks, int32_t num_pairs, kvq_caches caches,
                        kvq_scales scales, kvq_stream_t stream);

/*
 * kvq_device_errors -- synchronize `stream`, then return the sticky device
 * error bits of the current device in *bits_out; clear them if `clear` != 0.
 */
int kvq_device_errors(uint32_t *bits_out, int32_t clear, kvq_stream_t stream);

/* Human-readable text of a kvq_status (static storage). */
const char *kvq_status_string(int32_t status);

/*
 * kvq_paged_decode_noalloc -- kvq_paged_decode for callers that cannot
 * allocate device memory at the call (for example code hosted by an engine
 * or plugin framework that owns all device memory, or a serving loop that
 * must not take the allocator's locks).  The pages have no counterpart of
 * this call: it only changes where the split-K scratch lives.
 *
 * Same arguments and results as kvq_paged_decode, without the workspace.
 * The scratch is one static device array of KVQ_NOALLOC_SCRATCH_BYTES that
 * every GPU which loads the library holds until the process exits.  A shape
 * whose workspace (kvq_decode_workspace_size) is larger is rejected with
 * KVQ_ERR_WORKSPACE before anything is enqueued.  The call allocates
 * nothing.  Its first call on a device looks up the array's device address
 * (set-up done once per device, with that device current); make that first
 * call before any stream capture.  All calls share the array: calls whose
 * work overlaps on the GPU (e.g. on two streams at once) race on it and must
 * be ordered by the caller.  Nothing in it needs to start at zero.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (32u << 20)
int kvq_paged_decode_noalloc(const void *q_bf16, int32_t batch, int32_t num_q_heads,
                             const kvq_format *fmt, kvq_caches caches, kvq_scales scales,
                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                             const int32_t *context_lens, int32_t max_context_len, float *out,
                             kvq_stream_t stream);

/* Library version, e.g. 110 for 0.1.10. */
int32_t kvq_version(void);

/* Identity of the sources this library was built from: a hash over every
 * file of the kernel source directory and this header, fixed at build time
 * (static storage; "unknown" when the build did not set it).  Lets a caller
 * check that the loaded library matches the sources it was given. */
const char *kvq_build_id(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
