// Paged decode attention over the quantized cache (sm_103a): split kernel and
// split-reduce kernel.  Included by the per-format translation units.
//
// What it computes: "PidokuInfra 12 KV Cache Quantization", §5 The kernel
// side -- for every KV block, load the codes and scales, dequantize in
// registers (x_hat = x_q * s, "Use Less Memory", §2.1), form q·kᵀ, and return
// softmax(q·kᵀ / sqrt(d)) · V ("PidokuInfra 12", K is more sensitive than V);
// blocks come from the sequence's block table (PagedAttention, "Quantized KV
// caches in production"); query head h reads kv head h / G (GQA, "KV Cache
// Quantization" glossary).
//
// Work split.  All cached blocks of the batch form one global list (sequence
// by sequence, through the block tables).  CTA c of P takes the contiguous
// range [c*T/P, (c+1)*T/P), so every CTA streams the same number of blocks
// whatever the context mix; a CTA that crosses a sequence boundary emits one
// partial softmax state per sequence piece.  Partial (b, c) lives in workspace
// slot b + c, which is collision free because the CTAs covering sequence b+1
// start at or after the last CTA covering b.  The reduce kernel merges the
// partials of each (sequence, query head) with the usual max/sum rescaling.
//
// Per CTA: one producer warp and one consumer warp per kv head.  The producer
// walks the CTA's blocks, looks up block ids, and issues per-head TMA tile
// loads of the K and V codes (a 16 x row_bytes box of the 4-D cache tensor,
// written with the 128/64/32-byte swizzle) plus 1-D bulk copies of the
// block's scales, into a ring of NS shared-memory stages guarded by
// full/empty mbarriers.  Consumer warp h turns its head's codes into exact
// f16 values in registers and runs both contractions on the tensor cores
// (mma.sync m16n8k16, FP32 accumulate):
//
//   S   = Q' K^T : M = 16 rows (8 query-row slots, high and low f16 parts of
//                  q, or of q * s_c for per-channel K), N = 8 tokens, K = d.
//   O^T = V^T P'': M = 16 channels, N = 8 columns (P'' high/low parts),
//                  K = 16 tokens.  P'' = p * s_v * 2^F, split into f16
//                  high + low parts, so the V scales are exact to ~22 bits.
//
// The f16 forms of the codes are exact (|INT8| <= 127, INT4 <= 7, every
// E4M3 value), q is exact as an f16 pair after a power-of-two row scaling,
// so the only roundings are FP32 accumulation, exp2 and the ~2^-22 of the
// high/low splits.  The S accumulator fragment is re-used as the P fragment
// of the PV product (same thread owns the same tokens), so scores never
// leave registers.
#pragma once

#include <type_traits>

#include "common.cuh"
#include "kvq_internal.h"
#include "quantize_rows.cuh"

namespace kvq {

constexpr int kMaxHeadsPerCta = 8;  // one consumer warp per kv head
constexpr int kDecodeMaxRegs = 96;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kNoScale = 1 << 20;   // "no V scale seen yet" exponent sentinel
// Cap on the V exponent F so that 2^F is one normal float; it only binds for
// V scales below 2^-87, whose contributions sit far under any output ulp.
constexpr int kMaxVExp = 100;
// Online softmax: the running maximum m is raised only when a score exceeds it
// by more than this (log2 units), so a probability exp2(z - m) is at most 2
// and P'' = p s_v 2^F stays below 2^15, inside the f16 range.
constexpr float kLazyMax = 1.0f;
// While F is unset, any positive V scale (the smallest subnormal and up) sets it.
constexpr float kVThr0 = 0x1p-149f;

template <int D, int KF, int VF>
struct DecodeTraits {
  static constexpr int BS = kBlockSize;
  static constexpr bool KINT4 = (KF == K_INT4_TOK);
  static constexpr bool KINT2 = (KF == K_INT2_CHAN);
  static constexpr int KROW = KINT4 ? D / 2 : (KINT2 ? D / 4 : D);  // K code bytes per row
  static constexpr int VROW = (VF == V_INT4_G32) ? D / 2 : (VF == V_INT2_G32 ? D / 4 : D);
  static constexpr int KBOX = BS * KROW;
  static constexpr int VBOX = BS * VROW;
  static constexpr int NKS = D / 16;                              // QK k-steps
  static constexpr int NKG = NKS / 4;                             // 16-byte K loads per row
  static constexpr int NCH = D / 32;                              // 32-channel PV chunks
  static constexpr bool KCHAN = (KF == K_INT8_CHAN || KF == K_INT2_CHAN);
  // INT2 per-channel K: with q_max = 1 a channel scale is the channel's BF16
  // absmax, so s_c 2^eb is exact in f16 and the scales go into the K
  // operand (one f16 multiply per pair) instead of into a per-block Q'
  static constexpr bool KSCL = (KF == K_INT2_CHAN);
  static constexpr bool KFP8 = (KF == K_FP8_TOK);
  static constexpr bool VINT4 = (VF == V_INT4_G32);
  static constexpr bool VINT2 = (VF == V_INT2_G32);
  static constexpr bool VGRP = VINT4 || VINT2;                    // group-32 V scales
  static constexpr bool VFP8 = (VF == V_FP8_TOK);
  static constexpr int VGROUPS = VGRP ? D / 32 : 1;               // V scales per (token, head)
  // Four group scales per (token, head) (16 bytes): each head's [16 tokens][4]
  // scales arrive by a TMA tile load, head-major in shared memory, so the four
  // lanes of a row slot (consecutive tokens) read different banks.  The
  // cache's own [token][head][group] order puts every token's scales for one
  // head in the same four banks.
  static constexpr bool VS_TMA = (VGROUPS == 4);

  // byte layout of one pipeline stage (H kv heads)
  __host__ __device__ static constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }
  __host__ __device__ static uint32_t kc_off(int) { return 0; }
  __host__ __device__ static uint32_t vc_off(int H) { return align1k(H * KBOX); }
  __host__ __device__ static uint32_t ks_off(int H) { return vc_off(H) + H * VBOX; }
  __host__ __device__ static uint32_t ks_bytes(int H) { return KCHAN ? H * D * 4 : BS * H * 4; }
  __host__ __device__ static uint32_t vs_off(int H) { return (ks_off(H) + ks_bytes(H) + 127u) & ~127u; }
  __host__ __device__ static uint32_t vs_bytes(int H) { return BS * H * VGROUPS * 4; }
  __host__ __device__ static uint32_t stage_bytes(int H) { return align1k(vs_off(H) + vs_bytes(H)); }
  // After the stages: each head's query staging, D / 16 units of 8 bytes
  // per (row slot, lane-in-row), unit-major, with 8 row slots in the wide
  // layout and 4 in the packed one (per-channel K: the row-scaled BF16
  // query; per-token K: the f16 Q' fragments); then, for per-channel K, the
  // block's scaled channel scales (D floats per head).
  __host__ __device__ static constexpr uint32_t qst_unit(bool wide) { return wide ? 256u : 128u; }
  __host__ __device__ static uint32_t qst_bytes(bool wide) { return NKS * qst_unit(wide); }
  // Staged query units of 16 bytes (high part, low part or zero, for both
  // pairs) load as one MMA operand fragment with no register moves: the
  // rotated cache (real low parts), 2-bit per-channel K and per-token K with
  // group-scaled V.  FP8 / INT8 per-token V keep 8-byte units (high parts
  // only): their larger stages would lose a pipeline stage to the extra
  // staging.
  __host__ __device__ static constexpr bool q_wide_units(bool rot) { return rot || KSCL || (!KCHAN && VGRP); }
  __host__ __device__ static uint32_t aux_bytes(int H, bool wide, bool rot) {
    return H * (qst_bytes(wide) * (q_wide_units(rot) ? 2u : 1u) + (KCHAN ? D * 4 : 0));
  }
  __host__ __device__ static uint32_t tx_bytes(int H) {
    return H * (KBOX + VBOX) + ks_bytes(H) + vs_bytes(H);
  }
};

// Token permutation inside an 8-token MMA tile: row slot r of the B operand
// reads token PI(r).  With the 128-byte swizzle this keeps every 16-byte
// shared load of K and every 4-byte load of V free of bank conflicts.
__device__ __forceinline__ int PI(int r) { return (r >> 1) | ((r & 1) << 2); }

// x * 2^e for |e| up to ~250, exact when the result is a normal float.
__device__ __forceinline__ float scale_pow2(float x, int e) {
  const int e1 = e / 2;
  return x * pow2i(e1) * pow2i(e - e1);
}

// floor(log2(x)) for finite x > 0 (subnormals included).
__device__ __forceinline__ int ilog2f(float x) {
  const int bits = __float_as_int(x);
  const int ex = (bits >> 23) & 0xFF;
  if (ex != 0) return ex - 127;
  return -127 - __clz(bits & 0x7FFFFF) + 9;  // subnormal: 2^-149 * mantissa
}

// Last index b in [0, B) with cum[b] <= g (cum non-decreasing, g < cum[B]).
__device__ __forceinline__ int seq_of(const int *cum, int B, int g) {
  int lo = 0, hi = B;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cum[mid] <= g) lo = mid; else hi = mid;
  }
  return lo;
}

// ---------------------------------------------------------------------------
// code -> f16 conversions (exact)
// ---------------------------------------------------------------------------
// K: one 32-bit word = 4 channels of one token -> (ch0, ch1), (ch2, ch3).
template <bool FP8>
__device__ __forceinline__ void k_word_to_f16(uint32_t w, uint32_t &b0, uint32_t &b1) {
  if constexpr (FP8) {
    e4m3x4_to_f16x2x2(w, b0, b1);
  } else {
    // 0x64 00 | (code ^ 0x80) is the f16 value 1024 + code + 128
    const uint32_t u = w ^ 0x80808080u;
    b0 = hsub2_u32(prmt(u, 0x64646464u, 0x4140u), 0x64806480u);
    b1 = hsub2_u32(prmt(u, 0x64646464u, 0x4342u), 0x64806480u);
  }
}

// 8-bit INT K, channels 0..3 of one token in w -> pairs (ch0, ch2), (ch1,
// ch3): byte ^ 0x80 under the f16 exponent of 1024 (one LOP3 per pair) is
// 1152 + code, and one subtract removes the offset.
__device__ __forceinline__ void k_int8_word_to_f16_02_13(uint32_t w, uint32_t &b02, uint32_t &b13) {
  b02 = hsub2_u32(and_xor(w, 0x00FF00FFu, 0x64806480u), 0x64806480u);
  b13 = hsub2_u32(and_xor(shr8_mul(w), 0x00FF00FFu, 0x64806480u), 0x64806480u);
}

// INT4 K: 16-bit word = 4 channels of one token (channel 2j in the low nibble
// of byte j) -> (ch0, ch1), (ch2, ch3).  Each byte is copied into both f16
// halves; the low half keeps the low nibble, the high half the high one
// (times 16), each XORed with 8 under the f16 exponent of 1024, and one FMA
// per pair removes the offsets: lo - 1032, hi / 16 - 72.
__device__ __forceinline__ void k_nibbles_to_f16(uint32_t h, uint32_t &b0, uint32_t &b1) {
  const uint32_t t0 = prmt(h, 0u, 0x4040u);  // byte 0 in both halves
  const uint32_t t1 = prmt(h, 0u, 0x4141u);  // byte 1 in both halves
  b0 = hfma2_u32(and_xor(t0, 0x00F0000Fu, 0x64806408u), 0x2C003C00u, 0xD480E408u);
  b1 = hfma2_u32(and_xor(t1, 0x00F0000Fu, 0x64806408u), 0x2C003C00u, 0xD480E408u);
}

// INT2 K: byte ss of w = 4 channels of one token (channel m in bits 2m, 2m+1)
// -> (ch0, ch1), (ch2, ch3).  The byte is copied into both f16 halves; each
// half keeps one 2-bit field (XOR 2) under the exponent of 1024 and one FMA
// per pair scales it down and removes the offset.
template <int SS>
__device__ __forceinline__ void k_crumbs_to_f16(uint32_t w, uint32_t &b0, uint32_t &b1) {
  const uint32_t t = prmt(w, 0u, 0x4040u | SS | (SS << 8));
  b0 = hfma2_u32(and_xor(t, 0x000C0003u, 0x64086402u), 0x34003C00u, 0xDC08E402u);
  b1 = hfma2_u32(and_xor(t, 0x00C00030u, 0x64806420u), 0x24002C00u, 0xCC80D420u);
}

// INT2 V: bytes of tokens ta and tb (4 channels each) -> p[k] =
// f16x2(code[ta][k], code[tb][k]).
__device__ __forceinline__ void v_crumbs_to_f16(uint32_t ha, uint32_t hb, uint32_t (&p)[4]) {
  const uint32_t u = prmt(ha, hb, 0x5410u);  // ta in the low half, tb in the high half
  p[0] = hfma2_u32(and_xor(u, 0x00030003u, 0x64026402u), 0x3C003C00u, 0xE402E402u);
  p[1] = hfma2_u32(and_xor(u, 0x000C000Cu, 0x64086408u), 0x34003400u, 0xDC08DC08u);
  p[2] = hfma2_u32(and_xor(u, 0x00300030u, 0x64206420u), 0x2C002C00u, 0xD420D420u);
  p[3] = hfma2_u32(and_xor(u, 0x00C000C0u, 0x64806480u), 0x24002400u, 0xCC80CC80u);
}

// 8-bit V: words of tokens ta and tb (same 4 channels) -> pairs
// (ta, tb) for channels 0..3: p[k] = f16x2(code[ta][k], code[tb][k]).
template <bool FP8>
__device__ __forceinline__ void v_words_to_f16(uint32_t wa, uint32_t wb, uint32_t (&p)[4]) {
  const uint32_t x = prmt(wa, wb, 0x5140u);  // a0 b0 a1 b1
  const uint32_t y = prmt(wa, wb, 0x7362u);  // a2 b2 a3 b3
  if constexpr (FP8) {
    e4m3x4_to_f16x2x2(x, p[0], p[1]);
    e4m3x4_to_f16x2x2(y, p[2], p[3]);
  } else {
    const uint32_t xu = x ^ 0x80808080u, yu = y ^ 0x80808080u;
    p[0] = hsub2_u32(prmt(xu, 0x64646464u, 0x4140u), 0x64806480u);
    p[1] = hsub2_u32(prmt(xu, 0x64646464u, 0x4342u), 0x64806480u);
    p[2] = hsub2_u32(prmt(yu, 0x64646464u, 0x4140u), 0x64806480u);
    p[3] = hsub2_u32(prmt(yu, 0x64646464u, 0x4342u), 0x64806480u);
  }
}

// 8-bit V from a transposed ldmatrix register: bytes (ta c, ta c+1, tb c,
// tb c+1) -> lo = f16x2(code[ta][c], code[tb][c]), hi = the same for c + 1.
template <bool FP8>
__device__ __forceinline__ void v_byte_pairs_to_f16(uint32_t x, uint32_t &lo, uint32_t &hi) {
  if constexpr (FP8) {
    e4m3x4_to_f16x2x2(prmt(x, x, 0x3120u), lo, hi);
  } else {
    // 0x64 00 | (code ^ 0x80) is the f16 value 1024 + code + 128
    const uint32_t u = x ^ 0x80808080u;
    lo = hsub2_u32(prmt(u, 0x64646464u, 0x4240u), 0x64806480u);
    hi = hsub2_u32(prmt(u, 0x64646464u, 0x4341u), 0x64806480u);
  }
}

// INT4 V: the 16-bit words of tokens ta (low half of u) and tb (high half),
// 4 nibbles = channels 0..3 each -> p[k] = f16x2(code[ta][k], code[tb][k]).
__device__ __forceinline__ void v_nibble_pairs_to_f16(uint32_t u, uint32_t (&p)[4]) {
  const uint32_t u8 = shr8_mul(u);
  // nibble n ^ 8 in the f16 mantissa: 0x6400 | (n ^ 8) = 1024 + (n ^ 8)
  p[0] = hsub2_u32(and_xor(u, 0x000F000Fu, 0x64086408u), 0x64086408u);
  p[2] = hsub2_u32(and_xor(u8, 0x000F000Fu, 0x64086408u), 0x64086408u);
  // nibble in bits 4..7: 1024 + 16 (n ^ 8); x / 16 - 72 = (n ^ 8) - 8
  p[1] = hfma2_u32(and_xor(u, 0x00F000F0u, 0x64806480u), 0x2C002C00u, 0xD480D480u);
  p[3] = hfma2_u32(and_xor(u8, 0x00F000F0u, 0x64806480u), 0x2C002C00u, 0xD480D480u);
}

__device__ __forceinline__ void v_nibbles_to_f16(uint32_t ha, uint32_t hb, uint32_t (&p)[4]) {
  v_nibble_pairs_to_f16(prmt(ha, hb, 0x5410u), p);
}

// ---------------------------------------------------------------------------
// fused write: the step's new token of each sequence whose last block this
// CTA reads is quantized here, before any of the CTA's TMA loads
// ---------------------------------------------------------------------------
// Sequence b's last block (global index cum[b + 1] - 1) belongs to exactly one
// CTA's range, and that CTA is the only reader of it in this launch, so the
// owner writes token ctx_b - 1 (slot table[b][(ctx_b - 1) / 16] * 16 +
// (ctx_b - 1) % 16) with the row quantizer of the quantize-write kernel, then
// fences its generic-proxy writes against the async proxy; the caller's
// barrier follows.  Per-token K only (per-channel K blocks take no appends).
template <int D, int KF, int VF, int HT, bool ROT>
__device__ void fused_write_new_tokens(const DecodeArgs &a, const int *cum, int g0, int g1, int H, int warp,
                                       int nwarps) {
  constexpr int KDT = (KF == K_FP8_TOK) ? KVQ_FP8_E4M3FN : (KF == K_INT4_TOK ? KVQ_INT4 : KVQ_INT8);
  constexpr int VDT = (VF == V_FP8_TOK) ? KVQ_FP8_E4M3FN
                      : (VF == V_INT4_G32 ? KVQ_INT4 : (VF == V_INT2_G32 ? KVQ_INT2 : KVQ_INT8));
  constexpr int VGROUP = (VF == V_INT4_G32 || VF == V_INT2_G32) ? 32 : D;
  const int lane = threadIdx.x & 31;
  const int b0 = seq_of(cum, a.B, g0), b1 = seq_of(cum, a.B, g1 - 1);
  for (int b = b0 + warp; b <= b1; b += nwarps) {
    const int last = cum[b + 1] - 1;  // empty sequences: last < cum[b]
    if (last < cum[b] || last < g0 || last >= g1) continue;
    const int t = __ldg(a.ctx + b) - 1;  // >= 0: the sequence has blocks
    const int blk = __ldg(a.tables + static_cast<int64_t>(b) * a.max_blocks + t / kBlockSize);
    if (blk < 0 || blk >= a.num_blocks) {
      if (lane == 0) set_error(a.err, KVQ_DEVERR_BLOCK_RANGE);
      continue;
    }
    const int64_t sl = static_cast<int64_t>(blk) * kBlockSize + t % kBlockSize;
    const int64_t row0 = static_cast<int64_t>(b) * H * (D / 8);
    uint4 v[TokenRows<D>::NST];
    load_token_rows<D, HT>(reinterpret_cast<const uint4 *>(a.knew) + row0, H, v);
    quantize_loaded_token<D, KDT, D, HT, ROT>(v, sl, H, a.kc_w, a.ks_w, a.rot_signs);
    load_token_rows<D, HT>(reinterpret_cast<const uint4 *>(a.vnew) + row0, H, v);
    quantize_loaded_token<D, VDT, VGROUP, HT, ROT>(v, sl, H, a.vc_w, a.vs_w, a.rot_signs);
  }
  fence_proxy_async_global();
}

// ---------------------------------------------------------------------------
// the split kernel
// ---------------------------------------------------------------------------
// Two CTAs of 9 warps per SM need <= 96 registers per thread (an SM
// sub-partition holds 16K registers and receives up to 5 of the 18 warps).
// HT > 0 fixes the number of kv heads at compile time (every shared-memory
// offset then folds into an immediate); HT == 0 reads it from the arguments.
// ROT: rotated cache (per-token K only): the query is rotated and its low
// f16 parts staged too.
template <int D, int KF, int VF, bool WIDE, int HT, bool ROT>
__global__ void __maxnreg__(kDecodeMaxRegs)
    decode_split_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap smap,
                        const DecodeArgs a, const int nstages) {
  using T = DecodeTraits<D, KF, VF>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int H = HT > 0 ? HT : a.H;
  const int B = a.B;
  const uint32_t SB = T::stage_bytes(H);
  constexpr bool rot = ROT && !T::KCHAN;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + nstages * SB + T::aux_bytes(H, WIDE, rot));
  uint64_t *empty = full + nstages;
  int *info = reinterpret_cast<int *>(empty + nstages);
  int *cum = info + nstages;  // [B + 1]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], H);
    }
    mbar_init_fence();
  }
  // block counts per sequence (invalid contexts count as empty)
  if (warp == 0) {
    int carry = 0;
    if (lane == 0) cum[0] = 0;
    for (int base = 0; base < B; base += 32) {
      const int b = base + lane;
      int nb = 0;
      if (b < B) {
        const int ctx = __ldg(a.ctx + b);
        // with a full-precision tail only the complete blocks are cached and
        // need block table entries
        const bool tail = a.res_k != nullptr;
        const bool bad = ctx < 0 || (tail ? ctx / kBlockSize > a.max_blocks : ctx > a.max_blocks * kBlockSize) ||
                         ctx > a.max_ctx;
        if (bad && blockIdx.x == 0) set_error(a.err, KVQ_DEVERR_CONTEXT_RANGE);
        nb = bad ? 0 : (tail ? ctx / kBlockSize : (ctx + kBlockSize - 1) / kBlockSize);
      }
      int v = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      if (b < B) cum[b + 1] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();

  const int total = cum[B];
  const int P = a.nctas;
  const int c = blockIdx.x;
  const int g0 = static_cast<int>((static_cast<int64_t>(c) * total) / P);
  const int g1 = static_cast<int>((static_cast<int64_t>(c + 1) * total) / P);
  if (c == 0) {
    // the reduce kernel reads the prefix sums from the workspace
    for (int k = threadIdx.x; k <= B; k += blockDim.x) a.ws_cum[k] = cum[k];
  }
  if (g0 >= g1) return;
  if constexpr (!T::KCHAN) {
    if (a.knew != nullptr) {
      fused_write_new_tokens<D, KF, VF, HT, ROT>(a, cum, g0, g1, H, warp, H + 1);
      __syncthreads();
    }
  }

  if (warp == H) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&kmap);
      prefetch_tensormap(&vmap);
      if constexpr (T::VS_TMA) prefetch_tensormap(&smap);
    }
    const uint32_t tx = T::tx_bytes(H);
    int issued = 0;
    bool abort = false;
    int stage = 0;        // ring position of iteration `issued`
    uint32_t ph = 0;      // its phase parity
    for (int base = g0; base < g1 && !abort; base += 32) {
      const int gl = base + lane;
      int phys = -1;
      if (gl < g1) {
        const int bl = seq_of(cum, B, gl);
        phys = __ldg(a.tables + static_cast<int64_t>(bl) * a.max_blocks + (gl - cum[bl]));
      }
      const int n = min(32, g1 - base);
      for (int k = 0; k < n; ++k) {
        if (!__all_sync(0xffffffffu, mbar_wait(&empty[stage], ph ^ 1))) {
          if (lane == 0) set_error(a.err, KVQ_DEVERR_TIMEOUT);
          abort = true;
          break;
        }
        const int pb = __shfl_sync(0xffffffffu, phys, k);
        const bool valid = pb >= 0 && pb < a.num_blocks;
        uint8_t *st = smem + stage * SB;
        if (lane == 0) info[stage] = valid ? pb : -1;
        if (valid) {
          if (lane == 0) mbar_arrive_expect_tx(&full[stage], tx);
          __syncwarp();
          if (lane < H) {
            tma_load_4d(st + T::kc_off(H) + lane * T::KBOX, &kmap, 0, lane, 0, pb, &full[stage]);
            tma_load_4d(st + T::vc_off(H) + lane * T::VBOX, &vmap, 0, lane, 0, pb, &full[stage]);
            if constexpr (T::VS_TMA)
              tma_load_4d(st + T::vs_off(H) + lane * (kBlockSize * 16), &smap, 0, lane, 0, pb, &full[stage]);
          } else if (lane == 16) {
            const int64_t ksrc = static_cast<int64_t>(pb) * (T::ks_bytes(H) / 4);
            bulk_g2s(st + T::ks_off(H), a.ks + ksrc, T::ks_bytes(H), &full[stage]);
          } else if (!T::VS_TMA && lane == 17) {
            const int64_t vsrc = static_cast<int64_t>(pb) * (T::vs_bytes(H) / 4);
            bulk_g2s(st + T::vs_off(H), a.vs + vsrc, T::vs_bytes(H), &full[stage]);
          }
        } else if (lane == 0) {
          set_error(a.err, KVQ_DEVERR_BLOCK_RANGE);
          mbar_arrive(&full[stage]);
        }
        ++issued;
        if (++stage == nstages) {
          stage = 0;
          ph ^= 1;
        }
      }
    }
    // drain: the CTA must not exit with copies in flight
    const int first = issued > nstages ? issued - nstages : 0;
    for (int it = first; it < issued; ++it) {
      if (!__all_sync(0xffffffffu, mbar_wait(&full[it % nstages], (it / nstages) & 1))) {
        if (lane == 0) set_error(a.err, KVQ_DEVERR_TIMEOUT);
        break;
      }
    }
    return;
  }
  if (warp > H) return;

  // -------------------------------------------------------------- consumers
  const int h = warp;
  const int G = a.G;
  const int r = lane >> 2;  // row slot / channel row / B column
  const int i = lane & 3;   // k-slot group
  // row slot r: which query head of the group, and whether it carries the
  // high or the low f16 part of P'' in the PV product (packed layout, G <= 4:
  // columns [0, G) high, [G, 2G) low; wide layout: every column g = r is
  // multiplied twice, once with the high and once with the low part)
  const bool active = WIDE ? (r < G) : (r < 2 * G);
  const int gq = active ? (WIDE ? r : r % G) : 0;
  const bool lo_role = !WIDE && active && r >= G;

  // tokens this thread owns in S / P: n-tile 0 columns 2i, 2i+1 and n-tile 1
  int tk[4];
  tk[0] = i;        // PI(2i)
  tk[1] = i + 4;    // PI(2i + 1)
  tk[2] = i + 8;
  tk[3] = i + 12;

  uint32_t qraw[T::NKG][8];   // raw BF16 q (per-channel K rebuilds Q' per block)
  float o[T::NCH][2][4];      // O^T accumulators
  float m = -INFINITY, l = 0.f, rowscale = 0.f;
  // scores are formed relative to m (z - m in one FMA: mneg = -m); before the
  // first block of a piece m is -inf, mneg 0 and every score passes zth
  float mneg = 0.f, zth = -INFINITY;
  int F = kNoScale;
  float pf = 1.f;  // 2^F
  // packed layout: 2^F, or 0 for inactive row slots (their P'' is zero)
  float pfa = (WIDE || active) ? 1.f : 0.f;
  float vthr = kVThr0;  // V scales at or above this move F
  const float inv_sqrt_d = rsqrtf(static_cast<float>(D));

  // The query side of S lives in shared memory, not in registers (which the
  // O accumulators and the V path need).  Per-token K: the f16 Q' fragments,
  // written once per sequence piece.  Per-channel K (KIVI): the row-scaled
  // query as f16 (INT8 codes: pairs (c, c + 2), (c + 1, c + 3)), from which
  // the Q' fragments are rebuilt inside every block's S product.  This lane's D / 8 values (K-step order) form D / 16 units of
  // 8 bytes, unit u at qst + QU u, conflict free (a rotated cache stores the
  // high and low f16 parts of a unit side by side, 16 bytes, which load as
  // one S operand fragment: units at qst + 2 QU u).  In the packed layout row
  // slots r and r + G carry the same query and read one staged row; inactive
  // row slots read a zero row.  The block's scaled channel scales s' sit in
  // the head's D-float area (INT8 codes: per 4-channel unit the f16 pairs
  // s_h (c, c + 2), s_h (c + 1, c + 3), s_l (c, c + 2), s_l (c + 1, c + 3))
  // with 16-byte unit k stored at k ^ ((k >> 3) & 1), so the four lanes of a
  // row slot read four different bank groups.
  constexpr uint32_t QU = T::qst_unit(WIDE);
  const int srow = WIDE ? r : (active ? gq : G);  // G <= 3 when a row is inactive
  const bool qwriter = WIDE || r < G || r == 2 * G;
  constexpr bool Q2 = T::q_wide_units(rot);
  constexpr uint32_t QS = Q2 ? 2 * QU : QU;  // unit stride of this lane's staged query
  const uint32_t qst =
      smem_u32(smem + nstages * SB) + (Q2 ? 2u : 1u) * (h * T::qst_bytes(WIDE) + 8 * (4 * srow + i));
  uint32_t sw0 = 0, sw1 = 0, sown = 0, kcs0 = 0;
  int er = 0;  // row pre-scale exponent
  // per-channel K: the block exponent eb in use, as 2^eb, and the scale bit
  // patterns that end it (8-bit codes: some s 2^eb at or above 2^8, or every
  // s 2^eb below 2^3; 2-bit codes: 2^15 and 2^10)
  float fbk = 1.f;
  uint32_t ebhi = 0u, eblo = 0u;
  if constexpr (T::KSCL) {
    // f16 scales s' of channels 4 lane .. + 3 at byte 8 lane; the lanes of
    // row slot r read channels 16 (i + 4 kg) + 4 ss .. + 3 at sw0 + 128 kg + 8 ss
    const uint32_t sst = smem_u32(smem + nstages * SB) + (Q2 ? 2u : 1u) * H * T::qst_bytes(WIDE) + h * (D * 4);
    sw0 = sst + 32 * i;
    sown = sst + 8 * lane;
    kcs0 = smem_u32(smem + T::ks_off(H)) + h * (D * 4) + 16 * lane;
  } else if constexpr (T::KCHAN) {
    const uint32_t sst = smem_u32(smem + nstages * SB) + (Q2 ? 2u : 1u) * H * T::qst_bytes(WIDE) + h * (D * 4);
    sw0 = sst + 64 * i + 16 * (i >> 1);        // units with ss even
    sw1 = sst + 64 * i + 16 * ((i >> 1) ^ 1);  // units with ss odd
    sown = sst + 16 * (lane ^ ((lane >> 3) & 1));
    kcs0 = smem_u32(smem + T::ks_off(H)) + h * (D * 4) + 16 * lane;
  }

  // per-token K: Q' = q fragments with a power-of-two row scaling; returns
  // the exponent by which the staged values exceed the query (with a
  // rotated cache, the staged values are H (sigma q) 2^e and the query is
  // H (sigma q) / d, so log2 d is added)
  auto build_q = [&]() -> int {
    float qs[T::NKG][16];
#pragma unroll
    for (int kg = 0; kg < T::NKG; ++kg) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        qs[kg][2 * e] = bf16lo_to_f32(qraw[kg][e]);
        qs[kg][2 * e + 1] = bf16hi_to_f32(qraw[kg][e]);
      }
    }
    if constexpr (rot) {
      // H (sigma q) over the row's D channels: this lane holds the 16-channel
      // chunks i + 4 kg; stages 1..8 inside a chunk, 16 and 32 across the
      // row's lanes (chunk i xor 1, 2), 64 between the lane's two chunks
#pragma unroll
      for (int kg = 0; kg < T::NKG; ++kg) {
        const int ci = i + 4 * kg;
        const uint32_t sb = (a.rot_signs[ci >> 1] >> (16 * (ci & 1))) & 0xFFFFu;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          qs[kg][c] = __uint_as_float(__float_as_uint(qs[kg][c]) ^ (((sb >> c) & 1u) << 31));
#pragma unroll
        for (int hh = 1; hh < 16; hh <<= 1)
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (!(c & hh)) {
              const float x = qs[kg][c], y = qs[kg][c + hh];
              qs[kg][c] = x + y;
              qs[kg][c + hh] = x - y;
            }
#pragma unroll
        for (int m = 1; m < 4; m <<= 1) {
          const bool upper = (i & m) != 0;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float p = __shfl_xor_sync(0xffffffffu, qs[kg][c], m);
            qs[kg][c] = upper ? p - qs[kg][c] : qs[kg][c] + p;
          }
        }
      }
      if constexpr (T::NKG == 2) {
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float x = qs[0][c], y = qs[1][c];
          qs[0][c] = x + y;
          qs[1][c] = x - y;
        }
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int kg = 0; kg < T::NKG; ++kg)
#pragma unroll
      for (int c = 0; c < 16; ++c) amax = fmaxf(amax, fabsf(qs[kg][c]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const int e = (amax > 0.f) ? 14 - ilog2f(amax) : 0;
#pragma unroll
    for (int kg = 0; kg < T::NKG; ++kg) {
#pragma unroll
      for (int ss = 0; ss < 4; ++ss) {
        if constexpr (rot) {
          // rotated q carries up to 24 bits: high and low f16 parts
          uint32_t h01, l01, h23, l23;
          split_f16x2(scale_pow2(qs[kg][4 * ss], e), scale_pow2(qs[kg][4 * ss + 1], e), h01, l01);
          split_f16x2(scale_pow2(qs[kg][4 * ss + 2], e), scale_pow2(qs[kg][4 * ss + 3], e), h23, l23);
          if (qwriter)
            sts128(qst + QS * (4 * kg + ss), active ? h01 : 0u, active ? l01 : 0u, active ? h23 : 0u,
                   active ? l23 : 0u);
        } else {
          // BF16 q times 2^e is exact in f16 down to 2^-32 of the row maximum
          // (8 significant bits); the low parts (rows r + 8) are zero
          const uint32_t h01 = f32x2_to_f16x2(scale_pow2(qs[kg][4 * ss], e), scale_pow2(qs[kg][4 * ss + 1], e));
          const uint32_t h23 = f32x2_to_f16x2(scale_pow2(qs[kg][4 * ss + 2], e), scale_pow2(qs[kg][4 * ss + 3], e));
          if (qwriter) {
            if constexpr (Q2)
              sts128(qst + QS * (4 * kg + ss), active ? h01 : 0u, 0u, active ? h23 : 0u, 0u);
            else
              sts64(qst + QU * (4 * kg + ss), active ? h01 : 0u, active ? h23 : 0u);
          }
        }
      }
    }
    return rot ? e + ((D == 128) ? 7 : 6) : e;
  };

  auto start_segment = [&](int b) {
    const uint16_t *qrow = a.q + (static_cast<int64_t>(b) * a.Hq + h * G + gq) * D;
#pragma unroll
    for (int kg = 0; kg < T::NKG; ++kg) {
      const uint4 *p = reinterpret_cast<const uint4 *>(qrow + 16 * (i + 4 * kg));
      const uint4 z4 = make_uint4(0u, 0u, 0u, 0u);
      const uint4 w0 = active ? __ldg(p) : z4, w1 = active ? __ldg(p + 1) : z4;
      qraw[kg][0] = w0.x; qraw[kg][1] = w0.y; qraw[kg][2] = w0.z; qraw[kg][3] = w0.w;
      qraw[kg][4] = w1.x; qraw[kg][5] = w1.y; qraw[kg][6] = w1.z; qraw[kg][7] = w1.w;
    }
    if constexpr (T::KCHAN && !T::KSCL) {
      // Scale each row by 2^er so that its max |q| falls in [2^6, 2^7); the
      // block's channel scales are brought below 2^8, so every product
      // q~ s' stays below 2^15 (f16 range).  The staged values are f16,
      // exact for BF16 q down to 2^-17 (8 significant bits), as the pairs
      // (c, c + 2) and (c + 1, c + 3) of each 4-channel unit: the order in
      // which the 8-bit K codes convert (k_int8_word_to_f16_02_13).
      float rmax = 0.f;
#pragma unroll
      for (int kg = 0; kg < T::NKG; ++kg)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          rmax = fmaxf(rmax, fmaxf(fabsf(bf16lo_to_f32(qraw[kg][e])), fabsf(bf16hi_to_f32(qraw[kg][e]))));
      rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, 1));
      rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, 2));
      er = (rmax > 0.f) ? 6 - ilog2f(rmax) : 0;
      ebhi = 0u;  // the piece's first block sets eb and the row scale
      __syncwarp();  // the previous piece's last block has read the staging
#pragma unroll
      for (int kg = 0; kg < T::NKG; ++kg)
#pragma unroll
        for (int ss = 0; ss < 4; ++ss) {
          const uint32_t v0 = qraw[kg][2 * ss], v1 = qraw[kg][2 * ss + 1];  // (c0, c1), (c2, c3)
          const float q0 = scale_pow2(bf16lo_to_f32(v0), er), q1 = scale_pow2(bf16hi_to_f32(v0), er);
          const float q2 = scale_pow2(bf16lo_to_f32(v1), er), q3 = scale_pow2(bf16hi_to_f32(v1), er);
          if (qwriter) sts64(qst + QU * (4 * kg + ss), f32x2_to_f16x2(q0, q2), f32x2_to_f16x2(q1, q3));
        }
      __syncwarp();
    } else {
      __syncwarp();  // the previous piece's last block has read the staging
      const int e = build_q();
      __syncwarp();
      rowscale = scale_pow2(inv_sqrt_d * kLog2e, -e);
      er = e;  // K-side per-channel scales: the block adds its own exponent
      ebhi = 0u;
    }
#pragma unroll
    for (int cc = 0; cc < T::NCH; ++cc)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int k = 0; k < 4; ++k) o[cc][mt][k] = 0.f;
    m = -INFINITY;
    mneg = 0.f;
    zth = -INFINITY;
    l = 0.f;
    F = kNoScale;
    vthr = kVThr0;
    pf = 1.f;
    pfa = (WIDE || active) ? 1.f : 0.f;
  };

  // channel held in O^T row (r for k even, r + 8 for k odd) of chunk cc,
  // m-tile k / 2
  auto chan = [&](int cc, int k) -> int {
    if constexpr (T::VGRP) {
      return 32 * cc + 4 * r + k;
    } else if constexpr (T::VROW == 128) {
      return 16 * (2 * cc + (k >> 1)) + 2 * r + (k & 1);  // m-tile 2 cc + k / 2 = one 16-byte chunk
    } else {
      return 16 * (cc + (T::VROW / 32) * (r >> 2)) + 4 * (r & 3) + k;
    }
  };

  auto flush = [&](int b) {
    const int64_t slot = static_cast<int64_t>(b) + blockIdx.x;
    float lt = l + __shfl_xor_sync(0xffffffffu, l, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    const int64_t rec = slot * H + h;
    if (i == 0) {
      a.ws_ml[(rec * 8 + r) * 2 + 0] = m;
      a.ws_ml[(rec * 8 + r) * 2 + 1] = lt;
    }
    const bool none = (F == kNoScale);
#pragma unroll
    for (int cc = 0; cc < T::NCH; ++cc) {
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        float v0 = none ? 0.f : scale_pow2(o[cc][mt][0], -F);
        float v1 = none ? 0.f : scale_pow2(o[cc][mt][1], -F);
        float v2 = none ? 0.f : scale_pow2(o[cc][mt][2], -F);
        float v3 = none ? 0.f : scale_pow2(o[cc][mt][3], -F);
        // partial O^T stored column-major: [slot][head][column][channel]
        float *c0 = a.ws_o + (rec * 8 + 2 * i) * D;
        float *c1 = c0 + D;
        c0[chan(cc, 2 * mt)] = v0;
        c1[chan(cc, 2 * mt)] = v1;
        c0[chan(cc, 2 * mt + 1)] = v2;
        c1[chan(cc, 2 * mt + 1)] = v3;
      }
    }
  };

  int g = g0;
  int b = seq_of(cum, B, g0);
  int j = g0 - cum[b];
  int ctx_b = __ldg(a.ctx + b);
  int gend = min(cum[b + 1], g1);  // where the current sequence piece ends
  start_segment(b);

  // Shared-memory addresses of this warp's head in stage 0 (stage s adds
  // s * SB), with the thread's swizzled offsets folded in.  Box bases are
  // 1024-byte aligned, so the 16-byte chunk XOR of the swizzle can be applied
  // to base + offset directly.
  //  K (128-byte rows): 16-byte load (n-tile nt, k-group kg) of token
  //    8 nt + PI(r), logical chunk i + 4 kg -> (kofs ^ 64 kg) + 1024 nt.
  //  V (8-bit, 128-byte rows): one transposed x4 ldmatrix per two 16-byte
  //    chunks 2 cc, 2 cc + 1 (m-tiles; 16-bit elements = 2 channels), row
  //    order as for INT4 below, matrices (chunk 2 cc, tokens 0..7), (2 cc,
  //    8..15), (2 cc + 1, 0..7), (2 cc + 1, 8..15); lane (r, i) receives
  //    channels 2r, 2r + 1 of each chunk for its token pairs; address
  //    vofs0 ^ 32 cc.
  //  V (INT4, 64-byte rows): one transposed 8 x 8 ldmatrix per 8 tokens and
  //    chunk cc (16-bit elements = 4 channels): lane l gives the address of
  //    row l % 8 of matrix l / 8 (tokens 0..7, 8..15), row 2j being token j
  //    and row 2j + 1 token j + 4 of the eight, so lane (r, i) receives
  //    channels 4r .. 4r + 3 of chunk cc for tokens tk[0], tk[1] (matrix 0)
  //    and tk[2], tk[3] (matrix 1), already paired as the conversion wants
  //    them; address vofs0 ^ 16 cc.
  const int pr = PI(r);
  const uint32_t kofs = (T::KROW == 128) ? static_cast<uint32_t>(128 * pr + 16 * (i ^ pr)) : 0u;
  uint32_t vofs0 = 0;
  if constexpr (T::VINT4 && T::VROW == 64) {
    const int j = lane & 7;
    const int tok = (j >> 1) + 4 * (j & 1) + 8 * ((lane >> 3) & 1);
    vofs0 = 64 * tok + 16 * ((tok >> 1) & 3);
  } else if constexpr (!T::VINT4 && T::VROW == 128) {
    const int j = lane & 7;
    const int tok = (j >> 1) + 4 * (j & 1) + 8 * ((lane >> 3) & 1);
    vofs0 = 128 * tok + 16 * ((lane >> 4) ^ (tok & 7));
  }
  const uint32_t kbase0 = smem_u32(smem + T::kc_off(H) + h * T::KBOX) + kofs;
  const uint32_t vbase0 = smem_u32(smem + T::vc_off(H) + h * T::VBOX);
  const uint32_t ksb0 = smem_u32(smem + T::ks_off(H)) + (i * H + h) * 4;
  // V scales of token i + 4k: [token][head][group] (bulk copy) or
  // [head][token][group] (TMA, four groups)
  const uint32_t vsb0 = smem_u32(smem + T::vs_off(H)) +
                        (T::VS_TMA ? (h * kBlockSize + i) * 16 : (i * H + h) * T::VGROUPS * 4);
  int stage = 0;
  uint32_t ph = 0;
  uint32_t soff = 0;  // stage * SB

  for (; g < g1; ++g) {
    if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], ph))) {
      if (lane == 0) set_error(a.err, KVQ_DEVERR_TIMEOUT);
      break;
    }
    const int pb = info[stage];
    if (pb >= 0) {
      const uint32_t kbase = kbase0 + soff;
      const uint32_t vbase = vbase0 + soff;
      const uint32_t ksb = ksb0 + soff;
      const uint32_t vsb = vsb0 + soff;
      const int nvalid = min(kBlockSize, ctx_b - kBlockSize * j);
      // The block body is instantiated twice: every block but a sequence's
      // last is full and runs without any of the masking that positions
      // past the context need (partial = false removes it at compile time).
      auto process = [&](auto partial_tag) {
        constexpr bool partial = decltype(partial_tag)::value;
        // K: load of the 16 channels 16 (i + 4 kg) .. + 15 of token 8 nt + PI(r)
        // (16 bytes for 8-bit codes, 8 bytes for INT4)
        auto kaddr = [&](int nt, int kg) -> uint32_t {
          constexpr int CB = T::KINT2 ? 4 : (T::KINT4 ? 8 : 16);
          return (T::KROW == 128) ? ((kbase ^ (64u * kg)) + 1024u * nt)
                                  : kbase + swz<T::KROW>((8 * nt + pr) * T::KROW + CB * (i + 4 * kg));
        };

        // Positions past the context (cache rows that may hold any bytes,
        // FP8 NaN patterns included) must add nothing: their scores become
        // -inf below, and their V codes and V scales are zeroed in shared
        // memory before the block's loads.
        if constexpr (partial) {
          const int nz = (kBlockSize - nvalid) * (T::VROW / 16);
          for (int u = lane; u < nz; u += 32) sts128(vbase + nvalid * T::VROW + 16 * u, 0u, 0u, 0u, 0u);
          for (int t = nvalid + lane; t < kBlockSize; t += 32) {
            if constexpr (T::VS_TMA) {
              sts128(vsb - 16u * i + 16u * t, 0u, 0u, 0u, 0u);  // [head][token][4 groups]
            } else {
#pragma unroll
              for (int gi = 0; gi < T::VGROUPS; ++gi)  // [token][head][group]
                sts32(vsb - 4u * T::VGROUPS * (i * H) + 4u * ((t * H) * T::VGROUPS + gi), 0u);
            }
          }
          // the producer refills this stage through the async proxy
          fence_proxy_async_shared();
          __syncwarp();
        }
        // ---- S = Q' K^T
        float sacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int k = 0; k < 4; ++k) sacc[nt][k] = 0.f;
        if constexpr (T::KSCL) {
          // s' = s_c 2^eb in f16 with the block's largest s' in [2^10, 2^15)
          // (eb puts a block maximum in [2^14, 2^15)); K' = code s' is exact
          // (codes -1, 0, 1; BF16 scales down to 2^-27 of the largest), the
          // staged query carries 2^er, so the row scale takes 2^-(er + eb)
          float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
          if (lane < D / 4) {
            const uint4 u = lds128(kcs0 + soff);
            sc = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
          }
          // eb carries over while the block's largest s' stays in [2^10, 2^15)
          // (lane-local votes, as for the 8-bit codes below)
          const uint32_t lmaxb = max(max(__float_as_uint(sc.x), __float_as_uint(sc.y)),
                                     max(__float_as_uint(sc.z), __float_as_uint(sc.w)));
          if (__any_sync(0xffffffffu, lmaxb >= ebhi) || !__any_sync(0xffffffffu, lmaxb >= eblo)) {
            const uint32_t smaxb = warp_max_u32(lmaxb);
            const int eb = smaxb ? min(14 - ilog2f(__uint_as_float(smaxb)), kMaxVExp) : 0;
            fbk = pow2i(eb);
            ebhi = (15 - eb > 127) ? 0x7F800000u : __float_as_uint(pow2i(15 - eb));
            eblo = __float_as_uint(pow2i(10 - eb));
            rowscale = scale_pow2(inv_sqrt_d * kLog2e, -min(er + eb, 250));
          }
          const float fb = fbk;
          mul_f32x2(sc.x, sc.y, fb, fb, sc.x, sc.y);
          mul_f32x2(sc.z, sc.w, fb, fb, sc.z, sc.w);
          if (lane < D / 4) sts64(sown, f32x2_to_f16x2(sc.x, sc.y), f32x2_to_f16x2(sc.z, sc.w));
          __syncwarp();
#pragma unroll
          for (int kg = 0; kg < T::NKG; ++kg) {
            const uint32_t w0 = lds32(kaddr(0, kg)), w1 = lds32(kaddr(1, kg));
#pragma unroll
            for (int ss = 0; ss < 4; ++ss) {
              const uint4 qf = lds128(qst + QS * (4 * kg + ss));  // rows r + 8 zero
              const uint2 sv = lds64(sw0 + 128u * kg + 8u * ss);
              const uint32_t fr[4] = {qf.x, qf.y, qf.z, qf.w};
              uint32_t b0, b1, c0, c1;
              if (ss == 0) { k_crumbs_to_f16<0>(w0, b0, b1); k_crumbs_to_f16<0>(w1, c0, c1); }
              else if (ss == 1) { k_crumbs_to_f16<1>(w0, b0, b1); k_crumbs_to_f16<1>(w1, c0, c1); }
              else if (ss == 2) { k_crumbs_to_f16<2>(w0, b0, b1); k_crumbs_to_f16<2>(w1, c0, c1); }
              else { k_crumbs_to_f16<3>(w0, b0, b1); k_crumbs_to_f16<3>(w1, c0, c1); }
              mma_f16(sacc[0], fr, hmul2_u32(b0, sv.x), hmul2_u32(b1, sv.y));
              mma_f16(sacc[1], fr, hmul2_u32(c0, sv.x), hmul2_u32(c1, sv.y));
            }
          }
        } else if constexpr (T::KCHAN) {
          // The block's channel scales of this head, s' = s_c 2^eb with the
          // largest s' in [2^3, 2^8) (eb puts a block maximum in [2^7, 2^8)
          // and is kept while later maxima stay in the window), as f16 pairs
          // s' ~ s_h + s_l (s_h = RN(s'), s_l = RN(s' - s_h): ~22 bits).
          // Against the staged query (max |q~| < 2^7) every product q~ s' is
          // below 2^15.  The S operand Q' = q~ s' is rebuilt per block by f16
          // FMAs as high and low parts (rows r and r + 8): h = RN(q~ s_h);
          // q~ s_h - h is exact in one FMA (at most 8 significant bits left);
          // l = RN(q~ s_h - h + q~ s_l).  h + l carries q~ s' to ~2^-21 (only
          // products below 2^-23 of the largest can lose low bits to the f16
          // subnormal range).
          float4 sc = make_float4(0.f, 0.f, 0.f, 0.f);
          if (lane < D / 4) {
            const uint4 u = lds128(kcs0 + soff);
            sc = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z), __uint_as_float(u.w));
          }
          // eb carries over from the previous block while the block's largest
          // s 2^eb stays in [2^3, 2^8) (products below 2^15, at most 4 bits of
          // headroom given up at the bottom); otherwise the block maximum sets
          // it anew.  Scales are >= 0: their bit patterns order like their
          // values, and the lane-local tests need no warp maximum.
          const uint32_t lmaxb = max(max(__float_as_uint(sc.x), __float_as_uint(sc.y)),
                                     max(__float_as_uint(sc.z), __float_as_uint(sc.w)));
          if (__any_sync(0xffffffffu, lmaxb >= ebhi) || !__any_sync(0xffffffffu, lmaxb >= eblo)) {
            const uint32_t smaxb = warp_max_u32(lmaxb);
            const int eb = smaxb ? min(7 - ilog2f(__uint_as_float(smaxb)), 126) : 0;
            fbk = pow2i(eb);
            ebhi = (8 - eb > 127) ? 0x7F800000u : __float_as_uint(pow2i(8 - eb));
            eblo = __float_as_uint(pow2i(3 - eb));
            rowscale = scale_pow2(inv_sqrt_d * kLog2e, max(-250, min(250, -(eb + er))));
          }
          const float fb = fbk;
          float s0, s1, s2, s3;
          mul_f32x2(sc.x, sc.y, fb, fb, s0, s1);
          mul_f32x2(sc.z, sc.w, fb, fb, s2, s3);
          uint32_t h02, h13, l02, l13;
          split_f16x2(s0, s2, h02, l02);
          split_f16x2(s1, s3, h13, l13);
          if (lane < D / 4) sts128(sown, h02, h13, l02, l13);
          __syncwarp();
#pragma unroll
          for (int kg = 0; kg < T::NKG; ++kg) {
            const uint4 w0 = lds128(kaddr(0, kg));
            const uint4 w1 = lds128(kaddr(1, kg));
            const uint32_t k0[4] = {w0.x, w0.y, w0.z, w0.w};
            const uint32_t k1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int ss = 0; ss < 4; ++ss) {
              // channels c = 16 (i + 4 kg) + 4 ss .. + 3 of row slot r: query
              // pairs (c, c + 2), (c + 1, c + 3), then s_h and s_l of the same
              const uint2 qw = lds64(qst + QU * (4 * kg + ss));
              const uint4 sv = lds128(((ss & 1) ? sw1 : sw0) + 256u * kg + 32u * (ss >> 1));
              uint32_t fr[4];
              fr[0] = hmul2_u32(qw.x, sv.x);
              fr[1] = hfma2_u32(qw.x, sv.z, hfma2_negc_u32(qw.x, sv.x, fr[0]));
              fr[2] = hmul2_u32(qw.y, sv.y);
              fr[3] = hfma2_u32(qw.y, sv.w, hfma2_negc_u32(qw.y, sv.y, fr[2]));
              uint32_t b0, b1;
              k_int8_word_to_f16_02_13(k0[ss], b0, b1);
              mma_f16(sacc[0], fr, b0, b1);
              k_int8_word_to_f16_02_13(k1[ss], b0, b1);
              mma_f16(sacc[1], fr, b0, b1);
            }
          }
        } else if constexpr (T::KINT4) {
#pragma unroll
          for (int kg = 0; kg < T::NKG; ++kg) {
            const uint2 w0 = lds64(kaddr(0, kg));
            const uint2 w1 = lds64(kaddr(1, kg));
#pragma unroll
            for (int ss = 0; ss < 4; ++ss) {
              // rows r + 8: the low parts (zero unless the cache is rotated)
              uint4 f;
              if constexpr (Q2) {
                f = lds128(qst + QS * (4 * kg + ss));
              } else {
                const uint2 qh = lds64(qst + QU * (4 * kg + ss));
                f = make_uint4(qh.x, 0u, qh.y, 0u);
              }
              const uint32_t fr[4] = {f.x, f.y, f.z, f.w};
              const int sh = 16 * (ss & 1);
              uint32_t b0, b1;
              k_nibbles_to_f16(((ss < 2) ? w0.x : w0.y) >> sh, b0, b1);
              mma_f16(sacc[0], fr, b0, b1);
              k_nibbles_to_f16(((ss < 2) ? w1.x : w1.y) >> sh, b0, b1);
              mma_f16(sacc[1], fr, b0, b1);
            }
          }
        } else {
#pragma unroll
          for (int kg = 0; kg < T::NKG; ++kg) {
            const uint4 w0 = lds128(kaddr(0, kg));
            const uint4 w1 = lds128(kaddr(1, kg));
            const uint32_t k0[4] = {w0.x, w0.y, w0.z, w0.w};
            const uint32_t k1[4] = {w1.x, w1.y, w1.z, w1.w};
#pragma unroll
            for (int ss = 0; ss < 4; ++ss) {
              // rows r + 8: the low parts (zero unless the cache is rotated)
              uint4 f;
              if constexpr (Q2) {
                f = lds128(qst + QS * (4 * kg + ss));
              } else {
                const uint2 qh = lds64(qst + QU * (4 * kg + ss));
                f = make_uint4(qh.x, 0u, qh.y, 0u);
              }
              const uint32_t fr[4] = {f.x, f.y, f.z, f.w};
              uint32_t b0, b1;
              k_word_to_f16<T::KFP8>(k0[ss], b0, b1);
              mma_f16(sacc[0], fr, b0, b1);
              k_word_to_f16<T::KFP8>(k1[ss], b0, b1);
              mma_f16(sacc[1], fr, b0, b1);
            }
          }
        }

        // ---- scores (log2 domain), mask, block max
        float z[4];
        // rows r + 8 of Q' hold low parts (rotated cache, 8-bit per-channel
        // K) or zeros, which add nothing
        constexpr bool qlow = rot || (T::KCHAN && !T::KSCL);
        z[0] = qlow ? sacc[0][0] + sacc[0][2] : sacc[0][0];
        z[1] = qlow ? sacc[0][1] + sacc[0][3] : sacc[0][1];
        z[2] = qlow ? sacc[1][0] + sacc[1][2] : sacc[1][0];
        z[3] = qlow ? sacc[1][1] + sacc[1][3] : sacc[1][1];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          float sk = rowscale;
          if constexpr (!T::KCHAN) sk *= ldsf(ksb + 16 * H * k);  // token tk[k] = i + 4k
          float zs = fmaf(z[k], sk, mneg);  // z - m
          if constexpr (partial) zs = (tk[k] < nvalid) ? zs : -INFINITY;
          z[k] = zs;
        }
        const float zmax = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));  // this lane's tokens

        // ---- V scales of this thread's tokens and their maximum
        float vsc[4][T::VGROUPS];
        float vmax = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // token tk[k] = i + 4k: ((tk H + h) VGROUPS + gi) * 4 bytes; a token's
          // group scales are contiguous and load as one vector (the stage
          // always holds all 16 tokens' scales: every lane loads, and a partial
          // block then zeroes the scales of positions past the context)
          const uint32_t sa = vsb + (T::VS_TMA ? 64u * k : 16u * H * T::VGROUPS * k);
          if constexpr (T::VGROUPS == 4) {
            const uint4 u = lds128(sa);
            vsc[k][0] = __uint_as_float(u.x);
            vsc[k][1] = __uint_as_float(u.y);
            vsc[k][2] = __uint_as_float(u.z);
            vsc[k][3] = __uint_as_float(u.w);
          } else if constexpr (T::VGROUPS == 2) {
            const uint2 u = lds64(sa);
            vsc[k][0] = __uint_as_float(u.x);
            vsc[k][1] = __uint_as_float(u.y);
          } else {
            vsc[k][0] = ldsf(sa);
          }
        }
        if constexpr (T::VS_TMA && WIDE) {
          // the eight lanes of a token column hold the same 64 scales: for
          // the test, lane r reads two of them (token i + 4 (r / 2), groups
          // 2 (r % 2), + 1); this measured faster in the wide layout and
          // slower in the packed one
          const uint2 u = lds64(vsb + 64u * (r >> 1) + 8u * (r & 1));
          vmax = fmaxf(__uint_as_float(u.x), __uint_as_float(u.y));
        } else {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
#pragma unroll
            for (int gi = 0; gi < T::VGROUPS; ++gi) vmax = fmaxf(vmax, vsc[k][gi]);
          }
        }

        // ---- rescale the running state when a score passes m + kLazyMax (so
        // the probabilities stay at most 2^kLazyMax) or when a V scale reaches
        // 2^(14 - F), i.e. the block's exponent 13 - floor(log2 max s_v) would
        // be below F.  Both tests are lane-local; the row maxima (shuffles) and
        // the block's V-scale maximum (every row slot holds the same 16 tokens'
        // scales, >= 0, so their bit patterns order like the values) are only
        // formed when the warp rescales.
        if (__any_sync(0xffffffffu, zmax > zth || vmax >= vthr)) {
          float mb = fmaxf(zmax, __shfl_xor_sync(0xffffffffu, zmax, 1));
          mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
          // the row's scores move by dz (absolute on a piece's first block)
          const bool first = (m == -INFINITY);
          const float dz = first ? mb : fmaxf(mb, 0.f);
          const float m_new = first ? mb : m + dz;
#pragma unroll
          for (int k = 0; k < 4; ++k) z[k] -= dz;
          const float wv = __uint_as_float(warp_max_u32(__float_as_uint(vmax)));
          const int F_blk = (wv > 0.f) ? min(13 - ilog2f(wv), kMaxVExp) : kNoScale;
          const float alpha = first ? 0.f : fast_exp2(-dz);
          const int F_new = min(F, F_blk);
          l *= alpha;
          const float a0 = __shfl_sync(0xffffffffu, alpha, 4 * (2 * i));
          const float a1 = __shfl_sync(0xffffffffu, alpha, 4 * (2 * i + 1));
          const int df = (F == kNoScale) ? 0 : F_new - F;
          const float c0 = scale_pow2(a0, df), c1 = scale_pow2(a1, df);
#pragma unroll
          for (int cc = 0; cc < T::NCH; ++cc)
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
              o[cc][mt][0] *= c0;
              o[cc][mt][1] *= c1;
              o[cc][mt][2] *= c0;
              o[cc][mt][3] *= c1;
            }
          m = m_new;
          mneg = -m_new;
          zth = kLazyMax;
          F = F_new;
          if (F != kNoScale) {
            pf = pow2i(F);
            pfa = (WIDE || active) ? pf : 0.f;
            vthr = (14 - F > 127) ? INFINITY : pow2i(14 - F);
          }
        }

        // ---- probabilities
        float p[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) p[k] = fast_exp2(z[k]);
        l += (p[0] + p[1]) + (p[2] + p[3]);
        float pp[4];  // p * 2^F (exact: a power-of-two product); 0 in inactive packed slots
        const float pfw = WIDE ? pf : pfa;
        mul_f32x2(p[0], p[1], pfw, pfw, pp[0], pp[1]);
        mul_f32x2(p[2], p[3], pfw, pfw, pp[2], pp[3]);

        // ---- O^T += V^T P''   (P'' = p * s_v * 2^F as f16 high + low parts)
        // per-token V scales: one product per token, split into both parts
        auto p_frag = [&](uint32_t &bh0, uint32_t &bh1, uint32_t &bl0, uint32_t &bl1) {
          float q0, q1, q2, q3;
          mul_f32x2(pp[0], pp[1], vsc[0][0], vsc[1][0], q0, q1);
          mul_f32x2(pp[2], pp[3], vsc[2][0], vsc[3][0], q2, q3);
          split_f16x2(q0, q1, bh0, bl0);
          split_f16x2(q2, q3, bh1, bl1);
        };
        // group scales: the products p s_v 2^F of every (token, group) are
        // formed in place, once per block (two groups of one token per packed
        // multiply); chunk cc then takes group cc of its four tokens.  In the
        // packed layout a row slot needs only its own part of P'' (high for
        // columns < G, low for columns G .. 2G - 1, zero for inactive slots):
        // x, or x - f16(x) when lo_m = 1, rounded to f16.
        if constexpr (T::VGRP) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int gi = 0; gi < T::VGROUPS; gi += 2)
              mul_f32x2(pp[k], pp[k], vsc[k][gi], vsc[k][gi + 1], vsc[k][gi], vsc[k][gi + 1]);
        }
        const float lo_m = lo_role ? 1.f : 0.f;
        auto p_part = [&](int gi, uint32_t &b0, uint32_t &b1) {
          b0 = part_f16x2(vsc[0][gi], vsc[1][gi], lo_m);
          b1 = part_f16x2(vsc[2][gi], vsc[3][gi], lo_m);
        };
        // wide layout: both parts of group gi (the residuals are exact in FP32)
        auto p_split = [&](int gi, uint32_t &bh0, uint32_t &bh1, uint32_t &bl0, uint32_t &bl1) {
          const float q0 = vsc[0][gi], q1 = vsc[1][gi], q2 = vsc[2][gi], q3 = vsc[3][gi];
          bh0 = f32x2_to_f16x2(q0, q1);
          bl0 = f32x2_to_f16x2(q0 - f16lo_to_f32(bh0), q1 - f16hi_to_f32(bh0));
          bh1 = f32x2_to_f16x2(q2, q3);
          bl1 = f32x2_to_f16x2(q2 - f16lo_to_f32(bh1), q3 - f16hi_to_f32(bh1));
        };
        uint32_t th0 = 0u, th1 = 0u, tl0 = 0u, tl1 = 0u;  // per-token V: one fragment for all chunks
        if constexpr (!T::VGRP) p_frag(th0, th1, tl0, tl1);
        const uint32_t va0 = vbase + vofs0;
#pragma unroll
        for (int cc = 0; cc < T::NCH; ++cc) {
          uint32_t bh0 = th0, bh1 = th1, bl0 = tl0, bl1 = tl1;
          if constexpr (T::VGRP && WIDE) p_split(cc, bh0, bh1, bl0, bl1);  // group scale of chunk cc
          if constexpr (T::VGRP && !WIDE) p_part(cc, bh0, bh1);           // this slot's part, in bh
          uint32_t afr[2][4];
          if constexpr (T::VINT2) {
            // byte 8 cc + r of token row tk[k] = i + 4k (this lane's 4 channels
            // of group cc): in the 32-byte swizzle the row's 128-byte line is
            // k, so the chunk bit flips for odd k and every offset is a constant
            // from vbase + 32 i + r
            static_assert(T::VROW == 32, "INT2 V rows are 32 bytes");
            const uint32_t vb = vbase + 32u * i + r;
            const uint32_t h0 = lds8(vb + (8u * cc));
            const uint32_t h1 = lds8(vb + 128u + ((8u * cc) ^ 16u));
            const uint32_t h2 = lds8(vb + 256u + (8u * cc));
            const uint32_t h3 = lds8(vb + 384u + ((8u * cc) ^ 16u));
            uint32_t p01[4], p23[4];
            v_crumbs_to_f16(h0, h1, p01);
            v_crumbs_to_f16(h2, h3, p23);
            afr[0][0] = p01[0]; afr[0][1] = p01[1]; afr[0][2] = p23[0]; afr[0][3] = p23[1];
            afr[1][0] = p01[2]; afr[1][1] = p01[3]; afr[1][2] = p23[2]; afr[1][3] = p23[3];
          } else if constexpr (T::VINT4) {
            uint32_t p01[4], p23[4];
            if constexpr (T::VROW == 64) {
              uint32_t u01, u23;
              ldsm_x2_trans(va0 ^ (16u * cc), u01, u23);
              v_nibble_pairs_to_f16(u01, p01);
              v_nibble_pairs_to_f16(u23, p23);
            } else {
              const uint32_t off = 16 * cc + 2 * r;
              const uint32_t h0 = lds16(vbase + swz<T::VROW>(tk[0] * T::VROW + off));
              const uint32_t h1 = lds16(vbase + swz<T::VROW>(tk[1] * T::VROW + off));
              const uint32_t h2 = lds16(vbase + swz<T::VROW>(tk[2] * T::VROW + off));
              const uint32_t h3 = lds16(vbase + swz<T::VROW>(tk[3] * T::VROW + off));
              v_nibbles_to_f16(h0, h1, p01);
              v_nibbles_to_f16(h2, h3, p23);
            }
            afr[0][0] = p01[0]; afr[0][1] = p01[1]; afr[0][2] = p23[0]; afr[0][3] = p23[1];
            afr[1][0] = p01[2]; afr[1][1] = p01[3]; afr[1][2] = p23[2]; afr[1][3] = p23[3];
          } else if constexpr (T::VROW == 128) {
            uint32_t m0, m1, m2, m3;
            ldsm_x4_trans(va0 ^ (32u * cc), m0, m1, m2, m3);
            v_byte_pairs_to_f16<T::VFP8>(m0, afr[0][0], afr[0][1]);
            v_byte_pairs_to_f16<T::VFP8>(m1, afr[0][2], afr[0][3]);
            v_byte_pairs_to_f16<T::VFP8>(m2, afr[1][0], afr[1][1]);
            v_byte_pairs_to_f16<T::VFP8>(m3, afr[1][2], afr[1][3]);
          } else {
            const uint32_t off = 16 * (cc + (T::VROW / 32) * (r >> 2)) + 4 * (r & 3);
            const uint32_t w0 = lds32(vbase + swz<T::VROW>(tk[0] * T::VROW + off));
            const uint32_t w1 = lds32(vbase + swz<T::VROW>(tk[1] * T::VROW + off));
            const uint32_t w2 = lds32(vbase + swz<T::VROW>(tk[2] * T::VROW + off));
            const uint32_t w3 = lds32(vbase + swz<T::VROW>(tk[3] * T::VROW + off));
            uint32_t p01[4], p23[4];
            v_words_to_f16<T::VFP8>(w0, w1, p01);
            v_words_to_f16<T::VFP8>(w2, w3, p23);
            afr[0][0] = p01[0]; afr[0][1] = p01[1]; afr[0][2] = p23[0]; afr[0][3] = p23[1];
            afr[1][0] = p01[2]; afr[1][1] = p01[3]; afr[1][2] = p23[2]; afr[1][3] = p23[3];
          }
#pragma unroll
          for (int mt = 0; mt < 2; ++mt) {
            if constexpr (WIDE) {
              mma_f16(o[cc][mt], afr[mt], bh0, bh1);
              mma_f16(o[cc][mt], afr[mt], bl0, bl1);
            } else if constexpr (T::VGRP) {
              mma_f16(o[cc][mt], afr[mt], bh0, bh1);
            } else {
              const uint32_t b0 = lo_role ? bl0 : bh0;  // zero for inactive slots
              const uint32_t b1 = lo_role ? bl1 : bh1;
              mma_f16(o[cc][mt], afr[mt], b0, b1);
            }
          }
        }
      };
      if (nvalid < kBlockSize)
        process(std::true_type{});
      else
        process(std::false_type{});
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);
    soff += SB;
    if (++stage == nstages) {
      stage = 0;
      ph ^= 1;
      soff = 0;
    }

    // ---- advance; flush at the end of a sequence piece
    ++j;
    if (g + 1 == gend) {
      flush(b);
      if (g + 1 < g1) {
        ++b;
        while (cum[b + 1] == cum[b]) ++b;
        j = 0;
        ctx_b = __ldg(a.ctx + b);
        gend = min(cum[b + 1], g1);
        start_segment(b);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// split-reduce: one warp per (sequence, query head)
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256) decode_reduce_kernel(const DecodeArgs a, const int *__restrict__ cum) {
  const int warp = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (warp >= a.B * a.Hq) return;
  const int b = warp / a.Hq;
  const int hq = warp % a.Hq;
  const int h = hq / a.G;
  const int g = hq % a.G;
  constexpr int CPL = D / 32;  // channels per lane
  float *outp = a.out + static_cast<int64_t>(warp) * D + lane * CPL;
  const int c0b = cum[b], c1b = cum[b + 1];
  float acc[CPL];
#pragma unroll
  for (int k = 0; k < CPL; ++k) acc[k] = 0.f;
  float L = 0.f;
  float mx = -INFINITY;
  if (c1b > c0b) {
    const int total = cum[a.B];
    const int P = a.nctas;
    // CTA holding global block x: min(P - 1, floor(((x + 1) P - 1) / total))
    auto cta_of = [&](int x) -> int {
      const int64_t v = ((static_cast<int64_t>(x) + 1) * P - 1) / total;
      return static_cast<int>(v < P - 1 ? v : P - 1);
    };
    const int s0 = cta_of(c0b), ns = cta_of(c1b - 1) - s0 + 1;
    const bool packed = 2 * a.G <= 8;  // columns g (high) and g + G (low)
    // pass 1: lanes read the partial (m, l) pairs in parallel; the first 32
    // stay in registers for pass 2
    float m_own = -INFINITY, l_own = 0.f;
    for (int s = lane; s < ns; s += 32) {
      const int64_t rec = (static_cast<int64_t>(b) + s0 + s) * a.H + h;
      const float2 ml = *reinterpret_cast<const float2 *>(a.ws_ml + (rec * 8 + g) * 2);
      if (s == lane) {
        m_own = ml.x;
        l_own = ml.y;
      }
      mx = fmaxf(mx, ml.x);
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (mx != -INFINITY) {
      // pass 2: weights per split (lane s), then the weighted sum of the
      // partial outputs with every lane on its channels, eight partials'
      // loads in flight at a time
      constexpr int U = 8;
      for (int base = 0; base < ns; base += 32) {
        float w = 0.f;
        if (base + lane < ns) {
          float ms = m_own, ls = l_own;
          if (base > 0) {
            const int64_t rec = (static_cast<int64_t>(b) + s0 + base + lane) * a.H + h;
            const float2 ml = *reinterpret_cast<const float2 *>(a.ws_ml + (rec * 8 + g) * 2);
            ms = ml.x;
            ls = ml.y;
          }
          w = exp2f(ms - mx);
          L += w * ls;
        }
        const int n = min(32, ns - base);
        for (int k0 = 0; k0 < n; k0 += U) {
          float v[U][CPL];
#pragma unroll
          for (int u = 0; u < U; ++u) {
#pragma unroll
            for (int q = 0; q < CPL; ++q) v[u][q] = 0.f;
            if (k0 + u < n) {
              const int64_t rec = (static_cast<int64_t>(b) + s0 + base + k0 + u) * a.H + h;
              const float *col = a.ws_o + (rec * 8 + g) * D + lane * CPL;
              if constexpr (CPL == 4) {
                const float4 x = *reinterpret_cast<const float4 *>(col);
                v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
                if (packed) {
                  const float4 y = *reinterpret_cast<const float4 *>(col + a.G * D);
                  v[u][0] += y.x; v[u][1] += y.y; v[u][2] += y.z; v[u][3] += y.w;
                }
              } else {
#pragma unroll
                for (int q = 0; q < CPL; ++q) v[u][q] = col[q] + (packed ? col[a.G * D + q] : 0.f);
              }
            }
          }
#pragma unroll
          for (int u = 0; u < U; ++u) {
            // lanes at or past n hold w = 0 and their v is zero
            const float wk = __shfl_sync(0xffffffffu, w, (k0 + u) & 31);
#pragma unroll
            for (int q = 0; q < CPL; ++q) acc[q] += wk * v[u][q];
          }
        }
      }
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    }
  }
  if (a.res_k != nullptr) {
    // per-channel K with a full-precision tail: the residual rows 0 .. nt - 1
    // hold positions [n - nt, n); merged into (mx, L, acc) token by token
    const int n = __ldg(a.ctx + b);
    const bool bad = n < 0 || n / kBlockSize > a.max_blocks || n > a.max_ctx;
    const int nt = bad ? 0 : n % kBlockSize;
    if (nt > 0) {
      const uint16_t *qp = a.q + static_cast<int64_t>(warp) * D + lane * CPL;
      float qf[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) qf[c] = __uint_as_float(static_cast<uint32_t>(qp[c]) << 16);
      const float zscale = rsqrtf(static_cast<float>(D)) * kLog2e;
      for (int t = 0; t < nt; ++t) {
        const int64_t row = ((static_cast<int64_t>(b) * kBlockSize + t) * a.H + h) * D + lane * CPL;
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) dot += qf[c] * __uint_as_float(static_cast<uint32_t>(a.res_k[row + c]) << 16);
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        const float z = dot * zscale;
        const float m_new = fmaxf(mx, z);
        const float keep = exp2f(mx - m_new);  // 0 while nothing was seen
        const float p = exp2f(z - m_new);
        L = L * keep + p;
#pragma unroll
        for (int c = 0; c < CPL; ++c)
          acc[c] = acc[c] * keep + p * __uint_as_float(static_cast<uint32_t>(a.res_v[row + c]) << 16);
        mx = m_new;
      }
    }
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
  float o[CPL];
#pragma unroll
  for (int k = 0; k < CPL; ++k) o[k] = acc[k] * inv;
  if (a.rot) {
    // rotated cache: the merged output is in the rotated basis; return
    // sigma * (H o') / d.  This lane holds channels CPL lane .. + CPL - 1:
    // butterfly stages below CPL inside the lane, the others across lanes.
#pragma unroll
    for (int hh = 1; hh < CPL; hh <<= 1)
#pragma unroll
      for (int k = 0; k < CPL; ++k)
        if (!(k & hh)) {
          const float x = o[k], y = o[k + hh];
          o[k] = x + y;
          o[k + hh] = x - y;
        }
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int k = 0; k < CPL; ++k) {
        const float p = __shfl_xor_sync(0xffffffffu, o[k], m);
        o[k] = upper ? p - o[k] : o[k] + p;
      }
    }
    constexpr float kInvD = 1.f / D;  // a power of two
#pragma unroll
    for (int k = 0; k < CPL; ++k) {
      const int ch = lane * CPL + k;
      const uint32_t neg = (a.rot_signs[ch >> 5] >> (ch & 31)) & 1u;
      o[k] = __uint_as_float(__float_as_uint(o[k] * kInvD) ^ (neg << 31));
    }
  }
#pragma unroll
  for (int k = 0; k < CPL; ++k) outp[k] = o[k];
}

}  // namespace kvq
