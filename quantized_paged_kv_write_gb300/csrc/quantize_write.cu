// Quantize-on-write into the paged KV cache (sm_103a).
//
// What it computes: "Use Less Memory: Quantization and Offloading", §2.1
// Symmetric Quantization Formula (s = max|x| / q_max, x_q = clip(round(x/s)))
// and §5 Exercise 1, per scale group, stored in the cache layout of
// "PidokuInfra 12 KV Cache Quantization", §5 Where the scales live.  Per-channel
// K (KIVI, "Quantized KV caches in production", Numerical Formats; "PidokuInfra
// 12", K is more sensitive than V) takes the absmax of each (kv_head, channel)
// over the tokens written into one block.
//
// Design.  The op is a pure stream (per (token, head): read 2 x head_dim BF16
// of K and of V, write codes and scales), so the kernel is laid out for HBM
// and for few instructions per byte.  A warp takes one token at a time and
// all of its heads: a half-warp (head_dim 128) or a quarter-warp (64) owns a
// row, one 16-byte vector per lane, and all of the token's rows are loaded
// before any is processed (up to 64 bytes per lane in flight; 32 warps per
// SM).  The absmax is a shuffle reduction over the lanes of the scale group.
//
// Exactness.  Every scale is RN(absmax / q_max) and every code is the rounding
// (cvt.rni for INT, cvt.rn.satfinite.e4m3x2 for FP8) of the correctly rounded
// quotient RN(x / s), bit for bit, without a division per element:
//   * the scale uses s0 = RN(a * RN(1/q)), s = fma(fma(-s0, q, a), RN(1/q), s0),
//     which equals RN(a / q) for every BF16 absmax a and q in {127, 7, 448}
//     (checked exhaustively by tests/test_scale_sequence.py);
//   * the quotient uses y = rcp.approx(s) (relative error below 2^-23): the
//     exact products x RN(y (1 -/+ 2^-20)) lie on either side of RN(x / s),
//     and the code is monotone in the quotient, so equal codes at both ends
//     are the code (INT: one FMA per end into the rounding constant
//     1.5 * 2^23; FP8: the ends' conversions).  Per-channel K tests the
//     distance of RN(x * y) to the nearest half-integer instead.  Otherwise (a
//     few elements in 10^4, next to a rounding decision) the group is redone
//     with IEEE division.
// K and V share one launch when they run the same code (the first CTAs of the
// grid take K, the rest V), else they go in two launches.
#include "common.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 4;   // 64 registers per thread -> 4 x 256 threads resident
constexpr int kMaxHeads = 8;

template <int DT>
struct QConst;
template <>
struct QConst<KVQ_INT8> {
  static constexpr float q = 127.0f;
  static constexpr float inv = 0x1.020408p-7f;  // RN(1/127)
  static constexpr int qi = 127;
};
template <>
struct QConst<KVQ_INT4> {
  static constexpr float q = 7.0f;
  static constexpr float inv = 0x1.24924ap-3f;  // RN(1/7)
  static constexpr int qi = 7;
};
template <>
struct QConst<KVQ_FP8_E4M3FN> {
  static constexpr float q = 448.0f;
  static constexpr float inv = 0x1.24924ap-9f;  // RN(1/448)
};

// s = RN(a / q) for a BF16 absmax a (see the header comment).
template <int DT>
__device__ __forceinline__ float scale_of(float a) {
  const float s0 = __fmul_rn(a, QConst<DT>::inv);
  const float rho = __fmaf_rn(-s0, QConst<DT>::q, a);
  return __fmaf_rn(rho, QConst<DT>::inv, s0);
}

__device__ __forceinline__ float rcp_approx(float s) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(s));
  return y;
}

__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
  unsigned short r;
  // the first source goes to the upper byte
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ int qint(float r, int qmax) {
  int q = __float2int_rn(r);  // cvt.rni: round half to even
  return min(max(q, -qmax), qmax);
}

// The fast paths need 1/s to be a normal number: s >= 2^-125.
constexpr float kMinFastScale = 0x1p-125f;

// Fast-path bracket.  y = rcp.approx(s) has relative error below 2^-23, so
// with y_lo = RN(y (1 - 2^-20)) and y_hi = RN(y (1 + 2^-20)) the exact
// products x y_lo and x y_hi lie strictly on either side of RN(x / s) (the
// factors 1 -/+ 2^-20 outweigh the 2^-23 + 2 * 2^-24 of the reciprocal and
// the two roundings).  The code is a monotone function of the quotient, so
// equal codes at both ends are the code of RN(x / s); otherwise the group is
// redone with IEEE division.
constexpr float kBracketDown = 0x1.ffffe0p-1f;  // 1 - 2^-20
constexpr float kBracketUp = 0x1.000010p+0f;    // 1 + 2^-20

__device__ __forceinline__ void fma_f32x2(float a0, float a1, float b0, float b1, float c0, float c1, float &d0,
                                          float &d1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// INT codes of a pair: t = RN(x y + 1.5 * 2^23) in one FMA holds rint(x y)
// of the exact product (ties to even: 1.5 * 2^23 is even and the sum's ulp
// is 1) in its low mantissa bits, so the two's complement byte or nibble of
// the code is the low byte or nibble of t's bits.  In the fast path
// |x y_hi| < q_max + 1/2, so no clamp is needed.  `diff` collects the bits
// where the codes at the two ends differ.
__device__ __forceinline__ void int_pair_bracket(float x0, float x1, float ylo, float yhi, uint32_t &c0,
                                                 uint32_t &c1, uint32_t &diff) {
  const float kM = 0x1.8p23f;
  float l0, l1, h0, h1;
  fma_f32x2(x0, x1, ylo, ylo, kM, kM, l0, l1);
  fma_f32x2(x0, x1, yhi, yhi, kM, kM, h0, h1);
  c0 = __float_as_uint(l0);
  c1 = __float_as_uint(l1);
  diff |= (c0 ^ __float_as_uint(h0)) | (c1 ^ __float_as_uint(h1));
}

// FP8 codes of a pair: the codes of r = x y and of the two ends; the ends'
// codes equal r's whenever they equal each other.
__device__ __forceinline__ uint32_t fp8_pair_bracket(float x0, float x1, float y, float ylo, float yhi,
                                                     uint32_t &diff) {
  float r0, r1, l0, l1, h0, h1;
  mul_f32x2(x0, x1, y, y, r0, r1);
  mul_f32x2(x0, x1, ylo, ylo, l0, l1);
  mul_f32x2(x0, x1, yhi, yhi, h0, h1);
  const uint32_t c = fp8x2(r0, r1);
  diff |= (fp8x2(l0, l1) ^ c) | (fp8x2(h0, h1) ^ c);
  return c;
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]);

// The exact path: IEEE division for every element (kept out of line so the
// streaming loop stays small; the 8 BF16 values come by value in v).
template <int DT>
__device__ __noinline__ uint2 quantize8_exact(uint4 v, float s) {
  float f[8];
  unpack8(v, f);
  uint2 out;
  if constexpr (DT == KVQ_FP8_E4M3FN) {
    uint32_t b[4];
    for (int j = 0; j < 4; ++j) b[j] = fp8x2(__fdiv_rn(f[2 * j], s), __fdiv_rn(f[2 * j + 1], s));
    out.x = b[0] | (b[1] << 16);
    out.y = b[2] | (b[3] << 16);
  } else {
    constexpr int QM = QConst<DT>::qi;
    uint32_t w0 = 0, w1 = 0;
    for (int j = 0; j < 8; ++j) {
      const uint32_t q = static_cast<uint32_t>(qint(__fdiv_rn(f[j], s), QM));
      if constexpr (DT == KVQ_INT8) {
        if (j < 4) w0 |= (q & 0xFFu) << (8 * j); else w1 |= (q & 0xFFu) << (8 * (j - 4));
      } else {
        w0 |= (q & 0xFu) << (4 * j);
      }
    }
    out.x = w0;
    out.y = w1;
  }
  return out;
}

// Per-channel K, exact path for one row of a lane: `n` channels (2 or 4)
// packed as BF16 in w0 (and w1), each with its own scale; IEEE division.
__device__ __noinline__ uint32_t channel_row_exact(uint32_t w0, uint32_t w1, float s0, float s1, float s2,
                                                   float s3, int n) {
  const float x[4] = {bf16lo_to_f32(w0), bf16hi_to_f32(w0), bf16lo_to_f32(w1), bf16hi_to_f32(w1)};
  const float s[4] = {s0, s1, s2, s3};
  uint32_t w = 0;
  for (int c = 0; c < n; ++c) {
    const int q = s[c] == 0.f ? 0 : qint(__fdiv_rn(x[c], s[c]), 127);
    w |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * c);
  }
  return w;
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
  f[0] = bf16lo_to_f32(v.x);
  f[1] = bf16hi_to_f32(v.x);
  f[2] = bf16lo_to_f32(v.y);
  f[3] = bf16hi_to_f32(v.y);
  f[4] = bf16lo_to_f32(v.z);
  f[5] = bf16hi_to_f32(v.z);
  f[6] = bf16lo_to_f32(v.w);
  f[7] = bf16hi_to_f32(v.w);
}

// Codes of 8 consecutive values with scale s > 0, packed: INT8/FP8 -> 8 bytes
// (uint2), INT4 -> 4 bytes in .x (element 2j in the low nibble of byte j).
template <int DT>
__device__ __forceinline__ uint2 quantize8(const uint4 &v, const float (&f)[8], float s) {
  uint2 out;
  const float y = rcp_approx(s);
  const float ylo = y * kBracketDown, yhi = y * kBracketUp;
  uint32_t diff = 0;
  if constexpr (DT == KVQ_FP8_E4M3FN) {
    uint32_t b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = fp8_pair_bracket(f[2 * j], f[2 * j + 1], y, ylo, yhi, diff);
    out.x = b[0] | (b[1] << 16);
    out.y = b[2] | (b[3] << 16);
  } else {
    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) int_pair_bracket(f[2 * j], f[2 * j + 1], ylo, yhi, c[2 * j], c[2 * j + 1], diff);
    if constexpr (DT == KVQ_INT8) {
      // low bytes of c[0..3] and c[4..7]
      out.x = prmt(prmt(c[0], c[1], 0x0040u), prmt(c[2], c[3], 0x0040u), 0x5410u);
      out.y = prmt(prmt(c[4], c[5], 0x0040u), prmt(c[6], c[7], 0x0040u), 0x5410u);
    } else {
      // low nibbles, element 2j in the low nibble of byte j
      const uint32_t b0 = (c[0] & 0xFu) | ((c[1] & 0xFu) << 4);
      const uint32_t b1 = (c[2] & 0xFu) | ((c[3] & 0xFu) << 4);
      const uint32_t b2 = (c[4] & 0xFu) | ((c[5] & 0xFu) << 4);
      const uint32_t b3 = (c[6] & 0xFu) | ((c[7] & 0xFu) << 4);
      out.x = prmt(prmt(b0, b1, 0x0040u), prmt(b2, b3, 0x0040u), 0x5410u);
      out.y = 0;
    }
  }
  if (diff != 0u || s < kMinFastScale) out = quantize8_exact<DT>(v, s);
  return out;
}

// One tensor with per-token scales: PER_TOKEN_HEAD when GROUP == D, else
// PER_TOKEN_GROUP with GROUP channels per scale.  Warp `wid` of `nw` takes
// tokens wid, wid + nw, ...; RPW rows (heads) per warp step.  HT > 0 fixes the
// number of kv heads at compile time.  Pointers are formed once per token;
// every row of the token is then a constant offset.
template <int D, int DT, int GROUP, int HT>
__device__ void quantize_token_rows(const uint4 *__restrict__ x, const int64_t *__restrict__ slots,
                                    int64_t ntok, int h_rt, int64_t nslots, uint8_t *__restrict__ cache,
                                    float *__restrict__ scale, unsigned int *err, int64_t wid, int64_t nw) {
  constexpr int LPR = D / 8;                          // lanes per row
  constexpr int RPW = 32 / LPR;                       // rows per warp step
  constexpr int NST = (kMaxHeads + RPW - 1) / RPW;    // warp steps per token at most
  constexpr int LPG = GROUP / 8;                      // lanes per scale group
  constexpr int NG = D / GROUP;                       // scale groups per row
  constexpr int ROWB = (DT == KVQ_INT4) ? D / 2 : D;  // code bytes per row
  constexpr int BPL = ROWB / LPR;                     // code bytes per lane
  const int H = HT > 0 ? HT : h_rt;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR;
  const int lr = lane % LPR;
  const uint4 *xl = x + sub * LPR + lr;

  for (int64_t t = wid; t < ntok; t += nw) {
    // all of the token's rows first, then its slot
    const uint4 *xt = xl + t * H * LPR;
    uint4 v[NST];
#pragma unroll
    for (int st = 0; st < NST; ++st) {
      const int h = st * RPW + sub;
      v[st] = (h < H) ? __ldcs(xt + st * RPW * LPR) : make_uint4(0, 0, 0, 0);
    }
    const int64_t sl = __ldg(slots + t);
    if (sl < 0) continue;
    if (sl >= nslots) {
      if (lane == 0) set_error(err, KVQ_DEVERR_SLOT_RANGE);
      continue;
    }
    // row (sl, head sub) of the cache: (block * bs + offset) * H + head
    uint8_t *crow = cache + (sl * H + sub) * ROWB + lr * BPL;
    float *srow = scale + (sl * H + sub) * NG + lr / LPG;
#pragma unroll
    for (int st = 0; st < NST; ++st) {
      if (st * RPW >= H) break;
      const int h = st * RPW + sub;
      float f[8];
      unpack8(v[st], f);
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(f[j]));
#pragma unroll
      for (int m = LPG / 2; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
      if (h >= H) continue;
      const float s = scale_of<DT>(a);
      uint2 q = make_uint2(0, 0);
      if (s != 0.f) q = quantize8<DT>(v[st], f, s);
      if constexpr (DT == KVQ_INT4) {
        *reinterpret_cast<uint32_t *>(crow + st * RPW * ROWB) = q.x;
      } else {
        __stcs(reinterpret_cast<uint2 *>(crow + st * RPW * ROWB), q);
      }
      if (lr % LPG == 0) srow[st * RPW * NG] = s;
    }
  }
}

// Per-channel K: a "run" is a maximal sequence of adjacent tokens whose slots
// fall in one physical block (at most 16 tokens).  A warp task is (chunk of
// 32 tokens, head), head-minor.  The warp loads the 64 slots from the chunk
// on (one coalesced load per lane and half), finds the runs that start in the
// chunk with a ballot, and for each reduces every channel's absmax over the
// run's rows of its head, writes the block's [head, D] scales and the run's
// codes.  CPL channels per lane.
template <int D, int HT>
__device__ void quantize_block_channel(const uint16_t *__restrict__ x, const int64_t *__restrict__ slots,
                                       int64_t ntok, int h_rt, int64_t nslots, uint8_t *__restrict__ cache,
                                       float *__restrict__ scale, unsigned int *err, int64_t wid,
                                       int64_t nw) {
  constexpr int CPL = D / 32;
  constexpr int WPR = CPL / 2;  // BF16 words per lane per row
  const int H = HT > 0 ? HT : h_rt;
  const int lane = threadIdx.x & 31;
  const int64_t nchunks = (ntok + 31) / 32;
  for (int64_t task = wid; task < nchunks * H; task += nw) {
    const int64_t chunk = task / H;
    const int h = static_cast<int>(task - chunk * H);
    const int64_t t0 = chunk * 32;
    // slots of tokens t0 + lane (a) and t0 + 32 + lane (b); -1 if none
    const int64_t ta = t0 + lane, tb = t0 + 32 + lane;
    const int64_t sa = ta < ntok ? __ldg(slots + ta) : -1;
    const int64_t sb = tb < ntok ? __ldg(slots + tb) : -1;
    const int64_t sprev0 = (lane == 0 && t0 > 0) ? __ldg(slots + t0 - 1) : -1;
    const bool va = sa >= 0 && sa < nslots, vb = sb >= 0 && sb < nslots;
    if (h == 0 && sa >= nslots) set_error(err, KVQ_DEVERR_SLOT_RANGE);
    const int64_t ba = va ? sa / kBlockSize : -1, bb = vb ? sb / kBlockSize : -1;
    int64_t bprev = __shfl_up_sync(0xffffffffu, ba, 1);
    if (lane == 0) bprev = (sprev0 >= 0 && sprev0 < nslots) ? sprev0 / kBlockSize : -1;
    uint32_t starts = __ballot_sync(0xffffffffu, va && ba != bprev);
    while (starts) {
      const int s = __ffs(starts) - 1;
      starts &= starts - 1;
      const int64_t blk = __shfl_sync(0xffffffffu, ba, s);
      // run length: tokens s, s+1, ... of the 64 in the same block, at most 16
      const uint64_t same = (static_cast<uint64_t>(__ballot_sync(0xffffffffu, bb == blk)) << 32) |
                            __ballot_sync(0xffffffffu, ba == blk);
      const uint64_t from = same >> s;
      const int n = min(kBlockSize, __ffsll(static_cast<long long>(~from)) - 1);
      const int64_t ts = t0 + s;
      // the run's rows stay packed between the absmax pass and the code pass
      uint32_t raw[kBlockSize][WPR];
      float a[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) a[c] = 0.f;
#pragma unroll
      for (int j = 0; j < kBlockSize; ++j) {
        if (j < n) {
          const uint16_t *p = x + ((ts + j) * H + h) * D + lane * CPL;
          if constexpr (CPL == 4) {
            const uint2 w = __ldcs(reinterpret_cast<const uint2 *>(p));
            raw[j][0] = w.x;
            raw[j][WPR - 1] = w.y;
          } else {
            raw[j][0] = __ldcs(reinterpret_cast<const unsigned int *>(p));
          }
#pragma unroll
          for (int c = 0; c < CPL; ++c) {
            const uint32_t w = raw[j][c / 2];
            a[c] = fmaxf(a[c], fabsf((c & 1) ? bf16hi_to_f32(w) : bf16lo_to_f32(w)));
          }
        }
      }
      float sc[CPL], y[CPL];
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        sc[c] = scale_of<KVQ_INT8>(a[c]);
        y[c] = rcp_approx(sc[c]);
      }
      float *sp = scale + (blk * H + h) * D + lane * CPL;
      if constexpr (CPL == 4) {
        *reinterpret_cast<float4 *>(sp) = make_float4(sc[0], sc[1], sc[2], sc[3]);
      } else {
        *reinterpret_cast<float2 *>(sp) = make_float2(sc[0], sc[1]);
      }
#pragma unroll
      for (int j = 0; j < kBlockSize; ++j) {
        if (j < n) {
          const int pj = s + j;  // position among the 64 tokens
          const int64_t slj = pj < 32 ? __shfl_sync(__activemask(), sa, pj & 31)
                                      : __shfl_sync(__activemask(), sb, pj & 31);
          // channel pairs through the packed fast path; a row next to a
          // rounding decision (or with a tiny scale) is redone exactly
          uint32_t cw[CPL];
          float dmin = 1.0f;
#pragma unroll
          for (int c = 0; c < CPL; c += 2) {
            const uint32_t rw = raw[j][c / 2];
            float r0, r1;
            mul_f32x2(bf16lo_to_f32(rw), bf16hi_to_f32(rw), y[c], y[c + 1], r0, r1);
            const float kM = 0x1.8p23f;
            float t0, t1, n0, n1, d0, d1;
            add_f32x2(r0, r1, kM, kM, t0, t1);
            sub_f32x2(t0, t1, kM, kM, n0, n1);
            sub_f32x2(r0, r1, n0, n1, d0, d1);
            dmin = fminf(dmin, fminf(fabsf(fabsf(d0) - 0.5f), fabsf(fabsf(d1) - 0.5f)));
            // a zero scale (all-zero channel) gives code 0: t = 1.5 * 2^23 + 0
            cw[c] = sc[c] == 0.f ? 0u : __float_as_uint(t0);
            cw[c + 1] = sc[c + 1] == 0.f ? 0u : __float_as_uint(t1);
          }
          bool exact = dmin < 0x1p-14f;
#pragma unroll
          for (int c = 0; c < CPL; ++c) exact |= sc[c] != 0.f && sc[c] < kMinFastScale;
          uint32_t w;
          if constexpr (CPL == 4) {
            w = prmt(prmt(cw[0], cw[1], 0x0040u), prmt(cw[2], cw[3], 0x0040u), 0x5410u);
          } else {
            w = prmt(cw[0], cw[1], 0x0040u) & 0xFFFFu;
          }
          if (exact) {
            if constexpr (CPL == 4) {
              w = channel_row_exact(raw[j][0], raw[j][WPR - 1], sc[0], sc[1], sc[2], sc[CPL - 1], 4);
            } else {
              w = channel_row_exact(raw[j][0], 0u, sc[0], sc[1], 0.f, 0.f, 2);
            }
          }
          uint8_t *cp = cache + (slj * H + h) * D + lane * CPL;
          if constexpr (CPL == 4) {
            *reinterpret_cast<uint32_t *>(cp) = w;
          } else {
            *reinterpret_cast<uint16_t *>(cp) = static_cast<uint16_t>(w);
          }
        }
      }
    }
  }
}

template <int D, int HT>
__device__ __forceinline__ void run_k(int kf, const QuantizeArgs &a, int64_t wid, int64_t nw) {
  if (kf == K_INT8_TOK)
    quantize_token_rows<D, KVQ_INT8, D, HT>(reinterpret_cast<const uint4 *>(a.k), a.slots, a.ntok, a.H,
                                        a.nslots, a.kc, a.ks, a.err, wid, nw);
  else if (kf == K_FP8_TOK)
    quantize_token_rows<D, KVQ_FP8_E4M3FN, D, HT>(reinterpret_cast<const uint4 *>(a.k), a.slots, a.ntok, a.H,
                                              a.nslots, a.kc, a.ks, a.err, wid, nw);
  else
    quantize_block_channel<D, HT>(reinterpret_cast<const uint16_t *>(a.k), a.slots, a.ntok, a.H, a.nslots,
                              a.kc, a.ks, a.err, wid, nw);
}

template <int D, int HT>
__device__ __forceinline__ void run_v(int vf, const QuantizeArgs &a, int64_t wid, int64_t nw) {
  if (vf == V_INT8_TOK)
    quantize_token_rows<D, KVQ_INT8, D, HT>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                        a.nslots, a.vc, a.vs, a.err, wid, nw);
  else if (vf == V_FP8_TOK)
    quantize_token_rows<D, KVQ_FP8_E4M3FN, D, HT>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                              a.nslots, a.vc, a.vs, a.err, wid, nw);
  else
    quantize_token_rows<D, KVQ_INT4, 32, HT>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                         a.nslots, a.vc, a.vs, a.err, wid, nw);
}

// CTAs [0, k_blocks) quantize K, the rest quantize V.
template <int D, int KF, int VF, int HT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) quantize_write_kernel(QuantizeArgs a, int k_blocks) {
  const int warps = kThreads / 32;
  if (static_cast<int>(blockIdx.x) < k_blocks) {
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32;
    run_k<D, HT>(KF, a, wid, static_cast<int64_t>(k_blocks) * warps);
  } else {
    const int vb = gridDim.x - k_blocks;
    const int64_t wid = static_cast<int64_t>(blockIdx.x - k_blocks) * warps + threadIdx.x / 32;
    run_v<D, HT>(VF, a, wid, static_cast<int64_t>(vb) * warps);
  }
}

template <int D, int KF, int VF>
cudaError_t launch(const QuantizeArgs &a, int sms, cudaStream_t stream) {
  // one warp task per token (per-channel K: per 32-token chunk and head)
  const int warps = kThreads / 32;
  const int64_t need_v = (a.ntok + warps - 1) / warps;
  const int64_t need_k = (KF == K_INT8_CHAN) ? ((a.ntok + 31) / 32 * a.H + warps - 1) / warps : need_v;
  const int64_t cap = static_cast<int64_t>(sms) * kCtasPerSm;  // one resident wave
  // eight kv heads (Llama-3 8B / 70B layers) get a compile-time head count
  auto go = [&](int64_t kb, int64_t vb) {
    if (kb + vb <= 0) return;
    if (a.H == 8)
      quantize_write_kernel<D, KF, VF, 8><<<static_cast<unsigned>(kb + vb), kThreads, 0, stream>>>(
          a, static_cast<int>(kb));
    else
      quantize_write_kernel<D, KF, VF, 0><<<static_cast<unsigned>(kb + vb), kThreads, 0, stream>>>(
          a, static_cast<int>(kb));
  };
  constexpr bool same_code = (KF == K_INT8_TOK && VF == V_INT8_TOK) || (KF == K_FP8_TOK && VF == V_FP8_TOK);
  if (same_code || need_k + need_v <= cap) {
    // one launch: K and V run the same code (or the write is small); K and
    // V move about the same bytes, so the resident CTAs are split evenly
    int64_t kb = need_k, vb = need_v;
    if (kb + vb > cap) {
      kb = cap / 2;
      kb = kb < 1 ? 1 : (kb > need_k ? need_k : kb);
      vb = cap - kb;
      vb = vb > need_v ? need_v : vb;
    }
    go(kb, vb);
  } else {
    // different code for K and V: two launches, so the warps of an SM share
    // one instruction stream
    go(need_k < cap ? need_k : cap, 0);
    go(0, need_v < cap ? need_v : cap);
  }
  return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_d(int kf, int vf, const QuantizeArgs &a, int sms, cudaStream_t s) {
#define KVQ_QW_CASE(KF, VF) \
  if (kf == KF && vf == VF) return launch<D, KF, VF>(a, sms, s);
  KVQ_QW_CASE(K_INT8_TOK, V_INT8_TOK)
  KVQ_QW_CASE(K_INT8_TOK, V_FP8_TOK)
  KVQ_QW_CASE(K_INT8_TOK, V_INT4_G32)
  KVQ_QW_CASE(K_FP8_TOK, V_INT8_TOK)
  KVQ_QW_CASE(K_FP8_TOK, V_FP8_TOK)
  KVQ_QW_CASE(K_FP8_TOK, V_INT4_G32)
  KVQ_QW_CASE(K_INT8_CHAN, V_INT8_TOK)
  KVQ_QW_CASE(K_INT8_CHAN, V_FP8_TOK)
  KVQ_QW_CASE(K_INT8_CHAN, V_INT4_G32)
#undef KVQ_QW_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_quantize_write(int head_dim, int kf, int vf, const QuantizeArgs &a, int sms,
                                  cudaStream_t stream) {
  if (head_dim == 128) return dispatch_d<128>(kf, vf, a, sms, stream);
  if (head_dim == 64) return dispatch_d<64>(kf, vf, a, sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
