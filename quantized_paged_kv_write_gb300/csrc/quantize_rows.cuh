// Row quantizer shared by the quantize-write kernel and the fused
// write + decode path (sm_103a): per-(token, head) and per-(token, group)
// symmetric quantization of BF16 rows into codes and FP32 scales.
//
// What it computes: "Use Less Memory: Quantization and Offloading", §2.1
// Symmetric Quantization Formula (s = max|x| / q_max, x_q = clip(round(x/s)))
// per scale group, stored in the cache layout of "PidokuInfra 12 KV Cache
// Quantization", §5 Where the scales live.
//
// Exactness.  Every scale is RN(absmax / q_max) and every code is the rounding
// (round half to even for INT, satfinite RNE to E4M3 for FP8) of the correctly
// rounded quotient RN(x / s), bit for bit, without a division per element:
//   * the scale uses s0 = RN(a * RN(1/q)), s = fma(fma(-s0, q, a), RN(1/q), s0),
//     which equals RN(a / q) for every BF16 absmax a and q in {127, 7, 448}
//     (checked exhaustively by tests/test_scale_sequence.py);
//   * the quotient uses Markstein's correction step (P. Markstein, "Computation
//     of elementary functions on the IBM RISC System/6000 processor", IBM J.
//     Res. Dev. 34(1), 1990; the division theorem of Muller et al., Handbook
//     of Floating-Point Arithmetic): with y = RN(1/s) (IEEE rcp.rn, once per
//     scale group), q0 = RN(x y), the residual r = x - q0 s is exact in one
//     FMA and RN(q0 + r y) = RN(x / s).  The kernels carry it negated,
//     n = -y: q0' = RN(x n), r = fma(q0', s, x), q1' = fma(r, n, q0') =
//     -RN(x / s), which also keeps the sign of a zero quotient (x = -0 gives
//     q1' = +0, the code's sign is flipped back at the end);
//     tests/test_quotient_sequence.py checks the sequence against IEEE
//     division for every BF16 x with |x| <= a, every BF16 absmax a in
//     [1, 2) (the result is invariant under scaling a and x by a power of
//     two) and edge exponents.  Scales below 2^-82 (an absmax below ~2^-75,
//     where a residual could be subnormal) take IEEE division.
#pragma once

#include "common.cuh"

namespace kvq {
namespace {

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
struct QConst<KVQ_INT2> {
  static constexpr float q = 1.0f;
  static constexpr float inv = 1.0f;  // RN(1/1)
  static constexpr int qi = 1;
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

// The division-free quotients need s >= 2^-82: below it a residual of a
// quotient the codes distinguish from 0 could fall under the binary32
// subnormal quantum (such scales mean an absmax below ~2^-75; they take IEEE
// division).
constexpr float kMinFastScale = 0x1p-82f;

// -RN(x / s) for a pair (x0, x1) with one scale each (s0, s1), given
// n = -RN(1 / s) (Markstein's correction step, see the header comment).
__device__ __forceinline__ void neg_quotient_pair(float x0, float x1, float s0, float s1, float n0, float n1,
                                                  float &q0, float &q1) {
  float a0, a1, r0, r1;
  mul_f32x2(x0, x1, n0, n1, a0, a1);          // q0' = RN(x n)
  fma_f32x2(a0, a1, s0, s1, x0, x1, r0, r1);  // r = x + q0' s, exact
  fma_f32x2(r0, r1, n0, n1, a0, a1, q0, q1);  // RN(q0' + r n) = -RN(x / s)
}

// Two's complement INT codes of a pair from their negated quotients:
// t = RN(1.5 * 2^23 - q') holds rint(-q') (ties to even: 1.5 * 2^23 is even
// and the sum's ulp is 1) in its low mantissa bits, so the code's byte or
// nibble is the low byte or nibble of t's bits.  |q'| <= q_max (1 + 2^-23)
// rounds to at most q_max: no clamp is needed.
__device__ __forceinline__ void int_codes_pair(float q0, float q1, uint32_t &c0, uint32_t &c1) {
  const float kM = 0x1.8p23f;
  float t0, t1;
  sub_f32x2(kM, kM, q0, q1, t0, t1);
  c0 = __float_as_uint(t0);
  c1 = __float_as_uint(t1);
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]);

// The exact path: IEEE division for every element.
template <int DT>
__device__ __forceinline__ uint2 codes8_exact(const float (&f)[8], float s) {
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
      } else if constexpr (DT == KVQ_INT2) {
        w0 |= (q & 0x3u) << (2 * j);
      } else {
        w0 |= (q & 0xFu) << (4 * j);
      }
    }
    out.x = w0;
    out.y = w1;
  }
  return out;
}

// Kept out of line so the streaming loop stays small; the 8 values come by
// value (BF16 in v; FP32 bits in a, b for rotated rows).
template <int DT>
__device__ __noinline__ uint2 quantize8_exact(uint4 v, float s) {
  float f[8];
  unpack8(v, f);
  return codes8_exact<DT>(f, s);
}
template <int DT>
__device__ __noinline__ uint2 quantize8_exact_f32(uint4 a, uint4 b, float s) {
  const float f[8] = {__uint_as_float(a.x), __uint_as_float(a.y), __uint_as_float(a.z), __uint_as_float(a.w),
                      __uint_as_float(b.x), __uint_as_float(b.y), __uint_as_float(b.z), __uint_as_float(b.w)};
  return codes8_exact<DT>(f, s);
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

// Codes of 8 consecutive values with scale s >= 2^-125 (n = -RN(1/s)),
// packed: INT8/FP8 -> 8 bytes (uint2), INT4 -> 4 bytes in .x (element 2j in
// the low nibble of byte j), INT2 -> 2 bytes in .x.
template <int DT>
__device__ __forceinline__ uint2 codes8(const float (&f)[8], float s, float n) {
  float q[8];
#pragma unroll
  for (int j = 0; j < 4; ++j) neg_quotient_pair(f[2 * j], f[2 * j + 1], s, s, n, n, q[2 * j], q[2 * j + 1]);
  uint2 out;
  if constexpr (DT == KVQ_FP8_E4M3FN) {
    // E4M3 of -RN(x / s), then every byte's sign flipped back
    out.x = (fp8x2(q[0], q[1]) | (fp8x2(q[2], q[3]) << 16)) ^ 0x80808080u;
    out.y = (fp8x2(q[4], q[5]) | (fp8x2(q[6], q[7]) << 16)) ^ 0x80808080u;
  } else {
    uint32_t c[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) int_codes_pair(q[2 * j], q[2 * j + 1], c[2 * j], c[2 * j + 1]);
    if constexpr (DT == KVQ_INT8) {
      // low bytes of c[0..3] and c[4..7]
      out.x = prmt(prmt(c[0], c[1], 0x0040u), prmt(c[2], c[3], 0x0040u), 0x5410u);
      out.y = prmt(prmt(c[4], c[5], 0x0040u), prmt(c[6], c[7], 0x0040u), 0x5410u);
    } else if constexpr (DT == KVQ_INT2) {
      // element 4j + m in bits 2m .. 2m + 1 of byte j (16 bits in .x)
      uint32_t w = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) w |= (c[j] & 0x3u) << (2 * j);
      out.x = w;
      out.y = 0;
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
  return out;
}

// -RN(1 / s) for a scale s > 0.
__device__ __forceinline__ float neg_recip(float s) { return -__frcp_rn(s); }

template <int DT>
__device__ __forceinline__ uint2 quantize8(const uint4 &v, const float (&f)[8], float s) {
  if (s < kMinFastScale) return quantize8_exact<DT>(v, s);
  return codes8<DT>(f, s, neg_recip(s));
}

// Same for FP32 values (rotated rows).
template <int DT>
__device__ __forceinline__ uint2 quantize8_f32(const float (&f)[8], float s) {
  if (s < kMinFastScale)
    return quantize8_exact_f32<DT>(make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                                              __float_as_uint(f[3])),
                                   make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]),
                                              __float_as_uint(f[7])),
                                   s);
  return codes8<DT>(f, s, neg_recip(s));
}

// Walsh-Hadamard rotation of one row held by LPR lanes, 8 consecutive values
// per lane (values 8 lr .. 8 lr + 7): y = H (sigma * x) by the radix-2
// butterfly, stages 1, 2, 4 inside the lane, then 8, 16, ... across lanes
// (lane xor m), each (a, b) -> (a + b, a - b) with a the lower index, so that
// every FP32 rounding matches the plain butterfly.  sigma: bit c of the
// 128-bit sign mask set means -1.  All lanes of the warp must call it.
template <int LPR>
__device__ __forceinline__ void rotate_row8(float (&f)[8], int lr, const uint32_t (&signs)[4]) {
  const uint32_t sb = (signs[lr >> 2] >> (8 * (lr & 3))) & 0xFFu;
#pragma unroll
  for (int j = 0; j < 8; ++j) f[j] = __uint_as_float(__float_as_uint(f[j]) ^ (((sb >> j) & 1u) << 31));
#pragma unroll
  for (int h = 1; h < 8; h <<= 1)
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (!(j & h)) {
        const float a = f[j], b = f[j + h];
        f[j] = a + b;
        f[j + h] = a - b;
      }
#pragma unroll
  for (int m = 1; m < LPR; m <<= 1) {
    const bool upper = (lr & m) != 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p = __shfl_xor_sync(0xffffffffu, f[j], m);
      f[j] = upper ? p - f[j] : f[j] + p;
    }
  }
}

// One token of one tensor: a half-warp (head_dim 128) or a quarter-warp (64)
// owns a row, one 16-byte vector per lane; RPW rows (heads) go per warp step.
template <int D>
struct TokenRows {
  static constexpr int LPR = D / 8;                       // lanes per row
  static constexpr int RPW = 32 / LPR;                    // rows per warp step
  static constexpr int NST = (kMaxHeads + RPW - 1) / RPW;  // warp steps per token at most
};

// Load all H rows of one token (BF16 [H, D] at xtok) into v, one vector per
// lane and warp step.  Executed by a whole warp.
template <int D, int HT>
__device__ __forceinline__ void load_token_rows(const uint4 *__restrict__ xtok, int H,
                                                uint4 (&v)[TokenRows<D>::NST]) {
  using R = TokenRows<D>;
  const int lane = threadIdx.x & 31;
  const uint4 *xl = xtok + (lane / R::LPR) * R::LPR + lane % R::LPR;
#pragma unroll
  for (int st = 0; st < R::NST; ++st) {
    const int h = st * R::RPW + lane / R::LPR;
    v[st] = (h < H) ? __ldcs(xl + st * R::RPW * R::LPR) : make_uint4(0, 0, 0, 0);
  }
}

// Quantize the loaded rows of one token into cache row slot sl (in range):
// codes at (sl * H + head) * row_bytes, scales at (sl * H + head) * NG.
// PER_TOKEN_HEAD when GROUP == D, else PER_TOKEN_GROUP with GROUP channels
// per scale.  Executed by a whole warp; the absmax is a shuffle reduction
// over the lanes of the scale group.
// With ROT, every row is first rotated (rotate_row8) and quantized from its
// FP32 values, the scale by IEEE division.
template <int D, int DT, int GROUP, int HT, bool ROT>
__device__ __forceinline__ void quantize_loaded_token(const uint4 (&v)[TokenRows<D>::NST], int64_t sl, int H,
                                                      uint8_t *__restrict__ cache, float *__restrict__ scale,
                                                      const uint32_t (&signs)[4]) {
  using R = TokenRows<D>;
  constexpr int LPG = GROUP / 8;                      // lanes per scale group
  constexpr int NG = D / GROUP;                       // scale groups per row
  constexpr int ROWB = (DT == KVQ_INT4) ? D / 2 : (DT == KVQ_INT2 ? D / 4 : D);  // code bytes per row
  constexpr int BPL = ROWB / R::LPR;                  // code bytes per lane
  const int lane = threadIdx.x & 31;
  const int sub = lane / R::LPR;
  const int lr = lane % R::LPR;
  // row (sl, head sub) of the cache: (block * bs + offset) * H + head
  uint8_t *crow = cache + (sl * H + sub) * ROWB + lr * BPL;
  float *srow = scale + (sl * H + sub) * NG + lr / LPG;
#pragma unroll
  for (int st = 0; st < R::NST; ++st) {
    if (st * R::RPW >= H) break;
    const int h = st * R::RPW + sub;
    float f[8];
    unpack8(v[st], f);
    if constexpr (ROT) rotate_row8<R::LPR>(f, lr, signs);
    float a = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(f[j]));
#pragma unroll
    for (int m = LPG / 2; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
    if (h >= H) continue;
    float s;
    if constexpr (ROT) s = __fdiv_rn(a, QConst<DT>::q);
    else s = scale_of<DT>(a);
    uint2 q = make_uint2(0, 0);
    if (s != 0.f) {
      if constexpr (ROT) q = quantize8_f32<DT>(f, s);
      else q = quantize8<DT>(v[st], f, s);
    }
    if constexpr (DT == KVQ_INT4) {
      *reinterpret_cast<uint32_t *>(crow + st * R::RPW * ROWB) = q.x;
    } else if constexpr (DT == KVQ_INT2) {
      *reinterpret_cast<uint16_t *>(crow + st * R::RPW * ROWB) = static_cast<uint16_t>(q.x);
    } else {
      __stcs(reinterpret_cast<uint2 *>(crow + st * R::RPW * ROWB), q);
    }
    if (lr % LPG == 0) srow[st * R::RPW * NG] = s;
  }
}

}  // namespace
}  // namespace kvq
