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
//   * the quotient uses r = RN(x * y) with y = rcp.approx(s) (relative error
//     below 2^-23): |r - RN(x / s)| < 2^-21.9 |r|, so whenever every value that
//     close to r rounds to the same code, that is the code; otherwise (a few
//     elements in 10^4, next to a rounding decision) the element is redone
//     with IEEE division.
// K and V share one launch: the first CTAs of the grid take K, the rest V.
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

// INT: |E| <= q_max (1 + 2^-22) <= 127.1, so |r - RN(E)| < 127.1 * 2^-21.9
// < 2^-14; rint(RN(E)) == rint(r) unless r is within 2^-14 of a half-integer
// (then `near` is set and the caller redoes the group exactly).
__device__ __forceinline__ int qint_fast(float x, float y, int qmax, bool &near) {
  const float r = x * y;
  const float n = rintf(r);
  near |= fabsf(fabsf(r - n) - 0.5f) < 0x1p-14f;
  return min(max(static_cast<int>(n), -qmax), qmax);
}

// Packed FP32 pair multiply (Blackwell f32x2): {a0, a1} * {b0, b1}, each
// product rounded to nearest even like the scalar multiply.
__device__ __forceinline__ void mul_f32x2(float a0, float a1, float b0, float b1, float &d0, float &d1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// FP8: RNE-satfinite conversion is monotone; r (1 -/+ 2^-20), each rounded,
// still bracket RN(E), so equal codes at both ends are the code of RN(E);
// otherwise `diff` is nonzero and the caller redoes the group exactly.
__device__ __forceinline__ uint32_t fp8x2_fast(float x0, float x1, float y, uint32_t &diff) {
  const float kDown = 0x1.ffffe0p-1f;  // 1 - 2^-20
  const float kUp = 0x1.000010p+0f;    // 1 + 2^-20
  float r0, r1, l0, l1, h0, h1;
  mul_f32x2(x0, x1, y, y, r0, r1);
  mul_f32x2(r0, r1, kDown, kDown, l0, l1);
  mul_f32x2(r0, r1, kUp, kUp, h0, h1);
  const uint32_t c = fp8x2(r0, r1);
  const uint32_t lo = fp8x2(l0, l1);
  const uint32_t hi = fp8x2(h0, h1);
  diff |= (lo ^ c) | (hi ^ c);
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
  bool exact = s < kMinFastScale;
  if constexpr (DT == KVQ_FP8_E4M3FN) {
    uint32_t diff = 0, b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = fp8x2_fast(f[2 * j], f[2 * j + 1], y, diff);
    out.x = b[0] | (b[1] << 16);
    out.y = b[2] | (b[3] << 16);
    exact |= diff != 0u;
  } else {
    constexpr int QM = QConst<DT>::qi;
    int q[8];
    bool near = false;
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = qint_fast(f[j], y, QM, near);
    if constexpr (DT == KVQ_INT8) {
      out.x = (q[0] & 0xFF) | ((q[1] & 0xFF) << 8) | ((q[2] & 0xFF) << 16) | (static_cast<uint32_t>(q[3]) << 24);
      out.y = (q[4] & 0xFF) | ((q[5] & 0xFF) << 8) | ((q[6] & 0xFF) << 16) | (static_cast<uint32_t>(q[7]) << 24);
    } else {
      uint32_t w = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) w |= (static_cast<uint32_t>(q[j]) & 0xFu) << (4 * j);
      out.x = w;
      out.y = 0;
    }
    exact |= near;
  }
  if (exact) out = quantize8_exact<DT>(v, s);
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
// fall in one physical block.  The warp owning (run start, head) reduces each
// channel's absmax over the run's rows, writes the block's [head, D] scales
// and the run's codes.  CPL channels per lane.
template <int D>
__device__ void quantize_block_channel(const uint16_t *__restrict__ x, const int64_t *__restrict__ slots,
                                       int64_t ntok, int H, int64_t nslots, uint8_t *__restrict__ cache,
                                       float *__restrict__ scale, unsigned int *err, int64_t wid,
                                       int64_t nw) {
  constexpr int CPL = D / 32;
  constexpr int WPR = CPL / 2;  // BF16 words per lane per row
  const int lane = threadIdx.x & 31;
  for (int64_t t = wid; t < ntok; t += nw) {
    const int64_t sl = __ldg(slots + t);
    if (sl < 0) continue;
    if (sl >= nslots) {
      if (lane == 0) set_error(err, KVQ_DEVERR_SLOT_RANGE);
      continue;
    }
    const int64_t blk = sl / kBlockSize;
    if (t > 0) {
      const int64_t prev = __ldg(slots + t - 1);
      if (prev >= 0 && prev < nslots && prev / kBlockSize == blk) continue;  // not a run start
    }
    int n = 1;
    while (n < kBlockSize && t + n < ntok) {
      const int64_t nx = __ldg(slots + t + n);
      if (nx < 0 || nx >= nslots || nx / kBlockSize != blk) break;
      ++n;
    }
    for (int h = 0; h < H; ++h) {
    // the run's rows stay packed between the absmax pass and the code pass
    uint32_t raw[kBlockSize][WPR];
    float a[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) a[c] = 0.f;
#pragma unroll
    for (int j = 0; j < kBlockSize; ++j) {
      if (j < n) {
        const uint16_t *p = x + ((t + j) * H + h) * D + lane * CPL;
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
    float s[CPL], y[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      s[c] = scale_of<KVQ_INT8>(a[c]);
      y[c] = rcp_approx(s[c]);
    }
    float *sp = scale + (blk * H + h) * D + lane * CPL;
    if constexpr (CPL == 4) {
      *reinterpret_cast<float4 *>(sp) = make_float4(s[0], s[1], s[2], s[3]);
    } else {
      *reinterpret_cast<float2 *>(sp) = make_float2(s[0], s[1]);
    }
#pragma unroll
    for (int j = 0; j < kBlockSize; ++j) {
      if (j < n) {
        const int64_t slj = __ldg(slots + t + j);
        uint32_t w = 0;
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const uint32_t rw = raw[j][c / 2];
          const float xv = (c & 1) ? bf16hi_to_f32(rw) : bf16lo_to_f32(rw);
          bool near = s[c] < kMinFastScale;
          int q = qint_fast(xv, y[c], 127, near);
          if (near) q = qint(__fdiv_rn(xv, s[c]), 127);
          if (s[c] == 0.f) q = 0;
          w |= (static_cast<uint32_t>(q) & 0xFFu) << (8 * c);
        }
        uint8_t *cp = cache + (slj * H + h) * D + lane * CPL;
        if constexpr (CPL == 4) {
          *reinterpret_cast<uint32_t *>(cp) = w;
        } else {
          *reinterpret_cast<uint16_t *>(cp) = static_cast<uint16_t>(w);
        }
      }
    }
    }  // heads
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
    quantize_block_channel<D>(reinterpret_cast<const uint16_t *>(a.k), a.slots, a.ntok, a.H, a.nslots,
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
  // one warp task per token for both tensors (per-channel K: tokens that do
  // not start a run exit after reading two slots)
  const int warps = kThreads / 32;
  const int64_t need_v = (a.ntok + warps - 1) / warps;
  const int64_t need_k = need_v;
  const int64_t cap = static_cast<int64_t>(sms) * kCtasPerSm;  // one resident wave
  int64_t kb = need_k, vb = need_v;
  if (kb + vb > cap) {
    // K and V move about the same bytes: split the resident CTAs evenly
    kb = cap / 2;
    kb = kb < 1 ? 1 : (kb > need_k ? need_k : kb);
    vb = cap - kb;
    vb = vb > need_v ? need_v : vb;
  }
  if (kb + vb <= 0) return cudaSuccess;
  // eight kv heads (Llama-3 8B / 70B layers) get a compile-time head count
  if (a.H == 8)
    quantize_write_kernel<D, KF, VF, 8><<<static_cast<unsigned>(kb + vb), kThreads, 0, stream>>>(
        a, static_cast<int>(kb));
  else
    quantize_write_kernel<D, KF, VF, 0><<<static_cast<unsigned>(kb + vb), kThreads, 0, stream>>>(
        a, static_cast<int>(kb));
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
