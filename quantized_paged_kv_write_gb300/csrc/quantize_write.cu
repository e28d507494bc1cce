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
// Design.  The op is a pure stream (read 2 x 2 x head_dim bytes of BF16 per
// (token, head), write codes and a scale), so the kernel is laid out for HBM:
// per-token rows are handled by a half-warp (head_dim 128) or a quarter-warp
// (head_dim 64), each lane owning one 16-byte vector of 8 BF16 values.  The
// absmax is a shuffle reduction over the lanes of the scale group, the scale
// is an IEEE correctly rounded division, and every code is the rounding of
// the correctly rounded quotient RN(x / s) (a reciprocal-based fast path is
// used only where it provably gives the same code, see below).  INT rounding
// is cvt.rni (ties to even), FP8 is cvt.rn.satfinite.e4m3x2.
// Each thread keeps UNROLL rows in flight to cover HBM latency; the grid is a
// multiple of the SM count and grid-strides over rows.  K and V are one
// launch: the first blocks of the grid take K rows, the rest V rows.
#include "common.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 4;  // 64 registers per thread -> 4 x 256 threads resident
constexpr int kUnroll = 4;

template <int DT>
struct QMax;
template <>
struct QMax<KVQ_INT8> {
  static constexpr float v = 127.0f;
};
template <>
struct QMax<KVQ_INT4> {
  static constexpr float v = 7.0f;
};
template <>
struct QMax<KVQ_FP8_E4M3FN> {
  static constexpr float v = 448.0f;
};

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

// ---------------------------------------------------------------------------
// Rounded quotients without a division per element.
//
// With y = RN(1/s) (one correctly rounded reciprocal per scale group) and
// r = RN(x * y), the exact quotient E = x / s satisfies
//   r = E (1 + e1)(1 + e2),  |e1|, |e2| <= 2^-24,
// and the correctly rounded quotient R = RN(E) = E (1 + e3), |e3| <= 2^-24,
// so |r - R| <= 3.01 * 2^-24 |E| < 2^-22 |r| as long as 1/s is a finite normal
// number (s >= 2^-125; smaller scales take the division path for the whole
// group).  Whenever every value within that distance of r rounds to the same
// code, that code is the code of R -- the code the correctly rounded division
// gives.  Otherwise (near a rounding decision, a few elements in 10^4) the
// element is recomputed with IEEE division.  The result is bit-identical to
// rounding RN(x / s).
// ---------------------------------------------------------------------------
constexpr float kMinFastScale = 0x1p-125f;

// INT: rint(R) == rint(r) unless r lies within 2^-15 of a half-integer
// (|E| <= 127 (1 + 2^-22) here, so |r - R| <= 2.3e-5 < 2^-15).
__device__ __forceinline__ int qint_fast(float x, float s, float y, int qmax) {
  const float r = x * y;
  const float n = rintf(r);
  const float f = fabsf(r - n);  // exact: r and n are within 1/2
  if (fabsf(f - 0.5f) < 0x1p-15f) return qint(__fdiv_rn(x, s), qmax);
  return min(max(static_cast<int>(n), -qmax), qmax);
}

// FP8: RNE-satfinite conversion is monotone, so if r (1 - 2^-21) and
// r (1 + 2^-21) (each rounded, still bracketing R) give the same code, R does.
__device__ __forceinline__ uint32_t fp8x2_fast(float x0, float x1, float s, float y) {
  const float r0 = x0 * y, r1 = x1 * y;
  const float kDown = 0x1.fffff0p-1f;  // 1 - 2^-21
  const float kUp = 0x1.000008p+0f;    // 1 + 2^-21
  const uint32_t c = fp8x2(r0, r1);
  const uint32_t a = fp8x2(r0 * kDown, r1 * kDown);
  const uint32_t b = fp8x2(r0 * kUp, r1 * kUp);
  if (a == c && b == c) return c;
  return fp8x2(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
}

// Quantize 8 consecutive FP32 values with scale s (s > 0) and pack them:
// INT8/FP8 -> 8 bytes (uint2), INT4 -> 4 bytes (low nibble first).
template <int DT>
__device__ __forceinline__ uint2 quantize8(const float (&f)[8], float s) {
  uint2 out;
  const bool fast = s >= kMinFastScale;
  const float y = __frcp_rn(s);
  if constexpr (DT == KVQ_FP8_E4M3FN) {
    uint32_t b[4];
    if (fast) {
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = fp8x2_fast(f[2 * j], f[2 * j + 1], s, y);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = fp8x2(__fdiv_rn(f[2 * j], s), __fdiv_rn(f[2 * j + 1], s));
    }
    out.x = b[0] | (b[1] << 16);
    out.y = b[2] | (b[3] << 16);
  } else {
    constexpr int QM = (DT == KVQ_INT8) ? 127 : 7;
    int q[8];
    if (fast) {
#pragma unroll
      for (int j = 0; j < 8; ++j) q[j] = qint_fast(f[j], s, y, QM);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) q[j] = qint(__fdiv_rn(f[j], s), QM);
    }
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

// One tensor, per-token scales (PER_TOKEN_HEAD when GROUP == D, else
// PER_TOKEN_GROUP with GROUP channels per scale).  Rows are r = t * H + h,
// contiguous in the BF16 input.  `wid` / `nw` enumerate the warps working
// on this tensor.
template <int D, int DT, int GROUP>
__device__ void quantize_token_rows(const uint4 *__restrict__ x, const int64_t *__restrict__ slots,
                                    int64_t ntok, int H, int64_t nslots, uint8_t *__restrict__ cache,
                                    float *__restrict__ scale, unsigned int *err, int64_t wid, int64_t nw) {
  constexpr int LPR = D / 8;          // lanes per row
  constexpr int RPW = 32 / LPR;       // rows per warp step
  constexpr int LPG = GROUP / 8;      // lanes per scale group
  constexpr int NG = D / GROUP;       // scale groups per row
  constexpr int ROWB = (DT == KVQ_INT4) ? D / 2 : D;
  const int lane = threadIdx.x & 31;
  const int sub = lane / LPR;         // which row of the warp step
  const int lr = lane % LPR;          // lane within the row
  const int64_t rows = ntok * H;
  const int64_t step = nw * RPW;

  for (int64_t base = wid * RPW; base < rows; base += step * kUnroll) {
    uint4 v[kUnroll];
    int64_t slot[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t r = base + u * step + sub;
      v[u] = make_uint4(0, 0, 0, 0);
      slot[u] = -1;
      if (r < rows) {
        v[u] = __ldcs(x + r * LPR + lr);
        slot[u] = __ldg(slots + r / H);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t r = base + u * step + sub;
      float f[8];
      unpack8(v[u], f);
      float a = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) a = fmaxf(a, fabsf(f[j]));
#pragma unroll
      for (int m = LPG / 2; m >= 1; m >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, m));
      if (r >= rows) continue;
      const int64_t sl = slot[u];
      if (sl < 0) continue;
      if (sl >= nslots) {
        if (lr == 0) set_error(err, KVQ_DEVERR_SLOT_RANGE);
        continue;
      }
      const int h = static_cast<int>(r % H);
      const int64_t orow = sl * H + h;  // (block * bs + offset) * H + h
      const float s = __fdiv_rn(a, QMax<DT>::v);
      uint2 q = make_uint2(0, 0);
      if (s != 0.f) q = quantize8<DT>(f, s);
      if constexpr (DT == KVQ_INT4) {
        reinterpret_cast<uint32_t *>(cache + orow * ROWB)[lr] = q.x;
      } else {
        __stcs(reinterpret_cast<uint2 *>(cache + orow * ROWB) + lr, q);
      }
      if (lr % LPG == 0) scale[orow * NG + lr / LPG] = s;
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
  const int lane = threadIdx.x & 31;
  const int64_t tasks = ntok * H;
  for (int64_t task = wid; task < tasks; task += nw) {
    const int64_t t = task / H;
    const int h = static_cast<int>(task % H);
    const int64_t sl = __ldg(slots + t);
    if (sl < 0) continue;
    if (sl >= nslots) {
      if (lane == 0 && h == 0) set_error(err, KVQ_DEVERR_SLOT_RANGE);
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
    // load the run's rows: this lane's CPL channels of head h
    // the run's rows stay packed (CPL BF16 per row in CPL/2 words) between
    // the absmax pass and the quantize pass
    constexpr int WPR = CPL / 2;
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
    float s[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) s[c] = __fdiv_rn(a[c], 127.0f);
    float y[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) y[c] = __frcp_rn(s[c]);
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
          const int q = (s[c] == 0.f) ? 0
                        : (s[c] >= kMinFastScale ? qint_fast(xv, s[c], y[c], 127)
                                                 : qint(__fdiv_rn(xv, s[c]), 127));
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
  }
}

template <int D>
__device__ __forceinline__ void run_k(int kf, const QuantizeArgs &a, int64_t wid, int64_t nw) {
  if (kf == K_INT8_TOK)
    quantize_token_rows<D, KVQ_INT8, D>(reinterpret_cast<const uint4 *>(a.k), a.slots, a.ntok, a.H,
                                        a.nslots, a.kc, a.ks, a.err, wid, nw);
  else if (kf == K_FP8_TOK)
    quantize_token_rows<D, KVQ_FP8_E4M3FN, D>(reinterpret_cast<const uint4 *>(a.k), a.slots, a.ntok, a.H,
                                              a.nslots, a.kc, a.ks, a.err, wid, nw);
  else
    quantize_block_channel<D>(reinterpret_cast<const uint16_t *>(a.k), a.slots, a.ntok, a.H, a.nslots,
                              a.kc, a.ks, a.err, wid, nw);
}

template <int D>
__device__ __forceinline__ void run_v(int vf, const QuantizeArgs &a, int64_t wid, int64_t nw) {
  if (vf == V_INT8_TOK)
    quantize_token_rows<D, KVQ_INT8, D>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                        a.nslots, a.vc, a.vs, a.err, wid, nw);
  else if (vf == V_FP8_TOK)
    quantize_token_rows<D, KVQ_FP8_E4M3FN, D>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                              a.nslots, a.vc, a.vs, a.err, wid, nw);
  else
    quantize_token_rows<D, KVQ_INT4, 32>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                         a.nslots, a.vc, a.vs, a.err, wid, nw);
}

// blocks [0, k_blocks) quantize K, the rest quantize V.
template <int D, int KF, int VF>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) quantize_write_kernel(QuantizeArgs a, int k_blocks) {
  const int warps = kThreads / 32;
  if (static_cast<int>(blockIdx.x) < k_blocks) {
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32;
    run_k<D>(KF, a, wid, static_cast<int64_t>(k_blocks) * warps);
  } else {
    const int vb = gridDim.x - k_blocks;
    const int64_t wid = static_cast<int64_t>(blockIdx.x - k_blocks) * warps + threadIdx.x / 32;
    run_v<D>(VF, a, wid, static_cast<int64_t>(vb) * warps);
  }
}

template <int D, int KF, int VF>
cudaError_t launch(const QuantizeArgs &a, int sms, cudaStream_t stream) {
  // work per tensor, in rows of D elements; per-channel K is one warp task
  // per (token, head), most of which exit after reading two slots
  const int64_t rows = a.ntok * a.H;
  constexpr int rows_per_block_step = (kThreads / 32) * (32 / (D / 8)) * kUnroll;
  const int64_t need_v = (rows + rows_per_block_step - 1) / rows_per_block_step;
  const int64_t need_k = (KF == K_INT8_CHAN) ? (rows + (kThreads / 32) - 1) / (kThreads / 32) : need_v;
  const int64_t cap = static_cast<int64_t>(sms) * kCtasPerSm;  // one resident wave
  int64_t kb = need_k, vb = need_v;
  if (kb + vb > cap) {
    // K and V move about the same bytes: split the resident blocks evenly
    kb = cap / 2;
    kb = kb < 1 ? 1 : (kb > need_k ? need_k : kb);
    vb = cap - kb;
    vb = vb > need_v ? need_v : vb;
  }
  if (kb + vb <= 0) return cudaSuccess;
  quantize_write_kernel<D, KF, VF><<<static_cast<unsigned>(kb + vb), kThreads, 0, stream>>>(
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
