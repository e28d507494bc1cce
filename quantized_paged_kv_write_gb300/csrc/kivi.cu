// Per-channel K caches that take appends (sm_103a): the tokens of a
// sequence's incomplete last block stay in full precision in a residual
// buffer; the token that completes a block triggers its quantization.
//
// What it computes: "Quantized KV caches in production: FP8 vs INT8 vs
// INT4", Numerical Formats (KIVI: K per channel, V per token) with the
// per-channel scale spanning a block's tokens ("PidokuInfra 12 KV Cache
// Quantization", K is more sensitive than V).  The residual row of position
// p is p % 16; the block is quantized exactly as kvq_quantize_write would
// quantize its 16 tokens written in one call.
//
// One CTA per sequence: its threads copy the new K and V rows into the
// residual; when the block is complete, warp h reduces head h's channels over
// the 16 rows (lane: D / 32 channels) and writes the block's [h, D] scales
// and codes with IEEE division (this runs once per 16 steps of a sequence);
// then the warps quantize the 16 V rows with the row quantizer of the
// quantize-write kernel.
#include "common.cuh"
#include "kvq_internal.h"
#include "quantize_rows.cuh"

namespace kvq {
namespace {

constexpr int kKvThreads = 256;

template <int D, int KF, int VF, int HT>
__global__ void __launch_bounds__(kKvThreads) kivi_append_kernel(const KiviAppendArgs a) {
  constexpr int VDT = (VF == V_FP8_TOK) ? KVQ_FP8_E4M3FN
                      : (VF == V_INT4_G32 ? KVQ_INT4 : (VF == V_INT2_G32 ? KVQ_INT2 : KVQ_INT8));
  constexpr int VGROUP = (VF == V_INT4_G32 || VF == V_INT2_G32) ? 32 : D;
  constexpr int CPL = D / 32;                      // K channels per lane
  constexpr int KBITS = (KF == K_INT2_CHAN) ? 2 : 8;
  constexpr int KQMAX = (KF == K_INT2_CHAN) ? 1 : 127;
  constexpr int KRB = D * KBITS / 8;               // K code bytes per row
  const int H = HT > 0 ? HT : a.H;
  const int b = blockIdx.x;
  const int n = __ldg(a.ctx + b);
  if (n < 1) return;
  if (n / kBlockSize > a.max_blocks) {  // only complete blocks need table entries
    if (threadIdx.x == 0) set_error(a.err, KVQ_DEVERR_CONTEXT_RANGE);
    return;
  }
  const int r = (n - 1) % kBlockSize;
  const int row16 = H * D / 8;  // 16-byte vectors per token (all heads)
  const uint4 *kn = reinterpret_cast<const uint4 *>(a.knew) + static_cast<int64_t>(b) * row16;
  const uint4 *vn = reinterpret_cast<const uint4 *>(a.vnew) + static_cast<int64_t>(b) * row16;
  uint4 *rk = reinterpret_cast<uint4 *>(a.res_k) + (static_cast<int64_t>(b) * kBlockSize + r) * row16;
  uint4 *rv = reinterpret_cast<uint4 *>(a.res_v) + (static_cast<int64_t>(b) * kBlockSize + r) * row16;
  for (int i = threadIdx.x; i < row16; i += kKvThreads) {
    rk[i] = kn[i];
    rv[i] = vn[i];
  }
  if (n % kBlockSize != 0) return;
  __syncthreads();  // the block's 16 residual rows are complete

  const int blk = __ldg(a.tables + static_cast<int64_t>(b) * a.max_blocks + (n - 1) / kBlockSize);
  if (blk < 0 || blk >= a.num_blocks) {
    if (threadIdx.x == 0) set_error(a.err, KVQ_DEVERR_BLOCK_RANGE);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint16_t *res_k = a.res_k + static_cast<int64_t>(b) * kBlockSize * H * D;
  // K: per (head, channel) over the 16 rows
  auto kval = [&](int t, int h, int c) -> float {
    return __uint_as_float(static_cast<uint32_t>(res_k[(static_cast<int64_t>(t) * H + h) * D + lane * CPL + c]) << 16);
  };
  for (int h = warp; h < H; h += kKvThreads / 32) {
    float amax[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) amax[c] = 0.f;
    for (int t = 0; t < kBlockSize; ++t)
#pragma unroll
      for (int c = 0; c < CPL; ++c) amax[c] = fmaxf(amax[c], fabsf(kval(t, h, c)));
    float s[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      s[c] = __fdiv_rn(amax[c], static_cast<float>(KQMAX));
      a.ks[(static_cast<int64_t>(blk) * H + h) * D + lane * CPL + c] = s[c];
    }
    for (int t = 0; t < kBlockSize; ++t) {
      uint32_t w = 0;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const int q = s[c] == 0.f ? 0 : qint(__fdiv_rn(kval(t, h, c), s[c]), KQMAX);
        w |= (static_cast<uint32_t>(q) & ((1u << KBITS) - 1u)) << (KBITS * c);
      }
      uint8_t *dst = a.kc + ((static_cast<int64_t>(blk) * kBlockSize + t) * H + h) * KRB + lane * (CPL * KBITS / 8);
      if constexpr (KBITS == 2) {
        *dst = static_cast<uint8_t>(w);
      } else if constexpr (CPL == 4) {
        *reinterpret_cast<uint32_t *>(dst) = w;
      } else {
        *reinterpret_cast<uint16_t *>(dst) = static_cast<uint16_t>(w);
      }
    }
  }
  // V: the 16 rows, one token per warp step
  const uint32_t no_signs[4] = {0u, 0u, 0u, 0u};
  for (int t = warp; t < kBlockSize; t += kKvThreads / 32) {
    uint4 v[TokenRows<D>::NST];
    load_token_rows<D, HT>(reinterpret_cast<const uint4 *>(a.res_v) + (static_cast<int64_t>(b) * kBlockSize + t) * row16,
                           H, v);
    quantize_loaded_token<D, VDT, VGROUP, HT, false>(v, static_cast<int64_t>(blk) * kBlockSize + t, H, a.vc, a.vs,
                                                     no_signs);
  }
}

template <int D, int KF, int VF>
cudaError_t launch_d_vf(const KiviAppendArgs &a, cudaStream_t stream) {
  if (a.H == 8)
    kivi_append_kernel<D, KF, VF, 8><<<a.B, kKvThreads, 0, stream>>>(a);
  else
    kivi_append_kernel<D, KF, VF, 0><<<a.B, kKvThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int D, int KF>
cudaError_t launch_d(int vf, const KiviAppendArgs &a, cudaStream_t stream) {
  if (vf == V_INT8_TOK) return launch_d_vf<D, KF, V_INT8_TOK>(a, stream);
  if (vf == V_FP8_TOK) return launch_d_vf<D, KF, V_FP8_TOK>(a, stream);
  if (vf == V_INT4_G32) return launch_d_vf<D, KF, V_INT4_G32>(a, stream);
  if constexpr (D == 128) {
    if (vf == V_INT2_G32) return launch_d_vf<D, KF, V_INT2_G32>(a, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_kivi_append(int head_dim, int kf, int vf, const KiviAppendArgs &a, cudaStream_t stream) {
  if (a.B <= 0) return cudaSuccess;
  if (head_dim == 128)
    return kf == K_INT2_CHAN ? launch_d<128, K_INT2_CHAN>(vf, a, stream) : launch_d<128, K_INT8_CHAN>(vf, a, stream);
  if (head_dim == 64 && kf == K_INT8_CHAN) return launch_d<64, K_INT8_CHAN>(vf, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
