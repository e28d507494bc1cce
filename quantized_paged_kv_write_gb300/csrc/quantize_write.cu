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
// (round half to even for INT, satfinite RNE to E4M3 for FP8) of the
// correctly rounded quotient RN(x / s), bit for bit, without a division per
// element: the scale by one FMA residual correction of RN(a * RN(1/q)), the
// quotients by Markstein's correction of RN(x * RN(1/s)) (quantize_rows.cuh
// gives the argument and the tests that check it).
// K and V share one launch when they run the same code (the first CTAs of the
// grid take K, the rest V), else they go in two launches.
#include "common.cuh"
#include "kvq_internal.h"
#include "quantize_rows.cuh"

namespace kvq {
namespace {

constexpr int kThreads = 256;
constexpr int kCtasPerSm = 4;   // 64 registers per thread -> 4 x 256 threads resident
// Per-channel K, exact path for one row of a lane: `n` channels (2 or 4)
// packed as BF16 in w0 (and w1), each with its own scale; IEEE division;
// codes of `bits` bits (8: INT8, q_max 127; 2: INT2, q_max 1).
__device__ __noinline__ uint32_t channel_row_exact(uint32_t w0, uint32_t w1, float s0, float s1, float s2,
                                                   float s3, int n, int bits) {
  const float x[4] = {bf16lo_to_f32(w0), bf16hi_to_f32(w0), bf16lo_to_f32(w1), bf16hi_to_f32(w1)};
  const float s[4] = {s0, s1, s2, s3};
  const int qmax = bits == 8 ? 127 : 1;
  const uint32_t mask = (1u << bits) - 1u;
  uint32_t w = 0;
  for (int c = 0; c < n; ++c) {
    const int q = s[c] == 0.f ? 0 : qint(__fdiv_rn(x[c], s[c]), qmax);
    w |= (static_cast<uint32_t>(q) & mask) << (bits * c);
  }
  return w;
}

// One tensor with per-token scales: warp `wid` of `nw` takes tokens wid,
// wid + nw, ...; all of a token's rows are loaded before its slot, then
// quantized (quantize_rows.cuh).  HT > 0 fixes the number of kv heads at
// compile time.
template <int D, int DT, int GROUP, int HT, bool ROT>
__device__ void quantize_token_rows(const uint4 *__restrict__ x, const int64_t *__restrict__ slots,
                                    int64_t ntok, int h_rt, int64_t nslots, uint8_t *__restrict__ cache,
                                    float *__restrict__ scale, unsigned int *err, int64_t wid, int64_t nw,
                                    const uint32_t (&signs)[4]) {
  const int H = HT > 0 ? HT : h_rt;
  const int lane = threadIdx.x & 31;
  for (int64_t t = wid; t < ntok; t += nw) {
    uint4 v[TokenRows<D>::NST];
    load_token_rows<D, HT>(x + t * H * (D / 8), H, v);
    const int64_t sl = __ldg(slots + t);
    if (sl < 0) continue;
    if (sl >= nslots) {
      if (lane == 0) set_error(err, KVQ_DEVERR_SLOT_RANGE);
      continue;
    }
    quantize_loaded_token<D, DT, GROUP, HT, ROT>(v, sl, H, cache, scale, signs);
  }
}

// Per-channel K: a "run" is a maximal sequence of adjacent tokens whose slots
// fall in one physical block (at most 16 tokens).  A warp task is (chunk of
// 32 tokens, head), head-minor.  The warp loads the 64 slots from the chunk
// on (one coalesced load per lane and half), finds the runs that start in the
// chunk with a ballot, and for each reduces every channel's absmax over the
// run's rows of its head, writes the block's [head, D] scales and the run's
// codes.  CPL channels per lane.  DT: INT8 or INT2 codes (INT2 with D = 128:
// a lane's four channels make one byte).
template <int D, int HT, int DT>
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
      // In place: token s + j of the 64 goes to row j of the block, as a
      // prefill or a chunk that starts on a block boundary writes it.  The
      // block's tokens must arrive as one such run (include/kvq.h); any other
      // run is still written (its rows found through their slots) and sets
      // KVQ_DEVERR_CHANNEL_RUN, once per run (head 0's task).
      const int64_t base_slot = blk * kBlockSize;
      const bool bad_a = lane >= s && lane < s + n && sa != base_slot + (lane - s);
      const bool bad_b = lane + 32 >= s && lane + 32 < s + n && sb != base_slot + (lane + 32 - s);
      const bool in_place = !__any_sync(0xffffffffu, bad_a || bad_b);
      if (!in_place && h == 0 && lane == 0) set_error(err, KVQ_DEVERR_CHANNEL_RUN);
      // Two passes over the run's rows: the absmax of each channel (on the
      // BF16 bit patterns with the sign cleared, which order like the
      // magnitudes, two channels per word), then the codes.  8-bit codes read
      // the rows again in the second pass (L1 hits: the first pass caches
      // them) instead of holding 16 rows in registers, which spilled; 2-bit
      // codes keep them in registers (measured faster).
      constexpr bool kReload = (DT == KVQ_INT8);
      auto row_words = [&](int j, bool last) {
        const uint16_t *p = x + ((ts + j) * H + h) * D + lane * CPL;
        uint2 w = make_uint2(0u, 0u);
        if constexpr (CPL == 4) {
          w = last ? __ldcs(reinterpret_cast<const uint2 *>(p)) : __ldca(reinterpret_cast<const uint2 *>(p));
        } else {
          w.x = last ? __ldcs(reinterpret_cast<const unsigned int *>(p))
                     : __ldca(reinterpret_cast<const unsigned int *>(p));
        }
        return w;
      };
      uint2 held[kReload ? 1 : kBlockSize];
      uint32_t am[WPR];
#pragma unroll
      for (int k = 0; k < WPR; ++k) am[k] = 0u;
#pragma unroll
      for (int j = 0; j < kBlockSize; ++j) {
        if (j < n) {
          const uint2 w = row_words(j, !kReload);
          if constexpr (!kReload) held[j] = w;
          am[0] = max_u16x2(am[0], w.x & 0x7FFF7FFFu);
          if constexpr (WPR == 2) am[1] = max_u16x2(am[1], w.y & 0x7FFF7FFFu);
        }
      }
      // scales s_c = RN(a_c / q_max) and n_c = -RN(1 / s_c) (0 for a zero
      // channel: its codes come out 0)
      float sc[CPL], ng[CPL];
      bool tiny = false;
#pragma unroll
      for (int c = 0; c < CPL; ++c) {
        const float a = (c & 1) ? bf16hi_to_f32(am[c / 2]) : bf16lo_to_f32(am[c / 2]);
        sc[c] = scale_of<DT>(a);
        ng[c] = sc[c] == 0.f ? 0.f : neg_recip(sc[c]);
        tiny |= sc[c] != 0.f && sc[c] < kMinFastScale;
      }
      float *sp = scale + (blk * H + h) * D + lane * CPL;
      if constexpr (CPL == 4) {
        *reinterpret_cast<float4 *>(sp) = make_float4(sc[0], sc[1], sc[2], sc[3]);
      } else {
        *reinterpret_cast<float2 *>(sp) = make_float2(sc[0], sc[1]);
      }
      constexpr int BITS = (DT == KVQ_INT2) ? 2 : 8;
      constexpr int RB = D * BITS / 8;  // code bytes per row
      uint8_t *const cbase = cache + (base_slot * H + h) * RB + lane * (CPL * BITS / 8);
#pragma unroll
      for (int j = 0; j < kBlockSize; ++j) {
        if (j < n) {
          // codes of the lane's channels: Markstein quotients (quantize_rows.cuh)
          const uint2 rwj = kReload ? row_words(j, true) : held[kReload ? 0 : j];
          const uint32_t raw[2] = {rwj.x, rwj.y};
          uint32_t cw[CPL];
#pragma unroll
          for (int c = 0; c < CPL; c += 2) {
            const uint32_t rw = raw[c / 2];
            float q0, q1;
            neg_quotient_pair(bf16lo_to_f32(rw), bf16hi_to_f32(rw), sc[c], sc[c + 1], ng[c], ng[c + 1], q0, q1);
            int_codes_pair(q0, q1, cw[c], cw[c + 1]);
          }
          uint32_t w;
          if constexpr (DT == KVQ_INT2) {
            w = (cw[0] & 3u) | ((cw[1] & 3u) << 2) | ((cw[2] & 3u) << 4) | ((cw[3] & 3u) << 6);
          } else if constexpr (CPL == 4) {
            w = prmt(prmt(cw[0], cw[1], 0x0040u), prmt(cw[2], cw[3], 0x0040u), 0x5410u);
          } else {
            w = prmt(cw[0], cw[1], 0x0040u) & 0xFFFFu;
          }
          if (tiny) {  // a scale below 2^-125: IEEE division
            if constexpr (CPL == 4) {
              w = channel_row_exact(raw[0], raw[1], sc[0], sc[1], sc[2], sc[CPL - 1], 4, BITS);
            } else {
              w = channel_row_exact(raw[0], 0u, sc[0], sc[1], 0.f, 0.f, 2, BITS);
            }
          }
          int64_t row = j;
          if (!in_place) {
            const int pj = s + j;  // position among the 64 tokens
            const int64_t slj = pj < 32 ? __shfl_sync(0xffffffffu, sa, pj & 31)
                                        : __shfl_sync(0xffffffffu, sb, pj & 31);
            row = slj - base_slot;
          }
          uint8_t *cp = cbase + row * H * RB;
          if constexpr (DT == KVQ_INT2) {
            *cp = static_cast<uint8_t>(w);
          } else if constexpr (CPL == 4) {
            *reinterpret_cast<uint32_t *>(cp) = w;
          } else {
            *reinterpret_cast<uint16_t *>(cp) = static_cast<uint16_t>(w);
          }
        }
      }
    }
  }
}

template <int D, int HT, bool ROT>
__device__ __forceinline__ void run_k(int kf, const QuantizeArgs &a, int64_t wid, int64_t nw) {
  if (kf == K_INT8_TOK)
    quantize_token_rows<D, KVQ_INT8, D, HT, ROT>(reinterpret_cast<const uint4 *>(a.k), a.slots, a.ntok, a.H,
                                        a.nslots, a.kc, a.ks, a.err, wid, nw, a.rot_signs);
  else if (kf == K_FP8_TOK)
    quantize_token_rows<D, KVQ_FP8_E4M3FN, D, HT, ROT>(reinterpret_cast<const uint4 *>(a.k), a.slots, a.ntok, a.H,
                                              a.nslots, a.kc, a.ks, a.err, wid, nw, a.rot_signs);
  else if (kf == K_INT4_TOK)
    quantize_token_rows<D, KVQ_INT4, D, HT, ROT>(reinterpret_cast<const uint4 *>(a.k), a.slots, a.ntok, a.H,
                                        a.nslots, a.kc, a.ks, a.err, wid, nw, a.rot_signs);
  else if (kf == K_INT2_CHAN) {
    if constexpr (D == 128)
      quantize_block_channel<D, HT, KVQ_INT2>(reinterpret_cast<const uint16_t *>(a.k), a.slots, a.ntok, a.H,
                                              a.nslots, a.kc, a.ks, a.err, wid, nw);
  } else {
    quantize_block_channel<D, HT, KVQ_INT8>(reinterpret_cast<const uint16_t *>(a.k), a.slots, a.ntok, a.H,
                                            a.nslots, a.kc, a.ks, a.err, wid, nw);
  }
}

template <int D, int HT, bool ROT>
__device__ __forceinline__ void run_v(int vf, const QuantizeArgs &a, int64_t wid, int64_t nw) {
  if (vf == V_INT8_TOK)
    quantize_token_rows<D, KVQ_INT8, D, HT, ROT>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                        a.nslots, a.vc, a.vs, a.err, wid, nw, a.rot_signs);
  else if (vf == V_FP8_TOK)
    quantize_token_rows<D, KVQ_FP8_E4M3FN, D, HT, ROT>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                              a.nslots, a.vc, a.vs, a.err, wid, nw, a.rot_signs);
  else if (vf == V_INT4_G32)
    quantize_token_rows<D, KVQ_INT4, 32, HT, ROT>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                         a.nslots, a.vc, a.vs, a.err, wid, nw, a.rot_signs);
  else if constexpr (D == 128)
    quantize_token_rows<D, KVQ_INT2, 32, HT, ROT>(reinterpret_cast<const uint4 *>(a.v), a.slots, a.ntok, a.H,
                                         a.nslots, a.vc, a.vs, a.err, wid, nw, a.rot_signs);
}

// CTAs [0, k_blocks) quantize K, the rest quantize V.
template <int D, int KF, int VF, int HT, bool ROT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) quantize_write_kernel(QuantizeArgs a, int k_blocks) {
  const int warps = kThreads / 32;
  if (static_cast<int>(blockIdx.x) < k_blocks) {
    const int64_t wid = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32;
    run_k<D, HT, ROT>(KF, a, wid, static_cast<int64_t>(k_blocks) * warps);
  } else {
    const int vb = gridDim.x - k_blocks;
    const int64_t wid = static_cast<int64_t>(blockIdx.x - k_blocks) * warps + threadIdx.x / 32;
    run_v<D, HT, ROT>(VF, a, wid, static_cast<int64_t>(vb) * warps);
  }
}

template <int D, int KF, int VF>
cudaError_t launch(const QuantizeArgs &a, int sms, cudaStream_t stream) {
  // one warp task per token (per-channel K: per 32-token chunk and head)
  const int warps = kThreads / 32;
  const int64_t need_v = (a.ntok + warps - 1) / warps;
  const int64_t need_k = (KF == K_INT8_CHAN || KF == K_INT2_CHAN) ? ((a.ntok + 31) / 32 * a.H + warps - 1) / warps
                                                                 : need_v;
  const int64_t cap = static_cast<int64_t>(sms) * kCtasPerSm;  // one resident wave
  // eight kv heads (Llama-3 8B / 70B layers) get a compile-time head count
  auto go = [&](int64_t kb, int64_t vb) {
    if (kb + vb <= 0) return;
    if constexpr (KF != K_INT8_CHAN && KF != K_INT2_CHAN) {
      if (a.rot) {  // rotated rows: a runtime head count only
        quantize_write_kernel<D, KF, VF, 0, true><<<static_cast<unsigned>(kb + vb), kThreads, 0, stream>>>(
            a, static_cast<int>(kb));
        return;
      }
    }
    if (a.H == 8)
      quantize_write_kernel<D, KF, VF, 8, false><<<static_cast<unsigned>(kb + vb), kThreads, 0, stream>>>(
          a, static_cast<int>(kb));
    else
      quantize_write_kernel<D, KF, VF, 0, false><<<static_cast<unsigned>(kb + vb), kThreads, 0, stream>>>(
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
  KVQ_QW_CASE(K_INT4_TOK, V_INT8_TOK)
  KVQ_QW_CASE(K_INT4_TOK, V_FP8_TOK)
  KVQ_QW_CASE(K_INT4_TOK, V_INT4_G32)
  if constexpr (D == 128) {  // INT2 rows: head_dim 128
    KVQ_QW_CASE(K_INT8_TOK, V_INT2_G32)
    KVQ_QW_CASE(K_FP8_TOK, V_INT2_G32)
    KVQ_QW_CASE(K_INT8_CHAN, V_INT2_G32)
    KVQ_QW_CASE(K_INT4_TOK, V_INT2_G32)
    KVQ_QW_CASE(K_INT2_CHAN, V_INT8_TOK)
    KVQ_QW_CASE(K_INT2_CHAN, V_FP8_TOK)
    KVQ_QW_CASE(K_INT2_CHAN, V_INT4_G32)
    KVQ_QW_CASE(K_INT2_CHAN, V_INT2_G32)
  }
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
