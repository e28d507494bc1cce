// Internal interfaces between the C-ABI layer (kvq_api.cu) and the kernel
// translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

struct QuantizeArgs {
  const void *k;          // BF16 [ntok, H, D]
  const void *v;          // BF16 [ntok, H, D]
  const int64_t *slots;   // [ntok]
  int64_t ntok;
  int H;
  int64_t nslots;         // num_blocks * block_size
  uint8_t *kc, *vc;       // code caches
  float *ks, *vs;         // scale arrays
  unsigned int *err;      // sticky error word of this device
  int rot = 0;            // 1: Walsh-Hadamard rotation of every row (include/kvq.h)
  uint32_t rot_signs[4] = {0u, 0u, 0u, 0u};
};

cudaError_t launch_quantize_write(int head_dim, int kf, int vf, const QuantizeArgs &a, int sms,
                                  cudaStream_t stream);

struct DecodeArgs {
  const uint16_t *q;           // BF16 [B, Hq, D]
  const float *ks;             // K scales (layout by granularity)
  const float *vs;             // V scales
  const int32_t *tables;       // [B, max_blocks]
  const int32_t *ctx;          // [B]
  float *ws_o;                 // partial O^T, column-major: [slots, H, 8, D]
  float *ws_ml;                // partial (m, l): [slots, H, 8, 2]
  int *ws_cum;                 // block-count prefix sums [B + 1]
  float *out;                  // [B, Hq, D]
  unsigned int *err;
  int64_t num_blocks;
  int B, Hq, H, G;
  int max_blocks;
  int max_ctx;
  int nctas;                   // P: CTAs of the split kernel
  int rot = 0;                 // 1: rotated cache (include/kvq.h): rotate q, rotate the output back
  uint32_t rot_signs[4] = {0u, 0u, 0u, 0u};
  // Fused write (kvq_write_decode): the step's new K and V, one token per
  // sequence at position ctx - 1, BF16 [B, H, D]; null for a plain decode.
  const uint16_t *knew = nullptr, *vnew = nullptr;
  // Per-channel K with a full-precision tail (kvq_kivi_decode): the split
  // covers the complete blocks only; the reduce adds the residual rows
  // [16 floor(n / 16), n), BF16 [B, 16, H, D]; null otherwise.
  const uint16_t *res_k = nullptr, *res_v = nullptr;
  uint8_t *kc_w = nullptr, *vc_w = nullptr;  // code caches (written)
  float *ks_w = nullptr, *vs_w = nullptr;    // scales (written)
};

// Launch plan of the split kernel for one shape on the current device.
struct DecodePlan {
  int nstages = 0;       // pipeline depth
  size_t smem = 0;       // dynamic shared memory bytes
  int threads = 0;       // 32 * (H + 1)
  int ctas_per_sm = 0;   // occupancy
  int max_ctas = 0;      // SMs * ctas_per_sm: bound of P, sizes the workspace
};

// TMA descriptors of one decode call: K and V code caches (one (block, head)
// tile per load) and, for INT4 V with four group scales per row, the V scale
// array (one (block, head) [16 tokens][4] tile per load; otherwise a copy of
// v, unused).
struct DecodeMaps {
  CUtensorMap k, v, vs;
};


// Block prefetch from the host pool (prefetch.cu).  Piece sizes are in
// 16-byte vectors per block; host pointers are device-accessible addresses of
// pinned host memory.
struct PrefetchArgs {
  const int32_t *src, *dst;  // [n] host block, device block slot
  int64_t n;
  int64_t host_nb, dev_nb;
  const uint4 *hk, *hv, *hks, *hvs;
  uint4 *dk, *dv, *dks, *dvs;
  int64_t kb16, vb16, ksb16, vsb16;
  unsigned int *err;
};
cudaError_t launch_prefetch(const PrefetchArgs &a, int sms, cudaStream_t stream);

// Append to a per-channel K cache with a full-precision tail (kivi.cu).
struct KiviAppendArgs {
  const uint16_t *knew, *vnew;   // BF16 [B, H, D]: one token per sequence
  uint16_t *res_k, *res_v;       // BF16 [B, 16, H, D] residual rows
  const int32_t *tables;         // [B, max_blocks]
  const int32_t *ctx;            // [B] lengths after the append (0: none)
  uint8_t *kc, *vc;
  float *ks, *vs;
  unsigned int *err;
  int64_t num_blocks;
  int B, H, max_blocks;
};
cudaError_t launch_kivi_append(int head_dim, int kf, int vf, const KiviAppendArgs &a, cudaStream_t stream);

// (dispatch lives in kvq_api.cu)

// Per-format entry points defined in the decode_k*.cu translation units.
template <int KF>
cudaError_t plan_decode_kf(int head_dim, int vf, int H, int G, int B, bool rot, DecodePlan *plan);
template <int KF>
cudaError_t launch_decode_kf(int head_dim, int vf, const DecodeArgs &a, const DecodePlan &plan,
                             const DecodeMaps &maps, cudaStream_t stream);

}  // namespace kvq
