// Prefetch of offloaded cache blocks from pinned host memory into device
// block slots (sm_103a).
//
// What it computes: "Use Less Memory: Quantization and Offloading", §3 (CPU
// RAM holds the KV blocks that do not fit in HBM) and §4 Pipelining and
// Latency Overlap (the blocks the next step needs are copied into a second
// set of GPU buffers while the current step computes).  Block src[i] of the
// host pool (codes and scales, in the cache's own per-block layout) goes to
// block slot dst[i] of the device cache, unchanged.
//
// Design.  One kernel gathers all pairs: a CTA owns one of a block's four
// pieces (K codes, V codes, K scales, V scales; each a multiple of 16 bytes)
// for pairs i, i + grid, ..., read straight from host memory over the
// CPU-GPU link into HBM, two 16-byte loads in flight per thread before the
// stores.
// A launch stands in for one small copy per piece and block.  The grid is
// about one CTA per SM, with no shared memory, at most 40 registers per
// thread and the decode's L1 / shared split, so a CTA fits on an SM beside the
// two CTAs of a running decode (their 96 registers x 288 threads x 2 leave
// room for 256 x 40): the prefetch overlaps the decode instead of queueing
// behind it or in front of it.
#include <atomic>

#include "common.cuh"
#include "kvq_internal.h"

namespace kvq {
namespace {

constexpr int kPfThreads = 256;
constexpr int kPfUnroll = 2;

// n16 vectors of one block piece (under 2^31)
__device__ __forceinline__ void copy_vecs(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int n16) {
  for (int base = threadIdx.x; base < n16; base += kPfThreads * kPfUnroll) {
    uint4 v[kPfUnroll];
#pragma unroll
    for (int u = 0; u < kPfUnroll; ++u) {
      const int k = base + u * kPfThreads;
      if (k < n16) v[u] = src[k];
    }
#pragma unroll
    for (int u = 0; u < kPfUnroll; ++u) {
      const int k = base + u * kPfThreads;
      if (k < n16) dst[k] = v[u];
    }
  }
}

// at most 40 registers per thread (6 CTAs' worth per SM), so that a CTA fits
// beside two decode CTAs
// CTA (x, piece): piece 0..3 = K codes, V codes, K scales, V scales; pairs
// x, x + gridDim.x, ...
__global__ void __launch_bounds__(kPfThreads, 6) prefetch_blocks_kernel(const PrefetchArgs a) {
  const int piece = blockIdx.y;
  const uint4 *hs = piece == 0 ? a.hk : piece == 1 ? a.hv : piece == 2 ? a.hks : a.hvs;
  uint4 *ds = piece == 0 ? a.dk : piece == 1 ? a.dv : piece == 2 ? a.dks : a.dvs;
  const int64_t n16 = piece == 0 ? a.kb16 : piece == 1 ? a.vb16 : piece == 2 ? a.ksb16 : a.vsb16;
  for (int64_t i = blockIdx.x; i < a.n; i += gridDim.x) {
    const int32_t s = a.src[i], d = a.dst[i];
    if (s < 0 || s >= a.host_nb || d < 0 || d >= a.dev_nb) {
      if (threadIdx.x == 0 && piece == 0) set_error(a.err, KVQ_DEVERR_BLOCK_RANGE);
      continue;
    }
    copy_vecs(hs + s * n16, ds + d * n16, static_cast<int>(n16));
  }
}

constexpr int kPfMaxDevices = 64;
std::atomic<bool> g_carveout_set[kPfMaxDevices];

}  // namespace

cudaError_t launch_prefetch(const PrefetchArgs &a, int sms, cudaStream_t stream) {
  if (a.n <= 0) return cudaSuccess;
  // about one CTA per SM in all (a quarter of them per piece)
  const int64_t per_piece = (sms / 4 > 0) ? sms / 4 : 1;
  const int64_t ctas = a.n < per_piece ? a.n : per_piece;
  // the same L1 / shared split as the decode kernel, so that the two can share
  // an SM (an SM runs one split at a time)
  // (a function attribute is per device: set once on each)
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kPfMaxDevices) return cudaErrorInvalidDevice;
  if (!g_carveout_set[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(prefetch_blocks_kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    g_carveout_set[dev].store(true, std::memory_order_release);
  }
  prefetch_blocks_kernel<<<dim3(static_cast<unsigned>(ctas), 4), kPfThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace kvq
