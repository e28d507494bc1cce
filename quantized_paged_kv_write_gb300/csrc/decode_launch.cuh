// Host-side plan and launch of the paged decode kernels for one K format.
// Included once per K format (decode_k*.cu) so the template instances build
// in parallel.
#pragma once

#include <atomic>

#include "paged_decode_impl.cuh"

namespace kvq {

namespace detail {

// Shared memory per CTA to stay at two resident CTAs per SM (228 KB per SM,
// 1 KB reserved per CTA).
constexpr size_t kSmemPerCtaTarget = 112 * 1024;
constexpr int kMaxStages = 6;

template <int D, int KF, int VF, bool WIDE, int HT, bool ROT>
cudaError_t plan_one(int H, int B, DecodePlan *plan) {
  constexpr bool rot = ROT;
  using T = DecodeTraits<D, KF, VF>;
  const size_t sb = T::stage_bytes(H);
  const size_t fixed = 1024 /* alignment slack */ + T::aux_bytes(H, WIDE, rot) + 16 * kMaxStages /* barriers */ +
                       4 * kMaxStages /* info */ + 4 * (static_cast<size_t>(B) + 1) /* prefix sums */;
  int ns = static_cast<int>((kSmemPerCtaTarget - fixed) / sb);
  if (ns > kMaxStages) ns = kMaxStages;
  if (ns < 2) ns = 2;
  size_t smem = fixed + ns * sb;
  auto kern = decode_split_kernel<D, KF, VF, WIDE, HT, ROT>;
  int dev = 0, sms = 0, occ = 0, optin = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess) return e;
  if (smem > static_cast<size_t>(optin)) return cudaErrorInvalidConfiguration;
  // Once per device and kernel instance: allow launches up to the opt-in
  // maximum (plans for different batches share the kernel, so the bound must
  // cover all of them) and ask for all of the unified L1/shared array as
  // shared memory (two CTAs per SM).
  static std::atomic<unsigned long long> attr_done{0};
  if (!((attr_done.load(std::memory_order_acquire) >> dev) & 1ull)) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, optin)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
    attr_done.fetch_or(1ull << dev, std::memory_order_acq_rel);
  }
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int threads = 32 * (H + 1);
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem)) != cudaSuccess) return e;
  if (occ < 1) return cudaErrorInvalidConfiguration;
  plan->nstages = ns;
  plan->smem = smem;
  plan->threads = threads;
  plan->ctas_per_sm = occ;
  plan->max_ctas = sms * occ;
  return cudaSuccess;
}

template <int D, int KF, int VF, bool WIDE, int HT, bool ROT>
cudaError_t launch_one(const DecodeArgs &a, const DecodePlan &plan, const DecodeMaps &m, cudaStream_t stream) {
  if (a.nctas > 0) {
    decode_split_kernel<D, KF, VF, WIDE, HT, ROT>
        <<<a.nctas, plan.threads, plan.smem, stream>>>(m.k, m.v, m.vs, a, plan.nstages);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int warps = a.B * a.Hq;
  decode_reduce_kernel<D><<<(warps + 7) / 8, 256, 0, stream>>>(a, a.ws_cum);
  return cudaGetLastError();
}

template <int D, int KF, bool WIDE, int HT, bool ROT>
cudaError_t plan_vf_h(int vf, int H, int B, DecodePlan *plan) {
  if (vf == V_INT8_TOK) return plan_one<D, KF, V_INT8_TOK, WIDE, HT, ROT>(H, B, plan);
  if (vf == V_FP8_TOK) return plan_one<D, KF, V_FP8_TOK, WIDE, HT, ROT>(H, B, plan);
  if (vf == V_INT4_G32) return plan_one<D, KF, V_INT4_G32, WIDE, HT, ROT>(H, B, plan);
  if constexpr (D == 128) {
    if (vf == V_INT2_G32) return plan_one<D, KF, V_INT2_G32, WIDE, HT, ROT>(H, B, plan);
  }
  return cudaErrorInvalidValue;
}

// eight kv heads (Llama-3 8B / 70B layers) get a compile-time head count;
// a rotated cache (per-token K only) runs with a runtime head count
template <int D, int KF, bool WIDE>
cudaError_t plan_vf(int vf, int H, int B, bool rot, DecodePlan *plan) {
  if constexpr (KF != K_INT8_CHAN && KF != K_INT2_CHAN) {
    if (rot) return plan_vf_h<D, KF, WIDE, 0, true>(vf, H, B, plan);
  }
  return H == 8 ? plan_vf_h<D, KF, WIDE, 8, false>(vf, H, B, plan) : plan_vf_h<D, KF, WIDE, 0, false>(vf, H, B, plan);
}

template <int D, int KF, bool WIDE, int HT, bool ROT>
cudaError_t launch_vf_h(int vf, const DecodeArgs &a, const DecodePlan &plan, const DecodeMaps &m,
                        cudaStream_t stream) {
  if (vf == V_INT8_TOK) return launch_one<D, KF, V_INT8_TOK, WIDE, HT, ROT>(a, plan, m, stream);
  if (vf == V_FP8_TOK) return launch_one<D, KF, V_FP8_TOK, WIDE, HT, ROT>(a, plan, m, stream);
  if (vf == V_INT4_G32) return launch_one<D, KF, V_INT4_G32, WIDE, HT, ROT>(a, plan, m, stream);
  if constexpr (D == 128) {
    if (vf == V_INT2_G32) return launch_one<D, KF, V_INT2_G32, WIDE, HT, ROT>(a, plan, m, stream);
  }
  return cudaErrorInvalidValue;
}

template <int D, int KF, bool WIDE>
cudaError_t launch_vf(int vf, const DecodeArgs &a, const DecodePlan &plan, const DecodeMaps &m,
                      cudaStream_t stream) {
  if constexpr (KF != K_INT8_CHAN && KF != K_INT2_CHAN) {
    if (a.rot) return launch_vf_h<D, KF, WIDE, 0, true>(vf, a, plan, m, stream);
  }
  return a.H == 8 ? launch_vf_h<D, KF, WIDE, 8, false>(vf, a, plan, m, stream)
                  : launch_vf_h<D, KF, WIDE, 0, false>(vf, a, plan, m, stream);
}

}  // namespace detail

template <int KF>
cudaError_t plan_decode_kf(int head_dim, int vf, int H, int G, int B, bool rot, DecodePlan *plan) {
  const bool wide = G > 4;
  if (head_dim == 128)
    return wide ? detail::plan_vf<128, KF, true>(vf, H, B, rot, plan)
                : detail::plan_vf<128, KF, false>(vf, H, B, rot, plan);
  if constexpr (KF != K_INT2_CHAN) {  // INT2 rows: head_dim 128
    if (head_dim == 64)
      return wide ? detail::plan_vf<64, KF, true>(vf, H, B, rot, plan)
                  : detail::plan_vf<64, KF, false>(vf, H, B, rot, plan);
  }
  return cudaErrorInvalidValue;
}

template <int KF>
cudaError_t launch_decode_kf(int head_dim, int vf, const DecodeArgs &a, const DecodePlan &plan,
                             const DecodeMaps &m, cudaStream_t stream) {
  const bool wide = a.G > 4;
  if (head_dim == 128)
    return wide ? detail::launch_vf<128, KF, true>(vf, a, plan, m, stream)
                : detail::launch_vf<128, KF, false>(vf, a, plan, m, stream);
  if constexpr (KF != K_INT2_CHAN) {
    if (head_dim == 64)
      return wide ? detail::launch_vf<64, KF, true>(vf, a, plan, m, stream)
                  : detail::launch_vf<64, KF, false>(vf, a, plan, m, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace kvq
