// The C ABI of libkvq (declared in include/kvq.h): argument checks, format
// decoding, tensor-map encoding and kernel launches.  Nothing here computes
// on the host; every step of the path runs in the kernels.
#include <mutex>
#include <unordered_map>

#include "common.cuh"
#include "kvq_internal.h"

namespace {

using namespace kvq;

// The sticky device error word, one per device (kernels receive its address).
__device__ unsigned int g_kvq_errors = 0;

constexpr int kMaxDevices = 64;
unsigned int *g_err_addr[kMaxDevices] = {};
std::mutex g_err_mu;

cudaError_t error_word(unsigned int **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_err_mu);
  if (!g_err_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_kvq_errors);
    if (e != cudaSuccess) return e;
    g_err_addr[dev] = static_cast<unsigned int *>(p);
  }
  *out = g_err_addr[dev];
  return cudaSuccess;
}

int sm_count(int *sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Decodes and checks a format; on success sets the kernel format codes.
int decode_format(const kvq_format *f, int *kf, int *vf) {
  if (!f) return KVQ_ERR_INVALID_ARG;
  if (f->rotation != KVQ_ROT_NONE && f->rotation != KVQ_ROT_HADAMARD) return KVQ_ERR_INVALID_ARG;
  if (f->num_blocks < 0 || f->num_kv_heads < 1) return KVQ_ERR_INVALID_ARG;
  if (f->block_size != kBlockSize) return KVQ_ERR_UNSUPPORTED;
  if (f->head_dim != 64 && f->head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (f->num_kv_heads > 8) return KVQ_ERR_UNSUPPORTED;
  if (f->k_gran == KVQ_PER_TOKEN_HEAD && f->k_dtype == KVQ_INT8) *kf = K_INT8_TOK;
  else if (f->k_gran == KVQ_PER_TOKEN_HEAD && f->k_dtype == KVQ_FP8_E4M3FN) *kf = K_FP8_TOK;
  else if (f->k_gran == KVQ_PER_BLOCK_CHANNEL && f->k_dtype == KVQ_INT8) *kf = K_INT8_CHAN;
  else if (f->k_gran == KVQ_PER_TOKEN_HEAD && f->k_dtype == KVQ_INT4) *kf = K_INT4_TOK;
  else if (f->k_gran == KVQ_PER_BLOCK_CHANNEL && f->k_dtype == KVQ_INT2 && f->head_dim == 128) *kf = K_INT2_CHAN;
  else return KVQ_ERR_UNSUPPORTED;
  if (f->v_gran == KVQ_PER_TOKEN_HEAD && f->v_dtype == KVQ_INT8) *vf = V_INT8_TOK;
  else if (f->v_gran == KVQ_PER_TOKEN_HEAD && f->v_dtype == KVQ_FP8_E4M3FN) *vf = V_FP8_TOK;
  else if (f->v_gran == KVQ_PER_TOKEN_GROUP && f->v_dtype == KVQ_INT4 && f->v_group == 32) *vf = V_INT4_G32;
  else if (f->v_gran == KVQ_PER_TOKEN_GROUP && f->v_dtype == KVQ_INT2 && f->v_group == 32 && f->head_dim == 128)
    *vf = V_INT2_G32;
  else return KVQ_ERR_UNSUPPORTED;
  if (f->rotation == KVQ_ROT_HADAMARD && (*kf == K_INT8_CHAN || *kf == K_INT2_CHAN)) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

cudaError_t plan_decode_uncached(int D, int kf, int vf, int H, int G, int B, bool rot, DecodePlan *plan) {
  if (kf == K_INT8_TOK) return plan_decode_kf<K_INT8_TOK>(D, vf, H, G, B, rot, plan);
  if (kf == K_FP8_TOK) return plan_decode_kf<K_FP8_TOK>(D, vf, H, G, B, rot, plan);
  if (kf == K_INT8_CHAN) return plan_decode_kf<K_INT8_CHAN>(D, vf, H, G, B, rot, plan);
  if (kf == K_INT4_TOK) return plan_decode_kf<K_INT4_TOK>(D, vf, H, G, B, rot, plan);
  if (kf == K_INT2_CHAN) return plan_decode_kf<K_INT2_CHAN>(D, vf, H, G, B, rot, plan);
  return cudaErrorInvalidValue;
}

// Launch plans are computed once per (device, kernel instance, batch): the
// kernel attributes, the SM count and the occupancy query stay off the
// per-call path.  The map is bounded (cleared when full).
struct PlanKey {
  int dev, D, kf, vf, H, G, B, rot;
  bool operator==(const PlanKey &o) const {
    return dev == o.dev && D == o.D && kf == o.kf && vf == o.vf && H == o.H && G == o.G && B == o.B && rot == o.rot;
  }
};
struct PlanKeyHash {
  size_t operator()(const PlanKey &k) const {
    size_t h = 1469598103934665603ull;
    for (int x : {k.dev, k.D, k.kf, k.vf, k.H, k.G, k.B, k.rot}) h = (h ^ static_cast<uint32_t>(x)) * 1099511628211ull;
    return h;
  }
};
constexpr size_t kMaxPlans = 1024;
std::unordered_map<PlanKey, DecodePlan, PlanKeyHash> g_plans;
std::mutex g_plan_mu;

cudaError_t plan_decode(int D, int kf, int vf, int H, int G, int B, bool rot, DecodePlan *plan) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const PlanKey key{dev, D, kf, vf, H, G, B, rot ? 1 : 0};
  {
    std::lock_guard<std::mutex> lk(g_plan_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) {
      *plan = it->second;
      return cudaSuccess;
    }
  }
  DecodePlan p;
  if ((e = plan_decode_uncached(D, kf, vf, H, G, B, rot, &p)) != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_plan_mu);
  if (g_plans.size() >= kMaxPlans) g_plans.clear();
  g_plans.emplace(key, p);
  *plan = p;
  return cudaSuccess;
}

cudaError_t launch_decode(int D, int kf, int vf, const DecodeArgs &a, const DecodePlan &plan,
                          const DecodeMaps &m, cudaStream_t s) {
  if (kf == K_INT8_TOK) return launch_decode_kf<K_INT8_TOK>(D, vf, a, plan, m, s);
  if (kf == K_FP8_TOK) return launch_decode_kf<K_FP8_TOK>(D, vf, a, plan, m, s);
  if (kf == K_INT8_CHAN) return launch_decode_kf<K_INT8_CHAN>(D, vf, a, plan, m, s);
  if (kf == K_INT4_TOK) return launch_decode_kf<K_INT4_TOK>(D, vf, a, plan, m, s);
  if (kf == K_INT2_CHAN) return launch_decode_kf<K_INT2_CHAN>(D, vf, a, plan, m, s);
  return cudaErrorInvalidValue;
}

// Workspace layout: [partial O^T][partial (m, l)][prefix sums], 256-aligned.
struct WsLayout {
  size_t o_off, ml_off, cum_off, total;
};

WsLayout ws_layout(int B, int H, int D, int max_ctas) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t slots = static_cast<size_t>(B) + static_cast<size_t>(max_ctas);
  WsLayout w;
  w.o_off = 0;
  w.ml_off = al(slots * H * D * 8 * sizeof(float));
  w.cum_off = w.ml_off + al(slots * H * 8 * 2 * sizeof(float));
  w.total = w.cum_off + al((static_cast<size_t>(B) + 1) * sizeof(int));
  return w;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 4-D map over a code cache [num_blocks, bs, H, row_bytes] (uint8) with a
// box of one (block, head) tile: 16 rows of row_bytes.
int encode_cache_map(CUtensorMap *map, const void *base, int64_t nb, int H, int row_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KVQ_ERR_CUDA;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(kBlockSize), static_cast<cuuint64_t>(nb)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(row_bytes),
                                 static_cast<cuuint64_t>(row_bytes) * H,
                                 static_cast<cuuint64_t>(row_bytes) * H * kBlockSize};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(row_bytes), 1, static_cast<cuuint32_t>(kBlockSize), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = row_bytes >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVQ_OK : KVQ_ERR_CUDA;
}

// 4-D map over INT4 V group scales [num_blocks, bs, H, 4] (float32) with a
// box of one (block, head) tile: 16 tokens x 4 groups (256 bytes).
int encode_vscale_map(CUtensorMap *map, const float *base, int64_t nb, int H) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KVQ_ERR_CUDA;
  const cuuint64_t dims[4] = {4, static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(kBlockSize),
                              static_cast<cuuint64_t>(nb)};
  const cuuint64_t strides[3] = {16, static_cast<cuuint64_t>(16) * H,
                                 static_cast<cuuint64_t>(16) * H * kBlockSize};
  const cuuint32_t box[4] = {4, 1, static_cast<cuuint32_t>(kBlockSize), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVQ_OK : KVQ_ERR_CUDA;
}

// The descriptors of one decode call.
int encode_decode_maps_uncached(DecodeMaps *m, const kvq_caches &caches, const kvq_scales &scales, int64_t nb,
                                int H, int D, int kf, int vf) {
  const int krow = (kf == K_INT4_TOK) ? D / 2 : (kf == K_INT2_CHAN ? D / 4 : D);
  const int vrow = (vf == V_INT4_G32) ? D / 2 : (vf == V_INT2_G32 ? D / 4 : D);
  int st;
  if ((st = encode_cache_map(&m->k, caches.k_cache, nb, H, krow)) != KVQ_OK) return st;
  if ((st = encode_cache_map(&m->v, caches.v_cache, nb, H, vrow)) != KVQ_OK) return st;
  if ((vf == V_INT4_G32 || vf == V_INT2_G32) && D / 32 == 4) return encode_vscale_map(&m->vs, scales.v_scale, nb, H);
  m->vs = m->v;
  return KVQ_OK;
}

// The tensor maps of the last few caches, so that a serving loop over the
// same cache encodes them once: keyed by the cache and scale pointers and
// the shape and format they were encoded for.
struct MapEntry {
  bool used = false;
  int dev = 0, H = 0, D = 0, kf = 0, vf = 0;
  int64_t nb = 0;
  const void *kc = nullptr, *vc = nullptr;
  const float *vs = nullptr;
  DecodeMaps maps;
};
constexpr int kMapSlots = 16;
MapEntry g_maps[kMapSlots];
int g_map_next = 0;
std::mutex g_map_mu;

int encode_decode_maps(DecodeMaps *m, const kvq_caches &caches, const kvq_scales &scales, int64_t nb, int H, int D,
                       int kf, int vf) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KVQ_ERR_CUDA;
  {
    std::lock_guard<std::mutex> lk(g_map_mu);
    for (const MapEntry &e : g_maps) {
      if (e.used && e.dev == dev && e.kc == caches.k_cache && e.vc == caches.v_cache && e.vs == scales.v_scale &&
          e.nb == nb && e.H == H && e.D == D && e.kf == kf && e.vf == vf) {
        *m = e.maps;
        return KVQ_OK;
      }
    }
  }
  DecodeMaps fresh;
  const int st = encode_decode_maps_uncached(&fresh, caches, scales, nb, H, D, kf, vf);
  if (st != KVQ_OK) return st;
  std::lock_guard<std::mutex> lk(g_map_mu);
  MapEntry &e = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapSlots;
  e.used = true;
  e.dev = dev;
  e.H = H;
  e.D = D;
  e.kf = kf;
  e.vf = vf;
  e.nb = nb;
  e.kc = caches.k_cache;
  e.vc = caches.v_cache;
  e.vs = scales.v_scale;
  e.maps = fresh;
  *m = fresh;
  return KVQ_OK;
}

}  // namespace

extern "C" {

int32_t kvq_version(void) { return 110; }

#ifndef KVQ_BUILD_ID
#define KVQ_BUILD_ID "unknown"
#endif
const char *kvq_build_id(void) { return KVQ_BUILD_ID; }

const char *kvq_status_string(int32_t status) {
  switch (status) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported format or shape";
    case KVQ_ERR_WORKSPACE: return "workspace too small";
    case KVQ_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

int kvq_quantize_write(const void *k_bf16, const void *v_bf16, const int64_t *slot_mapping,
                       int64_t num_tokens, const kvq_format *fmt, kvq_caches caches, kvq_scales scales,
                       kvq_stream_t stream) {
  int kf = 0, vf = 0;
  int st = decode_format(fmt, &kf, &vf);
  if (st != KVQ_OK) return st;
  if (num_tokens < 0) return KVQ_ERR_INVALID_ARG;
  if (num_tokens == 0) return KVQ_OK;
  if (!k_bf16 || !v_bf16 || !slot_mapping || !caches.k_cache || !caches.v_cache || !scales.k_scale ||
      !scales.v_scale)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_bf16) || !aligned16(v_bf16) || !aligned16(caches.k_cache) || !aligned16(caches.v_cache) ||
      !aligned16(scales.k_scale) || !aligned16(scales.v_scale) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return KVQ_ERR_INVALID_ARG;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return KVQ_ERR_CUDA;
  int sms = 0;
  if ((st = sm_count(&sms)) != KVQ_OK) return st;
  QuantizeArgs a;
  a.k = k_bf16;
  a.v = v_bf16;
  a.slots = slot_mapping;
  a.ntok = num_tokens;
  a.H = fmt->num_kv_heads;
  a.nslots = fmt->num_blocks * fmt->block_size;
  a.kc = static_cast<uint8_t *>(caches.k_cache);
  a.vc = static_cast<uint8_t *>(caches.v_cache);
  a.ks = scales.k_scale;
  a.vs = scales.v_scale;
  a.err = err;
  a.rot = fmt->rotation;
  for (int w = 0; w < 4; ++w) a.rot_signs[w] = fmt->rotation_signs[w];
  return launch_quantize_write(fmt->head_dim, kf, vf, a, sms, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

static int check_decode_shape(const kvq_format *fmt, int32_t batch, int32_t num_q_heads, int *kf, int *vf) {
  int st = decode_format(fmt, kf, vf);
  if (st != KVQ_OK) return st;
  if (batch < 0 || num_q_heads < 1) return KVQ_ERR_INVALID_ARG;
  if (num_q_heads % fmt->num_kv_heads != 0) return KVQ_ERR_INVALID_ARG;
  const int G = num_q_heads / fmt->num_kv_heads;
  if (G > 8) return KVQ_ERR_UNSUPPORTED;
  if (batch > 8192) return KVQ_ERR_UNSUPPORTED;
  return KVQ_OK;
}

int kvq_decode_workspace_size(const kvq_format *fmt, int32_t batch, int32_t num_q_heads,
                              int32_t max_context_len, size_t *bytes) {
  int kf = 0, vf = 0;
  int st = check_decode_shape(fmt, batch, num_q_heads, &kf, &vf);
  if (st != KVQ_OK) return st;
  if (!bytes || max_context_len < 0) return KVQ_ERR_INVALID_ARG;
  DecodePlan plan;
  if (plan_decode(fmt->head_dim, kf, vf, fmt->num_kv_heads, num_q_heads / fmt->num_kv_heads, batch,
                  fmt->rotation != 0, &plan) !=
      cudaSuccess)
    return KVQ_ERR_CUDA;
  *bytes = ws_layout(batch, fmt->num_kv_heads, fmt->head_dim, plan.max_ctas).total;
  return KVQ_OK;
}

// The decode entry points with a caller workspace; k_new / v_new non-null
// fuse the write of each sequence's new token (kvq_write_decode).
static int run_decode(const void *q_bf16, int32_t batch, int32_t num_q_heads, const kvq_format *fmt,
                      kvq_caches caches, kvq_scales scales, const int32_t *block_tables,
                      int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t max_context_len,
                      float *out, void *workspace, size_t workspace_bytes, kvq_stream_t stream,
                      const void *k_new, const void *v_new, const void *res_k = nullptr,
                      const void *res_v = nullptr) {
  int kf = 0, vf = 0;
  int st = check_decode_shape(fmt, batch, num_q_heads, &kf, &vf);
  if (st != KVQ_OK) return st;
  const bool tail = res_k != nullptr || res_v != nullptr;
  if (tail) {
    if (kf != K_INT8_CHAN && kf != K_INT2_CHAN) return KVQ_ERR_UNSUPPORTED;  // the tail belongs to per-channel K
    if (!res_k || !res_v || !aligned16(res_k) || !aligned16(res_v)) return KVQ_ERR_INVALID_ARG;
  }
  const bool fused = k_new != nullptr || v_new != nullptr;
  if (fused) {
    if (kf == K_INT8_CHAN || kf == K_INT2_CHAN) return KVQ_ERR_UNSUPPORTED;  // per-channel K blocks take no appends
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return KVQ_ERR_INVALID_ARG;
  }
  if (batch == 0) return KVQ_OK;
  if (!q_bf16 || !caches.k_cache || !caches.v_cache || !scales.k_scale || !scales.v_scale || !block_tables ||
      !context_lens || !out || !workspace)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q_bf16) || !aligned16(caches.k_cache) || !aligned16(caches.v_cache) ||
      !aligned16(scales.k_scale) || !aligned16(scales.v_scale) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return KVQ_ERR_INVALID_ARG;
  if (max_blocks_per_seq < 1 || max_context_len < 0) return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * max_blocks_per_seq >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  if (fmt->num_blocks < 1 || fmt->num_blocks >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  const int H = fmt->num_kv_heads, D = fmt->head_dim, G = num_q_heads / H;
  DecodePlan plan;
  if (plan_decode(D, kf, vf, H, G, batch, fmt->rotation != 0, &plan) != cudaSuccess) return KVQ_ERR_CUDA;
  const WsLayout wl = ws_layout(batch, H, D, plan.max_ctas);
  if (workspace_bytes < wl.total) return KVQ_ERR_WORKSPACE;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return KVQ_ERR_CUDA;

  DecodeMaps maps;
  if ((st = encode_decode_maps(&maps, caches, scales, fmt->num_blocks, H, D, kf, vf)) != KVQ_OK) return st;

  // CTAs: one resident wave, but no more than one per 4 blocks of the
  // largest possible batch
  const int64_t ctx_cap = max_context_len < max_blocks_per_seq * kBlockSize ? max_context_len
                                                                             : max_blocks_per_seq * kBlockSize;
  const int64_t blocks_ub = static_cast<int64_t>(batch) * ((ctx_cap + kBlockSize - 1) / kBlockSize);
  int64_t P = (blocks_ub + 3) / 4;
  if (P > plan.max_ctas) P = plan.max_ctas;
  if (P < 1) P = 1;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  DecodeArgs a;
  a.q = static_cast<const uint16_t *>(q_bf16);
  a.ks = scales.k_scale;
  a.vs = scales.v_scale;
  a.tables = block_tables;
  a.ctx = context_lens;
  a.ws_o = reinterpret_cast<float *>(ws + wl.o_off);
  a.ws_ml = reinterpret_cast<float *>(ws + wl.ml_off);
  a.ws_cum = reinterpret_cast<int *>(ws + wl.cum_off);
  a.out = out;
  a.err = err;
  a.num_blocks = fmt->num_blocks;
  a.B = batch;
  a.Hq = num_q_heads;
  a.H = H;
  a.G = G;
  a.max_blocks = max_blocks_per_seq;
  a.max_ctx = max_context_len;
  a.nctas = static_cast<int>(P);
  a.rot = fmt->rotation;
  for (int w = 0; w < 4; ++w) a.rot_signs[w] = fmt->rotation_signs[w];
  if (tail) {
    a.res_k = static_cast<const uint16_t *>(res_k);
    a.res_v = static_cast<const uint16_t *>(res_v);
  }
  if (fused) {
    a.knew = static_cast<const uint16_t *>(k_new);
    a.vnew = static_cast<const uint16_t *>(v_new);
    a.kc_w = static_cast<uint8_t *>(caches.k_cache);
    a.vc_w = static_cast<uint8_t *>(caches.v_cache);
    a.ks_w = scales.k_scale;
    a.vs_w = scales.v_scale;
  }
  return launch_decode(D, kf, vf, a, plan, maps, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

int kvq_paged_decode(const void *q_bf16, int32_t batch, int32_t num_q_heads, const kvq_format *fmt,
                     kvq_caches caches, kvq_scales scales, const int32_t *block_tables,
                     int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t max_context_len,
                     float *out, void *workspace, size_t workspace_bytes, kvq_stream_t stream) {
  return run_decode(q_bf16, batch, num_q_heads, fmt, caches, scales, block_tables, max_blocks_per_seq,
                    context_lens, max_context_len, out, workspace, workspace_bytes, stream, nullptr, nullptr);
}

int kvq_write_decode(const void *q_bf16, const void *k_new_bf16, const void *v_new_bf16, int32_t batch,
                     int32_t num_q_heads, const kvq_format *fmt, kvq_caches caches, kvq_scales scales,
                     const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
                     int32_t max_context_len, float *out, void *workspace, size_t workspace_bytes,
                     kvq_stream_t stream) {
  if (!k_new_bf16 || !v_new_bf16) return KVQ_ERR_INVALID_ARG;
  return run_decode(q_bf16, batch, num_q_heads, fmt, caches, scales, block_tables, max_blocks_per_seq,
                    context_lens, max_context_len, out, workspace, workspace_bytes, stream, k_new_bf16,
                    v_new_bf16);
}

int kvq_kivi_decode(const void *q_bf16, int32_t batch, int32_t num_q_heads, const kvq_format *fmt,
                    kvq_caches caches, kvq_scales scales, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t max_context_len,
                    const void *res_k_bf16, const void *res_v_bf16, float *out, void *workspace,
                    size_t workspace_bytes, kvq_stream_t stream) {
  if (!res_k_bf16 || !res_v_bf16) return KVQ_ERR_INVALID_ARG;
  return run_decode(q_bf16, batch, num_q_heads, fmt, caches, scales, block_tables, max_blocks_per_seq,
                    context_lens, max_context_len, out, workspace, workspace_bytes, stream, nullptr, nullptr,
                    res_k_bf16, res_v_bf16);
}

int kvq_kivi_append(const void *k_new_bf16, const void *v_new_bf16, int32_t batch, const kvq_format *fmt,
                    kvq_caches caches, kvq_scales scales, const int32_t *block_tables,
                    int32_t max_blocks_per_seq, const int32_t *context_lens, void *res_k_bf16,
                    void *res_v_bf16, kvq_stream_t stream) {
  int kf = 0, vf = 0;
  int st = decode_format(fmt, &kf, &vf);
  if (st != KVQ_OK) return st;
  if (kf != K_INT8_CHAN && kf != K_INT2_CHAN) return KVQ_ERR_UNSUPPORTED;
  if (batch < 0 || max_blocks_per_seq < 1) return KVQ_ERR_INVALID_ARG;
  if (batch == 0) return KVQ_OK;
  if (!k_new_bf16 || !v_new_bf16 || !res_k_bf16 || !res_v_bf16 || !block_tables || !context_lens ||
      !caches.k_cache || !caches.v_cache || !scales.k_scale || !scales.v_scale)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_new_bf16) || !aligned16(v_new_bf16) || !aligned16(res_k_bf16) || !aligned16(res_v_bf16) ||
      !aligned16(caches.k_cache) || !aligned16(caches.v_cache) || !aligned16(scales.k_scale) ||
      !aligned16(scales.v_scale) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return KVQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(batch) * max_blocks_per_seq >= (int64_t(1) << 31)) return KVQ_ERR_UNSUPPORTED;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return KVQ_ERR_CUDA;
  KiviAppendArgs a;
  a.knew = static_cast<const uint16_t *>(k_new_bf16);
  a.vnew = static_cast<const uint16_t *>(v_new_bf16);
  a.res_k = static_cast<uint16_t *>(res_k_bf16);
  a.res_v = static_cast<uint16_t *>(res_v_bf16);
  a.tables = block_tables;
  a.ctx = context_lens;
  a.kc = static_cast<uint8_t *>(caches.k_cache);
  a.vc = static_cast<uint8_t *>(caches.v_cache);
  a.ks = scales.k_scale;
  a.vs = scales.v_scale;
  a.err = err;
  a.num_blocks = fmt->num_blocks;
  a.B = batch;
  a.H = fmt->num_kv_heads;
  a.max_blocks = max_blocks_per_seq;
  return launch_kivi_append(fmt->head_dim, kf, vf, a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? KVQ_OK
             : KVQ_ERR_CUDA;
}

// Device-accessible address of pinned host memory, or null.
static const void *host_device_ptr(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (at.type != cudaMemoryTypeHost || !at.devicePointer) return nullptr;
  return at.devicePointer;
}

// bytes of one block's scales for a granularity
static int64_t block_scale_bytes(int gran, int group, int H, int D) {
  if (gran == KVQ_PER_TOKEN_HEAD) return int64_t(kBlockSize) * H * 4;
  if (gran == KVQ_PER_TOKEN_GROUP) return int64_t(kBlockSize) * H * (D / group) * 4;
  return int64_t(H) * D * 4;
}

int kvq_prefetch_blocks(const kvq_format *fmt, kvq_caches host_caches, kvq_scales host_scales,
                        int64_t host_num_blocks, const int32_t *src_blocks, const int32_t *dst_blocks,
                        int32_t num_pairs, kvq_caches caches, kvq_scales scales, kvq_stream_t stream) {
  int kf = 0, vf = 0;
  int st = decode_format(fmt, &kf, &vf);
  if (st != KVQ_OK) return st;
  if (num_pairs < 0 || host_num_blocks < 0) return KVQ_ERR_INVALID_ARG;
  if (num_pairs == 0) return KVQ_OK;
  if (!src_blocks || !dst_blocks || !caches.k_cache || !caches.v_cache || !scales.k_scale || !scales.v_scale ||
      !host_caches.k_cache || !host_caches.v_cache || !host_scales.k_scale || !host_scales.v_scale)
    return KVQ_ERR_INVALID_ARG;
  if (!aligned16(caches.k_cache) || !aligned16(caches.v_cache) || !aligned16(scales.k_scale) ||
      !aligned16(scales.v_scale) || !aligned16(host_caches.k_cache) || !aligned16(host_caches.v_cache) ||
      !aligned16(host_scales.k_scale) || !aligned16(host_scales.v_scale) ||
      (reinterpret_cast<uintptr_t>(src_blocks) & 3u) || (reinterpret_cast<uintptr_t>(dst_blocks) & 3u))
    return KVQ_ERR_INVALID_ARG;
  const void *hk = host_device_ptr(host_caches.k_cache), *hv = host_device_ptr(host_caches.v_cache);
  const void *hks = host_device_ptr(host_scales.k_scale), *hvs = host_device_ptr(host_scales.v_scale);
  if (!hk || !hv || !hks || !hvs) return KVQ_ERR_INVALID_ARG;  // not pinned host memory
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return KVQ_ERR_CUDA;
  const int H = fmt->num_kv_heads, D = fmt->head_dim;
  auto row_bytes = [D](int dt) -> int64_t { return dt == KVQ_INT4 ? D / 2 : (dt == KVQ_INT2 ? D / 4 : D); };
  const int64_t krow = row_bytes(fmt->k_dtype), vrow = row_bytes(fmt->v_dtype);
  PrefetchArgs a;
  a.src = src_blocks;
  a.dst = dst_blocks;
  a.n = num_pairs;
  a.host_nb = host_num_blocks;
  a.dev_nb = fmt->num_blocks;
  a.hk = static_cast<const uint4 *>(hk);
  a.hv = static_cast<const uint4 *>(hv);
  a.hks = static_cast<const uint4 *>(hks);
  a.hvs = static_cast<const uint4 *>(hvs);
  a.dk = static_cast<uint4 *>(caches.k_cache);
  a.dv = static_cast<uint4 *>(caches.v_cache);
  a.dks = reinterpret_cast<uint4 *>(scales.k_scale);
  a.dvs = reinterpret_cast<uint4 *>(scales.v_scale);
  a.kb16 = int64_t(kBlockSize) * H * krow / 16;
  a.vb16 = int64_t(kBlockSize) * H * vrow / 16;
  a.ksb16 = block_scale_bytes(fmt->k_gran, fmt->k_group, H, D) / 16;
  a.vsb16 = block_scale_bytes(fmt->v_gran, fmt->v_group, H, D) / 16;
  a.err = err;
  int sms = 0;
  if ((st = sm_count(&sms)) != KVQ_OK) return st;
  return launch_prefetch(a, sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

int kvq_device_errors(uint32_t *bits_out, int32_t clear, kvq_stream_t stream) {
  if (!bits_out) return KVQ_ERR_INVALID_ARG;
  unsigned int *err = nullptr;
  if (error_word(&err) != cudaSuccess) return KVQ_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  if (cudaMemcpyAsync(&v, err, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return KVQ_ERR_CUDA;
  if (clear && cudaMemsetAsync(err, 0, sizeof(unsigned int), s) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KVQ_ERR_CUDA;
  *bits_out = v;
  return KVQ_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the decode: code
// that runs under an engine or plugin host that owns all device memory and
// forbids allocation on the serving path, or latency-critical loops that
// must not take the allocator's locks or synchronizations.  For them the
// split-K scratch lives in one static device array, allocated when the
// library's module is loaded and held by every GPU that loads the library
// until the process exits.  The array is shared by every call: calls whose
// work overlaps on the GPU (for example on two streams at once) race on it,
// so such callers must order their calls.  Nothing in it has to start at
// zero (every partial the merge reads is written by the same call).
// ---------------------------------------------------------------------------
namespace {

__device__ __align__(256) static unsigned char g_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

void *g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

// Set-up, once per device with that device current: the device address of
// the array.  (In host code the array's name is only a host-side stand-in.)
cudaError_t noalloc_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" int kvq_paged_decode_noalloc(const void *q_bf16, int32_t batch, int32_t num_q_heads,
                                        const kvq_format *fmt, kvq_caches caches, kvq_scales scales,
                                        const int32_t *block_tables, int32_t max_blocks_per_seq,
                                        const int32_t *context_lens, int32_t max_context_len, float *out,
                                        kvq_stream_t stream) {
  void *scratch = nullptr;
  if (noalloc_scratch(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  // the decode with a workspace, on the static array; a shape that needs
  // more than the array holds is refused there with KVQ_ERR_WORKSPACE
  return run_decode(q_bf16, batch, num_q_heads, fmt, caches, scales, block_tables, max_blocks_per_seq,
                    context_lens, max_context_len, out, scratch, KVQ_NOALLOC_SCRATCH_BYTES, stream, nullptr,
                    nullptr);
}
