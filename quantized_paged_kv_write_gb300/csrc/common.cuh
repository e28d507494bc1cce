// Shared device helpers for the libkvq kernels (sm_103a): format codes,
// mbarrier / bulk-copy / TMA wrappers in inline PTX, BF16 and FP8 bit helpers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

// ---------------------------------------------------------------------------
// Cache-format codes used as template parameters.
// ---------------------------------------------------------------------------
enum KFmt : int { K_INT8_TOK = 0, K_FP8_TOK = 1, K_INT8_CHAN = 2, K_INT4_TOK = 3, K_INT2_CHAN = 4 };
enum VFmt : int { V_INT8_TOK = 0, V_FP8_TOK = 1, V_INT4_G32 = 2, V_INT2_G32 = 3 };

constexpr int kBlockSize = 16;

// Bounded waits: a wait gives up after this many clock64 ticks (~2 s at the
// GB300's SM clock), records KVQ_DEVERR_TIMEOUT and lets the kernel return.
constexpr long long kWaitTicks = 4000000000LL;

__device__ __forceinline__ void set_error(unsigned int *err, unsigned int bit) {
  if (err) atomicOr(err, bit);
}

// ---------------------------------------------------------------------------
// BF16 <-> FP32 (exact widening)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---------------------------------------------------------------------------
// shared-memory addresses and mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete; false on timeout.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitTicks) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// bulk copies global -> shared, completing on an mbarrier
// ---------------------------------------------------------------------------
// 1-D bulk copy: dst, src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Order this thread's earlier generic-proxy global writes before later
// async-proxy (TMA / bulk copy) accesses issued after a barrier.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 4-D tiled TMA load.  c0 (the innermost coordinate) is always 0 here.
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Byte offset inside a TMA box written with the 32/64/128-byte swizzle: the
// 16-byte chunk index (bits 4..6) is XORed with the 128-byte line index
// (bits 7..9), masked to the swizzle span.  The box base is 1024-aligned.
template <int ROW_BYTES>
__device__ __forceinline__ uint32_t swz(uint32_t off) {
  constexpr uint32_t mask = ROW_BYTES >= 128 ? 7u : (ROW_BYTES == 64 ? 3u : 1u);
  return off ^ (((off >> 7) & mask) << 4);
}

template <int ROW_BYTES>
constexpr CUtensorMapSwizzle swizzle_mode() {
  return ROW_BYTES >= 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                          : (ROW_BYTES == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

// ---------------------------------------------------------------------------
// shared loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t x) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(x) : "memory");
}
__device__ __forceinline__ void sts64(uint32_t addr, uint32_t x, uint32_t y) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}
// Two 8 x 8 matrices of 16-bit elements, transposed: lanes 0-7 give the row
// addresses of matrix 0, lanes 8-15 those of matrix 1 (16 contiguous bytes
// each); lane l receives, per matrix, the elements (row 2 (l % 4), column
// l / 4) in its low half and (row 2 (l % 4) + 1, column l / 4) in its high
// half.
__device__ __forceinline__ void ldsm_x2_trans(uint32_t addr, uint32_t &m0, uint32_t &m1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
               : "=r"(m0), "=r"(m1)
               : "r"(addr));
}
// Four transposed 8 x 8 matrices of 16-bit elements (lanes 8m .. 8m + 7 give
// the rows of matrix m), with the same per-matrix result layout.
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &m0, uint32_t &m1, uint32_t &m2,
                                              uint32_t &m3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(m0), "=r"(m1), "=r"(m2), "=r"(m3)
               : "r"(addr));
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds8(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
  unsigned short v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float ldsf(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// ---------------------------------------------------------------------------
// register-level code -> f16 conversions (exact)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// (a & b) ^ c in one LOP3 (truth table (0xF0 & 0xCC) ^ 0xAA = 0x6A).
__device__ __forceinline__ uint32_t and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// a * b - c in one rounding (f16x2): the negation folds into the FMA.
__device__ __forceinline__ uint32_t hfma2_negc_u32(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("{\n\t.reg .b32 t;\n\tneg.f16x2 t, %3;\n\tfma.rn.f16x2 %0, %1, %2, t;\n\t}"
      : "=r"(d)
      : "r"(a), "r"(b), "r"(c));
  return d;
}

// w >> 8 as the high word of w * 2^24 (a multiply, not a shift).
__device__ __forceinline__ uint32_t shr8_mul(uint32_t w) {
  uint32_t d;
  asm("mul.hi.u32 %0, %1, 16777216;" : "=r"(d) : "r"(w));
  return d;
}

// Per-half unsigned maximum of two packed 16-bit values.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Maximum of x over the 32 lanes of a fully active warp.
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t x) {
  uint32_t d;
  asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(d) : "r"(x));
  return d;
}

// Two E4M3 bytes (low 16 bits of w) -> f16x2, byte 0 in the low half.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
  uint32_t d;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(d) : "r"(w));
  return d;
}

// Four E4M3 bytes -> two f16x2: bytes 0, 1 -> lo, bytes 2, 3 -> hi.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two FP32 -> f16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t f32x2_to_f16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ float f16lo_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}
__device__ __forceinline__ float f16hi_to_f32(uint32_t h2) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(h2));
  return f;
}

// Packed FP32 pair arithmetic (Blackwell f32x2): each lane is rounded to
// nearest even exactly like the scalar instruction.
__device__ __forceinline__ void mul_f32x2(float a0, float a1, float b0, float b1, float &d0, float &d1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void add_f32x2(float a0, float a1, float b0, float b1, float &d0, float &d1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub_f32x2(float a0, float a1, float b0, float b1, float &d0, float &d1) {
  asm("{\n\t.reg .b64 a, b, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
      "sub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

__device__ __forceinline__ void fma_f32x2(float a0, float a1, float b0, float b1, float c0, float c1, float &d0,
                                          float &d1) {
  asm("{\n\t.reg .b64 a, b, c, d;\n\t"
      "mov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
      "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

// Split two FP32 values into f16 high parts and f16 residuals:
// x = f16(x) + f16(x - f16(x)) to ~22 bits (the residual is exact in FP32).
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  hi = f32x2_to_f16x2(x0, x1);
  float r0, r1;
  sub_f32x2(x0, x1, f16lo_to_f32(hi), f16hi_to_f32(hi), r0, r1);
  lo = f32x2_to_f16x2(r0, r1);
}

// One part of the same split: m = 0 gives the high part f16(x), m = 1 the
// low part f16(x - f16(x)) (the residual is exact in FP32, as above).
__device__ __forceinline__ uint32_t part_f16x2(float x0, float x1, float m) {
  const uint32_t h = f32x2_to_f16x2(x0, x1);
  const float y0 = fmaf(-m, f16lo_to_f32(h), x0);
  const float y1 = fmaf(-m, f16hi_to_f32(h), x1);
  return f32x2_to_f16x2(y0, y1);
}

// D += A * B for one m16n8k16 tile, f16 inputs, FP32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^k as a float for -126 <= k <= 127.
__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

}  // namespace kvq
