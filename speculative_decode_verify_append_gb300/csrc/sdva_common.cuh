// sdva_common.cuh -- shared device helpers of the verify-step kernels
// (sm_103a).  Conversions use PTX cvt instructions or exact bit
// re-interpretations; nothing here re-implements a CUDA math routine.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sdva.h"

namespace sdva {

constexpr int kPage = 64;       // tokens per page
constexpr int kHeadDim = 128;   // head dimension
constexpr int kMaxWindow = 16;  // 1 + up to 15 drafts

__device__ __forceinline__ void raise_status(int32_t* status, int32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// The cache arrays are read and written with 16-byte vectors and bulk copies.
inline bool cache_aligned(const sdva_kv_cache* c) {
  return ((reinterpret_cast<uintptr_t>(c->k_codes) | reinterpret_cast<uintptr_t>(c->v_codes) |
           reinterpret_cast<uintptr_t>(c->k_scales) | reinterpret_cast<uintptr_t>(c->v_scales)) &
          15u) == 0;
}

// ---------------------------------------------------------------------------
// FP8 E4M3 (OCP, "fn")
// ---------------------------------------------------------------------------
// Two fp32 values -> two E4M3 codes, round to nearest even, saturating to the
// largest finite value (PTX cvt.rn.satfinite.e4m3x2.f32).  `lo` lands in the
// low byte.
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// An E4M3 code re-read as fp16 bits: sign to bit 15, exponent and mantissa
// (7 bits) to bits 7..13.  E4M3 and binary16 share the layout of a
// sign-exponent-mantissa number whose subnormals continue the normals, and
// E4M3's exponent bias (7) is 8 below binary16's (15), so the fp16 number
// equals the E4M3 value times 2^-8 exactly, subnormals included.  (Codes
// 0x7F/0xFF, E4M3's NaN, read as 1.875 * 2^0 -- the encoder never writes them.)
// Four codes in a 32-bit word become two fp16x2 words.
__device__ __forceinline__ uint32_t e4m3x2_spread_to_f16x2(uint32_t spread) {
  // spread = b_lo | (b_hi << 16); each 16-bit lane -> ((b & 0x7f) << 7) | ((b & 0x80) << 8)
  return ((spread & 0x007F007Fu) << 7) | ((spread & 0x00800080u) << 8);
}
__device__ __forceinline__ void e4m3x4_to_f16x4_scaled(uint32_t codes, uint32_t& lo2, uint32_t& hi2) {
  lo2 = e4m3x2_spread_to_f16x2(__byte_perm(codes, 0u, 0x4140));  // bytes 0, 1
  hi2 = e4m3x2_spread_to_f16x2(__byte_perm(codes, 0u, 0x4342));  // bytes 2, 3
}

// Exact float value of an E4M3 code (used by the append's re-encode).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
  uint16_t h = (uint16_t)(((code & 0x7Fu) << 7) | ((code & 0x80u) << 8));
  return __half2float(__ushort_as_half(h)) * 256.0f;
}

// ---------------------------------------------------------------------------
// bf16 / fp16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two bf16 (packed) -> two fp16 (packed), round to nearest even.  Exact for
// |x| in [2^-17, 65504].
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  __half2 h = __floats2half2_rn(bf16_lo(w), bf16_hi(w));
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---------------------------------------------------------------------------
// shared memory / async copy primitives
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16 f16, row) * B(16x8 f16, col) + D, fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace sdva
