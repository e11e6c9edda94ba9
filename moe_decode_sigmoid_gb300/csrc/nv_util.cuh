// nv_util.cuh — NVFP4 (e2m1 values, e4m3 block scales) dequantisation and f16
// tensor-core helpers shared by the NVFP4 kernels.  The formats are the OCP
// Microscaling FP4 (E2M1) and OCP 8-bit floating point (E4M3FN) definitions;
// the conversions are PTX cvt instructions.
#pragma once

#include <cuda_fp16.h>

#include "common.cuh"

namespace flint {
namespace nvu {

// Eight e2m1 codes (one 32-bit word, code k in bits 4k..4k+3) -> four f16x2,
// each holding codes (2i, 2i+1) in its (low, high) halves.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t& p0, uint32_t& p1,
                                                uint32_t& p2, uint32_t& p3) {
  asm("{ .reg .b8 b0, b1, b2, b3;\n"
      "  mov.b32 {b0, b1, b2, b3}, %4;\n"
      "  cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "  cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "  cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "  cvt.rn.f16x2.e2m1x2 %3, b3; }"
      : "=r"(p0), "=r"(p1), "=r"(p2), "=r"(p3)
      : "r"(w));
}

// One E4M3 byte -> f16x2 with the scale in both halves.
__device__ __forceinline__ uint32_t e4m3_bcast_f16x2(uint32_t byte) {
  const uint16_t two = (uint16_t)(byte | (byte << 8));
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// f16x2 -> bf16x2, exact for the dequantised weights (<= 6 significant bits,
// inside bf16's range): each half through fp32.
__device__ __forceinline__ uint32_t bf2_of_h2(uint32_t h2) {
  const __half2 v = *reinterpret_cast<const __half2*>(&h2);
  const float2 f = __half22float2(v);
  return pack_bf2(f.x, f.y);
}

__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// True if one of 8 bf16 values (uint4) is beyond f16's range: |x| >= 2^16
// (bf16 magnitude bits >= 0x4780), an infinity or a NaN.  The conversion
// below would make it an f16 infinity.
__device__ __forceinline__ bool bf16x8_beyond_f16(const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  bool out = false;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    out |= (w[i] & 0x7fffu) >= 0x4780u || ((w[i] >> 16) & 0x7fffu) >= 0x4780u;
  return out;
}

// bf16 x 8 (uint4) -> f16 x 8 (uint4), same element order.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4& v) {
  uint4 r;
  r.x = f16x2_of(bf_lo(v.x), bf_hi(v.x));
  r.y = f16x2_of(bf_lo(v.y), bf_hi(v.y));
  r.z = f16x2_of(bf_lo(v.z), bf_hi(v.z));
  r.w = f16x2_of(bf_lo(v.w), bf_hi(v.w));
  return r;
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

}  // namespace nvu
}  // namespace flint
