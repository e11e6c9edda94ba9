// down_impl.cuh — the tensor-core down / combine step for a group of 5..8
// tokens, used by the fused small-batch kernel (its own CUDA-core path takes
// groups of up to 4 tokens).
//
// A CTA owns 16 output rows; the group's 16 Wd rows (16 KiB, contiguous) and
// fp32 h rows sit in one shared-memory slot.  mma.sync m16n8k16 with the Wd
// rows as M and the tokens as N; the fp32 h is split into two bf16 parts
// (hi + lo, two MMAs) so the operand keeps ~16 significant bits; warp w owns a
// 64-column K-slice; the 8 partial tiles are summed through shared memory and
// weighted into the CTA's accumulators.
#pragma once

#include "common.cuh"
#include "expert_common.cuh"
#include "kernels.h"

namespace flint {
namespace dn {
constexpr int RS = 16;                    // output rows per CTA
constexpr int WROW = I * 2;               // bytes of one Wd row
constexpr int WSTRIDE = WROW;             // the 16 rows are one contiguous copy
constexpr int WBYTES = RS * WSTRIDE;      // 16 KiB
constexpr int HROW = I * 4;               // bytes of one fp32 h row
constexpr int HSTRIDE = HROW;             // the group's h rows are one contiguous copy
constexpr int CWARPS = 8;
constexpr int RED_FLOATS = CWARPS * RS * GROUP_MAX;
constexpr int CC_MAX = 4;                 // larger groups take the tensor-core step
}  // namespace dn

namespace dn_impl {

struct DnCtx {
  float* red;           // [CWARPS][RS][GROUP_MAX] partial tiles
  float* acc;           // [B][RS] accumulators
  const int* pair_tok;  // shared memory
  const float* pair_w;  // shared memory
};

template <int NT>
__device__ __forceinline__ void group_mma(const DnCtx& c, const uint8_t* st, int pair0, int n) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  float acc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
  const uint8_t* rlo = st + g * dn::WSTRIDE + (warp * 64 + q * 8) * 2;
  const uint8_t* rhi = rlo + 8 * dn::WSTRIDE;
  const uint8_t* hs = st + dn::WBYTES + (warp * 64 + q * 8) * 4;
#pragma unroll
  for (int kb = 0; kb < 2; ++kb) {
    const uint4 alo = *reinterpret_cast<const uint4*>(rlo + kb * 64);
    const uint4 ahi = *reinterpret_cast<const uint4*>(rhi + kb * 64);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int slot = nt * 8 + g;
      // h (fp32) = hi + lo with both parts bf16: two MMAs keep ~16 bits of h.
      uint32_t b[4] = {0u, 0u, 0u, 0u}, l[4] = {0u, 0u, 0u, 0u};
      if (slot < n) {
        const float4 h0 = *reinterpret_cast<const float4*>(hs + slot * dn::HSTRIDE + kb * 128);
        const float4 h1 = *reinterpret_cast<const float4*>(hs + slot * dn::HSTRIDE + kb * 128 + 16);
        split_bf2(h0.x, h0.y, b[0], l[0]);
        split_bf2(h0.z, h0.w, b[1], l[1]);
        split_bf2(h1.x, h1.y, b[2], l[2]);
        split_bf2(h1.z, h1.w, b[3], l[3]);
      }
      mma_bf16(acc[nt], alo.x, ahi.x, alo.y, ahi.y, b[0], b[1]);
      mma_bf16(acc[nt], alo.z, ahi.z, alo.w, ahi.w, b[2], b[3]);
      mma_bf16(acc[nt], alo.x, ahi.x, alo.y, ahi.y, l[0], l[1]);
      mma_bf16(acc[nt], alo.z, ahi.z, alo.w, ahi.w, l[2], l[3]);
    }
  }
  float* red = c.red + warp * dn::RS * GROUP_MAX;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = nt * 8 + 2 * q;
    red[g * GROUP_MAX + col] = acc[nt][0];
    red[g * GROUP_MAX + col + 1] = acc[nt][1];
    red[(g + 8) * GROUP_MAX + col] = acc[nt][2];
    red[(g + 8) * GROUP_MAX + col + 1] = acc[nt][3];
  }
  named_sync(1, dn::CWARPS * 32);
  for (int i = threadIdx.x; i < dn::RS * n; i += dn::CWARPS * 32) {
    const int r = i & (dn::RS - 1), j = i >> 4;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < dn::CWARPS; ++w) s += c.red[(w * dn::RS + r) * GROUP_MAX + j];
    const int t = c.pair_tok[pair0 + j];
    const float wt = c.pair_w[pair0 + j];
    c.acc[t * dn::RS + r] += wt * s;
  }
  named_sync(1, dn::CWARPS * 32);
}

}  // namespace dn_impl
}  // namespace flint
