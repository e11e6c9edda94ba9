// down_impl.cuh — device code of the BF16 down / combine stage (see down.cu
// for the design); shared by the standalone down kernel and the fused
// small-batch kernel.
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
constexpr int THREADS = CWARPS * 32 + 32;
constexpr int RED_FLOATS = CWARPS * RS * GROUP_MAX;
constexpr int MAX_STAGES = 8;
constexpr int SMEM_CAP = 232448 - 1024;   // opt-in maximum minus static/slack
constexpr int CC_MAX = 4;
constexpr uint64_t DRAIN_NS = 2000000000ull;

__host__ __device__ inline int nmax_for(int B) { return B < GROUP_MAX ? B : GROUP_MAX; }
__host__ __device__ inline int stage_bytes(int B) { return WBYTES + nmax_for(B) * HSTRIDE; }
__host__ __device__ inline int fixed_bytes(int B) {
  return RED_FLOATS * 4 + B * RS * 4 + (int)sizeof(MetaSmem) + MAX_B * SLOTS * 4 +
         2 * MAX_STAGES * 8;
}
__host__ __device__ inline int nstages(int B) {
  int n = (SMEM_CAP - fixed_bytes(B)) / stage_bytes(B);
  return n > MAX_STAGES ? MAX_STAGES : n;
}
__host__ __device__ inline int smem_bytes(int B) {
  return nstages(B) * stage_bytes(B) + fixed_bytes(B);
}
}  // namespace dn

namespace dn_impl {

struct DnCtx {
  uint8_t* stages;
  uint32_t stages_addr;
  int stage_bytes, nstage;
  float* red;
  float* acc;  // [B][RS]
  uint32_t full0, empty0;
  uint64_t deadline;
  WsHeader* hdr;
  volatile int* abort_flag;
  const int* pair_tok;  // shared memory
  const float* pair_w;  // shared memory
};

__device__ __forceinline__ uint32_t full_bar(const DnCtx& c, int s) { return c.full0 + 8u * s; }
__device__ __forceinline__ uint32_t empty_bar(const DnCtx& c, int s) { return c.empty0 + 8u * s; }

__device__ __forceinline__ bool wait_full(const DnCtx& c, int slot, uint32_t parity) {
  if (*c.abort_flag) return false;
  if (mbar_wait(full_bar(c, slot), parity, c.deadline)) return true;
  *c.abort_flag = 1;
  set_error(c.hdr, DEV_TIMEOUT);
  return false;
}

// CUDA-core group of NTOK <= 4 tokens.  Warp w owns Wd rows 2w and 2w+1; lane
// l covers K elements [4l + 128m, 4l + 128m + 4), m = 0..3.  The lane's 32
// weights are unpacked once for all tokens, every token's two partial dots are
// formed first, then all the warp reductions run interleaved (no branch
// between them), then lane 0 applies the combine weights.
template <int NTOK>
__device__ __forceinline__ void group_cc(const DnCtx& c, const uint8_t* st, int pair0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint8_t* w0 = st + (2 * warp) * dn::WSTRIDE;
  const uint8_t* w1 = w0 + dn::WSTRIDE;
  float f0[16], f1[16];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint2 a0 = *reinterpret_cast<const uint2*>(w0 + (4 * lane + 128 * m) * 2);
    const uint2 a1 = *reinterpret_cast<const uint2*>(w1 + (4 * lane + 128 * m) * 2);
    f0[4 * m] = bf_lo(a0.x);
    f0[4 * m + 1] = bf_hi(a0.x);
    f0[4 * m + 2] = bf_lo(a0.y);
    f0[4 * m + 3] = bf_hi(a0.y);
    f1[4 * m] = bf_lo(a1.x);
    f1[4 * m + 1] = bf_hi(a1.x);
    f1[4 * m + 2] = bf_lo(a1.y);
    f1[4 * m + 3] = bf_hi(a1.y);
  }
  const uint8_t* hs = st + dn::WBYTES;
  float s0[NTOK], s1[NTOK];
#pragma unroll
  for (int i = 0; i < NTOK; ++i) {
    s0[i] = s1[i] = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float4 hv =
          *reinterpret_cast<const float4*>(hs + i * dn::HSTRIDE + (4 * lane + 128 * m) * 4);
      s0[i] = fmaf(f0[4 * m], hv.x, s0[i]);
      s0[i] = fmaf(f0[4 * m + 1], hv.y, s0[i]);
      s0[i] = fmaf(f0[4 * m + 2], hv.z, s0[i]);
      s0[i] = fmaf(f0[4 * m + 3], hv.w, s0[i]);
      s1[i] = fmaf(f1[4 * m], hv.x, s1[i]);
      s1[i] = fmaf(f1[4 * m + 1], hv.y, s1[i]);
      s1[i] = fmaf(f1[4 * m + 2], hv.z, s1[i]);
      s1[i] = fmaf(f1[4 * m + 3], hv.w, s1[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int i = 0; i < NTOK; ++i) {
      s0[i] += __shfl_xor_sync(0xffffffffu, s0[i], o);
      s1[i] += __shfl_xor_sync(0xffffffffu, s1[i], o);
    }
  }
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NTOK; ++i) {
      const int t = c.pair_tok[pair0 + i];
      const float wt = c.pair_w[pair0 + i];
      c.acc[t * dn::RS + 2 * warp] += wt * s0[i];
      c.acc[t * dn::RS + 2 * warp + 1] += wt * s1[i];
    }
  }
}

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

__device__ __forceinline__ void produce(const DnCtx& c, const int4* groups, int n_groups,
                                        const uint16_t* w2, const uint16_t* ws2, const float* h,
                                        int r0) {
  int it = 0;
  for (int gi = 0; gi < n_groups; ++gi) {
    const int4 grp = groups[gi];
    const int slot = it % c.nstage;
    if (it >= c.nstage) {
      const bool got = mbar_wait(empty_bar(c, slot), (uint32_t)((it / c.nstage) - 1) & 1u, c.deadline);
      if (!got || *c.abort_flag) {
        *c.abort_flag = 1;
        if (!got) set_error(c.hdr, DEV_TIMEOUT);
        break;
      }
    } else if (*c.abort_flag) {
      break;
    }
    const int n = grp.z;
    mbar_expect_tx(full_bar(c, slot), dn::RS * dn::WROW + n * dn::HROW);
    const uint32_t dst = c.stages_addr + slot * c.stage_bytes;
    const uint16_t* wb = (grp.x < E ? w2 + (size_t)grp.x * H * I : ws2 + (size_t)(grp.x - E) * H * I) +
                         (size_t)r0 * I;
    bulk_g2s(dst, wb, dn::WBYTES, full_bar(c, slot));
    bulk_g2s(dst + dn::WBYTES, h + (size_t)grp.y * I, n * dn::HROW, full_bar(c, slot));
    ++it;
  }
  const uint64_t drain = globaltimer_ns() + dn::DRAIN_NS;
  for (int j = it - c.nstage < 0 ? 0 : it - c.nstage; j < it; ++j)
    mbar_wait(full_bar(c, j % c.nstage), (uint32_t)(j / c.nstage) & 1u, drain);
}

}  // namespace dn_impl
}  // namespace flint
