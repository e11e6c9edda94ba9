// gateup_impl.cuh — device code of the BF16 gate/up stage (see gateup.cu for
// the design); shared by the standalone gate/up kernel and the fused
// small-batch kernel.
#pragma once

#include "common.cuh"
#include "expert_common.cuh"
#include "kernels.h"

namespace flint {
namespace gu {
constexpr int ROWS = 16;                        // 8 gate + 8 up rows
constexpr int ROW_BYTES = H * 2;                // 4 KiB (bf16)
constexpr int STAGE_BYTES = ROWS * ROW_BYTES;   // 64 KiB
constexpr int NSTAGE = 3;
constexpr int UNITS = I / 8;                    // units per group
constexpr int CWARPS = 8;
constexpr int THREADS = CWARPS * 32 + 32;
// CUDA cores for groups of at most 2 tokens; from 3 tokens on, the FMA work
// per weight byte would make a unit slower than its HBM transfer (measured:
// units of 3-4 tokens ran ~1.4x longer and unbalanced the CTAs), so those go
// to the tensor cores.
constexpr int CC_MAX = 2;
// activations buffer keeps room for 4 tokens (shared with other uses)
constexpr int XS_TOKENS = 4;
// Shared buffer: tensor-core partial tiles, the CUDA-core path's bf16
// activations, or the logits during local selection.
constexpr int RED_BYTES = CWARPS * ROWS * GROUP_MAX * 4;
constexpr int XS_BYTES = XS_TOKENS * H * 2;
constexpr int LOGIT_BYTES = LOCAL_SELECT_MAX_B * E * 4;
constexpr int BUF_BYTES = RED_BYTES > XS_BYTES ? (RED_BYTES > LOGIT_BYTES ? RED_BYTES : LOGIT_BYTES)
                                               : (XS_BYTES > LOGIT_BYTES ? XS_BYTES : LOGIT_BYTES);
constexpr size_t SMEM = (size_t)NSTAGE * STAGE_BYTES + BUF_BYTES + sizeof(MetaSmem) + 2 * NSTAGE * 8;
constexpr uint64_t DRAIN_NS = 2000000000ull;
}  // namespace gu

namespace gu_impl {

struct GuCtx {
  uint8_t* stages;
  float* buf;
  uint32_t stages_addr;
  uint32_t full0, empty0;
  uint64_t deadline;
  const uint16_t* x;
  const int* pair_tok;  // shared memory
  float* h;
  WsHeader* hdr;
  volatile int* abort_flag;
};

__device__ __forceinline__ uint32_t full_bar(const GuCtx& c, int s) { return c.full0 + 8u * s; }
__device__ __forceinline__ uint32_t empty_bar(const GuCtx& c, int s) { return c.empty0 + 8u * s; }

// Consumer-side wait for a filled stage.
__device__ __forceinline__ bool wait_full(const GuCtx& c, int slot, uint32_t parity) {
  if (*c.abort_flag) return false;
  if (mbar_wait(full_bar(c, slot), parity, c.deadline)) return true;
  *c.abort_flag = 1;
  set_error(c.hdr, DEV_TIMEOUT);
  return false;
}

// sum of 8 bf16 products w[k] * x[k], one short chain of mixed-precision FMAs
// (each product is exact in fp32; the sum is rounded in fp32).
__device__ __forceinline__ float dot8_bf16(const uint4& w, const uint4& x) {
  float s = 0.f;
  asm("{ .reg .b16 a0, a1, a2, a3, a4, a5, a6, a7, b0, b1, b2, b3, b4, b5, b6, b7;\n"
      "  mov.b32 {a0, a1}, %1;\n  mov.b32 {a2, a3}, %2;\n"
      "  mov.b32 {a4, a5}, %3;\n  mov.b32 {a6, a7}, %4;\n"
      "  mov.b32 {b0, b1}, %5;\n  mov.b32 {b2, b3}, %6;\n"
      "  mov.b32 {b4, b5}, %7;\n  mov.b32 {b6, b7}, %8;\n"
      "  fma.rn.f32.bf16 %0, a0, b0, %0;\n  fma.rn.f32.bf16 %0, a1, b1, %0;\n"
      "  fma.rn.f32.bf16 %0, a2, b2, %0;\n  fma.rn.f32.bf16 %0, a3, b3, %0;\n"
      "  fma.rn.f32.bf16 %0, a4, b4, %0;\n  fma.rn.f32.bf16 %0, a5, b5, %0;\n"
      "  fma.rn.f32.bf16 %0, a6, b6, %0;\n  fma.rn.f32.bf16 %0, a7, b7, %0; }"
      : "+f"(s)
      : "r"(w.x), "r"(w.y), "r"(w.z), "r"(w.w), "r"(x.x), "r"(x.y), "r"(x.z), "r"(x.w));
  return s;
}

// CUDA-core segment: units [u0, u1) of one group with NTOK tokens.  The
// group's bf16 activations are staged once in shared memory (the buffer is
// shared with the tensor-core reduction and the local selection; segments are
// separated by consumer barriers).
template <int NTOK>
__device__ __forceinline__ void seg_cc(const GuCtx& c, int u0, int u1, int pair0, int tok_base,
                                       int& it, bool& ok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* xs = reinterpret_cast<uint4*>(c.buf);  // [NTOK][H/8]
  named_sync(1, gu::CWARPS * 32);                // previous user of buf is done
#pragma unroll
  for (int i = 0; i < NTOK; ++i) {
    const int tok = tok_base >= 0 ? tok_base + i : c.pair_tok[pair0 + i];
    xs[i * (H / 8) + threadIdx.x] =
        __ldg(reinterpret_cast<const uint4*>(c.x + (size_t)tok * H) + threadIdx.x);
  }
  named_sync(1, gu::CWARPS * 32);
  for (int u = u0; u < u1; ++u) {
    const int blk = u & (gu::UNITS - 1);
    const int slot = it % gu::NSTAGE;
    float g[NTOK], v[NTOK];
#pragma unroll
    for (int i = 0; i < NTOK; ++i) g[i] = v[i] = 0.f;
    if (ok) ok = wait_full(c, slot, (uint32_t)(it / gu::NSTAGE) & 1u);
    if (ok) {
      const uint8_t* st = c.stages + slot * gu::STAGE_BYTES;
      const uint4* gr = reinterpret_cast<const uint4*>(st + warp * gu::ROW_BYTES);
      const uint4* ur = reinterpret_cast<const uint4*>(st + (8 + warp) * gu::ROW_BYTES);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4 wg[4], wu[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          wg[j] = gr[lane + 32 * (4 * half + j)];
          wu[j] = ur[lane + 32 * (4 * half + j)];
        }
#pragma unroll
        for (int i = 0; i < NTOK; ++i) {
          float pg[4], pu[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 xv = xs[i * (H / 8) + lane + 32 * (4 * half + j)];
            pg[j] = dot8_bf16(wg[j], xv);
            pu[j] = dot8_bf16(wu[j], xv);
          }
          g[i] += (pg[0] + pg[1]) + (pg[2] + pg[3]);
          v[i] += (pu[0] + pu[1]) + (pu[2] + pu[3]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(c, slot));
    ++it;
#pragma unroll
    for (int i = 0; i < NTOK; ++i) {
      const float gs = warp_sum(g[i]);
      const float vs = warp_sum(v[i]);
      if (lane == 0 && ok) store_h_split(c.h, (size_t)(pair0 + i), blk * 8 + warp, silu_mul(gs, vs));
    }
  }
}

// Tensor-core segment: units [u0, u1) of one group with n tokens, NT = ceil(n/8).
template <int NT>
__device__ __forceinline__ void seg_mma(const GuCtx& c, int u0, int u1, int pair0, int n,
                                        int tok_base, int& it, bool& ok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  named_sync(1, gu::CWARPS * 32);  // the previous user of buf is done
  uint4 bfr[NT][8];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int slot = nt * 8 + g;
    if (slot < n) {
      const int tok = tok_base >= 0 ? tok_base + slot : c.pair_tok[pair0 + slot];
      const uint16_t* row = c.x + (size_t)tok * H + warp * 256 + q * 8;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb)
        bfr[nt][kb] = __ldg(reinterpret_cast<const uint4*>(row + kb * 32));
    } else {
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) bfr[nt][kb] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  for (int u = u0; u < u1; ++u) {
    const int blk = u & (gu::UNITS - 1);
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
    const int slot = it % gu::NSTAGE;
    if (ok) ok = wait_full(c, slot, (uint32_t)(it / gu::NSTAGE) & 1u);
    if (ok) {
      const uint8_t* rlo =
          c.stages + slot * gu::STAGE_BYTES + g * gu::ROW_BYTES + (warp * 256 + q * 8) * 2;
      const uint8_t* rhi = rlo + 8 * gu::ROW_BYTES;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        const uint4 alo = *reinterpret_cast<const uint4*>(rlo + kb * 64);
        const uint4 ahi = *reinterpret_cast<const uint4*>(rhi + kb * 64);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint4 b = bfr[nt][kb];
          mma_bf16(acc[nt], alo.x, ahi.x, alo.y, ahi.y, b.x, b.y);
          mma_bf16(acc[nt], alo.z, ahi.z, alo.w, ahi.w, b.z, b.w);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty_bar(c, slot));
    ++it;
    float* red = c.buf + warp * gu::ROWS * GROUP_MAX;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int col = nt * 8 + 2 * q;
      red[g * GROUP_MAX + col] = acc[nt][0];
      red[g * GROUP_MAX + col + 1] = acc[nt][1];
      red[(g + 8) * GROUP_MAX + col] = acc[nt][2];
      red[(g + 8) * GROUP_MAX + col + 1] = acc[nt][3];
    }
    named_sync(1, gu::CWARPS * 32);
    {
      // thread (token slot j, row r): the 8 rows of a token are 8 adjacent
      // lanes, which store the token's h block together
      static_assert(gu::CWARPS * 32 / 8 >= GROUP_MAX, "one 8-lane group per token slot");
      const int j = threadIdx.x >> 3;
      const int r = threadIdx.x & 7;
      const int jr = j < n ? j : 0;
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int w = 0; w < gu::CWARPS; ++w) {
        gs += c.buf[(w * gu::ROWS + r) * GROUP_MAX + jr];
        us += c.buf[(w * gu::ROWS + r + 8) * GROUP_MAX + jr];
      }
      store_h_block8(c.h, (size_t)(pair0 + jr), blk, silu_mul(gs, us), j < n && ok);
    }
    named_sync(1, gu::CWARPS * 32);
  }
}

// Issues the stage of one unit (8 gate + 8 up rows of the expert at `base`,
// block `blk`); false if the ring could not be acquired (abort).
__device__ __forceinline__ bool issue_unit(const GuCtx& c, const uint16_t* base, int blk, int& it) {
  const int slot = it % gu::NSTAGE;
  bool got = true;
  if (it >= gu::NSTAGE)
    got = mbar_wait(empty_bar(c, slot), (uint32_t)((it / gu::NSTAGE) - 1) & 1u, c.deadline);
  // A consumer that gave up sets the flag before releasing its stage.
  if (!got || *c.abort_flag) {
    *c.abort_flag = 1;
    if (!got) set_error(c.hdr, DEV_TIMEOUT);
    return false;
  }
  mbar_expect_tx(full_bar(c, slot), gu::STAGE_BYTES);
  const uint32_t dst = c.stages_addr + slot * gu::STAGE_BYTES;
  bulk_g2s_stream(dst, base + (size_t)(blk * 8) * H, 8 * gu::ROW_BYTES, full_bar(c, slot));
  bulk_g2s_stream(dst + 8 * gu::ROW_BYTES, base + (size_t)(I + blk * 8) * H, 8 * gu::ROW_BYTES,
           full_bar(c, slot));
  ++it;
  return true;
}

// Never leave the CTA with copies still landing in its shared memory.
__device__ __forceinline__ void drain(const GuCtx& c, int it) {
  const uint64_t drain = globaltimer_ns() + gu::DRAIN_NS;
  for (int j = it - gu::NSTAGE < 0 ? 0 : it - gu::NSTAGE; j < it; ++j)
    mbar_wait(full_bar(c, j % gu::NSTAGE), (uint32_t)(j / gu::NSTAGE) & 1u, drain);
}

// The shared-expert groups do not depend on routing: in the decode chain
// ("early") their units are dealt round-robin over the CTAs and started
// before the wait for the router.  Every other unit is claimed after the wait
// (gateup.cu).
struct Plan {
  int nsg;        // shared groups per shared expert
  int nsu;        // shared units handled before the wait (early only)
};

__device__ __forceinline__ Plan plan_pre(int B, bool early) {
  Plan p;
  p.nsg = (B + GROUP_MAX - 1) / GROUP_MAX;
  p.nsu = early ? S * p.nsg * gu::UNITS : 0;
  return p;
}

// Shared unit j -> (shared expert, group, block) and its pairs / tokens.
struct SharedUnit {
  int s, gi, blk, pair0, n, tok0;
};
__device__ __forceinline__ SharedUnit shared_unit(int j, int B, int nsg) {
  SharedUnit u;
  const int sg = j / gu::UNITS;
  u.blk = j % gu::UNITS;
  u.s = sg / nsg;
  u.gi = sg % nsg;
  u.tok0 = u.gi * GROUP_MAX;
  u.n = min(GROUP_MAX, B - u.tok0);
  u.pair0 = B * TOPK + u.s * B + u.tok0;
  return u;
}

__device__ __forceinline__ void segment(const GuCtx& c, int u0, int u1, int pair0, int n,
                                        int tok_base, int& it, bool& ok) {
  if (n <= gu::CC_MAX) {
    switch (n) {
      case 1: seg_cc<1>(c, u0, u1, pair0, tok_base, it, ok); break;
      default: seg_cc<2>(c, u0, u1, pair0, tok_base, it, ok); break;
    }
  } else {
    switch ((n + 7) >> 3) {
      case 1: seg_mma<1>(c, u0, u1, pair0, n, tok_base, it, ok); break;
      case 2: seg_mma<2>(c, u0, u1, pair0, n, tok_base, it, ok); break;
      default: seg_mma<3>(c, u0, u1, pair0, n, tok_base, it, ok); break;
    }
  }
}

}  // namespace gu_impl
}  // namespace flint
