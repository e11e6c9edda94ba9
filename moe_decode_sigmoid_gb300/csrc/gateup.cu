// gateup.cu — gathered gate/up GEMV with fused SiLU-and-mul, BF16 weights.
//
// For every (expert, token-range) group built by the router and every token t
// in it:  h[pair(t), i] = silu(Wg[i] . x_t) * (Wu[i] . x_t),  i < 512, with
// silu(g) = g / (1 + exp(-g)) ("SiLU-and-mul": Flint on Intel Arc Pro B70,
// "norm.py: Triton kernels that assumed CUDA").  Only the selected experts'
// rows are read ("read only the selected experts' weights": vLLM Day-0 Support
// for Recursive's Flint, "Optimization Strategies").
//
// Work unit: one group x one block of 8 intermediate rows = the 8 gate rows
// plus the 8 matching up rows (64 KiB of weights).  Units are numbered
// group-major and each CTA takes one contiguous range of them, so every SM
// streams the same number of weight bytes.
//
// Per CTA: 8 consumer warps + 1 producer warp.  The producer's elected lane
// streams each unit as two 32 KiB stages (16 rows x 1024 columns) through a
// 6-stage shared-memory ring with cp.async.bulk (TMA) and mbarriers, so up to
// ~200 KiB per SM is in flight at once.  Rows land at a 2112-byte stride
// (= 64 mod 128) so the tensor-core fragment loads are bank-conflict free.
// Consumers, per group:
//   <= 4 tokens (the batch-1/8 case): CUDA cores.  Warp w owns gate row w and
//      up row w of the stage; each lane keeps its slice of the group's
//      activations in registers for the whole group and accumulates fp32.
//   5..24 tokens: mma.sync m16n8k16 (bf16 in, fp32 acc) with the 16 weight
//      rows as M and the tokens as N; warp w owns a 128-column K-slice; the
//      8 partial tiles are summed through shared memory.  Because each
//      fragment's K order is the same permutation for weights and
//      activations, both are loaded as plain 16-byte row chunks.
// Every wait is bounded by the workspace's limit.
#include "common.cuh"
#include "kernels.h"

namespace flint {
namespace gu {
constexpr int ROWS = 16;                        // 8 gate + 8 up rows
constexpr int KS = 1024;                        // columns per stage
constexpr int ROW_BYTES = KS * 2;               // bf16
constexpr int ROW_STRIDE = ROW_BYTES + 64;      // 64 mod 128
constexpr int STAGE_BYTES = ROWS * ROW_STRIDE;  // 33,792
constexpr int NSTAGE = 6;
constexpr int UNITS = I / 8;                    // units per group
constexpr int CWARPS = 8;
constexpr int THREADS = CWARPS * 32 + 32;
constexpr int CC_MAX = 4;
// Shared buffer: tensor-core partial tiles, or the CUDA-core path's activations.
constexpr int RED_FLOATS = (CWARPS * ROWS * GROUP_MAX > CC_MAX * H / 2) ? CWARPS * ROWS * GROUP_MAX
                                                                        : CC_MAX * H / 2;
constexpr size_t SMEM = (size_t)NSTAGE * STAGE_BYTES + RED_FLOATS * 4 + 2 * NSTAGE * 8;
constexpr uint64_t DRAIN_NS = 2000000000ull;
}  // namespace gu

namespace {

struct GuCtx {
  uint8_t* stages;
  float* red;
  uint32_t stages_addr;
  uint32_t full0, empty0;
  uint64_t deadline;
  const uint16_t* x;
  const int* pair_tok;
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

__device__ __forceinline__ void dot8x2(const uint4& wg, const uint4& wu, const uint4& x, float& ag,
                                       float& au) {
  const float x0 = bf_lo(x.x), x1 = bf_hi(x.x), x2 = bf_lo(x.y), x3 = bf_hi(x.y);
  const float x4 = bf_lo(x.z), x5 = bf_hi(x.z), x6 = bf_lo(x.w), x7 = bf_hi(x.w);
  ag = fmaf(bf_lo(wg.x), x0, ag); au = fmaf(bf_lo(wu.x), x0, au);
  ag = fmaf(bf_hi(wg.x), x1, ag); au = fmaf(bf_hi(wu.x), x1, au);
  ag = fmaf(bf_lo(wg.y), x2, ag); au = fmaf(bf_lo(wu.y), x2, au);
  ag = fmaf(bf_hi(wg.y), x3, ag); au = fmaf(bf_hi(wu.y), x3, au);
  ag = fmaf(bf_lo(wg.z), x4, ag); au = fmaf(bf_lo(wu.z), x4, au);
  ag = fmaf(bf_hi(wg.z), x5, ag); au = fmaf(bf_hi(wu.z), x5, au);
  ag = fmaf(bf_lo(wg.w), x6, ag); au = fmaf(bf_lo(wu.w), x6, au);
  ag = fmaf(bf_hi(wg.w), x7, ag); au = fmaf(bf_hi(wu.w), x7, au);
}

// CUDA-core segment: units [u0, u1) of one group with NTOK tokens.  The
// group's activations are staged once in shared memory (xs, which aliases the
// tensor-core reduction buffer; segments are separated by consumer barriers).
template <int NTOK>
__device__ __forceinline__ void seg_cc(const GuCtx& c, int u0, int u1, int pair0, int tok_base,
                                       int& it, bool& ok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4* xs = reinterpret_cast<uint4*>(c.red);
  named_sync(1, gu::CWARPS * 32);  // previous segment is done with xs
#pragma unroll
  for (int i = 0; i < NTOK; ++i) {
    const int tok = tok_base >= 0 ? tok_base + i : __ldcg(c.pair_tok + pair0 + i);
    const uint4* row = reinterpret_cast<const uint4*>(c.x + (size_t)tok * H);
    xs[i * (H / 8) + threadIdx.x] = __ldg(row + threadIdx.x);  // 256 threads x 16 B = one row
  }
  named_sync(1, gu::CWARPS * 32);
  for (int u = u0; u < u1; ++u) {
    const int blk = u & (gu::UNITS - 1);
    float ag[NTOK], au[NTOK];
#pragma unroll
    for (int i = 0; i < NTOK; ++i) ag[i] = au[i] = 0.f;
#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
      const int slot = it % gu::NSTAGE;
      if (ok) ok = wait_full(c, slot, (uint32_t)(it / gu::NSTAGE) & 1u);
      if (ok) {
        const uint8_t* st = c.stages + slot * gu::STAGE_BYTES;
        const uint4* gr = reinterpret_cast<const uint4*>(st + warp * gu::ROW_STRIDE);
        const uint4* ur = reinterpret_cast<const uint4*>(st + (8 + warp) * gu::ROW_STRIDE);
        const uint4* xk = xs + kh * (gu::KS / 8) + lane;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 wg = gr[lane + 32 * j];
          const uint4 wu = ur[lane + 32 * j];
#pragma unroll
          for (int i = 0; i < NTOK; ++i) dot8x2(wg, wu, xk[i * (H / 8) + 32 * j], ag[i], au[i]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(c, slot));
      ++it;
    }
#pragma unroll
    for (int i = 0; i < NTOK; ++i) {
      const float g = warp_sum(ag[i]);
      const float v = warp_sum(au[i]);
      if (lane == 0 && ok) c.h[(size_t)(pair0 + i) * I + blk * 8 + warp] = silu_mul(g, v);
    }
  }
}

// Tensor-core segment: units [u0, u1) of one group with n tokens, NT = ceil(n/8).
template <int NT>
__device__ __forceinline__ void seg_mma(const GuCtx& c, int u0, int u1, int pair0, int n,
                                        int tok_base, int& it, bool& ok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  named_sync(1, gu::CWARPS * 32);  // a preceding CUDA-core segment is done with xs
  uint4 bfr[NT][2][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int slot = nt * 8 + g;
    if (slot < n) {
      const int tok = tok_base >= 0 ? tok_base + slot : __ldcg(c.pair_tok + pair0 + slot);
      const uint16_t* row = c.x + (size_t)tok * H + warp * 128 + q * 8;
#pragma unroll
      for (int kh = 0; kh < 2; ++kh)
#pragma unroll
        for (int kb = 0; kb < 4; ++kb)
          bfr[nt][kh][kb] = __ldg(reinterpret_cast<const uint4*>(row + kh * gu::KS + kb * 32));
    } else {
#pragma unroll
      for (int kh = 0; kh < 2; ++kh)
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) bfr[nt][kh][kb] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  for (int u = u0; u < u1; ++u) {
    const int blk = u & (gu::UNITS - 1);
    float acc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
#pragma unroll
    for (int kh = 0; kh < 2; ++kh) {
      const int slot = it % gu::NSTAGE;
      if (ok) ok = wait_full(c, slot, (uint32_t)(it / gu::NSTAGE) & 1u);
      if (ok) {
        const uint8_t* rlo =
            c.stages + slot * gu::STAGE_BYTES + g * gu::ROW_STRIDE + (warp * 128 + q * 8) * 2;
        const uint8_t* rhi = rlo + 8 * gu::ROW_STRIDE;
#pragma unroll
        for (int kb = 0; kb < 4; ++kb) {
          const uint4 alo = *reinterpret_cast<const uint4*>(rlo + kb * 64);
          const uint4 ahi = *reinterpret_cast<const uint4*>(rhi + kb * 64);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const uint4 b = bfr[nt][kh][kb];
            mma_bf16(acc[nt], alo.x, ahi.x, alo.y, ahi.y, b.x, b.y);
            mma_bf16(acc[nt], alo.z, ahi.z, alo.w, ahi.w, b.z, b.w);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(c, slot));
      ++it;
    }
    float* red = c.red + warp * gu::ROWS * GROUP_MAX;
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
      const int r = threadIdx.x >> 5;  // 0..7
      const int j = threadIdx.x & 31;  // token slot (GROUP_MAX <= 32)
      if (j < n && ok) {
        float gs = 0.f, us = 0.f;
#pragma unroll
        for (int w = 0; w < gu::CWARPS; ++w) {
          gs += c.red[(w * gu::ROWS + r) * GROUP_MAX + j];
          us += c.red[(w * gu::ROWS + r + 8) * GROUP_MAX + j];
        }
        c.h[(size_t)(pair0 + j) * I + blk * 8 + r] = silu_mul(gs, us);
      }
    }
    named_sync(1, gu::CWARPS * 32);
  }
}

// Issues the two stages of one unit (8 gate + 8 up rows of expert `e`, block
// `blk`); false if the ring could not be acquired (abort).
__device__ __forceinline__ bool issue_unit(const GuCtx& c, const uint16_t* base, int blk, int& it) {
#pragma unroll 1
  for (int kh = 0; kh < 2; ++kh) {
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
    mbar_expect_tx(full_bar(c, slot), gu::ROWS * gu::ROW_BYTES);
    const uint32_t dst = c.stages_addr + slot * gu::STAGE_BYTES;
#pragma unroll 1
    for (int r = 0; r < gu::ROWS; ++r) {
      const int row = (r < 8 ? 0 : I) + blk * 8 + (r & 7);
      bulk_g2s(dst + r * gu::ROW_STRIDE, base + (size_t)row * H + kh * gu::KS, gu::ROW_BYTES,
               full_bar(c, slot));
    }
    ++it;
  }
  return true;
}

// Never leave the CTA with copies still landing in its shared memory.
__device__ __forceinline__ void drain(const GuCtx& c, int it) {
  const uint64_t drain = globaltimer_ns() + gu::DRAIN_NS;
  for (int j = it - gu::NSTAGE < 0 ? 0 : it - gu::NSTAGE; j < it; ++j)
    mbar_wait(full_bar(c, j % gu::NSTAGE), (uint32_t)(j / gu::NSTAGE) & 1u, drain);
}

// Which units a CTA runs.  Shared-expert groups do not depend on routing; in
// the decode chain ("early") they are dealt round-robin over the CTAs and
// started before the wait for the router, and the routed units are then split
// so that every CTA ends up with the same total.  Otherwise every group,
// shared ones included, is split evenly after the wait.
struct Plan {
  int nsg;        // shared groups per shared expert
  int nsu;        // shared units handled before the wait (early only)
  int r_begin, r_end;
};

__device__ __forceinline__ int shared_units_below(int c, int nsu, int G) {
  return c * (nsu / G) + min(c, nsu % G);
}

__device__ __forceinline__ Plan plan_pre(int B, bool early) {
  Plan p;
  p.nsg = (B + GROUP_MAX - 1) / GROUP_MAX;
  p.nsu = early ? S * p.nsg * gu::UNITS : 0;
  p.r_begin = p.r_end = 0;
  return p;
}

__device__ __forceinline__ void plan_post(Plan& p, int n_groups, bool early) {
  const int G = gridDim.x, c = blockIdx.x;
  if (!early) {
    const int n = n_groups * gu::UNITS;
    p.r_begin = (int)((long long)c * n / G);
    p.r_end = (int)((long long)(c + 1) * n / G);
    return;
  }
  const int nru = (n_groups - S * p.nsg) * gu::UNITS;
  const long long T = (long long)p.nsu + nru;
  auto R = [&](int cc) {
    long long r = cc * T / G - shared_units_below(cc, p.nsu, G);
    return (int)(r < 0 ? 0 : (r > nru ? nru : r));
  };
  p.r_begin = R(c);
  p.r_end = max(p.r_begin, R(c + 1));
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

__device__ __forceinline__ void produce(const GuCtx& c, const ExpertArgs& a, Plan& pl, bool early) {
  int it = 0;
  bool ok = true;
  for (int j = blockIdx.x; ok && j < pl.nsu; j += gridDim.x) {
    const SharedUnit su = shared_unit(j, a.B, pl.nsg);
    ok = issue_unit(c, a.w.ws13 + (size_t)su.s * (2 * I) * H, su.blk, it);
  }
  pdl_wait();     // routing and buckets come from the router kernel
  plan_post(pl, (int)__ldcg(&a.ws.hdr->n_groups), early);
  for (int u = pl.r_begin; ok && u < pl.r_end; ++u) {
    const int4 grp = __ldcg(a.ws.groups + (u / gu::UNITS));
    const uint16_t* base = grp.x < E ? a.w.w13 + (size_t)grp.x * (2 * I) * H
                                     : a.w.ws13 + (size_t)(grp.x - E) * (2 * I) * H;
    ok = issue_unit(c, base, u & (gu::UNITS - 1), it);
  }
  drain(c, it);
}

template <bool CC>
__device__ __forceinline__ void run_segment(const GuCtx& c, int u0, int u1, int pair0, int n,
                                            int tok_base, int& it, bool& ok) {
  if (CC) {
    switch (n) {
      case 1: seg_cc<1>(c, u0, u1, pair0, tok_base, it, ok); break;
      case 2: seg_cc<2>(c, u0, u1, pair0, tok_base, it, ok); break;
      case 3: seg_cc<3>(c, u0, u1, pair0, tok_base, it, ok); break;
      default: seg_cc<4>(c, u0, u1, pair0, tok_base, it, ok); break;
    }
  } else {
    switch ((n + 7) >> 3) {
      case 1: seg_mma<1>(c, u0, u1, pair0, n, tok_base, it, ok); break;
      case 2: seg_mma<2>(c, u0, u1, pair0, n, tok_base, it, ok); break;
      default: seg_mma<3>(c, u0, u1, pair0, n, tok_base, it, ok); break;
    }
  }
}

__device__ __forceinline__ void segment(const GuCtx& c, int u0, int u1, int pair0, int n,
                                        int tok_base, int& it, bool& ok) {
  if (n <= gu::CC_MAX) run_segment<true>(c, u0, u1, pair0, n, tok_base, it, ok);
  else run_segment<false>(c, u0, u1, pair0, n, tok_base, it, ok);
}

}  // namespace

__global__ void __launch_bounds__(gu::THREADS, 1) gateup_bf16_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  GuCtx c;
  c.stages = smem;
  c.red = reinterpret_cast<float*>(smem + gu::NSTAGE * gu::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(c.red + gu::RED_FLOATS);
  c.stages_addr = smem_addr(smem);
  c.full0 = smem_addr(bars);
  c.empty0 = smem_addr(bars + gu::NSTAGE);
  c.x = a.x;
  c.pair_tok = a.ws.pair_tok;
  c.h = a.ws.h;
  c.hdr = a.ws.hdr;
  c.abort_flag = &s_abort;
  if (threadIdx.x == 0) {
    for (int s = 0; s < gu::NSTAGE; ++s) {
      mbar_init(full_bar(c, s), 1);
      mbar_init(empty_bar(c, s), gu::CWARPS);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const bool early = a.early_shared != 0;
  Plan pl = plan_pre(a.B, early);
  c.deadline = wait_deadline(a.ws.hdr);
  if ((threadIdx.x >> 5) == gu::CWARPS) {
    if ((threadIdx.x & 31) == 0) produce(c, a, pl, early);
    pdl_trigger();
    return;
  }
  int it = 0;
  bool ok = true;
  for (int j = blockIdx.x; j < pl.nsu; j += gridDim.x) {
    const SharedUnit su = shared_unit(j, a.B, pl.nsg);
    // unit numbers inside a segment only serve as block indices (u & 63)
    segment(c, su.blk, su.blk + 1, su.pair0, su.n, su.tok0, it, ok);
  }
  pdl_wait();     // routing and buckets come from the router kernel
  pdl_trigger();  // the down kernel may start its prologue
  plan_post(pl, (int)__ldcg(&a.ws.hdr->n_groups), early);
  int u = pl.r_begin;
  while (u < pl.r_end) {
    const int gi = u / gu::UNITS;
    const int4 grp = __ldcg(a.ws.groups + gi);
    const int u1 = min(pl.r_end, (gi + 1) * gu::UNITS);
    segment(c, u, u1, grp.y, grp.z, -1, it, ok);
    u = u1;
  }
}

cudaError_t launch_gateup_bf16(const ExpertArgs& a, cudaStream_t stream, int num_sms) {
  static bool attr_set = false;  // idempotent; racing first calls set the same value
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(gateup_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gu::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms, 1, 1);
  cfg.blockDim = dim3(gu::THREADS, 1, 1);
  cfg.dynamicSmemBytes = gu::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gateup_bf16_kernel, a);
}

}  // namespace flint
