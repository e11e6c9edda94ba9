// down.cu — down GEMV fused with the routing-weighted combine, the shared-
// expert add and the residual add, BF16 weights.
//
//   out[t] = residual[t] + sum over groups g containing t of
//            w(t, g) * Wd_{expert(g)} h[pair(t, g)]
// where shared-expert groups carry weight 1.  The expert combine sits in the
// same kernel as the down GEMV, as on the pages' low-latency decode path
// ("fuses ... routing, and expert combine into neighboring GEMV kernels":
// vLLM Day-0 Support for Recursive's Flint, "Optimization Strategies").
//
// Row-slice-major: CTA b owns output rows [16b, 16b+16) of every token and
// walks all groups in order, so each weight byte is read by exactly one CTA,
// the combine needs no atomics, and the summation order is fixed (results are
// bitwise reproducible).  The producer streams, per group, the CTA's 16 rows
// of Wd (one contiguous 16 KiB copy) plus the group's h rows (fp32, one
// contiguous copy) through a shared-memory ring with cp.async.bulk; per-token
// accumulators live in shared memory.
//   <= 4 tokens: CUDA cores, warp w owns rows 2w and 2w+1.
//   5..24 tokens: mma.sync m16n8k16 with Wd rows as M and tokens as N; the
//      fp32 h is split into two bf16 parts (hi + lo, two MMAs) so the operand
//      keeps ~16 significant bits; warp w owns a 64-column K-slice.
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

namespace {

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

// 4 bf16 weights (uint2) . 4 fp32 activations.
__device__ __forceinline__ float dot4(const uint2& w, const float4& h, float acc) {
  acc = fmaf(bf_lo(w.x), h.x, acc);
  acc = fmaf(bf_hi(w.x), h.y, acc);
  acc = fmaf(bf_lo(w.y), h.z, acc);
  acc = fmaf(bf_hi(w.y), h.w, acc);
  return acc;
}

template <int NTOK>
__device__ __forceinline__ void group_cc(const DnCtx& c, const uint8_t* st, int pair0) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Lane l covers K elements [4l + 128m, 4l + 128m + 4), m = 0..3.
  const uint8_t* w0 = st + (2 * warp) * dn::WSTRIDE;
  const uint8_t* w1 = w0 + dn::WSTRIDE;
  uint2 a0[4], a1[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    a0[m] = *reinterpret_cast<const uint2*>(w0 + (4 * lane + 128 * m) * 2);
    a1[m] = *reinterpret_cast<const uint2*>(w1 + (4 * lane + 128 * m) * 2);
  }
  const uint8_t* hs = st + dn::WBYTES;
#pragma unroll
  for (int i = 0; i < NTOK; ++i) {
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float4 hv =
          *reinterpret_cast<const float4*>(hs + i * dn::HSTRIDE + (4 * lane + 128 * m) * 4);
      s0 = dot4(a0[m], hv, s0);
      s1 = dot4(a1[m], hv, s1);
    }
    s0 = warp_sum(s0);
    s1 = warp_sum(s1);
    if (lane == 0) {
      const int t = c.pair_tok[pair0 + i];
      const float wt = c.pair_w[pair0 + i];
      c.acc[t * dn::RS + 2 * warp] += wt * s0;
      c.acc[t * dn::RS + 2 * warp + 1] += wt * s1;
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

}  // namespace

__global__ void __launch_bounds__(dn::THREADS, 1) down_bf16_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  const int B = a.B;
  DnCtx c;
  c.nstage = dn::nstages(B);
  c.stage_bytes = dn::stage_bytes(B);
  c.stages = smem;
  c.stages_addr = smem_addr(smem);
  c.red = reinterpret_cast<float*>(smem + c.nstage * c.stage_bytes);
  c.acc = c.red + dn::RED_FLOATS;
  MetaSmem& meta = *reinterpret_cast<MetaSmem*>(c.acc + B * dn::RS);
  float* pair_w_s = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(&meta) + sizeof(MetaSmem));
  uint64_t* bars = reinterpret_cast<uint64_t*>(pair_w_s + MAX_B * SLOTS);
  c.full0 = smem_addr(bars);
  c.empty0 = smem_addr(bars + dn::MAX_STAGES);
  c.hdr = a.ws.hdr;
  c.abort_flag = &s_abort;
  c.pair_tok = meta.pair_tok;
  c.pair_w = pair_w_s;
  if (threadIdx.x == 0) {
    for (int s = 0; s < c.nstage; ++s) {
      mbar_init(full_bar(c, s), 1);
      mbar_init(empty_bar(c, s), dn::CWARPS);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < B * dn::RS; i += blockDim.x) c.acc[i] = 0.f;
  __syncthreads();
  const int r0 = blockIdx.x * dn::RS;
  c.deadline = wait_deadline(a.ws.hdr);
  pdl_wait();     // h, the group table and the pairs come from the preceding kernels
  const int warp = threadIdx.x >> 5;
  if (warp == dn::CWARPS) {
    named_sync(2, ALL_THREADS);  // routing metadata is in shared memory
    if ((threadIdx.x & 31) == 0) produce(c, meta.groups, meta.n_groups, a.w.w2, a.w.ws2, a.ws.h, r0);
    return;
  }
  fill_meta(a, false, meta, pair_w_s, nullptr, nullptr);
  pdl_trigger();
  named_sync(2, ALL_THREADS);
  const int n_groups = meta.n_groups;
  bool ok = true;
  for (int gi = 0; gi < n_groups; ++gi) {
    const int4 grp = meta.groups[gi];
    const int slot = gi % c.nstage;
    if (ok) ok = wait_full(c, slot, (uint32_t)(gi / c.nstage) & 1u);
    const uint8_t* st = c.stages + slot * c.stage_bytes;
    const int n = grp.z;
    if (n <= dn::CC_MAX) {
      if (ok) {
        switch (n) {
          case 1: group_cc<1>(c, st, grp.y); break;
          case 2: group_cc<2>(c, st, grp.y); break;
          case 3: group_cc<3>(c, st, grp.y); break;
          default: group_cc<4>(c, st, grp.y); break;
        }
      }
    } else {
      // Every consumer warp takes this branch for the group (uniform), so the
      // named barriers inside always see all consumer warps.
      switch ((n + 7) >> 3) {
        case 1: group_mma<1>(c, st, grp.y, ok ? n : 0); break;
        case 2: group_mma<2>(c, st, grp.y, ok ? n : 0); break;
        default: group_mma<3>(c, st, grp.y, ok ? n : 0); break;
      }
    }
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar(c, slot));
  }
  named_sync(1, dn::CWARPS * 32);
  if (!ok) return;
  for (int i = threadIdx.x; i < B * dn::RS; i += dn::CWARPS * 32) {
    const int t = i / dn::RS, r = i % dn::RS;
    const size_t o = (size_t)t * H + r0 + r;
    const float res = bf_lo((uint32_t)a.residual[o]);
    a.out[o] = f2bf(res + c.acc[i]);
  }
}

cudaError_t launch_down_bf16(const ExpertArgs& a, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(down_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, dn::SMEM_CAP);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(H / dn::RS, 1, 1);
  cfg.blockDim = dim3(dn::THREADS, 1, 1);
  cfg.dynamicSmemBytes = dn::smem_bytes(a.B);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, down_bf16_kernel, a);
}

}  // namespace flint
