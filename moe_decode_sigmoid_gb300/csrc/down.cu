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
#include "down_impl.cuh"
#include "expert_common.cuh"
#include "kernels.h"

namespace flint {
using namespace dn_impl;

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
