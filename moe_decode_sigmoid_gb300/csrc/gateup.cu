// gateup.cu — gathered gate/up GEMV with fused SiLU-and-mul, BF16 weights.
//
// For every (expert, token-range) group of the routing and every token t in
// it:  h[pair(t), i] = silu(Wg[i] . x_t) * (Wu[i] . x_t),  i < 512, with
// silu(g) = g / (1 + exp(-g)) ("SiLU-and-mul": Flint on Intel Arc Pro B70,
// "norm.py: Triton kernels that assumed CUDA").  Only the selected experts'
// rows are read ("read only the selected experts' weights": vLLM Day-0 Support
// for Recursive's Flint, "Optimization Strategies").
//
// Work unit: one group x one block of 8 intermediate rows = the 8 gate rows
// plus the 8 matching up rows: two contiguous 32 KiB runs of w13.  The units
// that need the routing are claimed from a workspace counter by the CTAs (one
// per SM) as they go -- guided self-scheduling: chunks of about remaining /
// (2 x #SMs) units, at most 8, down to single units at the end -- because SMs
// stream at different rates: with an equal static share the last CTA ended
// ~10 us after the median one at batch 128 (skewed routing), 5.5 us at 32.
//
// Per CTA: 8 consumer warps + 1 producer warp.  The producer's elected lane
// streams each unit as one 64 KiB stage -- two cp.async.bulk copies -- through
// a 3-stage shared-memory ring with full/empty mbarriers, so 192 KiB per SM is
// in flight.  The shared expert's units, which do not depend on routing, start
// before the router has finished (programmatic dependent launch).  Consumers,
// per group:
//   <= 2 tokens (most groups at batch 1/8): CUDA cores.  Warp w owns gate row w and
//      up row w; the group's bf16 activations are staged once in shared
//      memory; products are formed by fma.rn.f32.bf16 (bf16 x bf16 is exact in
//      fp32, accumulation in fp32), one independent partial sum per 16-byte
//      chunk so the FMA chains overlap.
//   3..24 tokens: mma.sync m16n8k16 (bf16 in, fp32 acc) with the 16 weight
//      rows as M (8 gate + 8 up: the same thread then holds g and u) and the
//      tokens as N; warp w owns a 256-column K-slice; the 8 partial tiles are
//      summed through shared memory.  Because each fragment's K order is the
//      same permutation for weights and activations, both are loaded as plain
//      16-byte row chunks.
// Every wait is bounded by the workspace's limit.
#include "common.cuh"
#include "expert_common.cuh"
#include "gateup_impl.cuh"
#include "kernels.h"

namespace flint {
using namespace gu_impl;

namespace {
constexpr int CLAIM_MAX = 8;  // units per claim at most

// Waits (bounded) until ring stage `it` is free again; false on a failed wait
// or an abort.
__device__ __forceinline__ bool stage_free(const GuCtx& c, int it) {
  bool got = true;
  if (it >= gu::NSTAGE)
    got = mbar_wait(empty_bar(c, it % gu::NSTAGE), (uint32_t)((it / gu::NSTAGE) - 1) & 1u,
                    c.deadline);
  if (!got || *c.abort_flag) {
    *c.abort_flag = 1;
    if (!got) set_error(c.hdr, DEV_TIMEOUT);
    return false;
  }
  return true;
}

__device__ __forceinline__ int claim_size(int remaining) {
  const int s = remaining / (2 * (int)gridDim.x);
  return s < 1 ? 1 : (s > CLAIM_MAX ? CLAIM_MAX : s);
}
}  // namespace

__global__ void __launch_bounds__(gu::THREADS, 1) gateup_bf16_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  __shared__ LocalSelectSmem s_sel;
  // the claimed chunk {first unit, units} that starts at ring stage s (or
  // {-1, 0}: no more), written before the stage's copies are issued
  __shared__ int2 s_chunk[gu::NSTAGE];
  GuCtx c;
  c.stages = smem;
  c.buf = reinterpret_cast<float*>(smem + gu::NSTAGE * gu::STAGE_BYTES);
  MetaSmem& meta = *reinterpret_cast<MetaSmem*>(smem + gu::NSTAGE * gu::STAGE_BYTES + gu::BUF_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(&meta) + sizeof(MetaSmem));
  c.stages_addr = smem_addr(smem);
  c.full0 = smem_addr(bars);
  c.empty0 = smem_addr(bars + gu::NSTAGE);
  c.x = a.x;
  c.pair_tok = meta.pair_tok;
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
  const int lane = threadIdx.x & 31;
  if ((threadIdx.x >> 5) == gu::CWARPS) {  // producer warp (lane 0 issues)
    int it = 0;
    bool ok = true;
    if (lane == 0)
      for (int j = blockIdx.x; ok && j < pl.nsu; j += gridDim.x) {
        const SharedUnit su = shared_unit(j, a.B, pl.nsg);
        ok = issue_unit(c, a.w.ws13 + (size_t)su.s * (2 * I) * H, su.blk, it);
      }
    __syncwarp();
    named_sync(2, ALL_THREADS);  // routing metadata is in shared memory
    if (lane == 0) {
      // Units [0, n) of the groups after the shared ones handled above (all
      // groups when none were); one claim is kept in flight ahead.
      const int n = (meta.n_groups - (early ? S * pl.nsg : 0)) * gu::UNITS;
      uint32_t* const claim = &a.ws.hdr->gu_claim;
      int sz = claim_size(n);
      int c0 = (int)atomicAdd(claim, (uint32_t)sz);
      int sz_next = claim_size(n - c0 - sz);
      int c_next = (int)atomicAdd(claim, (uint32_t)sz_next);
      int gi_cached = -1;
      const uint16_t* base = nullptr;
      while (ok && c0 < n) {
        const int e = min(n, c0 + sz);
        ok = stage_free(c, it);
        if (!ok) break;
        s_chunk[it % gu::NSTAGE] = make_int2(c0, e - c0);
        for (int u = c0; ok && u < e; ++u) {
          const int gi = u / gu::UNITS;
          if (gi != gi_cached) {
            const int4 grp = meta.groups[gi];
            base = grp.x < E ? a.w.w13 + (size_t)grp.x * (2 * I) * H
                             : a.w.ws13 + (size_t)(grp.x - E) * (2 * I) * H;
            gi_cached = gi;
          }
          ok = issue_unit(c, base, u & (gu::UNITS - 1), it);
        }
        c0 = c_next;
        sz = sz_next;
        if (c0 < n) {
          sz_next = claim_size(n - c0 - sz);
          c_next = (int)atomicAdd(claim, (uint32_t)sz_next);
        }
      }
      if (ok && stage_free(c, it)) {  // no more: the consumers stop at this stage
        s_chunk[it % gu::NSTAGE] = make_int2(-1, 0);
        mbar_arrive(full_bar(c, it % gu::NSTAGE));
        ++it;
      }
      // The last CTA done claiming resets the counter for the next call.
      __threadfence();
      if (atomicAdd(&a.ws.hdr->gu_done, 1u) == gridDim.x - 1) {
        atomicExch(claim, 0u);
        atomicExch(&a.ws.hdr->gu_done, 0u);
      }
      drain(c, it);
    }
    return;
  }
  int it = 0;
  bool ok = true;
  for (int j = blockIdx.x; j < pl.nsu; j += gridDim.x) {
    const SharedUnit su = shared_unit(j, a.B, pl.nsg);
    // unit numbers inside a segment only serve as block indices (u & 63)
    segment(c, su.blk, su.blk + 1, su.pair0, su.n, su.tok0, it, ok);
  }
  pdl_wait();     // the router's logits / routing
  named_sync(1, gu::CWARPS * 32);  // the last segment is done with buf
  fill_meta(a, a.local_select != 0, meta, nullptr, c.buf, &s_sel);
  pdl_trigger();  // the down kernel may start its prologue
  named_sync(2, ALL_THREADS);
  // the producer's chunks, in its order
  while (ok) {
    const int slot = it % gu::NSTAGE;
    if (!wait_full(c, slot, (uint32_t)(it / gu::NSTAGE) & 1u)) break;
    const int2 ch = s_chunk[slot];
    if (ch.x < 0) break;
    int u = ch.x;
    const int u1 = ch.x + ch.y;
    while (ok && u < u1) {
      const int gi = u / gu::UNITS;
      const int4 grp = meta.groups[gi];
      const int ue = min(u1, (gi + 1) * gu::UNITS);
      segment(c, u, ue, grp.y, grp.z, -1, it, ok);
      u = ue;
    }
  }
}

cudaError_t launch_gateup_bf16(const ExpertArgs& a, cudaStream_t stream, int num_sms) {
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t es = set_smem_limit_once(gateup_bf16_kernel, (int)gu::SMEM, smem_set);
  if (es != cudaSuccess) return es;
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
