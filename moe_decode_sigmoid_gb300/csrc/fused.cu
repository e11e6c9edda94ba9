// fused.cu — the whole BF16 decode MoE layer in one persistent kernel, for
// batches of at most LOCAL_SELECT_MAX_B (8) tokens: the pages' low-latency
// path for up to 8 requests, which fuses routing and the expert combine into
// the neighbouring GEMVs ("Low-Latency Decode Path": vLLM Day-0 Support for
// Recursive's Flint, "Optimization Strategies").
//
// One CTA per SM (cooperative launch, so all CTAs are co-resident), 8 consumer
// warps + 1 producer warp, the gate/up kernel's shared-memory layout:
//   1. router: each CTA dots its 1-2 router rows with the batch and writes the
//      logits; meanwhile the producer streams the shared expert's gate/up
//      units, which do not depend on routing, and the consumers compute them.
//   2. grid barrier 1 (logits complete); every CTA ranks and buckets the
//      batch itself in shared memory (identical results in every CTA).
//   3. gate/up of the routed units, split evenly over the CTAs; while these
//      stream, the producer also prefetches into L2 the down-projection rows
//      its CTA will need (cp.async.bulk.prefetch.L2).
//   4. grid barrier 2 (all h written).  CTAs 0..127 then run the row-slice-major
//      down projection + combine + shared expert + residual over their 16
//      output rows: the Wd slices are copied into the (now free) ring right
//      after the CTA's last gate/up unit, the h rows only after the barrier.
// The grid barriers are arrive/wait pairs on workspace counters with bounded
// spins; the last CTA to finish resets them.
#include "common.cuh"
#include "down_impl.cuh"
#include "expert_common.cuh"
#include "gateup_impl.cuh"
#include "kernels.h"

namespace flint {
namespace fz {
constexpr int THREADS = gu::THREADS;
constexpr int DN_NSTAGE = 6;
constexpr int DN_STAGE = dn::WBYTES + LOCAL_SELECT_MAX_B * dn::HROW;  // 32 KiB
static_assert(DN_NSTAGE * DN_STAGE <= gu::NSTAGE * gu::STAGE_BYTES, "down stages overlay the ring");
static_assert(dn::RED_FLOATS * 4 <= gu::BUF_BYTES, "down reduction fits in the shared buffer");
constexpr int DOWN_CTAS = H / dn::RS;
constexpr size_t SMEM = gu::SMEM;
constexpr uint64_t DRAIN_NS = 2000000000ull;
}  // namespace fz

namespace {

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier halves; all CTAs are co-resident (cooperative launch).
__device__ __forceinline__ void grid_arrive(uint32_t* ctr) {
  __threadfence();
  atomicAdd(ctr, 1u);
}
__device__ __forceinline__ bool grid_wait(const uint32_t* ctr, uint32_t target, uint64_t deadline) {
  while (ld_acquire(ctr) < target)
    if (globaltimer_ns() > deadline) return false;
  __threadfence();
  return true;
}

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float dot8(const uint4& a, const uint4& b, float acc) {
  acc = fmaf(bf_lo(a.x), bf_lo(b.x), acc);
  acc = fmaf(bf_hi(a.x), bf_hi(b.x), acc);
  acc = fmaf(bf_lo(a.y), bf_lo(b.y), acc);
  acc = fmaf(bf_hi(a.y), bf_hi(b.y), acc);
  acc = fmaf(bf_lo(a.z), bf_lo(b.z), acc);
  acc = fmaf(bf_hi(a.z), bf_hi(b.z), acc);
  acc = fmaf(bf_lo(a.w), bf_lo(b.w), acc);
  acc = fmaf(bf_hi(a.w), bf_hi(b.w), acc);
  return acc;
}

// Logits of experts [e_begin, e_end) for the whole batch (B <= 8), by the 8
// consumer warps: warp w takes expert base + w/4 and the K-quarter w%4.
__device__ __forceinline__ void router_slice(const RouterArgs& r, int e_begin, int e_end,
                                             float (*s_part)[4][8]) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int el = warp >> 2, qk = warp & 3;
  const int B = r.B;
  for (int base = e_begin; base < e_end; base += 2) {
    const int e = base + el;
    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] = 0.f;
    if (e < e_end) {
      const int c0 = qk * 64 + lane, c1 = c0 + 32;
      const uint4* wrow = reinterpret_cast<const uint4*>(r.wr + (size_t)e * H);
      const uint4 w0 = ldg_stream(wrow + c0), w1 = ldg_stream(wrow + c1);
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (t < B) {
          const uint4* xrow = reinterpret_cast<const uint4*>(r.x + (size_t)t * H);
          acc[t] = dot8(w1, __ldg(xrow + c1), dot8(w0, __ldg(xrow + c0), 0.f));
        }
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[t] = warp_sum(acc[t]);
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < 8; ++t) s_part[el][qk][t] = acc[t];
    }
    named_sync(1, CONSUMER_THREADS);
    if (tid < 16) {
      const int le = tid >> 3, t = tid & 7, ee = base + le;
      if (ee < e_end && t < B)
        r.ws.logits[(size_t)t * E + ee] =
            (s_part[le][0][t] + s_part[le][1][t]) + (s_part[le][2][t] + s_part[le][3][t]) +
            (r.bias ? __ldg(r.bias + ee) : 0.0f);
    }
    named_sync(1, CONSUMER_THREADS);
  }
}

}  // namespace

__global__ void __launch_bounds__(fz::THREADS, 1) moe_small_bf16_kernel(ExpertArgs a, RouterArgs r) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  __shared__ LocalSelectSmem s_sel;
  __shared__ float s_part[2][4][8];
  __shared__ float s_pair_w[LOCAL_SELECT_MAX_B * SLOTS];
  __shared__ float s_acc[LOCAL_SELECT_MAX_B * dn::RS];
  __shared__ __align__(8) uint64_t s_dn_bars[2 * fz::DN_NSTAGE];
  WsHeader* hdr = a.ws.hdr;
  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const int B = a.B;

  gu_impl::GuCtx c;
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
  c.hdr = hdr;
  c.abort_flag = &s_abort;

  dn_impl::DnCtx d;
  d.stages = smem;
  d.stages_addr = c.stages_addr;
  d.stage_bytes = fz::DN_STAGE;
  d.nstage = fz::DN_NSTAGE;
  d.red = c.buf;
  d.acc = s_acc;
  d.full0 = smem_addr(s_dn_bars);
  d.empty0 = smem_addr(s_dn_bars + fz::DN_NSTAGE);
  d.hdr = hdr;
  d.abort_flag = &s_abort;
  d.pair_tok = meta.pair_tok;
  d.pair_w = s_pair_w;

  if (tid == 0) {
    for (int s = 0; s < gu::NSTAGE; ++s) {
      mbar_init(gu_impl::full_bar(c, s), 1);
      mbar_init(gu_impl::empty_bar(c, s), gu::CWARPS);
    }
    for (int s = 0; s < fz::DN_NSTAGE; ++s) {
      mbar_init(dn_impl::full_bar(d, s), 1);
      mbar_init(dn_impl::empty_bar(d, s), dn::CWARPS);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < LOCAL_SELECT_MAX_B * dn::RS; i += blockDim.x) s_acc[i] = 0.f;
  __syncthreads();
  c.deadline = wait_deadline(hdr);
  d.deadline = c.deadline;
  gu_impl::Plan pl = gu_impl::plan_pre(B, true);
  const bool down_cta = cta < fz::DOWN_CTAS;
  const int r0 = cta * dn::RS;

  if ((tid >> 5) == gu::CWARPS) {  // ---------------- producer warp (lane 0 issues)
    int it = 0;
    bool ok = true;
    if (lane == 0)
      for (int j = cta; ok && j < pl.nsu; j += G) {
        const gu_impl::SharedUnit su = gu_impl::shared_unit(j, B, pl.nsg);
        ok = gu_impl::issue_unit(c, a.w.ws13 + (size_t)su.s * (2 * I) * H, su.blk, it);
      }
    __syncwarp();
    named_sync(2, ALL_THREADS);  // routing metadata is in shared memory
    if (lane != 0) return;
    gu_impl::plan_post(pl, meta.n_groups, true);
    const int ng = meta.n_groups;
    const int nu = pl.r_end - pl.r_begin;
    int pf = 0;  // down-row prefetches issued (one per group)
    int gi_cached = -1;
    const uint16_t* base = nullptr;
    for (int u = pl.r_begin; ok && u < pl.r_end; ++u) {
      const int gi = u / gu::UNITS;
      if (gi != gi_cached) {
        const int4 grp = meta.groups[gi];
        base = grp.x < E ? a.w.w13 + (size_t)grp.x * (2 * I) * H
                         : a.w.ws13 + (size_t)(grp.x - E) * (2 * I) * H;
        gi_cached = gi;
      }
      ok = gu_impl::issue_unit(c, base, u & (gu::UNITS - 1), it);
      // Interleave the L2 prefetches of this CTA's down rows with the units.
      const int upto = down_cta ? (nu > 0 ? (int)(((long long)(u - pl.r_begin + 1) * ng + nu - 1) / nu) : ng) : 0;
      for (; pf < upto && pf < ng; ++pf) {
        const int4 g2 = meta.groups[pf];
        const uint16_t* wb = (g2.x < E ? a.w.w2 + (size_t)g2.x * H * I
                                       : a.w.ws2 + (size_t)(g2.x - E) * H * I) + (size_t)r0 * I;
        prefetch_l2_bulk(wb, dn::WBYTES);
      }
    }
    if (down_cta)
      for (; pf < ng; ++pf) {
        const int4 g2 = meta.groups[pf];
        const uint16_t* wb = (g2.x < E ? a.w.w2 + (size_t)g2.x * H * I
                                       : a.w.ws2 + (size_t)(g2.x - E) * H * I) + (size_t)r0 * I;
        prefetch_l2_bulk(wb, dn::WBYTES);
      }
    // The ring is free once the consumers have released every gate/up stage.
    const uint64_t drain = globaltimer_ns() + fz::DRAIN_NS;
    for (int j = it - gu::NSTAGE < 0 ? 0 : it - gu::NSTAGE; j < it; ++j)
      if (!mbar_wait(gu_impl::empty_bar(c, j % gu::NSTAGE), (uint32_t)(j / gu::NSTAGE) & 1u, drain))
        ok = false;
    if (!ok || !down_cta) {
      if (!ok) {
        *c.abort_flag = 1;
        set_error(hdr, DEV_TIMEOUT);
      }
      return;
    }
    // Down: Wd slices first (from L2), h rows once every CTA has written h.
    int k = 0;
    bool h_ready = false;
    const int early = ng < fz::DN_NSTAGE ? ng : fz::DN_NSTAGE;
    for (int gi = 0; gi < ng; ++gi) {
      const int4 grp = meta.groups[gi];
      const int slot = gi % fz::DN_NSTAGE;
      if (gi >= fz::DN_NSTAGE) {
        if (!mbar_wait(dn_impl::empty_bar(d, slot), (uint32_t)((gi / fz::DN_NSTAGE) - 1) & 1u,
                       d.deadline) ||
            *d.abort_flag) {
          *d.abort_flag = 1;
          set_error(hdr, DEV_TIMEOUT);
          break;
        }
      }
      mbar_expect_tx(dn_impl::full_bar(d, slot), dn::WBYTES + grp.z * dn::HROW);
      const uint16_t* wb = (grp.x < E ? a.w.w2 + (size_t)grp.x * H * I
                                      : a.w.ws2 + (size_t)(grp.x - E) * H * I) + (size_t)r0 * I;
      bulk_g2s(d.stages_addr + slot * fz::DN_STAGE, wb, dn::WBYTES, dn_impl::full_bar(d, slot));
      if (!h_ready && gi + 1 < early) continue;
      if (!h_ready) {  // all early Wd copies are out; now wait for h
        if (!grid_wait(&hdr->grid_bar[1], (uint32_t)G, d.deadline)) {
          *d.abort_flag = 1;
          set_error(hdr, DEV_TIMEOUT);
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
        h_ready = true;
      }
      for (; k <= gi; ++k) {
        const int4 gk = meta.groups[k];
        bulk_g2s(d.stages_addr + (k % fz::DN_NSTAGE) * fz::DN_STAGE + dn::WBYTES,
                 a.ws.h + (size_t)gk.y * I, gk.z * dn::HROW, dn_impl::full_bar(d, k % fz::DN_NSTAGE));
      }
    }
    const uint64_t dr = globaltimer_ns() + fz::DRAIN_NS;
    for (int j = k - fz::DN_NSTAGE < 0 ? 0 : k - fz::DN_NSTAGE; j < k; ++j)
      mbar_wait(dn_impl::full_bar(d, j % fz::DN_NSTAGE), (uint32_t)(j / fz::DN_NSTAGE) & 1u, dr);
    return;
  }

  // ---------------- consumer warps
  if (r.stall_check && cta == 0 && tid == 0 &&
      *reinterpret_cast<volatile uint32_t*>(&hdr->stall_armed)) {
    // Test hook: wait for a flag that nothing sets; the bounded wait runs out
    // and records the timeout, exactly like a stuck pipeline wait would.
    const uint64_t deadline = wait_deadline(hdr);
    while (!*reinterpret_cast<volatile uint32_t*>(&hdr->stall_release)) {
      if (globaltimer_ns() > deadline) {
        set_error(hdr, DEV_TIMEOUT);
        break;
      }
    }
    hdr->stall_armed = 0;
  }
  // 1. router logits for this CTA's experts
  router_slice(r, (int)((long long)cta * E / G), (int)((long long)(cta + 1) * E / G), s_part);
  if (tid == 0) grid_arrive(&hdr->grid_bar[0]);
  int it = 0;
  bool ok = true;
  for (int j = cta; j < pl.nsu; j += G) {
    const gu_impl::SharedUnit su = gu_impl::shared_unit(j, B, pl.nsg);
    gu_impl::segment(c, su.blk, su.blk + 1, su.pair0, su.n, su.tok0, it, ok);
  }
  // 2. every CTA ranks and buckets the batch once all logits are in
  if (tid == 0 && !grid_wait(&hdr->grid_bar[0], (uint32_t)G, c.deadline)) {
    *c.abort_flag = 1;
    set_error(hdr, DEV_TIMEOUT);
  }
  named_sync(1, CONSUMER_THREADS);
  fill_meta(a, true, meta, s_pair_w, c.buf, &s_sel);
  named_sync(2, ALL_THREADS);
  // 3. routed gate/up units
  gu_impl::plan_post(pl, meta.n_groups, true);
  int u = pl.r_begin;
  while (u < pl.r_end) {
    const int gi = u / gu::UNITS;
    const int4 grp = meta.groups[gi];
    const int u1 = min(pl.r_end, (gi + 1) * gu::UNITS);
    gu_impl::segment(c, u, u1, grp.y, grp.z, -1, it, ok);
    u = u1;
  }
  named_sync(1, CONSUMER_THREADS);  // every h store of this CTA is issued
  if (tid == 0) grid_arrive(&hdr->grid_bar[1]);
  // 4. down + combine + shared expert + residual over this CTA's 16 rows
  if (down_cta) {
    const int ng = meta.n_groups;
    bool dok = ok;
    for (int gi = 0; gi < ng; ++gi) {
      const int4 grp = meta.groups[gi];
      const int slot = gi % fz::DN_NSTAGE;
      if (dok) dok = dn_impl::wait_full(d, slot, (uint32_t)(gi / fz::DN_NSTAGE) & 1u);
      const uint8_t* st = d.stages + slot * fz::DN_STAGE;
      const int n = grp.z;
      if (n <= dn::CC_MAX) {
        if (dok) {
          switch (n) {
            case 1: dn_impl::group_cc<1>(d, st, grp.y); break;
            case 2: dn_impl::group_cc<2>(d, st, grp.y); break;
            case 3: dn_impl::group_cc<3>(d, st, grp.y); break;
            default: dn_impl::group_cc<4>(d, st, grp.y); break;
          }
        }
      } else {
        dn_impl::group_mma<1>(d, st, grp.y, dok ? n : 0);  // n <= 8 here
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(dn_impl::empty_bar(d, slot));
    }
    named_sync(1, CONSUMER_THREADS);
    if (dok) {
      for (int i = tid; i < B * dn::RS; i += CONSUMER_THREADS) {
        const int t = i / dn::RS, rr = i % dn::RS;
        const size_t o = (size_t)t * H + r0 + rr;
        a.out[o] = f2bf(bf_lo((uint32_t)a.residual[o]) + s_acc[i]);
      }
    }
  }
  // The last CTA out resets the barrier counters for the next call (every
  // CTA has passed both barriers by the time it counts itself out).
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&hdr->grid_bar[2], 1u) == (uint32_t)G - 1) {
      hdr->grid_bar[0] = 0u;
      hdr->grid_bar[1] = 0u;
      hdr->grid_bar[2] = 0u;
      __threadfence();
    }
  }
}

cudaError_t launch_small_bf16(const ExpertArgs& a, const RouterArgs& r, cudaStream_t stream,
                              int num_sms) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(moe_small_bf16_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fz::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms, 1, 1);
  cfg.blockDim = dim3(fz::THREADS, 1, 1);
  cfg.dynamicSmemBytes = fz::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_small_bf16_kernel, a, r);
}

}  // namespace flint
