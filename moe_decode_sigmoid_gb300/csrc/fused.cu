// fused.cu — the whole BF16 decode MoE layer in one persistent kernel, for
// batches of at most LOCAL_SELECT_MAX_B (8) tokens: the pages' low-latency
// path for up to 8 requests, which fuses routing and the expert combine into
// the neighbouring GEMVs ("Low-Latency Decode Path": vLLM Day-0 Support for
// Recursive's Flint, "Optimization Strategies").
//
// One CTA per SM (its shared memory admits no second CTA, so the #SMs CTAs are
// all resident), 8 consumer warps + 1 producer warp.  The producer's lane 0
// feeds a ring of 32 KiB shared-memory slots with cp.async.bulk copies and
// tags each slot with what it holds; the consumers take the slots in order.
//
//   1. Router: the consumers dot the CTA's 1-2 router rows with the batch and
//      write the logits; one grid-wide arrive.  Meanwhile the producer streams
//      shared-expert gate/up units, which do not depend on routing.
//   2. Work queue: gate/up units (8 gate + 8 up rows of one group, two slots)
//      are claimed one at a time from a workspace counter -- the shared
//      expert's 64 units first, then the routed groups' in group order -- so
//      CTAs that stream faster take more units and groups finish roughly in
//      order.  The first claim past the shared units makes the producer post a
//      SELECT slot: the consumers wait for every CTA's logits, rank and bucket
//      the batch in shared memory (identical in every CTA) and hand the group
//      table to the producer.
//   3. Completion counters: after storing its h values of a unit, each
//      consumer warp adds 1 to its group's counter (release); the add is
//      deferred until the warp's next unit is computed or the warp runs idle,
//      so the fence finds the stores already done.  64 units x 8 warps = 512
//      marks a group's h complete.
//   4. Down: CTA b < 128 owns output rows [16b, 16b+16) of every token.  As
//      soon as a group is complete (acquire), its producer posts a DOWN slot:
//      the 16 rows of the expert's Wd (16 KiB) and the group's h rows, and the
//      consumers accumulate w(t, g) * (Wd h) per token: groups of <= 4 tokens
//      on CUDA cores into per-lane running sums (reduced once, at the end),
//      larger ones on tensor cores.
//      Down slots take priority over gate/up units, so the down projection
//      streams while gate/up is still running instead of after a grid
//      barrier.  Items run in a fixed order (the shared expert, then the
//      routed groups by expert), so results are reproducible bit for bit.
// Every wait is bounded by the workspace's limit; the last CTA out resets the
// workspace counters for the next call.
#include "common.cuh"
#include "down_impl.cuh"
#include "expert_common.cuh"
#include "gateup_impl.cuh"
#include "kernels.h"

namespace flint {
namespace fz {
constexpr int CW = 8;                          // consumer warps
constexpr int THREADS = (CW + 3) * 32;         // + producer, signalling and poll warps
constexpr int CT = CW * 32;                    // consumer threads
constexpr int SLOT = 32 * 1024;                // ring slot bytes
constexpr int NS = 5;                          // ring slots
constexpr int ROWB = H * 2;                    // one gate/up row (bf16), 4 KiB
constexpr int UNITS = I / 8;                   // gate/up units per group
constexpr int MAXB = LOCAL_SELECT_MAX_B;
constexpr int MAXG = MAXB * TOPK + S;          // groups at these batches (one shared group)
constexpr int NPAIR = MAXB * SLOTS;
constexpr int DONE_SHARED = 63;                // counter slot of the shared group
constexpr uint32_t DONE_TARGET = UNITS;        // finished units per group
constexpr int SIGQ = 8;                        // finished units in flight to the signalling warp
constexpr int DOWN_CTAS = H / dn::RS;          // 128 row-slice owners
constexpr int XS_BYTES = MAXB * H * 2;         // bf16 activations of the batch, 32 KiB
constexpr int RED_BYTES = CW * 16 * GROUP_MAX * 4;
constexpr int LOGIT_BYTES = MAXB * E * 4;
constexpr int BUF_BYTES = RED_BYTES > LOGIT_BYTES ? RED_BYTES : LOGIT_BYTES;
// Per-lane running sums of the CUDA-core down items: [token * 2 + row][thread],
// rows padded to 257 floats so that both the updates (one row, consecutive
// lanes) and the final per-row sums (16 lanes each) are free of bank conflicts.
constexpr int LACC_STRIDE = CW * 32 + 1;
constexpr int LACC_BYTES = MAXB * 2 * LACC_STRIDE * 4;
constexpr size_t SMEM = (size_t)NS * SLOT + XS_BYTES + BUF_BYTES + LACC_BYTES;
constexpr uint64_t DRAIN_NS = 2000000000ull;
enum : int { IT_GATE = 0, IT_UP = 1, IT_DOWN = 2, IT_SELECT = 3, IT_END = 4 };
static_assert(S == 1 && MAXB <= GROUP_MAX, "one shared group at these batches");
static_assert(MAXG <= DONE_SHARED, "routed groups and the shared group have distinct counters");
static_assert(dn::WBYTES + MAXB * dn::HROW <= SLOT, "a down item fits one slot");
static_assert(8 * ROWB == SLOT, "8 gate (or up) rows fill one slot");
static_assert(dn::RED_FLOATS * 4 <= BUF_BYTES, "down partial tiles fit the buffer");
}  // namespace fz

namespace {

// What a ring slot holds (written by the producer before it arms the slot).
struct Item {
  int kind;
  int blk;       // gate/up: block of 8 intermediate rows
  int pair0;     // first h row (pair) of the group
  int n;         // tokens in the group
  int tok0;      // gate/up of the shared group: first token (tokens are consecutive), else -1
  int done_idx;  // completion counter of the group
  int pad[2];
};

__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
__device__ __forceinline__ int ld_acquire_cta_shared(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta_shared(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// Non-blocking probe of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ bool grid_wait(const uint32_t* ctr, uint32_t target, uint64_t deadline) {
  while (ld_acquire(ctr) < target)
    if (globaltimer_ns() > deadline) return false;
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
      uint4 xv[8][2];  // every load of the tile in flight before any FMA
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const uint4* xrow = reinterpret_cast<const uint4*>(r.x + (size_t)t * H);
        xv[t][0] = t < B ? __ldg(xrow + c0) : make_uint4(0u, 0u, 0u, 0u);
        xv[t][1] = t < B ? __ldg(xrow + c1) : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[t] = dot8(w1, xv[t][1], dot8(w0, xv[t][0], 0.f));
#pragma unroll
      for (int t = 0; t < 8; ++t) acc[t] = warp_sum(acc[t]);
    }
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < 8; ++t) s_part[el][qk][t] = acc[t];
    }
    named_sync(1, fz::CT);
    if (tid < 16) {
      const int le = tid >> 3, t = tid & 7, ee = base + le;
      if (ee < e_end && t < B)
        r.ws.logits[(size_t)t * E + ee] =
            (s_part[le][0][t] + s_part[le][1][t]) + (s_part[le][2][t] + s_part[le][3][t]) +
            (r.bias ? __ldg(r.bias + ee) : 0.0f);
    }
    named_sync(1, fz::CT);
  }
}

// ---- consumer side -----------------------------------------------------------

__device__ __forceinline__ void release_slot(uint32_t empty_bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar);
}

// Finished gate/up units go to the signalling warp through a small ring of
// mbarriers (8 consumer-warp arrivals each, after the warps' h stores); it
// publishes them to the group counters, so no consumer warp waits on a
// GPU-scope fence.
struct Sig {
  uint32_t full0, free0;
  int* grp;
  uint64_t limit;
};
// gidx: the unit's group counter, -2 for a unit skipped after an abort, -1 at the end.
__device__ __forceinline__ void signal_unit(const Sig& s, int seq, int gidx) {
  const int j = seq & (fz::SIGQ - 1);
  if (seq >= fz::SIGQ && (threadIdx.x & 31) == 0)
    mbar_wait(s.free0 + 8u * j, (uint32_t)((seq / fz::SIGQ) - 1) & 1u, s.limit);
  __syncwarp();
  if ((threadIdx.x & 31) == 0) {
    if (threadIdx.x == 0) s.grp[j] = gidx;
    mbar_arrive(s.full0 + 8u * j);
  }
}

// Gate/up unit on CUDA cores (<= 2 tokens): warp w owns gate row w and up row
// w; the same arithmetic, in the same order, as the standalone gate/up kernel
// (gate and up chains interleaved: eight independent FMA chains per lane).
template <int NTOK>
__device__ __forceinline__ void unit_cc(const uint8_t* gs, const uint8_t* us, const uint4* xs,
                                        const int (&tok)[2], float* h, const Item& d, bool ok,
                                        uint32_t emA, uint32_t emB) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float g[NTOK], v[NTOK];
#pragma unroll
  for (int i = 0; i < NTOK; ++i) g[i] = v[i] = 0.f;
  if (ok) {
    const uint4* gr = reinterpret_cast<const uint4*>(gs + warp * fz::ROWB);
    const uint4* ur = reinterpret_cast<const uint4*>(us + warp * fz::ROWB);
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
          const uint4 xv = xs[tok[i] * (H / 8) + lane + 32 * (4 * half + j)];
          pg[j] = gu_impl::dot8_bf16(wg[j], xv);
          pu[j] = gu_impl::dot8_bf16(wu[j], xv);
        }
        g[i] += (pg[0] + pg[1]) + (pg[2] + pg[3]);
        v[i] += (pu[0] + pu[1]) + (pu[2] + pu[3]);
      }
    }
  }
  release_slot(emA);
  release_slot(emB);
  if (!ok) return;
#pragma unroll
  for (int i = 0; i < NTOK; ++i) {
    const float gsum = warp_sum(g[i]);
    const float vsum = warp_sum(v[i]);
    if (lane == 0) h[(size_t)(d.pair0 + i) * I + d.blk * 8 + warp] = silu_mul(gsum, vsum);
  }
}

// Down item on CUDA cores (<= 4 tokens): warp w owns Wd rows 2w and 2w+1 of
// the slice.  The lane's 32 weights are unpacked once and reused by every
// token; each lane adds w(t, g) times its partial dot product (16 columns) to
// its own running sum in shared memory -- the sums across lanes are taken
// once, when the output is written.
__device__ __forceinline__ void down_cc(const uint8_t* st, int pair0, int n, const int* pair_tok,
                                        const float* pair_w, float* lacc, bool ok, uint32_t em) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float s0[dn::CC_MAX], s1[dn::CC_MAX];
#pragma unroll
  for (int i = 0; i < dn::CC_MAX; ++i) s0[i] = s1[i] = 0.f;
  if (ok) {
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
#pragma unroll
    for (int i = 0; i < dn::CC_MAX; ++i) {
      if (i < n) {
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 hv = *reinterpret_cast<const float4*>(st + dn::WBYTES + i * dn::HSTRIDE +
                                                             (4 * lane + 128 * m) * 4);
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
    }
  }
  release_slot(em);
  if (!ok) return;
#pragma unroll
  for (int i = 0; i < dn::CC_MAX; ++i) {
    if (i < n) {
      const int t = pair_tok[pair0 + i];
      const float wt = pair_w[pair0 + i];
      float* acc = lacc + (2 * t) * fz::LACC_STRIDE + threadIdx.x;
      acc[0] = fmaf(wt, s0[i], acc[0]);
      acc[fz::LACC_STRIDE] = fmaf(wt, s1[i], acc[fz::LACC_STRIDE]);
    }
  }
}

// Gate/up unit on tensor cores (3..8 tokens): m16n8k16 with the 8 gate + 8 up
// rows as M and the tokens as N, warp w owns a 256-column K-slice; the same
// arithmetic as the standalone gate/up kernel.
__device__ __forceinline__ void unit_mma(const uint8_t* gs, const uint8_t* us, const uint16_t* xs,
                                         const int* pair_tok, float* buf, float* h, const Item& d,
                                         bool ok, uint32_t emA, uint32_t emB) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int n = d.n;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (ok) {
    uint4 bfr[8];
    if (g < n) {
      const int tok = d.tok0 >= 0 ? d.tok0 + g : pair_tok[d.pair0 + g];
      const uint16_t* row = xs + (size_t)tok * H + warp * 256 + q * 8;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) bfr[kb] = *reinterpret_cast<const uint4*>(row + kb * 32);
    } else {
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) bfr[kb] = make_uint4(0u, 0u, 0u, 0u);
    }
    const uint8_t* rlo = gs + g * fz::ROWB + (warp * 256 + q * 8) * 2;
    const uint8_t* rhi = us + g * fz::ROWB + (warp * 256 + q * 8) * 2;
#pragma unroll
    for (int kb = 0; kb < 8; ++kb) {
      const uint4 alo = *reinterpret_cast<const uint4*>(rlo + kb * 64);
      const uint4 ahi = *reinterpret_cast<const uint4*>(rhi + kb * 64);
      mma_bf16(acc, alo.x, ahi.x, alo.y, ahi.y, bfr[kb].x, bfr[kb].y);
      mma_bf16(acc, alo.z, ahi.z, alo.w, ahi.w, bfr[kb].z, bfr[kb].w);
    }
  }
  release_slot(emA);
  release_slot(emB);
  float* red = buf + warp * gu::ROWS * GROUP_MAX;
  const int col = 2 * q;
  red[g * GROUP_MAX + col] = acc[0];
  red[g * GROUP_MAX + col + 1] = acc[1];
  red[(g + 8) * GROUP_MAX + col] = acc[2];
  red[(g + 8) * GROUP_MAX + col + 1] = acc[3];
  named_sync(1, fz::CT);
  {
    const int r = warp, j = lane;  // row r of the block, token slot j
    if (j < n && ok) {
      float gsum = 0.f, usum = 0.f;
#pragma unroll
      for (int w = 0; w < fz::CW; ++w) {
        gsum += buf[(w * gu::ROWS + r) * GROUP_MAX + j];
        usum += buf[(w * gu::ROWS + r + 8) * GROUP_MAX + j];
      }
      h[(size_t)(d.pair0 + j) * I + d.blk * 8 + r] = silu_mul(gsum, usum);
    }
  }
  named_sync(1, fz::CT);  // buf is free again
}

// ---- producer side (lane 0 of the producer warp) -----------------------------

struct Prod {
  uint32_t full0, empty0, stages_addr;
  Item* desc;
  int it;
  uint64_t deadline;
  WsHeader* hdr;
  volatile int* abort_flag;
};

__device__ __forceinline__ bool take_slot(Prod& p, int& slot) {
  slot = p.it % fz::NS;
  if (p.it >= fz::NS &&
      !mbar_wait(p.empty0 + 8u * slot, (uint32_t)((p.it / fz::NS) - 1) & 1u, p.deadline)) {
    *p.abort_flag = 1;
    set_error(p.hdr, DEV_TIMEOUT);
    return false;
  }
  if (*p.abort_flag) return false;
  ++p.it;
  return true;
}

// A slot with no payload (SELECT / END): armed by a plain arrive.
__device__ __forceinline__ void post_marker(Prod& p, int kind) {
  const int slot = p.it % fz::NS;
  if (p.it >= fz::NS)  // END is posted even after an abort; wait out the drain bound
    mbar_wait(p.empty0 + 8u * slot, (uint32_t)((p.it / fz::NS) - 1) & 1u,
              p.deadline + fz::DRAIN_NS);
  ++p.it;
  Item d = {};
  d.kind = kind;
  p.desc[slot] = d;
  mbar_arrive(p.full0 + 8u * slot);
}

__device__ __forceinline__ bool post_gateup(Prod& p, const uint16_t* base, const Item& d) {
  int sa, sb;
  if (!take_slot(p, sa)) return false;
  p.desc[sa] = d;
  mbar_expect_tx(p.full0 + 8u * sa, fz::SLOT);
  bulk_g2s_stream(p.stages_addr + sa * fz::SLOT, base + (size_t)(d.blk * 8) * H, fz::SLOT,
                  p.full0 + 8u * sa);
  if (!take_slot(p, sb)) return false;  // the END posted next takes the up half's place
  Item du = d;
  du.kind = fz::IT_UP;
  p.desc[sb] = du;
  mbar_expect_tx(p.full0 + 8u * sb, fz::SLOT);
  bulk_g2s_stream(p.stages_addr + sb * fz::SLOT, base + (size_t)(I + d.blk * 8) * H, fz::SLOT,
           p.full0 + 8u * sb);
  return true;
}


}  // namespace

__global__ void __launch_bounds__(fz::THREADS, 1) moe_small_bf16_kernel(ExpertArgs a, RouterArgs r) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  __shared__ int s_ngroups;
  __shared__ int s_ready;  // down items whose groups are complete (poll warp -> producer)
  __shared__ Item s_desc[fz::NS];
  __shared__ int4 s_groups[fz::MAXG];
  __shared__ int s_pair_tok[fz::NPAIR];
  __shared__ float s_pair_w[fz::NPAIR];
  __shared__ float s_acc[fz::MAXB * dn::RS];  // this CTA's 16 output rows per token
  __shared__ LocalSelectSmem s_sel;
  __shared__ float s_part[2][4][8];
  __shared__ int s_hgrp[fz::SIGQ];
  // ring full / empty, SELECT done, finished-unit full / free, signalling done
  __shared__ __align__(8) uint64_t s_bars[2 * fz::NS + 1 + 2 * fz::SIGQ + 1];
  WsHeader* hdr = a.ws.hdr;
  uint32_t* done = hdr->group_done;
  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const int B = a.B;
  uint8_t* ring = smem;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + fz::NS * fz::SLOT);
  float* buf = reinterpret_cast<float*>(smem + fz::NS * fz::SLOT + fz::XS_BYTES);
  float* lacc = reinterpret_cast<float*>(smem + fz::NS * fz::SLOT + fz::XS_BYTES + fz::BUF_BYTES);
  const uint32_t full0 = smem_addr(s_bars), empty0 = smem_addr(s_bars + fz::NS);
  const uint32_t sel_bar = smem_addr(s_bars + 2 * fz::NS);
  const uint32_t hfull0 = smem_addr(s_bars + 2 * fz::NS + 1);
  const uint32_t hfree0 = hfull0 + 8u * fz::SIGQ;
  const uint32_t sig_done = hfree0 + 8u * fz::SIGQ;

  if (tid == 0) {
    for (int s = 0; s < fz::NS; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, fz::CW);
    }
    mbar_init(sel_bar, 1);
    for (int j = 0; j < fz::SIGQ; ++j) {
      mbar_init(hfull0 + 8u * j, fz::CW);
      mbar_init(hfree0 + 8u * j, 1);
    }
    mbar_init(sig_done, 1);
    s_abort = 0;
    s_ngroups = 0;
    s_ready = 0;
    fence_mbar_init();
  }
  for (int i = tid; i < fz::MAXB * dn::RS; i += blockDim.x) s_acc[i] = 0.f;
  for (int i = tid; i < fz::LACC_BYTES / 4; i += blockDim.x) lacc[i] = 0.f;
  __syncthreads();
  // Launched with programmatic serialization: the set-up above overlaps the
  // preceding kernel; x, the weights and the workspace are read only after it.
  pdl_wait();
  const uint64_t deadline = wait_deadline(hdr);
  const bool owner = cta < fz::DOWN_CTAS;
  const int r0 = cta * dn::RS;
  const int npairs = B * TOPK;

  if ((tid >> 5) == fz::CW) {  // ---------------- producer warp (lane 0 issues)
    if (lane != 0) return;
    Prod p;
    p.full0 = full0;
    p.empty0 = empty0;
    p.stages_addr = smem_addr(ring);
    p.desc = s_desc;
    p.it = 0;
    p.deadline = deadline;
    p.hdr = hdr;
    p.abort_flag = &s_abort;
    int u = (int)atomicAdd(&hdr->unit_next, 1u);    // unit being issued
    int nxt = (int)atomicAdd(&hdr->unit_next, 1u);  // claimed ahead
    bool meta = false, claims_open = true;
    int total = 0x7fffffff, ng = 0, ndn = 0;
    // Down items: the shared group first (its h is ready first), then the
    // routed groups in table order.  kw: items whose Wd copy is issued, kh:
    // items whose h copy is issued (kh <= kw; items in between were posted
    // ahead with only their Wd slice, once this CTA had no gate/up left).
    int kw = 0, kh = 0;
    int dslot[fz::NS];
    auto dn_group = [&](int kk) { return kk == 0 ? ng - 1 : kk - 1; };
    auto dn_item = [&](int kk, const uint16_t*& wd, const float*& hr) {
      const int4 grp = s_groups[dn_group(kk)];
      Item d = {};
      d.kind = fz::IT_DOWN;
      d.pair0 = grp.y;
      d.n = grp.z;
      wd = (grp.x < E ? a.w.w2 + (size_t)grp.x * H * I : a.w.ws2 + (size_t)(grp.x - E) * H * I) +
           (size_t)r0 * I;
      hr = a.ws.h + (size_t)grp.y * I;
      return d;
    };
    bool ok = true;
    while (ok && !s_abort) {
      // Down items whose groups the poll warp has seen complete.
      const int rdy = meta && kh < ndn ? ld_acquire_cta_shared(&s_ready) : 0;
      if (rdy > kh) {
        {
          // h of these groups was written by other CTAs (generic proxy); the
          // poll warp acquired it at GPU scope and this thread from the poll
          // warp at CTA scope.  Order it before the bulk (async-proxy) reads.
          asm volatile("fence.proxy.async.global;" ::: "memory");
          for (; ok && kh < rdy; ++kh) {
            const uint16_t* wd;
            const float* hr;
            const Item d = dn_item(kh, wd, hr);
            if (kh < kw) {  // Wd already on its way: add the h rows
              const int sl = dslot[kh % fz::NS];
              bulk_g2s(p.stages_addr + sl * fz::SLOT + dn::WBYTES, hr, d.n * dn::HROW,
                       p.full0 + 8u * sl);
            } else {
              int sl;
              if (!(ok = take_slot(p, sl))) break;
              p.desc[sl] = d;
              mbar_expect_tx(p.full0 + 8u * sl, dn::WBYTES + d.n * dn::HROW);
              bulk_g2s_stream(p.stages_addr + sl * fz::SLOT, wd, dn::WBYTES, p.full0 + 8u * sl);
              bulk_g2s(p.stages_addr + sl * fz::SLOT + dn::WBYTES, hr, d.n * dn::HROW,
                       p.full0 + 8u * sl);
              kw = kh + 1;
            }
          }
          continue;
        }
      }
      if (claims_open && u >= fz::UNITS && !meta) {
        post_marker(p, fz::IT_SELECT);
        if (!mbar_wait(sel_bar, 0u, deadline)) {
          s_abort = 1;
          set_error(hdr, DEV_TIMEOUT);
          break;
        }
        ng = s_ngroups;
        total = ng * fz::UNITS;  // the shared group's units and the routed ones
        ndn = owner ? ng : 0;
        meta = true;
        continue;
      }
      if (claims_open && u < total) {
        Item d = {};
        d.kind = fz::IT_GATE;
        const uint16_t* base;
        if (u < fz::UNITS) {  // shared expert: tokens 0..B-1, pairs after the routed ones
          d.blk = u;
          d.pair0 = npairs;
          d.n = B;
          d.tok0 = 0;
          d.done_idx = fz::DONE_SHARED;
          base = a.w.ws13;
        } else {
          const int ru = u - fz::UNITS;
          const int gi = ru / fz::UNITS;
          const int4 grp = s_groups[gi];
          d.blk = ru % fz::UNITS;
          d.pair0 = grp.y;
          d.n = grp.z;
          d.tok0 = -1;
          d.done_idx = gi;
          base = a.w.w13 + (size_t)grp.x * (2 * I) * H;
        }
        ok = post_gateup(p, base, d);
        u = nxt;
        nxt = (int)atomicAdd(&hdr->unit_next, 1u);
        continue;
      }
      claims_open = false;
      if (kh < ndn) {  // nothing left to stream but this CTA's down rows
        if (kw < ndn && kw - kh < fz::NS) {
          // post the next item's Wd slice now; its h follows once complete
          const uint16_t* wd;
          const float* hr;
          const Item d = dn_item(kw, wd, hr);
          int sl;
          if (!(ok = take_slot(p, sl))) break;
          p.desc[sl] = d;
          mbar_expect_tx(p.full0 + 8u * sl, dn::WBYTES + d.n * dn::HROW);
          bulk_g2s_stream(p.stages_addr + sl * fz::SLOT, wd, dn::WBYTES, p.full0 + 8u * sl);
          dslot[kw % fz::NS] = sl;
          ++kw;
          continue;
        }
        if (globaltimer_ns() > deadline) {
          s_abort = 1;
          set_error(hdr, DEV_TIMEOUT);
          break;
        }
        continue;  // spin on s_ready (shared memory)
      }
      break;
    }
    // Items posted with their Wd slice only still wait for h: on an abort,
    // complete them with the h rows as they are, so no copy stays pending.
    for (; kh < kw; ++kh) {
      const uint16_t* wd;
      const float* hr;
      const Item d = dn_item(kh, wd, hr);
      const int sl = dslot[kh % fz::NS];
      bulk_g2s(p.stages_addr + sl * fz::SLOT + dn::WBYTES, hr, d.n * dn::HROW, p.full0 + 8u * sl);
    }
    // The claim made ahead must have landed before the CTA counts itself out
    // (the last CTA out resets the counter): wait for its value.
    if (nxt < 0) s_abort = 1;
    post_marker(p, fz::IT_END);
    return;
  }

  if ((tid >> 5) == fz::CW + 2) {  // ---------------- poll warp (lane 0, row-slice owners)
    // Watches the completion counters of this CTA's down items in order (the
    // shared group first, then the routed groups), eight loads in flight at a
    // time, and publishes how many are complete; the GPU-scope acquire fence
    // is taken here, so the producer never waits on one.
    if (lane != 0 || !owner) return;
    while (!mbar_test(sel_bar, 0u))
      if (s_abort || globaltimer_ns() > deadline) return;
    const int ng = s_ngroups;
    int k = 0;
    while (k < ng && !s_abort) {
      uint32_t pw[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        pw[j] = k + j < ng ? ld_relaxed(done + (k + j == 0 ? fz::DONE_SHARED : k + j - 1)) : 0u;
      int rdy = 0;
      bool run = true;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        run = run && k + j < ng && pw[j] >= fz::DONE_TARGET;
        rdy += run ? 1 : 0;
      }
      if (rdy > 0) {
        fence_acq_rel_gpu();
        k += rdy;
        st_release_cta_shared(&s_ready, k);
      } else if (globaltimer_ns() > deadline) {
        break;
      }
    }
    return;
  }

  if ((tid >> 5) == fz::CW + 1) {  // ---------------- signalling warp (lane 0)
    if (lane != 0) return;
    // Publishes finished units in order, one release fence per batch of units
    // found finished (the consumers' h stores were ordered before their
    // arrivals on the unit's barrier, which this thread has observed).
    const uint64_t limit = deadline + fz::DRAIN_NS;
    int q = 0;
    bool end = false;
    while (!end) {
      if (!mbar_wait(hfull0 + 8u * (q & (fz::SIGQ - 1)), (uint32_t)(q / fz::SIGQ) & 1u, limit)) break;
      int n = 1;
      while (n < fz::SIGQ &&
             mbar_test(hfull0 + 8u * ((q + n) & (fz::SIGQ - 1)), (uint32_t)((q + n) / fz::SIGQ) & 1u))
        ++n;
      fence_acq_rel_gpu();
      int k = 0;
      for (; k < n; ++k) {
        const int gi = s_hgrp[(q + k) & (fz::SIGQ - 1)];
        if (gi == -1) {
          end = true;
          break;
        }
        if (gi >= 0) red_add_relaxed(done + gi, 1u);
      }
      for (int j = 0; j < k; ++j) mbar_arrive(hfree0 + 8u * ((q + j) & (fz::SIGQ - 1)));
      q += k;
    }
    __threadfence();  // the adds are performed before the CTA counts itself out
    mbar_arrive(sig_done);
    return;
  }

  // ---------------- consumer warps
  if (r.stall_check && cta == 0 && tid == 0 &&
      *reinterpret_cast<volatile uint32_t*>(&hdr->stall_armed)) {
    // Test hook: wait for a flag that nothing sets; the bounded wait runs out
    // and records the timeout, exactly like a stuck pipeline wait would.
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
  if (tid == 0) {
    __threadfence();
    atomicAdd(&hdr->grid_bar[0], 1u);
  }
  // the batch's activations, once (all loads in flight together)
  {
    uint4 v[fz::MAXB];
#pragma unroll
    for (int t = 0; t < fz::MAXB; ++t)
      v[t] = t < B ? __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)t * H) + tid)
                   : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int t = 0; t < fz::MAXB; ++t)
      if (t < B) reinterpret_cast<uint4*>(xs)[t * (H / 8) + tid] = v[t];
  }
  named_sync(1, fz::CT);  // xs is complete before any gate/up unit reads it

  dn_impl::DnCtx dc;
  dc.acc = s_acc;
  dc.red = buf;
  dc.pair_tok = s_pair_tok;
  dc.pair_w = s_pair_w;

  int it = 0, useq = 0;
  const uint64_t drain = deadline + fz::DRAIN_NS;
  Sig sig;
  sig.full0 = hfull0;
  sig.free0 = hfree0;
  sig.grp = s_hgrp;
  sig.limit = drain;
  while (true) {
    const int slot = it % fz::NS;
    const uint32_t par = (uint32_t)(it / fz::NS) & 1u;
    if (!mbar_wait(full0 + 8u * slot, par, deadline)) {
      s_abort = 1;
      set_error(hdr, DEV_TIMEOUT);
      if (!mbar_wait(full0 + 8u * slot, par, drain)) break;
    }
    const Item d = s_desc[slot];
    const bool ok = !s_abort;
    if (d.kind == fz::IT_END) break;
    if (d.kind == fz::IT_SELECT) {
      // 2. every CTA ranks and buckets the batch once all logits are in
      if (tid == 0 && !grid_wait(&hdr->grid_bar[0], (uint32_t)G, deadline)) {
        s_abort = 1;
        set_error(hdr, DEV_TIMEOUT);
      }
      named_sync(1, fz::CT);
      {
        float lv[fz::MAXB];
#pragma unroll
        for (int t = 0; t < fz::MAXB; ++t)
          lv[t] = t < B ? __ldcg(a.ws.logits + (size_t)t * E + tid) : 0.f;
#pragma unroll
        for (int t = 0; t < fz::MAXB; ++t)
          if (t < B) buf[t * E + tid] = lv[t];
      }
      named_sync(1, fz::CT);
      const int warp = tid >> 5;
      if (warp < B) {
        int ix;
        float wt;
        topk_warp<false>(buf + warp * E, ix, wt);
        if (lane < TOPK) {
          const int pp = warp * TOPK + lane;
          s_sel.idx[pp] = ix;
          s_sel.w[pp] = wt;
          if (cta == 0) {
            a.ws.topk_idx[pp] = ix;
            a.ws.topk_w[pp] = wt;
            if (a.user_idx) a.user_idx[pp] = ix;
            if (a.user_w) a.user_w[pp] = wt;
          }
        }
      }
      named_sync(1, fz::CT);
      bucket_small<fz::CT, 4>(B, s_sel.idx, s_sel.w, s_pair_tok, s_pair_w, s_groups, &s_ngroups,
                              s_sel.sc.off);
      named_sync(1, fz::CT);
      if (tid == 0) mbar_arrive(sel_bar);
      release_slot(empty0 + 8u * slot);
      ++it;
      continue;
    }
    if (d.kind == fz::IT_DOWN) {
      // 4. this CTA's 16 output rows of the group, weighted into the accumulators
      const uint8_t* st = ring + slot * fz::SLOT;
      const uint32_t em = empty0 + 8u * slot;
      if (d.n <= dn::CC_MAX) {
        down_cc(st, d.pair0, d.n, s_pair_tok, s_pair_w, lacc, ok, em);
      } else {
        dn_impl::group_mma<1>(dc, st, d.pair0, ok ? d.n : 0);  // n <= 8 here, into s_acc
        release_slot(em);
      }
      ++it;
      continue;
    }
    // 3. gate/up unit: gate rows in this slot, up rows in the next
    const int slot2 = (it + 1) % fz::NS;
    const uint32_t par2 = (uint32_t)((it + 1) / fz::NS) & 1u;
    bool ok2 = ok;
    if (!mbar_wait(full0 + 8u * slot2, par2, deadline)) {
      s_abort = 1;
      set_error(hdr, DEV_TIMEOUT);
      ok2 = false;
      if (!mbar_wait(full0 + 8u * slot2, par2, drain)) break;
    }
    if (s_desc[slot2].kind != fz::IT_UP) break;  // the producer gave up mid-unit (abort)
    const uint8_t* gs = ring + slot * fz::SLOT;
    const uint8_t* us = ring + slot2 * fz::SLOT;
    if (d.n <= gu::CC_MAX) {
      int tok[2];
      tok[0] = d.tok0 >= 0 ? d.tok0 : s_pair_tok[d.pair0];
      tok[1] = d.n > 1 ? (d.tok0 >= 0 ? d.tok0 + 1 : s_pair_tok[d.pair0 + 1]) : tok[0];
      if (d.n == 1)
        unit_cc<1>(gs, us, reinterpret_cast<const uint4*>(xs), tok, a.ws.h, d, ok2,
                   empty0 + 8u * slot, empty0 + 8u * slot2);
      else
        unit_cc<2>(gs, us, reinterpret_cast<const uint4*>(xs), tok, a.ws.h, d, ok2,
                   empty0 + 8u * slot, empty0 + 8u * slot2);
    } else {
      unit_mma(gs, us, xs, s_pair_tok, buf, a.ws.h, d, ok2, empty0 + 8u * slot,
               empty0 + 8u * slot2);
    }
    signal_unit(sig, useq++, ok2 ? d.done_idx : -2);
    it += 2;
  }
  signal_unit(sig, useq, -1);
  named_sync(1, fz::CT);
  if (owner && !s_abort) {
    // Thread pair (2s, 2s+1) finishes sum s = (warp w, token t, row r): each
    // adds 16 lanes' running sums, one shuffle joins the halves; the
    // tensor-core items' share is in s_acc.  Row 2w + r of the CTA's slice.
    const int sidx = tid >> 1, half = tid & 1;
    const int w = sidx >> 4, j = sidx & 15, t = j >> 1, rr = j & 1;
    const float* src = lacc + j * fz::LACC_STRIDE + w * 32 + half * 16;
    float v = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) v += src[k];
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    if (half == 0 && t < B) {
      const int row = 2 * w + rr;
      const size_t o = (size_t)t * H + r0 + row;
      a.out[o] = f2bf(bf_lo((uint32_t)a.residual[o]) + (v + s_acc[t * dn::RS + row]));
    }
  }
  // The last CTA out resets the counters for the next call (every CTA has
  // finished its claims, marks and polls by the time it counts itself out).
  if (tid == 0) {
    mbar_wait(sig_done, 0u, drain);
    __threadfence();
    if (atomicAdd(&hdr->grid_bar[2], 1u) == (uint32_t)G - 1) {
      hdr->grid_bar[0] = 0u;
      hdr->unit_next = 0u;
      for (int i = 0; i < 64; ++i) done[i] = 0u;
      hdr->grid_bar[2] = 0u;
      __threadfence();
    }
  }
}

cudaError_t launch_small_bf16(const ExpertArgs& a, const RouterArgs& r, cudaStream_t stream,
                              int num_sms) {
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t es = set_smem_limit_once(moe_small_bf16_kernel, (int)fz::SMEM, smem_set);
  if (es != cudaSuccess) return es;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms, 1, 1);
  cfg.blockDim = dim3(fz::THREADS, 1, 1);
  cfg.dynamicSmemBytes = fz::SMEM;
  cfg.stream = stream;
  // One CTA per SM: the kernel's shared memory (> half an SM's) allows no
  // second one, so the grid of #SMs CTAs is resident as soon as the SMs are
  // free; the grid-wide waits are bounded in any case.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_small_bf16_kernel, a, r);
}

}  // namespace flint
