// fused.cu — the whole BF16 decode MoE layer in one persistent kernel, for
// batches of at most SMALL_B (8) tokens: the pages' low-latency path for up to
// 8 requests, which fuses routing and the expert combine into the neighbouring
// GEMVs ("Low-Latency Decode Path": vLLM Day-0 Support for Recursive's Flint,
// "Optimization Strategies").
//
// One CTA per SM, all co-resident (cooperative launch), 8 consumer warps + a
// producer warp + a poll warp.  The producer's lane 0 feeds a ring of 32 KiB
// shared-memory slots with cp.async.bulk copies and tags each slot with what
// it holds; the consumers take the slots in order.
//
//   1. Router: the producer copies the CTA's 1-3 router rows into shared
//      memory as soon as the kernel starts (weights do not depend on the
//      preceding kernel); the consumers stage the batch's activations, dot
//      them with the rows and publish the logits as tagged words.  Meanwhile
//      the producer streams shared-expert gate/up units, which need no routing.
//   2. Selection: once every CTA has counted its logits in, each CTA reads all
//      of them, ranks every token (one warp per token) and buckets the pairs --
//      identical results in every CTA -- and hands the group table to the
//      producer and the poll warp.
//   3. Work queue: gate/up units (8 gate + 8 up rows of one group, two slots)
//      are claimed one at a time from a workspace counter -- the shared
//      expert's 64 units first, then the routed groups' in group order -- so
//      CTAs that stream faster take more units and groups finish roughly in
//      order.  The consumer warps store their h values as tagged words; the
//      last of them to finish a unit adds one to its group's counter, and 64
//      marks a group's h complete.
//   4. Down: CTA b < 128 owns output rows [16b, 16b+16) of every token.  The
//      poll warp watches the counters of its groups; as soon as one is
//      complete, the producer posts a DOWN item: the 16 rows of the expert's
//      Wd (16 KiB) and the group's tagged h rows (4 KiB per token; more than
//      4 tokens spill into a second slot), and the consumers confirm every h
//      word's tag and accumulate w(t, g) * (Wd h) per token: groups of <= 4
//      tokens on CUDA cores into per-lane running sums (reduced once, at the
//      end), larger ones on tensor cores.  Down items take priority over
//      gate/up units, so the down projection streams while gate/up is still
//      running.  Items run in a fixed order (the shared expert, then the
//      routed groups by expert), so results are reproducible bit for bit.
//
// No GPU-scope fence is taken on the data path: a fence waits for the SM's
// outstanding memory traffic, which while weights stream costs 1-3 us per
// hand-off.  Logits and h cross SMs as tagged words instead (call_tag), and
// the counters only say when to look.  The counters come in two sets used by
// alternate calls: a call clears the set of the next call, and CTA 0 advances
// the workspace's call counter at its end, so nothing is reset at the exit.
// Every wait is bounded by the workspace's limit.
#include "common.cuh"
#include "expert_common.cuh"
#include "gateup_impl.cuh"
#include "kernels.h"
#include "nv_util.cuh"

namespace flint {
namespace fz {
constexpr int CW = 8;                          // consumer warps
constexpr int PRODUCER = CW;                   // warp index of the producer
constexpr int POLL = CW + 1;                   // warp index of the poll warp
constexpr int THREADS = (CW + 2) * 32;
constexpr int CT = CW * 32;                    // consumer threads
constexpr int ROWB = H * 2;                    // one gate/up row (bf16), 4 KiB
constexpr int UNITS = I / 8;                   // gate/up units per group
constexpr int MAXB = SMALL_B;
constexpr int MAXG = MAXB * TOPK + S;          // groups at these batches (one shared group)
constexpr int NPAIR = MAXB * SLOTS;
constexpr int DONE_SHARED = SYNC_GROUPS - 1;   // counter of the shared group
constexpr int UCNT = 8;                        // unit-completion counts in flight
// Ready down items an owner may post between two of its gate/up units.  A
// claimed unit must not wait behind a long run of down items: its group would
// complete late for every owner, and their down items with it.
constexpr int DN_PER_UNIT = 3;
constexpr uint32_t DONE_TARGET = UNITS;        // unit marks per complete group
constexpr int RS = 16;                         // output rows per row-slice owner
constexpr int DOWN_CTAS = H / RS;              // 128 row-slice owners
constexpr int WROW = I * 2;                    // one Wd row (bf16)
constexpr int THROW = I * 8;                   // one tagged h row, 4 KiB
constexpr int CC_MAX = 4;                      // BF16 down items on CUDA cores up to this many tokens
constexpr int XS_BYTES = MAXB * H * 2;         // bf16 activations of the batch, 32 KiB
constexpr int RED_BYTES = CW * 16 * GROUP_MAX * 4;
constexpr int LOGIT_BYTES = MAXB * E * 4;
constexpr int RMAX = 3;                        // router rows per CTA (grids of >= 86 CTAs)
constexpr int RROW_BYTES = RMAX * H * 2;
constexpr int BUF_BYTES = RED_BYTES > LOGIT_BYTES ? (RED_BYTES > RROW_BYTES ? RED_BYTES : RROW_BYTES)
                                                  : (LOGIT_BYTES > RROW_BYTES ? LOGIT_BYTES : RROW_BYTES);
// Per-lane running sums of the CUDA-core down items: [token * 2 + row][thread],
// rows padded to 257 floats so that both the updates (one row, consecutive
// lanes) and the final per-row sums (16 lanes each) are free of bank conflicts.
constexpr int LACC_STRIDE = CW * 32 + 1;
constexpr int LACC_BYTES = MAXB * 2 * LACC_STRIDE * 4;
// Ring and down-slice layout of each weight format.
template <bool NV>
struct Geo;
template <>
struct Geo<false> {  // BF16: a gate/up unit is 2 slots (8 gate rows, 8 up rows)
  static constexpr int SLOT = 32 * 1024, NS = 5, UNIT_SLOTS = 2;
  static constexpr int WBYTES = RS * WROW;                  // Wd slice, 16 KiB
  static constexpr int HROWS_A = (SLOT - WBYTES) / THROW;   // h rows beside it: 4
};
template <>
struct Geo<true> {  // NVFP4: a gate/up unit is 1 slot (codes, then block scales)
  static constexpr int SLOT = 20 * 1024, NS = 8, UNIT_SLOTS = 1;
  static constexpr int QROW = H / 2, SFROW = H / 16;        // one gate/up row
  static constexpr int UNIT_BYTES = 16 * QROW + 16 * SFROW; // 18 KiB
  static constexpr int DQROW = I / 2, DSFROW = I / 16;      // one Wd row
  static constexpr int WQ = RS * DQROW;                     // slice codes, 4 KiB
  static constexpr int WBYTES = WQ + RS * DSFROW;           // + scales, 4.5 KiB
  static constexpr int HROWS_A = (SLOT - WBYTES) / THROW;   // h rows beside it: 3
};
template <bool NV>
constexpr size_t smem_bytes() {
  return (size_t)Geo<NV>::NS * Geo<NV>::SLOT + XS_BYTES + BUF_BYTES + LACC_BYTES;
}
constexpr uint64_t DRAIN_NS = 2000000000ull;
enum : int { IT_GATE = 0, IT_UP = 1, IT_DOWN = 2, IT_DOWN2 = 3, IT_END = 4 };
static_assert(S == 1 && MAXB <= GROUP_MAX, "one shared group at these batches");
static_assert(MAXG <= DONE_SHARED, "routed groups and the shared group have distinct counters");
static_assert(SYNC_LINES <= CT, "one thread clears each counter line");
static_assert(Geo<false>::HROWS_A == 4 && MAXB - 4 <= Geo<false>::SLOT / THROW,
              "a BF16 down item fits two slots");
static_assert(Geo<true>::HROWS_A == 3 && MAXB - 3 <= Geo<true>::SLOT / THROW,
              "an NVFP4 down item fits two slots");
static_assert(8 * ROWB == Geo<false>::SLOT, "8 gate (or up) rows fill one BF16 slot");
static_assert(Geo<true>::UNIT_BYTES <= Geo<true>::SLOT, "an NVFP4 unit fits one slot");
static_assert(Geo<true>::WBYTES % 16 == 0, "h rows start 16-byte aligned");
static_assert((E + RMAX - 1) / RMAX <= 86, "grids of 86 CTAs or more keep <= RMAX router rows");
static_assert(smem_bytes<false>() + 6 * 1024 <= 232448 && smem_bytes<true>() + 6 * 1024 <= 232448,
              "fits the opt-in shared memory of one SM");
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
  int expert;    // expert of the group (E + s for shared expert s)
  int pad;
};

__device__ __forceinline__ int ld_acquire_cta_shared(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta_shared(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
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

// Router scores of experts [e_begin, e_end) for the whole batch (B <= 8), by
// the 8 consumer warps from shared memory (router rows in `rows`, activations
// in xs): warp w takes expert base + w/4 and the K-quarter w%4.  Published as
// tagged words; the logit offsets join at ranking.
__device__ __forceinline__ void router_slice(int B, uint64_t* tlogits,
                                             const uint16_t* rows, const uint16_t* xs,
                                             int e_begin, int e_end, float (*s_part)[4][8],
                                             uint32_t tag) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int el = warp >> 2, qk = warp & 3;
  for (int base = e_begin; base < e_end; base += 2) {
    const int e = base + el;
    float acc[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) acc[t] = 0.f;
    if (e < e_end) {
      const int c0 = qk * 64 + lane, c1 = c0 + 32;
      const uint4* wrow = reinterpret_cast<const uint4*>(rows + (size_t)(e - e_begin) * H);
      const uint4 w0 = wrow[c0], w1 = wrow[c1];
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        if (t < B) {
          const uint4* xrow = reinterpret_cast<const uint4*>(xs + (size_t)t * H);
          acc[t] = dot8(w1, xrow[c1], dot8(w0, xrow[c0], 0.f));
        }
      }
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
        st_tagged(tlogits + (size_t)t * E + ee,
                  (s_part[le][0][t] + s_part[le][1][t]) + (s_part[le][2][t] + s_part[le][3][t]),
                  tag);
    }
    named_sync(1, fz::CT);
  }
}

// ---- consumer side -----------------------------------------------------------

__device__ __forceinline__ void release_slot(uint32_t empty_bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty_bar);
}

// After a warp's h stores of a unit: the last of the 8 consumer warps to get
// here puts one mark on the group's counter -- a hint; the readers confirm
// the tags.  The count lives in shared memory, one per unit sequence number
// modulo UCNT: a warp can be at most a few units ahead of another (the ring
// refills a slot only once all 8 warps have released it).
__device__ __forceinline__ void mark_unit(SyncLine* done, int done_idx, int* ucnt) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0 && atomicAdd(ucnt, 1) == fz::CW - 1) {
    *ucnt = 0;
    red_add_relaxed(&done[done_idx].v, 1u);
  }
}

// Gate/up unit on CUDA cores (<= 2 tokens): warp w owns gate row w and up row
// w; the same arithmetic, in the same order, as the standalone gate/up kernel
// (gate and up chains interleaved: eight independent FMA chains per lane).
template <int NTOK>
__device__ __forceinline__ void unit_cc(const uint8_t* gs, const uint8_t* us, const uint4* xs,
                                        const int (&tok)[2], uint64_t* th, const Item& d, bool ok,
                                        uint32_t emA, uint32_t emB, uint32_t tag, SyncLine* done,
                                        int* ucnt) {
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
    if (lane == 0)
      st_tagged(th + (size_t)(d.pair0 + i) * I + d.blk * 8 + warp, silu_mul(gsum, vsum), tag);
  }
  mark_unit(done, d.done_idx, ucnt);
}

template <bool SCALED>
__device__ __forceinline__ void unit_finish(const float (&acc)[4], float* buf, uint64_t* th,
                                            const Item& d, bool ok, uint32_t tag,
                                            SyncLine* done, int* ucnt, float ts_g, float ts_u);

// Gate/up unit on tensor cores (3..8 tokens): m16n8k16 with the 8 gate + 8 up
// rows as M and the tokens as N, warp w owns a 256-column K-slice; the same
// arithmetic as the standalone gate/up kernel.
__device__ __forceinline__ void unit_mma(const uint8_t* gs, const uint8_t* us, const uint16_t* xs,
                                         const int* pair_tok, float* buf, uint64_t* th,
                                         const Item& d, bool ok, uint32_t emA, uint32_t emB,
                                         uint32_t tag, SyncLine* done, int* ucnt) {
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
  unit_finish<false>(acc, buf, th, d, ok, tag, done, ucnt, 1.f, 1.f);
}

// The 8 warps' partial 16 x 8 tiles of a tensor-core unit summed through
// shared memory; row r of the block and token slot j go to thread (r, j),
// which stores h = silu(gate) * up (NVFP4: each sum times its tensor scale).
template <bool SCALED>
__device__ __forceinline__ void unit_finish(const float (&acc)[4], float* buf, uint64_t* th,
                                            const Item& d, bool ok, uint32_t tag,
                                            SyncLine* done, int* ucnt, float ts_g, float ts_u) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int n = d.n;
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
      if constexpr (SCALED) {
        gsum *= ts_g;
        usum *= ts_u;
      }
      st_tagged(th + (size_t)(d.pair0 + j) * I + d.blk * 8 + r, silu_mul(gsum, usum), tag);
    }
    if (ok) mark_unit(done, d.done_idx, ucnt);
  }
  named_sync(1, fz::CT);  // buf is free again
}

// Gate/up unit of NVFP4 weights, on tensor cores for every group size (the
// dequantisation, about one instruction per weight, dominates; the MMA then
// costs nothing extra).  The slot holds the 8 gate rows' codes, the 8 up
// rows' codes, then their block scales; the 16 rows are the MMA's M, the
// tokens its N.  Warp w owns a 256-column K-slice; thread q of a quad takes
// columns [32q + 128m, +32) for m = 0, 1 (16 contiguous code bytes per row),
// the f16 activations in shared memory follow the same order.  Each code
// times its E4M3 block scale is exact in f16.
__device__ __forceinline__ void unit_nv(const uint8_t* st, const uint16_t* xh,
                                        const int* pair_tok, float* buf, uint64_t* th,
                                        const Item& d, float ts_g, float ts_u, bool ok,
                                        uint32_t em, uint32_t tag, SyncLine* done, int* ucnt) {
  using Gm = fz::Geo<true>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (ok) {
    uint4 bfr[2][4];
    if (g < d.n) {
      const int tok = d.tok0 >= 0 ? d.tok0 + g : pair_tok[d.pair0 + g];
      const uint4* row = reinterpret_cast<const uint4*>(xh + (size_t)tok * H + warp * 256 + q * 32);
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) bfr[m][i] = row[m * 16 + i];
    } else {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) bfr[m][i] = make_uint4(0u, 0u, 0u, 0u);
    }
    const uint8_t* qlo = st + g * Gm::QROW + warp * 128 + q * 16;
    const uint8_t* qhi = qlo + 8 * Gm::QROW;
    const uint8_t* sfb = st + 16 * Gm::QROW;
    const uint4 slo = *reinterpret_cast<const uint4*>(sfb + g * Gm::SFROW + warp * 16);
    const uint4 shi = *reinterpret_cast<const uint4*>(sfb + (g + 8) * Gm::SFROW + warp * 16);
    const bool qh = (q >> 1) != 0;
#pragma unroll
    for (int m = 0; m < 2; ++m) {
      const uint4 clo = *reinterpret_cast<const uint4*>(qlo + m * 64);
      const uint4 chi = *reinterpret_cast<const uint4*>(qhi + m * 64);
      const uint32_t cl[4] = {clo.x, clo.y, clo.z, clo.w};
      const uint32_t ch[4] = {chi.x, chi.y, chi.z, chi.w};
      // columns 32q + 128m + 8i .. +8 are block 8m + 2q + i/2 of the warp's
      // 16: byte 2(q & 1) + i/2 of scale word 2m + q/2
      const uint32_t wl = m ? (qh ? slo.w : slo.z) : (qh ? slo.y : slo.x);
      const uint32_t wh = m ? (qh ? shi.w : shi.z) : (qh ? shi.y : shi.x);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int sh = 8 * (2 * (q & 1) + (i >> 1));
        const uint32_t scl = nvu::e4m3_bcast_f16x2((wl >> sh) & 0xffu);
        const uint32_t sch = nvu::e4m3_bcast_f16x2((wh >> sh) & 0xffu);
        uint32_t l0, l1, l2, l3, h0, h1, h2, h3;
        nvu::e2m1x8_to_f16x2(cl[i], l0, l1, l2, l3);
        nvu::e2m1x8_to_f16x2(ch[i], h0, h1, h2, h3);
        l0 = nvu::hmul2(l0, scl);
        l1 = nvu::hmul2(l1, scl);
        l2 = nvu::hmul2(l2, scl);
        l3 = nvu::hmul2(l3, scl);
        h0 = nvu::hmul2(h0, sch);
        h1 = nvu::hmul2(h1, sch);
        h2 = nvu::hmul2(h2, sch);
        h3 = nvu::hmul2(h3, sch);
        nvu::mma_f16(acc, l0, h0, l1, h1, bfr[m][i].x, bfr[m][i].y);
        nvu::mma_f16(acc, l2, h2, l3, h3, bfr[m][i].z, bfr[m][i].w);
      }
    }
  }
  release_slot(em);
  unit_finish<true>(acc, buf, th, d, ok, tag, done, ucnt, ts_g, ts_u);
}

// Shared context of the down items.
struct DnCtx {
  const int* pair_tok;  // shared memory
  const float* pair_w;  // shared memory
  float* lacc;          // CUDA-core running sums
  float* acc;           // [MAXB][RS] tensor-core accumulators
  float* red;           // [CW][RS][GROUP_MAX] partial tiles
  const uint64_t* th;   // tagged h (global), for words whose tag has not landed
  uint32_t tag;
  uint64_t deadline;
  WsHeader* hdr;
  volatile int* abort_flag;
};

// h value k of a token's row (copy in shared memory at hrow, the tagged row
// itself at src), confirmed against the call's tag.
__device__ __forceinline__ float h_settled(const DnCtx& c, const uint8_t* hrow,
                                           const uint64_t* src, int k) {
  uint64_t w = *reinterpret_cast<const uint64_t*>(hrow + (size_t)k * 8);
  if (!settle_tagged(w, src + k, c.tag, c.deadline)) {
    *c.abort_flag = 1;
    set_error(c.hdr, DEV_TIMEOUT);
  }
  return __uint_as_float((uint32_t)w);
}

// Down item on CUDA cores (<= 4 tokens): warp w owns Wd rows 2w and 2w+1 of
// the slice; lane l takes columns 2l + 64m (+1), m < 8, which makes every
// 128-bit load of tagged h words conflict-free.  The lane's 32 weights are
// unpacked once and reused by every token; each token's two dot products run
// as four independent chains; each lane adds w(t, g) times its partial sums to
// its own running sums in shared memory -- the sums across lanes are taken
// once, when the output is written.  A word whose tag has not landed sends
// the warp through the same arithmetic with every value confirmed from global
// memory (rare: the counters run behind the stores).
__device__ __forceinline__ void down_cc(const DnCtx& c, const uint8_t* st, int pair0, int n,
                                        bool ok, uint32_t em) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tok[fz::CC_MAX];
  float wt[fz::CC_MAX];
#pragma unroll
  for (int i = 0; i < fz::CC_MAX; ++i) {  // the bookkeeping loads go out first
    tok[i] = i < n ? c.pair_tok[pair0 + i] : 0;
    wt[i] = i < n ? c.pair_w[pair0 + i] : 0.f;
  }
  float s0[fz::CC_MAX], s1[fz::CC_MAX];
#pragma unroll
  for (int i = 0; i < fz::CC_MAX; ++i) s0[i] = s1[i] = 0.f;
  const uint32_t* w0 = reinterpret_cast<const uint32_t*>(st + (2 * warp) * fz::WROW);
  const uint32_t* w1 = w0 + fz::WROW / 4;
  if (ok) {
    float f0[16], f1[16];
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      const uint32_t a0 = w0[lane + 32 * m], a1 = w1[lane + 32 * m];
      f0[2 * m] = bf_lo(a0);
      f0[2 * m + 1] = bf_hi(a0);
      f1[2 * m] = bf_lo(a1);
      f1[2 * m + 1] = bf_hi(a1);
    }
    bool bad = false;
#pragma unroll
    for (int i = 0; i < fz::CC_MAX; ++i) {
      if (i < n) {
        const uint4* hr =
            reinterpret_cast<const uint4*>(st + fz::Geo<false>::WBYTES + i * fz::THROW);
        float e0 = 0.f, o0 = 0.f, e1 = 0.f, o1 = 0.f;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint4 hv = hr[lane + 32 * m];
          bad |= (hv.y != c.tag) | (hv.w != c.tag);
          const float h0 = __uint_as_float(hv.x), h1 = __uint_as_float(hv.z);
          e0 = fmaf(f0[2 * m], h0, e0);
          o0 = fmaf(f0[2 * m + 1], h1, o0);
          e1 = fmaf(f1[2 * m], h0, e1);
          o1 = fmaf(f1[2 * m + 1], h1, o1);
        }
        s0[i] = e0 + o0;
        s1[i] = e1 + o1;
      }
    }
    if (__any_sync(0xffffffffu, bad)) {
      // Same sums, same order; weights re-read from the slot so that no
      // register array is indexed at run time.
#pragma unroll
      for (int i = 0; i < fz::CC_MAX; ++i) {
        float e0 = 0.f, o0 = 0.f, e1 = 0.f, o1 = 0.f;
        if (i < n) {
          const uint8_t* hrow = st + fz::Geo<false>::WBYTES + i * fz::THROW;
          const uint64_t* src = c.th + (size_t)(pair0 + i) * I;
#pragma unroll 1
          for (int m = 0; m < 8; ++m) {
            const int k = 2 * lane + 64 * m;
            const uint32_t u0 = w0[lane + 32 * m], u1 = w1[lane + 32 * m];
            const float h0 = h_settled(c, hrow, src, k);
            const float h1 = h_settled(c, hrow, src, k + 1);
            e0 = fmaf(bf_lo(u0), h0, e0);
            o0 = fmaf(bf_hi(u0), h1, o0);
            e1 = fmaf(bf_lo(u1), h0, e1);
            o1 = fmaf(bf_hi(u1), h1, o1);
          }
        }
        s0[i] = e0 + o0;
        s1[i] = e1 + o1;
      }
    }
  }
  release_slot(em);
  if (!ok) return;
#pragma unroll
  for (int i = 0; i < fz::CC_MAX; ++i) {
    if (i < n) {
      float* acc = c.lacc + (2 * tok[i]) * fz::LACC_STRIDE + threadIdx.x;
      acc[0] = fmaf(wt[i], s0[i], acc[0]);
      acc[fz::LACC_STRIDE] = fmaf(wt[i], s1[i], acc[fz::LACC_STRIDE]);
    }
  }
}

// Down item on tensor cores (5..8 tokens, h rows 0..3 beside the Wd slice in
// slot A, rows 4.. in slot B): mma.sync m16n8k16 with the 16 Wd rows as M and
// the tokens as N; the fp32 h is split into two bf16 parts (hi + lo, two
// MMAs) so the operand keeps ~16 significant bits; warp w owns a 64-column
// K-slice; the 8 partial tiles are summed through shared memory and weighted
// into the CTA's accumulators.
__device__ __forceinline__ void down_mma(const DnCtx& c, const uint8_t* sa, const uint8_t* sb,
                                         int pair0, int n, bool ok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  const uint8_t* rlo = sa + g * fz::WROW + (warp * 64 + q * 8) * 2;
  const uint8_t* rhi = rlo + 8 * fz::WROW;
  using Gm = fz::Geo<false>;
  const uint8_t* hrow = g < Gm::HROWS_A ? sa + Gm::WBYTES + g * fz::THROW
                                        : sb + (g - Gm::HROWS_A) * fz::THROW;
  if (ok) {
#pragma unroll
    for (int kb = 0; kb < 2; ++kb) {
      const uint4 alo = *reinterpret_cast<const uint4*>(rlo + kb * 64);
      const uint4 ahi = *reinterpret_cast<const uint4*>(rhi + kb * 64);
      // h (fp32) = hi + lo with both parts bf16: two MMAs keep ~16 bits of h.
      uint32_t b[4] = {0u, 0u, 0u, 0u}, l[4] = {0u, 0u, 0u, 0u};
      if (g < n) {
        const int k0 = warp * 64 + kb * 32 + q * 8;
        float hv[8];
        bool bad = false;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w = *reinterpret_cast<const uint4*>(hrow + (size_t)(k0 + 2 * j) * 8);
          bad |= (w.y != c.tag) | (w.w != c.tag);
          hv[2 * j] = __uint_as_float(w.x);
          hv[2 * j + 1] = __uint_as_float(w.z);
        }
        if (bad) {
          const uint64_t* src = c.th + (size_t)(pair0 + g) * I;
#pragma unroll
          for (int j = 0; j < 8; ++j)
            hv[j] = h_settled(c, hrow, src, k0 + j);
        }
        split_bf2(hv[0], hv[1], b[0], l[0]);
        split_bf2(hv[2], hv[3], b[1], l[1]);
        split_bf2(hv[4], hv[5], b[2], l[2]);
        split_bf2(hv[6], hv[7], b[3], l[3]);
      }
      mma_bf16(acc, alo.x, ahi.x, alo.y, ahi.y, b[0], b[1]);
      mma_bf16(acc, alo.z, ahi.z, alo.w, ahi.w, b[2], b[3]);
      mma_bf16(acc, alo.x, ahi.x, alo.y, ahi.y, l[0], l[1]);
      mma_bf16(acc, alo.z, ahi.z, alo.w, ahi.w, l[2], l[3]);
    }
  }
  float* red = c.red + warp * fz::RS * GROUP_MAX;
  const int col = 2 * q;
  red[g * GROUP_MAX + col] = acc[0];
  red[g * GROUP_MAX + col + 1] = acc[1];
  red[(g + 8) * GROUP_MAX + col] = acc[2];
  red[(g + 8) * GROUP_MAX + col + 1] = acc[3];
  named_sync(1, fz::CT);
  if (ok) {
    for (int i = threadIdx.x; i < fz::RS * n; i += fz::CT) {
      const int r = i & (fz::RS - 1), j = i >> 4;
      float s = 0.f;
#pragma unroll
      for (int w = 0; w < fz::CW; ++w) s += c.red[(w * fz::RS + r) * GROUP_MAX + j];
      const int t = c.pair_tok[pair0 + j];
      const float wt = c.pair_w[pair0 + j];
      c.acc[t * fz::RS + r] += wt * s;
    }
  }
  named_sync(1, fz::CT);
}

// Down item of NVFP4 weights on CUDA cores (every group size; h rows 0..2
// beside the slice in slot A, rows 3.. in slot B).  Warp w owns rows 2w and
// 2w+1 of the 16-row slice; lane l takes columns 256hf + 8l .. +7 of each half
// hf: one code word and one block scale per row and half, dequantised once
// (exact in f16, then fp32).  The lane visits its four column pairs starting
// at pair (l >> 1) & 3 -- which makes every quarter-warp's 128-bit loads of
// tagged h words hit eight distinct bank groups -- and its code words are
// rotated by as many bytes to match.  Each token's two dot products run as
// four chains; the lane adds w(t, g) * ts times its partial sums to its own
// running sums, as the BF16 items do.
__device__ __forceinline__ void down_nv(const DnCtx& c, const uint8_t* sa, const uint8_t* sb,
                                        int pair0, int n, float ts, bool ok) {
  using Gm = fz::Geo<true>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int tok[fz::MAXB];
  float wt[fz::MAXB];
#pragma unroll
  for (int i = 0; i < fz::MAXB; ++i) {
    tok[i] = i < n ? c.pair_tok[pair0 + i] : 0;
    wt[i] = i < n ? c.pair_w[pair0 + i] * ts : 0.f;
  }
  if (!ok) return;
  const int rot = (lane >> 1) & 3;
  float f[2][2][8];  // [row][half][column pair j (visiting order), even/odd]
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int row = 2 * warp + rr;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t wv = *reinterpret_cast<const uint32_t*>(sa + row * Gm::DQROW + hf * 128 + 4 * lane);
      wv = __funnelshift_r(wv, wv, 8 * rot);
      const uint32_t sc = nvu::e4m3_bcast_f16x2(sa[Gm::WQ + row * Gm::DSFROW + 16 * hf + (lane >> 1)]);
      uint32_t pv[4];
      nvu::e2m1x8_to_f16x2(wv, pv[0], pv[1], pv[2], pv[3]);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t v = nvu::hmul2(pv[j], sc);
        const float2 fv = __half22float2(*reinterpret_cast<const __half2*>(&v));
        f[rr][hf][2 * j] = fv.x;
        f[rr][hf][2 * j + 1] = fv.y;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < fz::MAXB; ++i) {
    if (i < n) {
      const uint8_t* hrow = i < Gm::HROWS_A ? sa + Gm::WBYTES + i * fz::THROW
                                            : sb + (i - Gm::HROWS_A) * fz::THROW;
      const uint4* hr = reinterpret_cast<const uint4*>(hrow);
      float e0 = 0.f, o0 = 0.f, e1 = 0.f, o1 = 0.f;
      bool bad = false;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 hv = hr[128 * hf + 4 * lane + ((j + rot) & 3)];
          bad |= (hv.y != c.tag) | (hv.w != c.tag);
          const float h0 = __uint_as_float(hv.x), h1 = __uint_as_float(hv.z);
          e0 = fmaf(f[0][hf][2 * j], h0, e0);
          o0 = fmaf(f[0][hf][2 * j + 1], h1, o0);
          e1 = fmaf(f[1][hf][2 * j], h0, e1);
          o1 = fmaf(f[1][hf][2 * j + 1], h1, o1);
        }
      }
      if (__any_sync(0xffffffffu, bad)) {  // same sums, every value confirmed
        const uint64_t* src = c.th + (size_t)(pair0 + i) * I;
        e0 = o0 = e1 = o1 = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int k = 256 * hf + 8 * lane + 2 * ((j + rot) & 3);
            const float h0 = h_settled(c, hrow, src, k);
            const float h1 = h_settled(c, hrow, src, k + 1);
            e0 = fmaf(f[0][hf][2 * j], h0, e0);
            o0 = fmaf(f[0][hf][2 * j + 1], h1, o0);
            e1 = fmaf(f[1][hf][2 * j], h0, e1);
            o1 = fmaf(f[1][hf][2 * j + 1], h1, o1);
          }
        }
      }
      float* acc = c.lacc + (2 * tok[i]) * fz::LACC_STRIDE + threadIdx.x;
      acc[0] = fmaf(wt[i], e0 + o0, acc[0]);
      acc[fz::LACC_STRIDE] = fmaf(wt[i], e1 + o1, acc[fz::LACC_STRIDE]);
    }
  }
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

template <bool NV>
__device__ __forceinline__ bool take_slot(Prod& p, int& slot) {
  constexpr int NS = fz::Geo<NV>::NS;
  slot = p.it % NS;
  if (p.it >= NS &&
      !mbar_wait(p.empty0 + 8u * slot, (uint32_t)((p.it / NS) - 1) & 1u, p.deadline)) {
    *p.abort_flag = 1;
    set_error(p.hdr, DEV_TIMEOUT);
    return false;
  }
  if (*p.abort_flag) return false;
  ++p.it;
  return true;
}

// The END slot: armed by a plain arrive (posted even after an abort; waits
// out the drain bound for its slot).
template <bool NV>
__device__ __forceinline__ void post_end(Prod& p) {
  constexpr int NS = fz::Geo<NV>::NS;
  const int slot = p.it % NS;
  if (p.it >= NS)
    mbar_wait(p.empty0 + 8u * slot, (uint32_t)((p.it / NS) - 1) & 1u,
              p.deadline + fz::DRAIN_NS);
  ++p.it;
  Item d = {};
  d.kind = fz::IT_END;
  p.desc[slot] = d;
  mbar_arrive(p.full0 + 8u * slot);
}

// A gate/up unit (BF16: gate rows g and up rows u, 32 KiB each, in two slots;
// NVFP4: gate codes g, up codes u, gate scales gs, up scales us in one slot).
template <bool NV>
__device__ __forceinline__ bool post_gateup(Prod& p, const uint8_t* g, const uint8_t* u,
                                            const uint8_t* gs, const uint8_t* us, const Item& d) {
  using Gm = fz::Geo<NV>;
  int sa, sb;
  if (!take_slot<NV>(p, sa)) return false;
  p.desc[sa] = d;
  const uint32_t bar = p.full0 + 8u * sa, dst = p.stages_addr + sa * Gm::SLOT;
  if constexpr (NV) {
    mbar_expect_tx(bar, Gm::UNIT_BYTES);
    bulk_g2s_stream(dst, g, 8 * Gm::QROW, bar);
    bulk_g2s_stream(dst + 8 * Gm::QROW, u, 8 * Gm::QROW, bar);
    bulk_g2s_stream(dst + 16 * Gm::QROW, gs, 8 * Gm::SFROW, bar);
    bulk_g2s_stream(dst + 16 * Gm::QROW + 8 * Gm::SFROW, us, 8 * Gm::SFROW, bar);
    return true;
  } else {
    mbar_expect_tx(bar, Gm::SLOT);
    bulk_g2s_stream(dst, g, Gm::SLOT, bar);
    if (!take_slot<NV>(p, sb)) return false;  // the END posted next takes the up half's place
    Item du = d;
    du.kind = fz::IT_UP;
    p.desc[sb] = du;
    mbar_expect_tx(p.full0 + 8u * sb, Gm::SLOT);
    bulk_g2s_stream(p.stages_addr + sb * Gm::SLOT, u, Gm::SLOT, p.full0 + 8u * sb);
    return true;
  }
}

// A down item's slots: its Wd slice (issued now) and room for its tagged h
// rows (counted now, copied once the group is complete).  Returns false on
// abort; `sl` receives the slots (second -1 for items of <= 4 tokens).
// (BF16: the 16-row Wd slice wq; NVFP4: its codes wq and block scales wsf.)
template <bool NV>
__device__ __forceinline__ bool post_down_w(Prod& p, const Item& d, const uint8_t* wq,
                                            const uint8_t* wsf, int* sl) {
  using Gm = fz::Geo<NV>;
  sl[1] = -1;
  if (!take_slot<NV>(p, sl[0])) return false;
  const int na = d.n < Gm::HROWS_A ? d.n : Gm::HROWS_A;
  p.desc[sl[0]] = d;
  const uint32_t bar = p.full0 + 8u * sl[0], dst = p.stages_addr + sl[0] * Gm::SLOT;
  mbar_expect_tx(bar, Gm::WBYTES + na * fz::THROW);
  if constexpr (NV) {
    bulk_g2s_stream(dst, wq, Gm::WQ, bar);
    bulk_g2s_stream(dst + Gm::WQ, wsf, Gm::WBYTES - Gm::WQ, bar);
  } else {
    bulk_g2s_stream(dst, wq, Gm::WBYTES, bar);
  }
  if (d.n > Gm::HROWS_A) {
    if (!take_slot<NV>(p, sl[1])) return false;
    Item d2 = d;
    d2.kind = fz::IT_DOWN2;
    p.desc[sl[1]] = d2;
    mbar_expect_tx(p.full0 + 8u * sl[1], (d.n - Gm::HROWS_A) * fz::THROW);
  }
  return true;
}

template <bool NV>
__device__ __forceinline__ void post_down_h(Prod& p, const Item& d, const uint64_t* hr,
                                            const int* sl) {
  using Gm = fz::Geo<NV>;
  const int na = d.n < Gm::HROWS_A ? d.n : Gm::HROWS_A;
  bulk_g2s(p.stages_addr + sl[0] * Gm::SLOT + Gm::WBYTES, hr, na * fz::THROW,
           p.full0 + 8u * sl[0]);
  if (sl[1] >= 0)
    bulk_g2s(p.stages_addr + sl[1] * Gm::SLOT, hr + (size_t)na * I, (d.n - na) * fz::THROW,
             p.full0 + 8u * sl[1]);
}

}  // namespace

template <bool NV>
__device__ __forceinline__ void moe_small_body(ExpertArgs a, RouterArgs r) {
  using Gm = fz::Geo<NV>;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ int s_ngroups;
  __shared__ int s_ready;  // down items whose groups are complete (poll warp -> producer)
  __shared__ Item s_desc[Gm::NS];
  __shared__ int4 s_groups[fz::MAXG];
  __shared__ int s_pair_tok[fz::NPAIR];
  __shared__ float s_pair_w[fz::NPAIR];
  __shared__ float s_acc[fz::MAXB * fz::RS];  // this CTA's 16 output rows per token
  __shared__ LocalSelectSmem s_sel;
  __shared__ float s_part[2][4][8];
  __shared__ int s_ucnt[fz::UCNT];  // consumer warps done with recent units
  __shared__ int s_dslot[Gm::NS][2];  // producer: ring slots of its down items in flight
  // ring full / empty, router rows, selection done
  __shared__ __align__(8) uint64_t s_bars[2 * Gm::NS + 2];
  WsHeader* hdr = a.ws.hdr;
  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = a.B;
  uint8_t* ring = smem;
  uint16_t* xs = reinterpret_cast<uint16_t*>(smem + Gm::NS * Gm::SLOT);
  float* buf = reinterpret_cast<float*>(smem + Gm::NS * Gm::SLOT + fz::XS_BYTES);
  float* lacc = reinterpret_cast<float*>(smem + Gm::NS * Gm::SLOT + fz::XS_BYTES + fz::BUF_BYTES);
  const uint32_t full0 = smem_addr(s_bars), empty0 = smem_addr(s_bars + Gm::NS);
  const uint32_t rrow_bar = smem_addr(s_bars + 2 * Gm::NS);
  const uint32_t sel_bar = rrow_bar + 8u;
  const int e_begin = (int)((long long)cta * E / G), e_end = (int)((long long)(cta + 1) * E / G);

  if (warp == fz::PRODUCER && lane == 0) {
    for (int s = 0; s < Gm::NS; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, fz::CW);
    }
    mbar_init(rrow_bar, 1);
    mbar_init(sel_bar, 1);
    fence_mbar_init();
    // The router rows are weights: nothing the preceding kernel writes.
    const uint32_t rb = (uint32_t)(e_end - e_begin) * (H * 2);
    mbar_expect_tx(rrow_bar, rb);
    bulk_g2s_stream(smem_addr(buf), r.wr + (size_t)e_begin * H, rb, rrow_bar);
    s_abort = 0;
    s_ngroups = 0;
    s_ready = 0;
  }
  if (tid < fz::UCNT) s_ucnt[tid] = 0;
  for (int i = tid; i < fz::MAXB * fz::RS; i += blockDim.x) s_acc[i] = 0.f;
  for (int i = tid; i < fz::LACC_BYTES / 4; i += blockDim.x) lacc[i] = 0.f;
  __syncthreads();
  // Launched with programmatic serialization: the set-up above overlaps the
  // preceding kernel; x and the workspace are read only after it.
  pdl_wait();
  const uint64_t deadline = wait_deadline(hdr);
  const uint32_t epoch = __ldcg(&hdr->epoch);
  const uint32_t par = epoch & 1u, tag = call_tag(epoch);
  SyncLine* sync = hdr->sync[par];
  SyncLine* done = sync;  // completion counters: lines 0 .. SYNC_GROUPS-1
  const bool owner = cta < fz::DOWN_CTAS;
  const int r0 = cta * fz::RS;
  const int npairs = B * TOPK;

  if (warp == fz::PRODUCER) {  // ---------------- producer warp (lane 0 issues)
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
    uint32_t* claim = &sync[SYNC_UNIT].v;
    int u = (int)atomicAdd(claim, 1u);    // unit being issued
    int nxt = (int)atomicAdd(claim, 1u);  // claimed ahead
    bool meta = false, claims_open = true;
    int total = 0x7fffffff, ng = 0, ndn = 0;
    // Down items: the shared group first (its h is ready first), then the
    // routed groups in table order.  kw: items whose Wd copy is issued, kh:
    // items whose h copy is issued (kh <= kw; items in between were posted
    // ahead with only their Wd slice, once this CTA had no gate/up left).
    int kw = 0, kh = 0;
    int (*dslot)[2] = s_dslot;  // ring slots of the down items in flight
    const uint64_t* const th = a.ws.th;
    // Down item kk: the group's h rows and this CTA's slice of the expert's
    // Wd (BF16: wq; NVFP4: codes wq and block scales wsf).
    auto dn_item = [&](int kk, const uint8_t*& wq, const uint8_t*& wsf, const uint64_t*& hr) {
      const int4 grp = s_groups[kk == 0 ? ng - 1 : kk - 1];
      Item d = {};
      d.kind = fz::IT_DOWN;
      d.pair0 = grp.y;
      d.n = grp.z;
      d.expert = grp.x;
      const bool routed = grp.x < E;
      const size_t row0 = (size_t)(routed ? grp.x : grp.x - E) * H + r0;
      if constexpr (NV) {
        wq = (routed ? a.w.w2_q : a.w.ws2_q) + row0 * Gm::DQROW;
        wsf = (routed ? a.w.w2_sf : a.w.ws2_sf) + row0 * Gm::DSFROW;
      } else {
        wq = reinterpret_cast<const uint8_t*>((routed ? a.w.w2 : a.w.ws2) + row0 * I);
        wsf = nullptr;
      }
      hr = th + (size_t)grp.y * I;
      return d;
    };
    // Gate/up unit d of expert ex (E + s for shared expert s): its 8 gate and
    // 8 up rows.
    auto post_unit = [&](int ex, const Item& d) {
      const bool routed = ex < E;
      const size_t e = (size_t)(routed ? ex : ex - E);
      const size_t gr = (size_t)d.blk * 8, ur = (size_t)I + d.blk * 8;
      if constexpr (NV) {
        const uint8_t* qb = (routed ? a.w.w13_q : a.w.ws13_q) + e * (2 * I) * Gm::QROW;
        const uint8_t* sb = (routed ? a.w.w13_sf : a.w.ws13_sf) + e * (2 * I) * Gm::SFROW;
        return post_gateup<true>(p, qb + gr * Gm::QROW, qb + ur * Gm::QROW, sb + gr * Gm::SFROW,
                                 sb + ur * Gm::SFROW, d);
      } else {
        const uint16_t* base = (routed ? a.w.w13 : a.w.ws13) + e * (2 * I) * H;
        return post_gateup<false>(p, reinterpret_cast<const uint8_t*>(base + gr * H),
                                  reinterpret_cast<const uint8_t*>(base + ur * H), nullptr,
                                  nullptr, d);
      }
    };
    bool ok = true;
    int dn_budget = 0;  // ready down items still allowed before the claimed unit
    while (ok && !s_abort) {
      // Down items whose groups the poll warp has seen complete.
      const int rdy = meta && kh < ndn ? ld_acquire_cta_shared(&s_ready) : 0;
      const bool unit_pending = claims_open && (u < fz::UNITS || (meta && u < total));
      if (rdy > kh && (!unit_pending || dn_budget > 0)) {
        const uint8_t *wq, *wsf;
        const uint64_t* hr;
        const Item d = dn_item(kh, wq, wsf, hr);
        if (kh >= kw) {
          if (!(ok = post_down_w<NV>(p, d, wq, wsf, dslot[kh % Gm::NS]))) break;
          kw = kh + 1;
        }
        post_down_h<NV>(p, d, hr, dslot[kh % Gm::NS]);
        ++kh;
        --dn_budget;
        continue;
      }
      if (claims_open && u < fz::UNITS) {  // shared expert: tokens 0..B-1, pairs after the routed ones
        Item d = {};
        d.kind = fz::IT_GATE;
        d.blk = u;
        d.pair0 = npairs;
        d.n = B;
        d.tok0 = 0;
        d.done_idx = fz::DONE_SHARED;
        d.expert = E;
        ok = post_unit(E, d);
        u = nxt;
        nxt = (int)atomicAdd(claim, 1u);
        dn_budget = fz::DN_PER_UNIT;
        continue;
      }
      if (!meta) {
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
        const int ru = u - fz::UNITS;
        const int gi = ru / fz::UNITS;
        const int4 grp = s_groups[gi];
        Item d = {};
        d.kind = fz::IT_GATE;
        d.blk = ru % fz::UNITS;
        d.pair0 = grp.y;
        d.n = grp.z;
        d.tok0 = -1;
        d.done_idx = gi;
        d.expert = grp.x;
        ok = post_unit(grp.x, d);
        u = nxt;
        nxt = (int)atomicAdd(claim, 1u);
        dn_budget = fz::DN_PER_UNIT;
        continue;
      }
      claims_open = false;
      if (kh < ndn) {  // nothing left to stream but this CTA's down rows
        if (kw < ndn && kw - kh < Gm::NS - 1) {
          // post the next item's Wd slice now; its h follows once complete
          const uint8_t *wq, *wsf;
          const uint64_t* hr;
          const Item d = dn_item(kw, wq, wsf, hr);
          if (!(ok = post_down_w<NV>(p, d, wq, wsf, dslot[kw % Gm::NS]))) break;
          ++kw;
          continue;
        }
        if (globaltimer_ns() > deadline) {
          s_abort = 1;
          set_error(hdr, DEV_TIMEOUT);
          break;
        }
        __nanosleep(64);
        continue;  // wait for s_ready (shared memory)
      }
      break;
    }
    // Items posted with their Wd slice only still wait for h: on an abort,
    // complete them with the h rows as they are, so no copy stays pending.
    for (; kh < kw; ++kh) {
      const uint8_t *wq, *wsf;
      const uint64_t* hr;
      const Item d = dn_item(kh, wq, wsf, hr);
      post_down_h<NV>(p, d, hr, dslot[kh % Gm::NS]);
    }
    post_end<NV>(p);
    return;
  }

  if (warp == fz::POLL) {  // ---------------- poll warp (lane 0, row-slice owners)
    // Watches the completion counters of this CTA's down items in order (the
    // shared group first, then the routed groups), eight loads in flight at a
    // time, and publishes how many are complete.
    if (lane != 0 || !owner) return;
    while (!mbar_test(sel_bar, 0u))
      if (s_abort || globaltimer_ns() > deadline) return;
    const int ng = s_ngroups;
    int k = 0;
    while (k < ng && !s_abort) {
      uint32_t pw[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        pw[j] = k + j < ng ? ld_relaxed_u32(&done[k + j == 0 ? fz::DONE_SHARED : k + j - 1].v) : 0u;
      int rdy = 0;
      bool run = true;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        run = run && k + j < ng && pw[j] >= fz::DONE_TARGET;
        rdy += run ? 1 : 0;
      }
      if (rdy > 0) {
        k += rdy;
        st_release_cta_shared(&s_ready, k);
      } else if (globaltimer_ns() > deadline) {
        break;
      } else {
        __nanosleep(128);
      }
    }
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
        s_abort = 1;
        break;
      }
    }
    hdr->stall_armed = 0;
  }
  if (cta == 0 && tid < SYNC_LINES) {
    // The next call uses the other set of counters: clear it now (the last
    // call that used it has completed).
    hdr->sync[par ^ 1u][tid].v = 0u;
  }
  // 1. the batch's activations (all loads in flight together), then the
  //    router logits of this CTA's experts
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
  // Every word of the tagged regions carries this call's tag or the previous
  // call's: the rows this call does not use (tokens >= B) are stamped now with
  // a dead value, so a later call never meets a word older than one call.
  {
    const int gid = cta * fz::CT + tid, nthr = G * fz::CT;
    const int h_used = B * SLOTS * I, h_all = fz::MAXB * SLOTS * I;
    for (int i = h_used + gid; i < h_all; i += nthr) st_tagged(a.ws.th + i, 0.f, tag);
    for (int i = B * E + gid; i < fz::MAXB * E; i += nthr) st_tagged(a.ws.tlogits + i, 0.f, tag);
  }
  named_sync(1, fz::CT);
  if (!mbar_wait(rrow_bar, 0u, deadline)) {
    s_abort = 1;
    set_error(hdr, DEV_TIMEOUT);
  }
  router_slice(B, a.ws.tlogits, reinterpret_cast<const uint16_t*>(buf), xs, e_begin,
               e_end, s_part, tag);
  if constexpr (NV) {
    // The NVFP4 gate/up MMAs take the activations as f16 (exact for bf16
    // values inside f16's range; larger ones are reported, not clamped).
    bool big = false;
#pragma unroll
    for (int t = 0; t < fz::MAXB; ++t) {
      if (t < B) {
        uint4* v = reinterpret_cast<uint4*>(xs) + t * (H / 8) + tid;
        big |= nvu::bf16x8_beyond_f16(*v);
        *v = nvu::bf16x8_to_f16x8(*v);
      }
    }
    if (big) set_error(hdr, DEV_BAD_INPUT);
  }
  // 2. every CTA ranks and buckets the batch once all logits are in
  if (tid == 0) {
    red_add_relaxed(&sync[SYNC_ARRIVE].v, 1u);
    while (ld_relaxed_u32(&sync[SYNC_ARRIVE].v) < (uint32_t)G) {
      if (s_abort || globaltimer_ns() > deadline) {
        s_abort = 1;
        set_error(hdr, DEV_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
  }
  named_sync(1, fz::CT);
  {
    uint64_t lw[fz::MAXB];
#pragma unroll
    for (int t = 0; t < fz::MAXB; ++t) lw[t] = t < B ? ld_tagged(a.ws.tlogits + (size_t)t * E + tid) : 0u;
#pragma unroll
    for (int t = 0; t < fz::MAXB; ++t) {
      if (t < B) {
        if (!s_abort && !settle_tagged(lw[t], a.ws.tlogits + (size_t)t * E + tid, tag, deadline)) {
          s_abort = 1;
          set_error(hdr, DEV_TIMEOUT);
        }
        buf[t * E + tid] = __uint_as_float((uint32_t)lw[t]);
      }
    }
  }
  named_sync(1, fz::CT);
  if (warp < B) {
    int ix;
    float wt;
    topk_warp<false>(buf + warp * E, r.bias, r.bias_select_only != 0, ix, wt);
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
  if (cta == 0) {  // the routing tables, for the stage calls that may follow
    const int ng = s_ngroups;
    for (int i = tid; i < ng; i += fz::CT) a.ws.groups[i] = s_groups[i];
    for (int i = tid; i < B * SLOTS; i += fz::CT) {
      a.ws.pair_tok[i] = s_pair_tok[i];
      a.ws.pair_w[i] = s_pair_w[i];
    }
    if (tid == 0) hdr->n_groups = (uint32_t)ng;
  }

  DnCtx dc;
  dc.pair_tok = s_pair_tok;
  dc.pair_w = s_pair_w;
  dc.lacc = lacc;
  dc.acc = s_acc;
  dc.red = buf;
  dc.th = a.ws.th;
  dc.tag = tag;
  dc.deadline = deadline;
  dc.hdr = hdr;
  dc.abort_flag = &s_abort;

  // 3./4. the ring: gate/up units and this CTA's down items
  int it = 0, useq = 0;
  const uint64_t drain = deadline + fz::DRAIN_NS;
  while (true) {
    const int slot = it % Gm::NS;
    const uint32_t ph = (uint32_t)(it / Gm::NS) & 1u;
    if (!mbar_wait(full0 + 8u * slot, ph, deadline)) {
      s_abort = 1;
      set_error(hdr, DEV_TIMEOUT);
      if (!mbar_wait(full0 + 8u * slot, ph, drain)) break;
    }
    const Item d = s_desc[slot];
    const bool ok = !s_abort;
    if (d.kind == fz::IT_END) break;
    // both kinds may take a second slot
    const int slot2 = (it + 1) % Gm::NS;
    const uint32_t ph2 = (uint32_t)((it + 1) / Gm::NS) & 1u;
    if constexpr (NV) {
      const uint8_t* st = ring + slot * Gm::SLOT;
      const bool routed = d.expert < E;
      if (d.kind == fz::IT_DOWN) {
        const float ts = __ldg(routed ? a.w.w2_ts + d.expert : a.w.ws2_ts + (d.expert - E));
        if (d.n <= Gm::HROWS_A) {
          down_nv(dc, st, nullptr, d.pair0, d.n, ts, ok);
          release_slot(empty0 + 8u * slot);
          ++it;
          continue;
        }
        bool ok2 = ok;
        if (!mbar_wait(full0 + 8u * slot2, ph2, deadline)) {
          s_abort = 1;
          set_error(hdr, DEV_TIMEOUT);
          ok2 = false;
          if (!mbar_wait(full0 + 8u * slot2, ph2, drain)) break;
        }
        if (s_desc[slot2].kind != fz::IT_DOWN2) break;  // the producer gave up mid-item (abort)
        down_nv(dc, st, ring + slot2 * Gm::SLOT, d.pair0, d.n, ts, ok2);
        release_slot(empty0 + 8u * slot);
        release_slot(empty0 + 8u * slot2);
        it += 2;
        continue;
      }
      const float* ts13 = routed ? a.w.w13_ts + 2 * d.expert : a.w.ws13_ts + 2 * (d.expert - E);
      unit_nv(st, xs, s_pair_tok, buf, a.ws.th, d, __ldg(ts13), __ldg(ts13 + 1), ok,
              empty0 + 8u * slot, tag, done, &s_ucnt[useq]);
      useq = (useq + 1) & (fz::UCNT - 1);
      ++it;
      continue;
    }
    if (d.kind == fz::IT_DOWN) {
      const uint8_t* st = ring + slot * Gm::SLOT;
      if (d.n <= fz::CC_MAX) {
        down_cc(dc, st, d.pair0, d.n, ok, empty0 + 8u * slot);
        ++it;
        continue;
      }
      bool ok2 = ok;
      if (!mbar_wait(full0 + 8u * slot2, ph2, deadline)) {
        s_abort = 1;
        set_error(hdr, DEV_TIMEOUT);
        ok2 = false;
        if (!mbar_wait(full0 + 8u * slot2, ph2, drain)) break;
      }
      if (s_desc[slot2].kind != fz::IT_DOWN2) break;  // the producer gave up mid-item (abort)
      down_mma(dc, st, ring + slot2 * Gm::SLOT, d.pair0, d.n, ok2);
      release_slot(empty0 + 8u * slot);
      release_slot(empty0 + 8u * slot2);
      it += 2;
      continue;
    }
    // gate/up unit: gate rows in this slot, up rows in the next
    bool ok2 = ok;
    if (!mbar_wait(full0 + 8u * slot2, ph2, deadline)) {
      s_abort = 1;
      set_error(hdr, DEV_TIMEOUT);
      ok2 = false;
      if (!mbar_wait(full0 + 8u * slot2, ph2, drain)) break;
    }
    if (s_desc[slot2].kind != fz::IT_UP) break;  // the producer gave up mid-unit (abort)
    const uint8_t* gs = ring + slot * Gm::SLOT;
    const uint8_t* us = ring + slot2 * Gm::SLOT;
    if (d.n <= gu::CC_MAX) {
      int tok[2];
      tok[0] = d.tok0 >= 0 ? d.tok0 : s_pair_tok[d.pair0];
      tok[1] = d.n > 1 ? (d.tok0 >= 0 ? d.tok0 + 1 : s_pair_tok[d.pair0 + 1]) : tok[0];
      if (d.n == 1)
        unit_cc<1>(gs, us, reinterpret_cast<const uint4*>(xs), tok, a.ws.th, d, ok2,
                   empty0 + 8u * slot, empty0 + 8u * slot2, tag, done, &s_ucnt[useq]);
      else
        unit_cc<2>(gs, us, reinterpret_cast<const uint4*>(xs), tok, a.ws.th, d, ok2,
                   empty0 + 8u * slot, empty0 + 8u * slot2, tag, done, &s_ucnt[useq]);
    } else {
      unit_mma(gs, us, xs, s_pair_tok, buf, a.ws.th, d, ok2, empty0 + 8u * slot,
               empty0 + 8u * slot2, tag, done, &s_ucnt[useq]);
    }
    useq = (useq + 1) & (fz::UCNT - 1);
    it += 2;
  }
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
      a.out[o] = f2bf(bf_lo((uint32_t)a.residual[o]) + (v + s_acc[t * fz::RS + row]));
    }
  }
  // CTA 0 counts the call (also after a timeout, so that words a failed call
  // left behind never carry the next call's tag): every CTA read the counter
  // before it counted its logits in, and CTA 0 has seen all of them.
  if (cta == 0 && tid == 0) hdr->epoch = (epoch + 1u) & 0x7fffffffu;
}

__global__ void __launch_bounds__(fz::THREADS, 1) moe_small_bf16_kernel(ExpertArgs a, RouterArgs r) {
  moe_small_body<false>(a, r);
}
__global__ void __launch_bounds__(fz::THREADS, 1) moe_small_nvfp4_kernel(ExpertArgs a, RouterArgs r) {
  moe_small_body<true>(a, r);
}

bool small_supported(int num_sms) { return num_sms >= 86 && num_sms <= 1024; }

namespace {
template <bool NV>
cudaError_t launch_small(const ExpertArgs& a, const RouterArgs& r, cudaStream_t stream,
                         int num_sms) {
  static std::atomic<uint64_t> smem_set{0};
  constexpr size_t smem = fz::smem_bytes<NV>();
  void (*const kernel)(ExpertArgs, RouterArgs) = NV ? moe_small_nvfp4_kernel : moe_small_bf16_kernel;
  const cudaError_t es = set_smem_limit_once(kernel, (int)smem, smem_set);
  if (es != cudaSuccess) return es;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms, 1, 1);
  cfg.blockDim = dim3(fz::THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // One CTA per SM, all of them resident at once (the CTAs wait for each
  // other's logits and h): a cooperative launch, which the runtime refuses
  // rather than start a grid that cannot be co-resident.  Programmatic
  // serialization lets the set-up overlap the preceding kernel.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, a, r);
}
}  // namespace

cudaError_t launch_small_bf16(const ExpertArgs& a, const RouterArgs& r, cudaStream_t stream,
                              int num_sms) {
  return launch_small<false>(a, r, stream, num_sms);
}
cudaError_t launch_small_nvfp4(const ExpertArgs& a, const RouterArgs& r, cudaStream_t stream,
                               int num_sms) {
  return launch_small<true>(a, r, stream, num_sms);
}

}  // namespace flint
