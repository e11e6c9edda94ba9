// fused.cu — the whole BF16 decode MoE layer in one persistent kernel, for
// batches of at most SMALL_B (8) tokens: the pages'
// low-latency path for up to 8 requests, which fuses routing and the expert
// combine into the neighbouring GEMVs ("Low-Latency Decode Path": vLLM Day-0
// Support for Recursive's Flint, "Optimization Strategies").
//
// One CTA per SM, all co-resident (cooperative launch), 8 consumer warps + a
// producer warp + a poll warp.  The producer's lane 0 feeds a ring of
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
//      identical results in every CTA.
//   3. Work queue: every CTA claims units one at a time from one workspace
//      counter -- the shared expert's 64 gate/up units, the routed groups'
//      gate/up units in group order, then the down units of every group (the
//      shared group first) -- so CTAs that stream faster take more units.
//      A gate/up unit is 8 gate + 8 up rows of one group (two 32 KiB slots);
//      the consumer warps store h as tagged words and the last of them to
//      finish adds one to the group's completion counter (64 = the group's h
//      is complete).  A down unit is 64 Wd rows of one group's expert (two
//      slots of 32 rows) plus the group's h rows: its weights are copied as soon
//      as it is claimed, its h rows once the poll warp has seen the group
//      complete.  Every gate/up claim precedes every down claim, so no ring
//      waits on a unit queued behind it.
//   4. Each down unit writes y(p, row) = w(p) * (Wd h_p)[row] for its pairs p
//      as tagged words, each written once per call.  After its ring drains,
//      each CTA finishes its share of the output rows: out = residual + the
//      token's SLOTS y values in ascending pair order -- a fixed order, so
//      results are reproducible bit for bit whichever CTA computed what.
//
// No GPU-scope fence is taken on the data path: a fence waits for the SM's
// outstanding memory traffic, which while weights stream costs 1-3 us per
// hand-off.  Logits, h and y cross SMs as tagged words instead (call_tag),
// and the counters only say when to look.  The counters come in two sets used
// by alternate calls: a call clears the set of the next call, and CTA 0
// advances the workspace's call counter at its end, so nothing is reset at
// the exit.  Every wait is bounded by the workspace's limit.
#include "common.cuh"
#include "expert_common.cuh"
#include "gateup_impl.cuh"
#include "kernels.h"

namespace flint {
namespace fz {
constexpr int CW = 8;                          // consumer warps
constexpr int PRODUCER = CW;                   // warp index of the producer
constexpr int POLL = CW + 1;                   // warp index of the poll warp
constexpr int THREADS = (CW + 2) * 32;
constexpr int CT = CW * 32;                    // consumer threads
constexpr int ROWB = H * 2;                    // one gate/up row (bf16), 4 KiB
constexpr int MAXB = SMALL_B;
constexpr int MAXG = MAXB * TOPK + S;          // groups at these batches (one shared group)
constexpr int NPAIR = MAXB * SLOTS;
constexpr int DONE_SHARED = SYNC_GROUPS - 1;   // counter of the shared group
constexpr int WROW = I * 2;                    // one Wd row (bf16)
constexpr int THROW = I * 8;                   // one tagged h row, 4 KiB
constexpr int XS_BYTES = MAXB * H * 2;         // activations of the batch, 32 KiB
constexpr int UCNT = 8;                        // unit-completion counts in flight
constexpr int RED_BYTES = CW * 16 * GROUP_MAX * 4;
constexpr int LOGIT_BYTES = MAXB * E * 4;
constexpr int RMAX = 3;                        // router rows per CTA (grids of >= 86 CTAs)
constexpr int RROW_BYTES = RMAX * H * 2;
// router rows, then the batch's logits, then the gate/up units' partial tiles
constexpr int BUF_BYTES = RED_BYTES > LOGIT_BYTES ? (RED_BYTES > RROW_BYTES ? RED_BYTES : RROW_BYTES)
                                                  : (LOGIT_BYTES > RROW_BYTES ? LOGIT_BYTES : RROW_BYTES);
// Ring and unit layout.
struct Geo {
  static constexpr int SLOT = 32 * 1024, NS = 5;
  static constexpr int GR = 8;                              // gate/up unit: 8 gate + 8 up rows
  static constexpr int UNIT_SLOTS = 2;                      // gate rows | up rows
  static constexpr int DR = 64;                             // Wd rows per down unit
  static constexpr int DN_SLOTS = 2;                        // rows 0-31 | rows 32-63
};
constexpr int UNITS = I / Geo::GR;             // gate/up units per group
constexpr int ND = H / Geo::DR;                // down units per group
// Down units take their h rows from the activations' buffer, which the gate/up
// units no longer need by then, preceded by HDED rows of their own: a ring of
// HROWS contiguous tagged rows whose first HDED are free from the start (the
// first down units need not wait for the hand-over).
constexpr int HDED = 4;
constexpr int HDED_BYTES = HDED * THROW;
constexpr int HROWS = HDED + XS_BYTES / THROW;
// Ring row h0 + i (h0 < HROWS, i < MAXB), wrapped.
__device__ __forceinline__ int hring_row(int h0, int i) {
  const int r = h0 + i;
  return r >= HROWS ? r - HROWS : r;
}
constexpr size_t smem_bytes() {
  return (size_t)Geo::NS * Geo::SLOT + HDED_BYTES + XS_BYTES + BUF_BYTES;
}
constexpr int NQ = 8;                          // down units posted and not yet released
constexpr uint64_t DRAIN_NS = 2000000000ull;
enum : int { IT_GATE = 0, IT_UP = 1, IT_DOWN = 2, IT_DOWN2 = 3, IT_END = 4 };
static_assert(S == 1 && MAXB <= GROUP_MAX, "one shared group at these batches");
static_assert(MAXG <= DONE_SHARED, "routed groups and the shared group have distinct counters");
static_assert(DONE_SHARED < 64, "one bit per counter in a 64-bit mask");
static_assert(SYNC_LINES <= CT, "one thread clears each counter line");
static_assert(Geo::GR * ROWB == Geo::SLOT, "8 gate (or up) rows fill one slot");
static_assert(Geo::DR / 2 * WROW == Geo::SLOT, "32 Wd rows fill one slot");
static_assert(HROWS == 12 && MAXB <= HROWS, "a group's h rows fit the h ring");
static_assert(Geo::NS <= NQ, "every posted down unit has a queue entry");
static_assert(H % Geo::DR == 0, "row blocks tile H");
static_assert((E + RMAX - 1) / RMAX <= 86, "grids of 86 CTAs or more keep <= RMAX router rows");
static_assert(smem_bytes() + 6 * 1024 <= 232448, "fits the opt-in shared memory of one SM");
}  // namespace fz

namespace {

// What a ring slot holds (written by the producer before it arms the slot).
struct Item {
  int kind;
  int blk;       // gate/up: block of GR intermediate rows; down: block of DR output rows
  int pair0;     // first h row (pair) of the group
  int n;         // tokens in the group
  int tok0;      // gate/up of the shared group: first token (tokens are consecutive), else -1
  int done_idx;  // completion counter of the group
  int expert;    // expert of the group (E + s for shared expert s)
  int h0;        // down: the group's first row in the h ring
};

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

// Sums of four values over the 32 lanes of a warp in six shuffles: lane l
// ends with the sum of value ((l >> 4) & 1) * 2 + ((l >> 3) & 1).  Each lane
// keeps half of its values and adds its partner's copy of them (lanes l and
// l ^ 16, then l ^ 8), then the last three rounds add plainly.  A fixed
// pattern, so the sums are reproducible.
__device__ __forceinline__ float reduce4(float s0, float s1, float s2, float s3) {
  const int lane = threadIdx.x & 31;
  const bool up = (lane & 16) != 0, mid = (lane & 8) != 0;
  float a0 = up ? s2 : s0, a1 = up ? s3 : s1;
  const float b0 = up ? s0 : s2, b1 = up ? s1 : s3;
  a0 += __shfl_xor_sync(0xffffffffu, b0, 16);
  a1 += __shfl_xor_sync(0xffffffffu, b1, 16);
  float c = mid ? a1 : a0;
  c += __shfl_xor_sync(0xffffffffu, mid ? a0 : a1, 8);
  c += __shfl_xor_sync(0xffffffffu, c, 4);
  c += __shfl_xor_sync(0xffffffffu, c, 2);
  c += __shfl_xor_sync(0xffffffffu, c, 1);
  return c;
}

// Shared context of the down units.
struct DnCtx {
  const float* pair_w;  // shared memory
  const uint64_t* th;   // tagged h (global), for words whose tag has not landed
  uint64_t* ty;         // tagged y (global)
  uint32_t tag;
  uint64_t deadline;
  WsHeader* hdr;
  volatile int* abort_flag;
};

// Words k of a token's h row (q-th of `cnt`, columns given by col(q)) that do
// not carry the call's tag yet are confirmed from the row's global copy and
// written back into the shared copy (rare: the counters run behind the
// stores).
template <int CNT, class Col>
__device__ __forceinline__ void settle_words(const DnCtx& c, const uint8_t* hrow, const uint64_t* src,
                                             Col col) {
  uint64_t* sw = reinterpret_cast<uint64_t*>(const_cast<uint8_t*>(hrow));
#pragma unroll 1
  for (int q = 0; q < CNT; ++q) {
    const int k = col(q);
    uint64_t w = sw[k];
    if ((uint32_t)(w >> 32) != c.tag) {
      if (!settle_tagged(w, src + k, c.tag, c.deadline)) {
        *c.abort_flag = 1;
        set_error(c.hdr, DEV_TIMEOUT);
      }
      sw[k] = w;
    }
  }
}

// The down units below read token i's h row at ring row (d.h0 + i) mod
// HROWS of hb (hring_row), and write y(p, row) = w(p) * (Wd h_p)[row] as tagged
// words.
//
// BF16 down unit on CUDA cores: 64 Wd rows in two slots (rows 0-31 in sa,
// 32-63 in sb); warp w owns rows 4w .. 4w+3 of each slot; lane l takes
// columns 2l + 64m (+1), m < 8, which makes every 128-bit load of tagged h
// words conflict-free, and each h word serves all eight of the warp's rows.
// Each token's eight row sums run as sixteen chains and meet in two reduce4;
// lanes 0, 8, 16, 24 store the rows.
__device__ __forceinline__ void down_cc(const DnCtx& c, const uint8_t* sa, const uint8_t* sb,
                                        const uint8_t* hb, const Item& d, bool ok) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = d.n;
  if (!ok) return;
  const uint32_t* wa = reinterpret_cast<const uint32_t*>(sa + (4 * warp) * fz::WROW);
  const uint32_t* wb = reinterpret_cast<const uint32_t*>(sb + (4 * warp) * fz::WROW);
  uint32_t va[4][8], vb[4][8];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      va[r][m] = wa[r * (fz::WROW / 4) + lane + 32 * m];
      vb[r][m] = wb[r * (fz::WROW / 4) + lane + 32 * m];
    }
  const int row = d.blk * fz::Geo::DR + 4 * warp + (lane >> 3);
#pragma unroll
  for (int i = 0; i < fz::MAXB; ++i) {
    if (i < n) {
      const uint8_t* hrow = hb + fz::hring_row(d.h0, i) * fz::THROW;
      const uint4* hr = reinterpret_cast<const uint4*>(hrow);
      float ea[4], oa[4], eb[4], ob[4];
#pragma unroll 1
      for (int attempt = 0;; ++attempt) {
#pragma unroll
        for (int r = 0; r < 4; ++r) ea[r] = oa[r] = eb[r] = ob[r] = 0.f;
        bool bad = false;
#pragma unroll
        for (int m = 0; m < 8; ++m) {
          const uint4 hv = hr[lane + 32 * m];
          bad |= (hv.y != c.tag) | (hv.w != c.tag);
          const float h0 = __uint_as_float(hv.x), h1 = __uint_as_float(hv.z);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            ea[r] = fmaf(bf_lo(va[r][m]), h0, ea[r]);
            oa[r] = fmaf(bf_hi(va[r][m]), h1, oa[r]);
            eb[r] = fmaf(bf_lo(vb[r][m]), h0, eb[r]);
            ob[r] = fmaf(bf_hi(vb[r][m]), h1, ob[r]);
          }
        }
        if (attempt > 0 || !__any_sync(0xffffffffu, bad)) break;
        settle_words<16>(c, hrow, c.th + (size_t)(d.pair0 + i) * I,
                         [lane](int q) { return 2 * lane + 64 * (q >> 1) + (q & 1); });
        __syncwarp();
      }
      const float ya = reduce4(ea[0] + oa[0], ea[1] + oa[1], ea[2] + oa[2], ea[3] + oa[3]);
      const float yb = reduce4(eb[0] + ob[0], eb[1] + ob[1], eb[2] + ob[2], eb[3] + ob[3]);
      if ((lane & 7) == 0) {
        const float w = c.pair_w[d.pair0 + i];
        uint64_t* yp = c.ty + (size_t)(d.pair0 + i) * H + row;
        st_tagged(yp, w * ya, c.tag);
        st_tagged(yp + 32, w * yb, c.tag);
      }
    }
  }
}

// ---- producer side (lane 0 of the producer warp) -----------------------------

struct Prod {
  uint32_t full0, empty0, stages_addr;
  Item* desc;
  int it;  // ring iterations issued
};

// The next ring slot (the caller has seen it free).
__device__ __forceinline__ int next_slot(Prod& p) {
  return p.it++ % fz::Geo::NS;
}

// The END slot: armed by a plain arrive; waits out the drain bound for its
// slot (the consumers release every slot they take, also after an abort).
__device__ __forceinline__ void post_end(Prod& p, uint64_t deadline) {
  constexpr int NS = fz::Geo::NS;
  const int slot = p.it % NS;
  if (p.it >= NS)
    mbar_wait(p.empty0 + 8u * slot, (uint32_t)((p.it / NS) - 1) & 1u, deadline + fz::DRAIN_NS);
  ++p.it;
  Item d = {};
  d.kind = fz::IT_END;
  p.desc[slot] = d;
  mbar_arrive(p.full0 + 8u * slot);
}

// A gate/up unit: gate rows g and up rows u, 32 KiB each, in two slots.
__device__ __forceinline__ void post_gateup(Prod& p, const uint8_t* g, const uint8_t* u,
                                            const Item& d) {
  using Gm = fz::Geo;
  const int sa = next_slot(p);
  p.desc[sa] = d;
  const uint32_t bar = p.full0 + 8u * sa, dst = p.stages_addr + sa * Gm::SLOT;
  mbar_expect_tx(bar, Gm::SLOT);
  bulk_g2s_stream(dst, g, Gm::SLOT, bar);
  const int sb = next_slot(p);
  Item du = d;
  du.kind = fz::IT_UP;
  p.desc[sb] = du;
  mbar_expect_tx(p.full0 + 8u * sb, Gm::SLOT);
  bulk_g2s_stream(p.stages_addr + sb * Gm::SLOT, u, Gm::SLOT, p.full0 + 8u * sb);
}

// A down unit's 64 Wd rows wq, 32 per slot, copied now, and the tx count of
// its h rows, which post_down_h copies into the h ring once the group is
// complete.  Returns the slot whose barrier the h rows complete.
__device__ __forceinline__ int post_down_w(Prod& p, const Item& d, const uint8_t* wq) {
  using Gm = fz::Geo;
  const int sa = next_slot(p);
  p.desc[sa] = d;
  const uint32_t bar = p.full0 + 8u * sa, dst = p.stages_addr + sa * Gm::SLOT;
  mbar_expect_tx(bar, Gm::SLOT + d.n * fz::THROW);
  bulk_g2s_stream(dst, wq, Gm::SLOT, bar);
  const int sb = next_slot(p);
  Item d2 = d;
  d2.kind = fz::IT_DOWN2;
  p.desc[sb] = d2;
  mbar_expect_tx(p.full0 + 8u * sb, Gm::SLOT);
  bulk_g2s_stream(p.stages_addr + sb * Gm::SLOT, wq + Gm::SLOT, Gm::SLOT, p.full0 + 8u * sb);
  return sa;
}

// The group's h rows hr (tagged, n of them) into ring rows d.h0 .. (mod
// HROWS) of the h ring at hring, completing the unit's first slot.  Rows
// HDED and up lie in the activations' buffer: the caller has seen it handed
// over (h_needs_xs).
__device__ __forceinline__ bool h_needs_xs(const Item& d) {
  return d.h0 + d.n > fz::HDED;  // some row in [HDED, HROWS) (a wrap passes HDED first)
}
__device__ __forceinline__ void post_down_h(const Prod& p, const Item& d, const uint64_t* hr,
                                            uint32_t hring, int slot) {
  const int run = d.n < fz::HROWS - d.h0 ? d.n : fz::HROWS - d.h0;
  const uint32_t bar = p.full0 + 8u * slot;
  bulk_g2s(hring + d.h0 * fz::THROW, hr, run * fz::THROW, bar);
  if (run < d.n) bulk_g2s(hring, hr + (size_t)run * I, (d.n - run) * fz::THROW, bar);
}

__device__ __forceinline__ uint64_t ld_acquire_cta_shared_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.cta.shared::cta.u64 %0, [%1];" : "=l"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_cta_shared_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.cta.shared::cta.u64 [%0], %1;" ::"r"(smem_addr(p)), "l"(v) : "memory");
}

// The layer's input RMSNorm of rows 0 .. NR-1 of a batch staged as in the
// persistent kernel (consumer thread tid holds elements 8 tid .. 8 tid + 7 of
// every row; rows at or past the batch are zeros and are never stored), in
// the same arithmetic as the standalone RMSNorm kernel -- fp32 sum of squares
// in element order, warp_sum's butterfly, the 8 warp sums added in warp order,
// rsqrtf -- so x comes out bit for bit as that kernel writes it.  The rows'
// chains run side by side.
template <int NR>
__device__ __forceinline__ void input_rmsnorm(uint4 (&v)[fz::MAXB], float (*s_norm)[fz::CW],
                                              float eps, int lane, int warp) {
  float ss[NR];
#pragma unroll
  for (int t = 0; t < NR; ++t) {
    const uint4 u = v[t];
    const float f[8] = {bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y),
                        bf_lo(u.z), bf_hi(u.z), bf_lo(u.w), bf_hi(u.w)};
    ss[t] = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) ss[t] = fmaf(f[i], f[i], ss[t]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int t = 0; t < NR; ++t) ss[t] += __shfl_xor_sync(0xffffffffu, ss[t], o);
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < NR; ++t) s_norm[t][warp] = ss[t];
  }
  named_sync(1, fz::CT);
#pragma unroll
  for (int t = 0; t < NR; ++t) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < fz::CW; ++w) tot += s_norm[t][w];
    const float inv = rsqrtf(tot / (float)H + eps);
    const uint4 u = v[t];
    v[t] = make_uint4(pack_bf2(bf_lo(u.x) * inv, bf_hi(u.x) * inv),
                      pack_bf2(bf_lo(u.y) * inv, bf_hi(u.y) * inv),
                      pack_bf2(bf_lo(u.z) * inv, bf_hi(u.z) * inv),
                      pack_bf2(bf_lo(u.w) * inv, bf_hi(u.w) * inv));
  }
}

}  // namespace

// PRENORM: the rows at a.x are pre-norm activations (input_rmsnorm); a
// separate instance, so that the plain kernel's code stays as it is.
template <bool PRENORM>
__device__ __forceinline__ void moe_small_body(ExpertArgs a, RouterArgs r) {
  using Gm = fz::Geo;
  constexpr int ND = fz::ND;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ volatile int s_abort;
  __shared__ int s_ngroups;
  __shared__ uint64_t s_gmask;  // groups seen complete, by counter index (poll warp -> producer)
  __shared__ Item s_desc[Gm::NS];
  __shared__ int4 s_groups[fz::MAXG];
  __shared__ int s_pair_tok[fz::NPAIR];
  __shared__ float s_pair_w[fz::NPAIR];
  __shared__ int s_tokp[fz::MAXB][SLOTS];  // each token's pairs, ascending
  __shared__ LocalSelectSmem s_sel;
  __shared__ float s_part[2][4][8];
  __shared__ volatile int s_first_dn;  // ring iteration of this CTA's first down unit
  __shared__ int s_ucnt[fz::UCNT];     // consumer warps done with recent units
  // producer: down units posted, by post order -- the unit, the slot its h
  // rows complete, its ring iteration and the h ring's fill after it
  __shared__ Item s_pq[fz::NQ];
  __shared__ int s_pq_slot[fz::NQ], s_pq_it[fz::NQ], s_pq_hend[fz::NQ];
  // ring full / empty, router rows, selection done, activations' buffer free
  __shared__ __align__(8) uint64_t s_bars[2 * Gm::NS + 3];
  WsHeader* hdr = a.ws.hdr;
  const int G = gridDim.x, cta = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = a.B;
  uint8_t* ring = smem;
  uint8_t* hded = smem + Gm::NS * Gm::SLOT;  // h ring rows 0 .. HDED-1, then xs
  uint16_t* xs = reinterpret_cast<uint16_t*>(hded + fz::HDED_BYTES);
  float* buf = reinterpret_cast<float*>(hded + fz::HDED_BYTES + fz::XS_BYTES);
  const uint32_t full0 = smem_addr(s_bars), empty0 = smem_addr(s_bars + Gm::NS);
  const uint32_t rrow_bar = smem_addr(s_bars + 2 * Gm::NS);
  const uint32_t sel_bar = rrow_bar + 8u, xs_bar = rrow_bar + 16u;
  const int e_begin = (int)((long long)cta * E / G), e_end = (int)((long long)(cta + 1) * E / G);

  if (warp == fz::PRODUCER && lane == 0) {
    for (int s = 0; s < Gm::NS; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, fz::CW);
    }
    mbar_init(rrow_bar, 1);
    mbar_init(sel_bar, 1);
    mbar_init(xs_bar, fz::CW);
    fence_mbar_init();
    // The router rows are weights: nothing the preceding kernel writes.
    const uint32_t rb = (uint32_t)(e_end - e_begin) * (H * 2);
    mbar_expect_tx(rrow_bar, rb);
    bulk_g2s_stream(smem_addr(buf), r.wr + (size_t)e_begin * H, rb, rrow_bar);
    s_abort = 0;
    s_ngroups = 0;
    s_gmask = 0ull;
    s_first_dn = 0x7fffffff;
  }
  if (tid < fz::UCNT) s_ucnt[tid] = 0;
  __syncthreads();
  // Launched with programmatic serialization: the set-up above overlaps the
  // preceding kernel; x and the workspace are read only after it.
  pdl_wait();
  // The next kernel on the stream may launch now, its CTAs taking SMs as this
  // kernel's CTAs leave: what it does before its own wait (barrier set-up,
  // router-row copies) touches nothing this kernel uses.  -0.5 us per layer
  // chained at batch 1, -0.2 us at batch 8.
  pdl_trigger();
  const uint64_t deadline = wait_deadline(hdr);
  const uint32_t epoch = __ldcg(&hdr->epoch);
  const uint32_t par = epoch & 1u, tag = call_tag(epoch);
  SyncLine* sync = hdr->sync[par];
  SyncLine* done = sync;  // completion counters: lines 0 .. SYNC_GROUPS-1
  const int npairs = B * TOPK;

  if (warp == fz::PRODUCER) {  // ---------------- producer warp (lane 0 issues)
    if (lane != 0) return;
    Prod p;
    p.full0 = full0;
    p.empty0 = empty0;
    p.stages_addr = smem_addr(ring);
    p.desc = s_desc;
    p.it = 0;
    uint32_t* claim = &sync[SYNC_UNIT].v;
    int u = (int)atomicAdd(claim, 1u);    // unit to post next
    int nxt = (int)atomicAdd(claim, 1u);  // claimed ahead
    bool meta = false, xs_free = false;
    constexpr int UNITS = fz::UNITS;
    int ng = 0, total_gu = UNITS, total = 0x7fffffff;
    // Down units: [0, kh) have their h rows posted, [kh, kw) wait for them;
    // [0, kf) are known released (their h rows free again: hf).  hw: h rows
    // handed out.  rel: the last ring iteration known released.
    int kw = 0, kh = 0, kf = 0, hw = 0, hf = 0, rel = -1;
    const uint64_t* const th = a.ws.th;
    const uint32_t hring = smem_addr(hded);
    // true if the next `need` slots are free (the consumers release in ring
    // order: all 8 warps take every item in turn)
    auto slots_ok = [&](int need) {
      const int j = p.it + need - 1 - Gm::NS;  // the iteration that must be released
      if (j <= rel) return true;
      if (!mbar_test(empty0 + 8u * ((j + Gm::NS) % Gm::NS), (uint32_t)(j / Gm::NS) & 1u)) return false;
      rel = j;
      return true;
    };
    // retires the posted down units the consumers have released (their queue
    // entries and h rows are free again); a slot is tested only while it still
    // holds the iteration (later ones are posted only after rel passed it)
    auto reap = [&]() {
      while (kf < kw) {
        const int j = s_pq_it[kf % fz::NQ];
        if (j > rel && !mbar_test(empty0 + 8u * (j % Gm::NS), (uint32_t)(j / Gm::NS) & 1u)) break;
        hf = s_pq_hend[kf % fz::NQ];
        ++kf;
      }
    };
    while (!s_abort) {
      // 1. the oldest down unit waiting for h, once its group is complete and
      //    the consumers are done with the activations' buffer
      if (kh < kw) {
        const Item& pd = s_pq[kh % fz::NQ];
        if (!xs_free && h_needs_xs(pd)) xs_free = mbar_test(xs_bar, 0u);
        if ((xs_free || !h_needs_xs(pd)) &&
            ((ld_acquire_cta_shared_u64(&s_gmask) >> pd.done_idx) & 1ull)) {
          post_down_h(p, pd, th + (size_t)pd.pair0 * I, hring, s_pq_slot[kh % fz::NQ]);
          ++kh;
          continue;
        }
      }
      // 2. the next claimed unit, if its slots are free
      if (!meta && u >= UNITS) {  // beyond the shared expert: needs the routing
        if (!mbar_wait(sel_bar, 0u, deadline)) {
          s_abort = 1;
          set_error(hdr, DEV_TIMEOUT);
          break;
        }
        ng = s_ngroups;
        total_gu = ng * UNITS;  // the shared group's units and the routed ones
        total = total_gu + ng * ND;
        meta = true;
        continue;
      }
      bool posted = false;
      if (u < total_gu) {  // gate/up unit
        if (slots_ok(Gm::UNIT_SLOTS)) {
          Item d = {};
          d.kind = fz::IT_GATE;
          if (u < UNITS) {  // shared expert: tokens 0..B-1, pairs after the routed ones
            d.blk = u;
            d.pair0 = npairs;
            d.n = B;
            d.tok0 = 0;
            d.done_idx = fz::DONE_SHARED;
            d.expert = E;
          } else {
            const int ru = u - UNITS, gi = ru / UNITS;
            const int4 grp = s_groups[gi];
            d.blk = ru % UNITS;
            d.pair0 = grp.y;
            d.n = grp.z;
            d.tok0 = -1;
            d.done_idx = gi;
            d.expert = grp.x;
          }
          const bool routed = d.expert < E;
          const size_t e = (size_t)(routed ? d.expert : d.expert - E);
          const size_t gr = (size_t)d.blk * Gm::GR, ur = (size_t)I + d.blk * Gm::GR;
          const uint16_t* base = (routed ? a.w.w13 : a.w.ws13) + e * (2 * I) * H;
          post_gateup(p, reinterpret_cast<const uint8_t*>(base + gr * H),
                      reinterpret_cast<const uint8_t*>(base + ur * H), d);
          posted = true;
        }
      } else if (u < total) {  // down unit: group k (the shared group first), row block rb
        const int dc = u - total_gu, k = dc / ND, rb = dc % ND;
        const int4 grp = s_groups[k == 0 ? ng - 1 : k - 1];
        reap();
        if (kw - kf < fz::NQ && hw + grp.z - hf <= fz::HROWS && slots_ok(Gm::DN_SLOTS)) {
          Item d = {};
          d.kind = fz::IT_DOWN;
          d.blk = rb;
          d.pair0 = grp.y;
          d.n = grp.z;
          d.tok0 = -1;
          d.done_idx = k == 0 ? fz::DONE_SHARED : k - 1;
          d.expert = grp.x;
          d.h0 = hw % fz::HROWS;
          hw += grp.z;
          const bool routed = grp.x < E;
          const size_t row0 = (size_t)(routed ? grp.x : grp.x - E) * H + (size_t)rb * Gm::DR;
          const uint8_t* wq =
              reinterpret_cast<const uint8_t*>((routed ? a.w.w2 : a.w.ws2) + row0 * I);
          const int q = kw % fz::NQ;
          if (kw == 0) s_first_dn = p.it;  // from here on the consumers release xs
          s_pq[q] = d;
          s_pq_it[q] = p.it;
          s_pq_hend[q] = hw;
          s_pq_slot[q] = post_down_w(p, d, wq);
          ++kw;
          posted = true;
        }
      } else if (kh == kw) {
        break;  // every claimed unit is posted
      }
      if (posted) {
        u = nxt;
        nxt = (int)atomicAdd(claim, 1u);
        continue;
      }
      if (globaltimer_ns() > deadline) {
        s_abort = 1;
        set_error(hdr, DEV_TIMEOUT);
        break;
      }
      __nanosleep(32);
    }
    // Down units still waiting for h: on an abort, copy their h rows as they
    // are, so that no slot waits for bytes that never come.
    for (; kh < kw; ++kh)
      post_down_h(p, s_pq[kh % fz::NQ], th + (size_t)s_pq[kh % fz::NQ].pair0 * I, hring,
                  s_pq_slot[kh % fz::NQ]);
    post_end(p, deadline);
    return;
  }

  if (warp == fz::POLL) {  // ---------------- poll warp
    // Watches the completion counters of all groups (lane l: counters l and
    // l + 32) and publishes the set seen complete.  Every decision is taken
    // warp-wide (the ballots need all 32 lanes).
    while (!__any_sync(0xffffffffu, mbar_test(sel_bar, 0u)))
      if (__any_sync(0xffffffffu, s_abort || globaltimer_ns() > deadline)) return;
    const int ng = s_ngroups;
    const uint64_t want = ((1ull << (ng - 1)) - 1ull) | (1ull << fz::DONE_SHARED);
    const bool w_lo = (want >> lane) & 1ull, w_hi = (want >> (lane + 32)) & 1ull;
    bool d_lo = false, d_hi = false;
    uint64_t have = 0ull;
    while (have != want && !__any_sync(0xffffffffu, s_abort)) {
      const uint32_t c_lo = w_lo && !d_lo ? ld_relaxed_u32(&done[lane].v) : 0u;
      const uint32_t c_hi = w_hi && !d_hi ? ld_relaxed_u32(&done[lane + 32].v) : 0u;
      d_lo = d_lo || (w_lo && c_lo >= (uint32_t)fz::UNITS);
      d_hi = d_hi || (w_hi && c_hi >= (uint32_t)fz::UNITS);
      const uint64_t m = (uint64_t)__ballot_sync(0xffffffffu, d_lo) |
                         ((uint64_t)__ballot_sync(0xffffffffu, d_hi) << 32);
      if (m != have) {
        have = m;
        if (lane == 0) st_release_cta_shared_u64(&s_gmask, m);
      } else if (__any_sync(0xffffffffu, globaltimer_ns() > deadline)) {
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
    if constexpr (PRENORM) {
      __shared__ float s_norm[fz::MAXB][fz::CW];
      static_assert(PRENORM_FUSED_MAX_B <= fz::MAXB, "rows in registers");
      if (B == 1)
        input_rmsnorm<1>(v, s_norm, a.norm_eps, lane, warp);
      else
        input_rmsnorm<PRENORM_FUSED_MAX_B>(v, s_norm, a.norm_eps, lane, warp);
    }
#pragma unroll
    for (int t = 0; t < fz::MAXB; ++t)
      if (t < B) reinterpret_cast<uint4*>(xs)[t * (H / 8) + tid] = v[t];
  }
  // Every word of the tagged regions carries a recent call's tag: the rows
  // this call does not use (tokens >= B) are stamped with a dead value -- h
  // and logits every call, y one sixteenth of its rows per call -- so a later
  // call never meets a word old enough for its tag to come round again.
  {
    const int gid = cta * fz::CT + tid, nthr = G * fz::CT;
    const int h_used = B * SLOTS * I, h_all = fz::MAXB * SLOTS * I;
    for (int i = h_used + gid; i < h_all; i += nthr) st_tagged(a.ws.th + i, 0.f, tag);
    for (int i = B * E + gid; i < fz::MAXB * E; i += nthr) st_tagged(a.ws.tlogits + i, 0.f, tag);
    constexpr int YCH = H / 16;
    const int y0 = (int)(epoch & 15u) * YCH;
    for (int i = gid; i < (fz::MAXB - B) * SLOTS * YCH; i += nthr)
      st_tagged(a.ws.ty + (size_t)(B * SLOTS + i / YCH) * H + y0 + i % YCH, 0.f, tag);
  }
  named_sync(1, fz::CT);
  if (!mbar_wait(rrow_bar, 0u, deadline)) {
    s_abort = 1;
    set_error(hdr, DEV_TIMEOUT);
  }
  router_slice(B, a.ws.tlogits, reinterpret_cast<const uint16_t*>(buf), xs, e_begin,
               e_end, s_part, tag);
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
  dc.pair_w = s_pair_w;
  dc.th = a.ws.th;
  dc.ty = a.ws.ty;
  dc.tag = tag;
  dc.deadline = deadline;
  dc.hdr = hdr;
  dc.abort_flag = &s_abort;

  // 3. the ring: every consumer warp takes every item in ring order (gate/up
  //    units, then down units, then the END)
  int it = 0, useq = 0;
  bool xs_done = false;  // this warp has handed the activations' buffer over
  const uint64_t drain = deadline + fz::DRAIN_NS;
  const uint8_t* hb = hded;
  // Waits (warp-wide decision) for ring iteration j; false: give up the loop.
  auto wait_it = [&](int j) -> bool {
    const int slot = j % Gm::NS;
    const uint32_t ph = (uint32_t)(j / Gm::NS) & 1u;
    bool got;
    while (true) {
      // Every item from the first down unit on is a down unit (or the END):
      // this warp no longer reads the activations, and their buffer becomes
      // the h ring once every warp has said so.
      if (!xs_done && j >= s_first_dn) {
        xs_done = true;
        if (lane == 0) mbar_arrive(xs_bar);
      }
      if ((got = mbar_try_wait(full0 + 8u * slot, ph))) break;
      if (globaltimer_ns() > deadline) break;
    }
    if (__all_sync(0xffffffffu, got)) return true;
    s_abort = 1;
    set_error(hdr, DEV_TIMEOUT);
    return __all_sync(0xffffffffu, mbar_wait(full0 + 8u * slot, ph, drain));
  };
  while (true) {
    const int slot = it % Gm::NS;
    if (!wait_it(it)) break;
    const Item d = s_desc[slot];
    const bool ok = !s_abort;
    if (d.kind == fz::IT_END) break;
    const uint8_t* st = ring + slot * Gm::SLOT;
    // every unit takes two slots
    const int slot2 = (it + 1) % Gm::NS;
    if (!wait_it(it + 1)) break;
    const int k2 = s_desc[slot2].kind;
    if (k2 != (d.kind == fz::IT_DOWN ? fz::IT_DOWN2 : fz::IT_UP)) break;  // producer gave up (abort)
    const uint8_t* st2 = ring + slot2 * Gm::SLOT;
    const bool ok2 = !s_abort;
    if (d.kind == fz::IT_DOWN) {
      down_cc(dc, st, st2, hb, d, ok2);
      release_slot(empty0 + 8u * slot);
      release_slot(empty0 + 8u * slot2);
    } else {
      if (d.n <= gu::CC_MAX) {
        int tok[2];
        tok[0] = d.tok0 >= 0 ? d.tok0 : s_pair_tok[d.pair0];
        tok[1] = d.n > 1 ? (d.tok0 >= 0 ? d.tok0 + 1 : s_pair_tok[d.pair0 + 1]) : tok[0];
        if (d.n == 1)
          unit_cc<1>(st, st2, reinterpret_cast<const uint4*>(xs), tok, a.ws.th, d, ok2,
                     empty0 + 8u * slot, empty0 + 8u * slot2, tag, done, &s_ucnt[useq]);
        else
          unit_cc<2>(st, st2, reinterpret_cast<const uint4*>(xs), tok, a.ws.th, d, ok2,
                     empty0 + 8u * slot, empty0 + 8u * slot2, tag, done, &s_ucnt[useq]);
      } else {
        unit_mma(st, st2, xs, s_pair_tok, buf, a.ws.th, d, ok2, empty0 + 8u * slot,
                 empty0 + 8u * slot2, tag, done, &s_ucnt[useq]);
      }
      useq = (useq + 1) & (fz::UCNT - 1);
    }
    it += 2;
    (void)ok;
  }
  named_sync(1, fz::CT);
  // 4. this CTA's output rows: residual + the token's SLOTS y values in
  //    ascending pair order.  Warp t lists token t's pairs first (ballots).
  if (warp < B) {
    int cnt = 0;
    for (int base = 0; base < B * SLOTS; base += 32) {
      const int pr = base + lane;
      const bool mine = pr < B * SLOTS && s_pair_tok[pr] == warp;
      const uint32_t m = __ballot_sync(0xffffffffu, mine);
      const int k = cnt + __popc(m & ((1u << lane) - 1u));
      if (mine && k < SLOTS) s_tokp[warp][k] = pr;
      cnt += __popc(m);
    }
    if (cnt != SLOTS) {  // every token has SLOTS pairs; without them nothing is combined
      if (lane == 0) set_error(hdr, DEV_BAD_ROUTING);
      s_abort = 1;
    }
  }
  named_sync(1, fz::CT);
  if (!s_abort) {
    const int row_b = (int)((long long)cta * H / G), nr = (int)((long long)(cta + 1) * H / G) - row_b;
    for (int i = tid; i < B * nr; i += fz::CT) {
      const int t = i / nr, row = row_b + i % nr;
      uint64_t yw[SLOTS];
#pragma unroll
      for (int k = 0; k < SLOTS; ++k) yw[k] = ld_tagged(a.ws.ty + (size_t)s_tokp[t][k] * H + row);
      float v = 0.f;
#pragma unroll
      for (int k = 0; k < SLOTS; ++k) {
        const uint64_t* src = a.ws.ty + (size_t)s_tokp[t][k] * H + row;
        while ((uint32_t)(yw[k] >> 32) != tag) {  // not yet written: poll, bounded
          if (s_abort || globaltimer_ns() > deadline) {
            s_abort = 1;
            set_error(hdr, DEV_TIMEOUT);
            break;
          }
          __nanosleep(64);
          yw[k] = ld_tagged(src);
        }
        v += __uint_as_float((uint32_t)yw[k]);
      }
      const size_t o = (size_t)t * H + row;
      if (!s_abort) a.out[o] = f2bf(bf_lo((uint32_t)a.residual[o]) + v);
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
__global__ void __launch_bounds__(fz::THREADS, 1)
    moe_small_bf16_prenorm_kernel(ExpertArgs a, RouterArgs r) {
  moe_small_body<true>(a, r);
}

bool small_supported(int num_sms) { return num_sms >= 86 && num_sms <= 1024; }

namespace {
template <bool PRENORM>
cudaError_t launch_small(const ExpertArgs& a, const RouterArgs& r, cudaStream_t stream,
                         int num_sms) {
  static std::atomic<uint64_t> smem_set{0};
  constexpr size_t smem = fz::smem_bytes();
  void (*const kernel)(ExpertArgs, RouterArgs) =
      PRENORM ? moe_small_bf16_prenorm_kernel : moe_small_bf16_kernel;
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
  return a.prenorm ? launch_small<true>(a, r, stream, num_sms)
                   : launch_small<false>(a, r, stream, num_sms);
}

}  // namespace flint
