// down_ring.cuh — the large-batch down GEMV + routing-weighted combine +
// shared-expert add + residual add, as a template over the weight format
// (instantiated for BF16 weights in down.cu).
//
//   out[t] = residual[t] + sum over groups g containing t of
//            w(t, g) * Wd_{expert(g)} h[pair(t, g)]
// where shared-expert groups carry weight 1 (the expert combine sits in the
// down GEMV, as on the pages' low-latency decode path: vLLM Day-0 Support for
// Recursive's Flint, "Optimization Strategies").
//
// Row-slice-major: CTA b owns output rows [16b, 16b+16) of every token and
// walks all groups in order, so each weight byte is read by exactly one CTA
// and the combine needs no atomics.  Per group a producer lane copies the
// CTA's 16-row slice of the group's Wd (the format decides how) and the
// group's h rows (one bulk copy; the gate/up kernel stores them split into hi
// + lo parts and already swizzled by row) into a byte ring in shared memory:
// each group takes only the bytes it needs, so many groups are in flight per
// SM.  Two producer warps take alternate groups, each into its own half of
// the ring.
//
// Warp pair p (of 4) takes groups p, p + 4, p + 8, ...: mma.sync m16n8k16
// with the 16 Wd rows as M, the group's tokens as N (8 per tile) and K split
// between the pair's two warps (256 columns each); the hi and lo parts of h
// each take one MMA, so the operand keeps the fp32 h to ~16 significant bits
// (bf16 parts).  The odd warp hands its partial tiles to the even
// one through shared memory; the even warp applies the routing weights into
// the pair's own accumulator rows.  The four pairs work on four groups at once
// and never wait for each other; the four partial sums are added in a fixed
// order when the output is written, so results are bitwise reproducible.
//
// A weight format F provides: WBYTES (ring bytes of a group's weights,
// including the hand-over area at XCH), WCOPY (bytes its copies bring), NDESC,
// Maps (kernel parameter), issue() (the weight copies), Frag / load() / a()
// (the A fragment of step kk of a K half: block b(q, kk) of rows gq, gq + 8 as
// 8 halves each), mma() and scale() (a per-expert factor on the sums).  At
// step kk of K half kh every lane reads line 8 kh + kk of its h rows, so the
// h writer must place block b(q, kk) there (chunk pair q).
#pragma once

#include <cuda.h>  // CUtensorMap and its enums

#include "common.cuh"
#include "expert_common.cuh"
#include "kernels.h"

namespace flint {
namespace dring {

constexpr int RS = 16;                  // output rows per CTA
constexpr int HROW = I * 4;             // bytes of one split h row
constexpr int PAIRS = 4;                // consumer warp pairs; a pair takes one group at a time
constexpr int CW = 2 * PAIRS;           // consumer warps
constexpr int NPROD = 2;                // producer warps, each filling its own part of the ring
constexpr int PRODUCER = CW;            // first producer warp
constexpr int THREADS = (CW + NPROD) * 32;
constexpr int SMEM_CAP = 232448 - 1024; // opt-in maximum minus static/slack
constexpr int ALIGN = 1024;             // swizzled tensor copies land on 1 KiB boundaries
constexpr uint64_t DRAIN_NS = 2000000000ull;
static_assert(HROW % ALIGN == 0, "groups stay aligned in the ring");

// Groups the bucketing can form for a batch of B: per routed expert one per
// GROUP_MAX of its tokens, and the same for the shared expert(s).
__host__ __device__ inline int group_cap(int B) {
  const int routed = (TOPK * B + GROUP_MAX - 1) / GROUP_MAX + (TOPK * B < E ? TOPK * B : E);
  const int cap = routed + S * ((B + GROUP_MAX - 1) / GROUP_MAX);
  return cap < MAX_GROUPS ? cap : MAX_GROUPS;
}

template <class F>
struct Layout {
  // Every group's bytes are a multiple of ALIGN, so every group starts aligned.
  static_assert(F::WBYTES % ALIGN == 0, "groups stay aligned in the ring");
  static_assert(F::NDESC % PAIRS == 0, "descriptor reuse stays within one pair");
  static_assert(((GROUP_MAX + 7) / 8) * 4 * 32 * 4 + F::XCH <= F::WBYTES, "hand-over fits");
  __host__ __device__ static constexpr int group_bytes(int n) { return F::WBYTES + n * HROW; }
  // Shared memory after the ring: accumulators [PAIRS][B][RS] fp32, the group
  // table, the pairs' tokens and weights, the mbarriers.
  __host__ __device__ static int fixed_bytes(int B) {
    return PAIRS * B * RS * 4 + group_cap(B) * 16 + 2 * B * SLOTS * 4 + 2 * F::NDESC * 8;
  }
  __host__ __device__ static int ring_bytes(int B) {
    return ((SMEM_CAP - ALIGN - fixed_bytes(B)) / ALIGN) * ALIGN;
  }
  // Each producer's part of the ring.
  __host__ __device__ static int part_bytes(int B) { return (ring_bytes(B) / NPROD / ALIGN) * ALIGN; }
  __host__ static int smem_bytes(int B) { return ALIGN + ring_bytes(B) + fixed_bytes(B); }
  static_assert(MAX_B * RS * 4 * PAIRS + MAX_GROUPS * 16 + 2 * MAX_B * SLOTS * 4 +
                        2 * F::NDESC * 8 + ALIGN + NPROD * (F::WBYTES + GROUP_MAX * HROW + ALIGN) <=
                    SMEM_CAP,
                "each part of the ring holds the largest group at the largest batch");
  static_assert(F::NDESC % NPROD == 0 && PAIRS % NPROD == 0, "a pair's groups come from one producer");
};

struct DnMeta {
  const int4* groups;
  const int* pair_tok;
  const float* pair_w;
  int n_groups;
};

// 3-D tensor copy of weight bytes (L2 evict-first, like bulk_g2s_stream).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(l2_evict_first())
      : "memory");
}

// Position of each group in the ring, both as a monotonic byte count (for
// the free-space test) and as the offset in the ring.  A group never
// straddles the ring's end: if it would, it starts at the next wrap instead.
struct RingPos {
  uint32_t mono = 0, off = 0;
  uint32_t ring;
  __device__ explicit RingPos(uint32_t r) : ring(r) {}
  // Returns the group's ring offset; `start` gets its monotonic position.
  __device__ __forceinline__ uint32_t place(uint32_t need, uint32_t& start) {
    if (off + need > ring) {
      mono += ring - off;
      off = 0;
    }
    start = mono;
    const uint32_t o = off;
    mono += need;
    off += need;
    return o;
  }
};

template <int NDESC>
struct Ring {
  uint8_t* base;
  uint32_t base_addr, ring;
  uint32_t full0, empty0;
  __device__ uint32_t full(int g) const { return full0 + 8u * (uint32_t)(g % NDESC); }
  __device__ uint32_t empty(int g) const { return empty0 + 8u * (uint32_t)(g % NDESC); }
  __device__ static uint32_t parity(int g) { return (uint32_t)(g / NDESC) & 1u; }
};

// One lane of producer warp k (of NPROD): groups g = k, k + NPROD, ... into
// its own part [k * part, (k + 1) * part) of the ring.  Each producer's issue
// path (bookkeeping, then copy instructions that can stall until the SM's copy
// unit takes them) then overlaps the other's.  Group g is issued once its
// bytes and its mbarrier pair are free: the producer waits for its oldest
// unreleased groups, in issue order, until both hold.  It publishes the
// group's ring offset in goff[g % NDESC] before the arrival on the group's
// full barrier, so a consumer that has seen the barrier complete reads it
// there.
template <class F>
__device__ void produce(const Ring<F::NDESC>& R, const DnMeta& meta,
                        const typename F::Maps& maps, const ExpertArgs& a, int r0, int k,
                        uint32_t part, uint32_t* goff, volatile int* abort_flag,
                        uint64_t deadline) {
  constexpr int NDESC = F::NDESC;
  constexpr int WIN = NDESC / NPROD;  // groups of one producer in flight
  using RingT = Ring<NDESC>;
  WsHeader* hdr = a.ws.hdr;
  const int n_groups = meta.n_groups;
  const uint32_t base = (uint32_t)k * part;
  RingPos pos(part);
  uint32_t released = 0;  // position in the part up to which every byte is free again
  int rel = k;            // this producer's groups below rel are released
  // Part ends of the outstanding groups rel, rel + NPROD, ... in registers (a
  // shift register: every access is a static index), so that the wait loop's
  // chain has no shared-memory round trip besides the barrier test.
  uint32_t ends[WIN];
#pragma unroll
  for (int i = 0; i < WIN; ++i) ends[i] = 0;
  // The next descriptor is loaded one iteration ahead.
  int4 grp = k < n_groups ? meta.groups[k] : make_int4(0, 0, 0, 0);
  int g = k;
  for (; g < n_groups; g += NPROD) {
    const int4 cur = grp;
    if (g + NPROD < n_groups) grp = meta.groups[g + NPROD];
    const uint32_t need = (uint32_t)Layout<F>::group_bytes(cur.z);
    uint32_t start;
    const uint32_t off = pos.place(need, start);
    bool ok = true;
    while (rel < g && (g - rel >= NDESC || start + need - released > part)) {
      if (!mbar_wait(R.empty(rel), RingT::parity(rel), deadline)) {
        if (!*abort_flag) set_error(hdr, DEV_TIMEOUT);
        *abort_flag = 1;
        ok = false;
        break;
      }
      released = ends[0];
#pragma unroll
      for (int i = 0; i + 1 < WIN; ++i) ends[i] = ends[i + 1];
      rel += NPROD;
    }
    if (!ok || ((g / NPROD) % 16 == 0 && *abort_flag)) break;
    const int slot = (g - rel) / NPROD;  // < WIN
#pragma unroll
    for (int i = 0; i < WIN; ++i)
      if (i == slot) ends[i] = start + need;
    const uint32_t dst = R.base_addr + base + off;
    goff[g % NDESC] = base + off;
    mbar_expect_tx(R.full(g), (uint32_t)(F::WCOPY + cur.z * HROW));
    F::issue(maps, a, dst, cur, r0, R.full(g));
    bulk_g2s(dst + F::WBYTES, a.ws.h + (size_t)cur.y * I, cur.z * HROW, R.full(g));
  }
  // No copy may still be landing in shared memory when the CTA exits.
  const uint64_t drain = globaltimer_ns() + DRAIN_NS;
  for (int j = rel; j < g; j += NPROD) mbar_wait(R.full(j), RingT::parity(j), drain);
}

// Barrier over one warp pair (64 threads, barrier id) that also ANDs a flag
// across it: both warps always arrive, so neither can be left waiting.
__device__ __forceinline__ bool pair_sync_and(uint32_t id, bool v) {
  uint32_t r;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; bar.red.and.pred q, %2, 64, p; selp.u32 %0, 1, 0, q; }"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id)
      : "memory");
  return r != 0;
}

// One warp, half the K columns of one group of n <= 8 * NT tokens:
// d[nt] = Wd_slice[:, K half] * h[tokens, K half]^T for token tile nt.
// Lane (gq = lane / 4, q = lane % 4) holds Wd rows gq and gq + 8 and, at step
// kk, the 8 K columns of the format's block b(q, kk); h is read with the same
// K relabeling, so the products pair up as in the plain dot product.  The h
// rows sit in shared memory with 16-byte chunks XOR-permuted by the pair
// index mod 8, so each 8-lane phase of a 128-bit load touches 8 distinct
// banks.  hi and lo, and the two halves of each step, go to four independent
// accumulators so the MMA chains overlap; with one token tile, even and odd
// steps take separate sets as well (eight chains of four MMAs).
// d element e: (row, token column) = (gq, 2q), (gq, 2q+1), (gq+8, 2q), (gq+8, 2q+1).
template <class F, int NT>
__device__ __forceinline__ void group_half(const uint8_t* st, int n, int pair0, int khalf,
                                           float (&d)[NT][4]) {
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, q = lane & 3;
  constexpr int CH = NT == 1 ? 2 : 1;  // accumulator sets, taken by step kk % CH
  float acc[NT][CH][4][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int h = 0; h < CH; ++h)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        acc[nt][h][c][0] = acc[nt][h][c][1] = acc[nt][h][c][2] = acc[nt][h][c][3] = 0.f;
  typename F::Frag fr;
  F::load(st, gq, q, khalf, fr);
  // Token columns past n read token 0's row: their results are never used,
  // and the loads need no branch.
  const uint8_t* hrow[NT];
  int hx[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int slot = nt * 8 + gq < n ? nt * 8 + gq : 0;
    hrow[nt] = st + F::WBYTES + slot * HROW;
    hx[nt] = (pair0 + slot) & 7;
  }
#pragma unroll
  for (int kk = 0; kk < I / 64; ++kk) {
    const int kc = khalf * (I / 64) + kk;
    uint4 alo, ahi;
    F::a(st, fr, gq, q, khalf, kk, alo, ahi);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // hi and lo chunks of the same block (line kc of the row, chunk pair q)
      const uint8_t* hl = hrow[nt] + kc * 128;
      const uint4 b = *reinterpret_cast<const uint4*>(hl + (((2 * q) ^ hx[nt]) * 16));
      const uint4 l = *reinterpret_cast<const uint4*>(hl + (((2 * q + 1) ^ hx[nt]) * 16));
      float(&ac)[4][4] = acc[nt][kk % CH];
      F::mma(ac[0], alo.x, ahi.x, alo.y, ahi.y, b.x, b.y);
      F::mma(ac[1], alo.z, ahi.z, alo.w, ahi.w, b.z, b.w);
      F::mma(ac[2], alo.x, ahi.x, alo.y, ahi.y, l.x, l.y);
      F::mma(ac[3], alo.z, ahi.z, alo.w, ahi.w, l.z, l.w);
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = (acc[nt][0][0][e] + acc[nt][0][1][e]) + (acc[nt][0][2][e] + acc[nt][0][3][e]);
#pragma unroll
      for (int h = 1; h < CH; ++h)
        v += (acc[nt][h][0][e] + acc[nt][h][1][e]) + (acc[nt][h][2][e] + acc[nt][h][3][e]);
      d[nt][e] = v;
    }
}

// One group on one warp pair.  The odd warp hands its K-half tiles to the
// even warp in the format's hand-over area (bytes only the odd warp reads, or
// none); after the pair barrier the even warp adds them and applies the
// routing weight (times the format's per-expert scale) to the pair's
// accumulator rows.  Returns false (on both warps) if either warp's data wait
// failed.
template <class F, int NT>
__device__ __forceinline__ bool group_pair(uint8_t* st, bool ok, int n, int pair0, int khalf,
                                           uint32_t bar_id, float scale, float* acc_rows,
                                           const int* pair_tok, const float* pair_w) {
  const int lane = threadIdx.x & 31;
  const int gq = lane >> 2, q = lane & 3;
  float* xch = reinterpret_cast<float*>(st + F::XCH);
  float d[NT][4];
  if (ok) {
    group_half<F, NT>(st, n, pair0, khalf, d);
    if (khalf == 1) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) xch[(nt * 4 + e) * 32 + lane] = d[nt][e];
    }
  }
  if (!pair_sync_and(bar_id, ok)) return false;
  if (khalf == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) d[nt][e] += xch[(nt * 4 + e) * 32 + lane];
      // A group holds each token once, so the lanes' targets are distinct.
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int col = nt * 8 + 2 * q + e;
        if (col < n) {
          const int t = pair_tok[pair0 + col];
          const float wt = pair_w[pair0 + col] * scale;
          acc_rows[t * RS + gq] += wt * d[nt][e];
          acc_rows[t * RS + gq + 8] += wt * d[nt][2 + e];
        }
      }
    }
  }
  return true;
}

template <class F>
__global__ void __launch_bounds__(THREADS, 1)
    down_ring_kernel(ExpertArgs a, const __grid_constant__ typename F::Maps maps) {
  constexpr int NDESC = F::NDESC;
  using L = Layout<F>;
  using RingT = Ring<NDESC>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ int s_ngroups;
  __shared__ uint32_t s_goff[NDESC];  // ring offset of group g at g % NDESC
  volatile int* abort_flag = &s_abort;
  const int B = a.B;
  const uint32_t ring = (uint32_t)L::ring_bytes(B);
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + ALIGN - 1) & ~uint32_t(ALIGN - 1)) - raw_addr);
  float* accw = reinterpret_cast<float*>(smem + ring);  // [PAIRS][B][RS]
  const int gcap = group_cap(B);
  int4* groups_s = reinterpret_cast<int4*>(accw + PAIRS * B * RS);
  int* pair_tok_s = reinterpret_cast<int*>(groups_s + gcap);
  float* pair_w_s = reinterpret_cast<float*>(pair_tok_s + B * SLOTS);
  uint64_t* bars = reinterpret_cast<uint64_t*>(pair_w_s + B * SLOTS);
  RingT R;
  R.base = smem;
  R.base_addr = smem_addr(smem);
  R.ring = ring;
  R.full0 = smem_addr(bars);
  R.empty0 = smem_addr(bars + NDESC);
  if (threadIdx.x == 0) {
    for (int s = 0; s < NDESC; ++s) {
      mbar_init(R.full0 + 8u * s, 1);
      mbar_init(R.empty0 + 8u * s, 1);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  for (int i = threadIdx.x; i < PAIRS * B * RS; i += blockDim.x) accw[i] = 0.f;
  __syncthreads();
  const int r0 = blockIdx.x * RS;
  const uint64_t deadline = wait_deadline(a.ws.hdr);
  pdl_wait();  // h, the group table and the pairs come from the preceding kernels
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  DnMeta meta;
  meta.groups = groups_s;
  meta.pair_tok = pair_tok_s;
  meta.pair_w = pair_w_s;
  if (warp >= PRODUCER) {
    named_sync(2, THREADS);  // routing metadata is in shared memory
    meta.n_groups = s_ngroups;
    if (lane == 0)
      produce<F>(R, meta, maps, a, r0, warp - PRODUCER, (uint32_t)L::part_bytes(B), s_goff,
                 abort_flag, deadline);
    return;
  }
  // Routing metadata into shared memory: all loads first, then the stores,
  // so the round trips overlap.
  {
    constexpr int CT = CW * 32;
    constexpr int GR = (MAX_GROUPS + CT - 1) / CT;
    constexpr int PR = (MAX_B * SLOTS + CT - 1) / CT;
    int n = (int)__ldcg(&a.ws.hdr->n_groups);
    if (n > gcap) {  // more groups than the bucketing can form: inconsistent routing
      if (threadIdx.x == 0) set_error(a.ws.hdr, DEV_BAD_ROUTING);
      n = 0;
      *abort_flag = 1;
    }
    int4 gv[GR];
    int tv[PR];
    float wv[PR];
#pragma unroll
    for (int k = 0; k < GR; ++k) {
      const int i = threadIdx.x + k * CT;
      gv[k] = i < n ? __ldcg(a.ws.groups + i) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < PR; ++k) {
      const int i = threadIdx.x + k * CT;
      const bool in = i < B * SLOTS;
      tv[k] = in ? __ldcg(a.ws.pair_tok + i) : 0;
      wv[k] = in ? __ldcg(a.ws.pair_w + i) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < GR; ++k) {
      const int i = threadIdx.x + k * CT;
      if (i < n) groups_s[i] = gv[k];
    }
#pragma unroll
    for (int k = 0; k < PR; ++k) {
      const int i = threadIdx.x + k * CT;
      if (i < B * SLOTS) {
        pair_tok_s[i] = tv[k];
        pair_w_s[i] = wv[k];
      }
    }
    if (threadIdx.x == 0) s_ngroups = n;
  }
  pdl_trigger();
  named_sync(2, THREADS);
  const int n_groups = s_ngroups;
  const int pair = warp >> 1, khalf = warp & 1;
  float* my_acc = accw + pair * B * RS;
  const uint32_t bar_id = 3 + pair;
  for (int g = pair; g < n_groups; g += PAIRS) {
    const int4 grp = groups_s[g];
    bool ok = !*abort_flag && mbar_wait(R.full(g), RingT::parity(g), deadline);
    if (!ok && !*abort_flag) {
      set_error(a.ws.hdr, DEV_TIMEOUT);
      *abort_flag = 1;
    }
    // Read after the wait: the producer wrote it before its arrival.  (After
    // a failed wait the slot is not read.)
    uint8_t* st = smem + (ok ? *static_cast<volatile uint32_t*>(&s_goff[g % NDESC]) : 0u);
    const float sc = F::scale(a, grp.x);
    switch ((grp.z + 7) >> 3) {
      case 1:
        ok = group_pair<F, 1>(st, ok, grp.z, grp.y, khalf, bar_id, sc, my_acc, pair_tok_s, pair_w_s);
        break;
      case 2:
        ok = group_pair<F, 2>(st, ok, grp.z, grp.y, khalf, bar_id, sc, my_acc, pair_tok_s, pair_w_s);
        break;
      default:
        ok = group_pair<F, 3>(st, ok, grp.z, grp.y, khalf, bar_id, sc, my_acc, pair_tok_s, pair_w_s);
        break;
    }
    if (!ok) break;
    // Both warps' ring reads are done (they preceded the pair barrier).
    if (khalf == 0 && lane == 0) mbar_arrive(R.empty(g));
  }
  named_sync(1, CW * 32);
  if (*abort_flag) return;
  for (int i = threadIdx.x; i < B * RS; i += CW * 32) {
    const int t = i / RS, r = i % RS;
    float v = accw[i];
#pragma unroll
    for (int p = 1; p < PAIRS; ++p) v += accw[p * B * RS + i];
    const size_t o = (size_t)t * H + r0 + r;
    a.out[o] = f2bf(bf_lo((uint32_t)a.residual[o]) + v);
  }
}

// Launch (PDL-chained after the gate/up kernel); `maps` from F::make_maps.
template <class F>
cudaError_t launch_down_ring(const ExpertArgs& a, const typename F::Maps& maps, cudaStream_t stream) {
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t es = set_smem_limit_once(down_ring_kernel<F>, SMEM_CAP, smem_set);
  if (es != cudaSuccess) return es;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(H / RS, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = Layout<F>::smem_bytes(a.B);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, down_ring_kernel<F>, a, maps);
}

}  // namespace dring
}  // namespace flint
