// nvfp4.cu — NVFP4 weight-only (W4A16) expert kernels: gate/up + SiLU-and-mul
// and down + combine + shared + residual, with the weights dequantised in
// registers.  "run weight-only (W4A16) while maintaining BF16 activations":
// vLLM Day-0 Support for Recursive's Flint, "Flint Model Overview and
// Capabilities".
//
// Storage (per projection, rows x K): q = e2m1 codes, two per byte (low nibble
// = even k); sf = one OCP E4M3 scale per 16 consecutive k; ts = fp32 tensor
// scale.  W = e2m1(q) * e4m3(sf) * ts.
//
// The product e2m1 * e4m3 has at most 6 significant bits and lies in
// [2^-10, 2688], so it is EXACT in f16: each thread converts its fragment's
// codes with cvt.rn.f16x2.e2m1x2, multiplies by the block scale (f16x2, exact)
// and feeds mma.sync m16n8k16 f16 x f16 -> fp32.  bf16 activations convert to
// f16 exactly (8 significant bits; |x| inside f16's normal range); the tensor
// scale is applied to the fp32 sums.  h is stored scaled by 2^-8 as an f16
// pair hi + lo (~22 significant bits; |h| up to ~1.7e7, beyond which the
// gate/up kernel reports the input), so the down kernel feeds its dequantised
// f16 weights straight into f16 MMAs on both halves and undoes the scale on
// the sums.  Dequantisation costs about one instruction per weight, which is
// why this path uses the tensor cores for every group, including single-token
// ones: the FMAs then cost nothing on the CUDA cores that do the unpacking.
//
// The gate/up work decomposition and its TMA/mbarrier pipeline are those of
// the BF16 gate/up kernel (gate/up units are (group, 8 gate + 8 up rows)
// ranges split evenly over one CTA per SM); it stores h as f16 for the down
// kernel, which splits the work into (group, 128-row block) units and
// combines the partial sums per row block (see below).
#include <cuda_fp16.h>

#include "common.cuh"
#include "expert_common.cuh"
#include "kernels.h"
#include "nv_util.cuh"
#include "tmap.h"

namespace flint {
using namespace nvu;
namespace f4 {
constexpr int CWARPS = 8;
constexpr int THREADS = CWARPS * 32 + 32;
constexpr uint64_t DRAIN_NS = 2000000000ull;
// gate/up.  A stage holds one unit as four tensor-map copies with a 128-byte
// swizzle (16-byte chunk c of a 128-byte line stored at c ^ (line mod 8)):
// the 8 gate rows' codes as [column block L of 128 bytes][row r] lines, the 8
// up rows' codes the same, then the gate and up rows' scales as [row] lines.
constexpr int GU_QROW = H / 2;                       // 1024 code bytes per row
constexpr int GU_SFROW = H / 16;                     // 128 scale bytes per row
constexpr int GU_UPQ = 8 * GU_QROW;                  // offsets in a stage
constexpr int GU_SF = 16 * GU_QROW;
constexpr int GU_UPSF = GU_SF + 8 * GU_SFROW;
constexpr int GU_STAGE = 16 * GU_QROW + 16 * GU_SFROW;  // 18,432 (18 x 1 KiB)
constexpr int GU_NSTAGE = 10;
constexpr int GU_ALIGN = 1024;                       // swizzled copies land on 1 KiB boundaries
static_assert(GU_STAGE % GU_ALIGN == 0 && GU_SF % GU_ALIGN == 0 && GU_UPSF % GU_ALIGN == 0,
              "every copy starts on a 1 KiB boundary");
// A round takes up to GU_UB(NT) units of one group at once; their partial
// tiles [unit][warp][16 rows][NT * 8 tokens] share one reduction.
__host__ __device__ constexpr int gu_ub(int nt) { return nt == 1 ? 4 : nt == 2 ? 2 : 1; }
constexpr int GU_RED = 4 * CWARPS * 16 * 8;  // = 2 * CWARPS * 16 * 16 >= CWARPS * 16 * 24
static_assert(GU_RED >= 2 * CWARPS * 16 * 16 && GU_RED >= CWARPS * 16 * GROUP_MAX, "rounds fit");
// The reduction buffer doubles as the logits buffer of the local selection.
constexpr int GU_BUF = GU_RED * 4 > LOCAL_SELECT_MAX_B * E * 4 ? GU_RED * 4 : LOCAL_SELECT_MAX_B * E * 4;
constexpr size_t GU_SMEM =
    GU_ALIGN + (size_t)GU_NSTAGE * GU_STAGE + GU_BUF + sizeof(MetaSmem) + 2 * GU_NSTAGE * 8;
constexpr int UNITS = I / 8;
static_assert(GU_SMEM <= 232448, "the gate/up ring fits one CTA's shared memory");
}  // namespace f4

namespace {

struct Pipe {
  uint8_t* stages;
  uint32_t stages_addr;
  int stage_bytes, nstage;
  uint32_t full0, empty0;
  uint64_t deadline;
  WsHeader* hdr;
  volatile int* abort_flag;
};

__device__ __forceinline__ uint32_t full_bar(const Pipe& p, int s) { return p.full0 + 8u * s; }
__device__ __forceinline__ uint32_t empty_bar(const Pipe& p, int s) { return p.empty0 + 8u * s; }

__device__ __forceinline__ bool wait_full(const Pipe& p, int slot, uint32_t parity) {
  if (*p.abort_flag) return false;
  if (mbar_wait(full_bar(p, slot), parity, p.deadline)) return true;
  *p.abort_flag = 1;
  set_error(p.hdr, DEV_TIMEOUT);
  return false;
}

// Producer-side acquire of a free stage; false means stop issuing.
__device__ __forceinline__ bool acquire_stage(const Pipe& p, int it) {
  const int slot = it % p.nstage;
  bool got = true;
  if (it >= p.nstage)
    got = mbar_wait(empty_bar(p, slot), (uint32_t)((it / p.nstage) - 1) & 1u, p.deadline);
  if (!got || *p.abort_flag) {
    *p.abort_flag = 1;
    if (!got) set_error(p.hdr, DEV_TIMEOUT);
    return false;
  }
  return true;
}

__device__ __forceinline__ void drain(const Pipe& p, int it) {
  const uint64_t dl = globaltimer_ns() + f4::DRAIN_NS;
  for (int j = it - p.nstage < 0 ? 0 : it - p.nstage; j < it; ++j)
    mbar_wait(full_bar(p, j % p.nstage), (uint32_t)(j / p.nstage) & 1u, dl);
}

// Units [0, n) over the CTAs.  With fewer than min_per_cta units per CTA
// (small batches), CTA c takes the c-th of equal contiguous shares: each CTA's
// consumers then work through long runs of one group in full reduction rounds.
// Otherwise each CTA first takes a static chunk of min(8, n / (2 x #SMs))
// units and then claims the rest as it goes -- guided self-scheduling, as in
// the BF16 gate/up kernel (SMs stream at different rates, so equal static
// shares leave a tail): chunks of about remaining / (2 x #SMs) units (1..8,
// in multiples of ALIGN) from *claim, the first claim sent while the static
// chunk streams and the next one claimed ahead while plenty remains.  Each
// chunk {first unit, units}
// is published on its first stage in s_chunk, and a stage marked {-1, 0} ends
// the list; the last CTA done claiming resets the counters for the next call.
// Measured on GB300 (NVFP4 layer, chained): claimed gate/up units take skewed
// batch 128 from 183 to 165 us and claimed down units to 168 us (both: 150;
// 147 with gate/up chunks of whole reduction rounds), but cost 3-7 us at 1-8
// tokens, hence the per-kernel minimum.
__device__ __forceinline__ bool claims_used(int n, int min_per_cta) {
  return n >= min_per_cta * (int)gridDim.x;
}
__device__ __forceinline__ int static_begin(int n, int c) {
  return (int)((long long)c * n / gridDim.x);
}
constexpr int GU_CLAIM_MIN = 32, DN_CLAIM_MIN = 8;  // units per CTA
// gate/up chunks keep whole reduction rounds (4 units for groups of <= 8 tokens)
constexpr int GU_CLAIM_ALIGN = 4;

template <int ALIGN, class Issue>
__device__ __forceinline__ void produce_claimed(const Pipe& p, int n, int min_per_cta,
                                                uint32_t* claim, uint32_t* done, int2* s_chunk,
                                                Issue issue) {
  const int G = (int)gridDim.x, cta = (int)blockIdx.x;
  int it = 0;
  bool ok = true;
  auto run = [&](int c0, int e, bool publish) {  // issue units [c0, e)
    for (int u = c0; ok && u < e; ++u) {
      if (!acquire_stage(p, it)) {
        ok = false;
        break;
      }
      if (publish && u == c0) s_chunk[it % p.nstage] = make_int2(c0, e - c0);
      issue(u, it % p.nstage);
      ++it;
    }
  };
  if (!claims_used(n, min_per_cta)) {
    run(static_begin(n, cta), static_begin(n, cta + 1), false);
    drain(p, it);
    return;
  }
  auto size_for = [G](int rem) {  // a multiple of ALIGN in [ALIGN, 8]
    const int s = (rem / (2 * G)) / ALIGN * ALIGN;
    return s < ALIGN ? ALIGN : (s > 8 ? 8 : s);
  };
  const int f = min(8, n / (2 * G)) / ALIGN * ALIGN;
  const int base = G * f;  // claimed units start here
  int sz = size_for(n - base);
  int c0 = base + (int)atomicAdd(claim, (uint32_t)sz);
  run(cta * f, cta * f + f, true);
  while (ok && c0 < n) {
    const int e = min(n, c0 + sz);
    const int sz_next = size_for(n - e);
    const bool ahead = n - e > 2 * G;
    int c_next = ahead ? base + (int)atomicAdd(claim, (uint32_t)sz_next) : 0;
    run(c0, e, true);
    if (!ahead) c_next = base + (int)atomicAdd(claim, (uint32_t)sz_next);
    c0 = c_next;
    sz = sz_next;
  }
  __threadfence();
  if (atomicAdd(done, 1u) == (uint32_t)G - 1u) {
    atomicExch(claim, 0u);
    atomicExch(done, 0u);
  }
  if (ok && acquire_stage(p, it)) {  // no more: the consumers stop at this stage
    s_chunk[it % p.nstage] = make_int2(-1, 0);
    mbar_arrive(full_bar(p, it % p.nstage));
    ++it;
  }
  drain(p, it);
}

__device__ __forceinline__ void init_pipe(Pipe& p, uint8_t* smem, int stage_bytes, int nstage,
                                          uint64_t* bars, int max_stages, volatile int* abort_flag,
                                          WsHeader* hdr) {
  p.stages = smem;
  p.stages_addr = smem_addr(smem);
  p.stage_bytes = stage_bytes;
  p.nstage = nstage;
  p.full0 = smem_addr(bars);
  p.empty0 = smem_addr(bars + max_stages);
  p.abort_flag = abort_flag;
  p.hdr = hdr;
  if (threadIdx.x == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(full_bar(p, s), 1);
      mbar_init(empty_bar(p, s), f4::CWARPS);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
}

// ---------------------------------------------------------------- gate/up

// Units [u0, u1) of one group with n tokens, NT = ceil(n / 8), taken UB at a
// time: the warps compute their K-slice of every unit of the round (the
// units' dequantisation and MMAs interleave), then one reduction round sums
// the 8 warps' partial tiles of all of them.
template <int NT>
__device__ __forceinline__ void gu_segment(const Pipe& p, const ExpertArgs& a, const int* pair_tok,
                                           float* red, int u0,
                                           int u1, int expert, int pair0, int n, int& it,
                                           bool& ok) {
  constexpr int UB = f4::gu_ub(NT);
  constexpr int NC = NT * 8;  // token columns of a partial tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  named_sync(1, f4::CWARPS * 32);  // the previous segment is done with `red`
  // K order inside this warp's 256-column slice (its 128-byte code line):
  // thread q of a quad owns the 32 consecutive columns [64q + 32m, +32) for
  // m = 0, 1, i.e. 16-byte chunk 2q + m of the line; step (m, i) covers
  // columns 64q + 32m + 8i .. +8.  Under the swizzle, rows g and g + 1 of a
  // quarter-warp then read chunks of opposite parity: no bank conflicts.  The
  // activations follow the same order, so the MMA sums match.
  uint4 bfr[NT][2][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int slot = nt * 8 + g;
    if (slot < n) {
      const int tok = pair_tok[pair0 + slot];
      const uint4* row = reinterpret_cast<const uint4*>(a.x + (size_t)tok * H + warp * 256 + q * 64);
      bool big = false;
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 xv = __ldg(row + m * 4 + i);
          big |= bf16x8_beyond_f16(xv);
          bfr[nt][m][i] = bf16x8_to_f16x8(xv);
        }
      if (big) set_error(a.ws.hdr, DEV_BAD_INPUT);  // the activations run as f16 here
    } else {
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int i = 0; i < 4; ++i) bfr[nt][m][i] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  const float* ts = expert < E ? a.w.w13_ts + 2 * expert : a.w.ws13_ts + 2 * (expert - E);
  const float ts_g = __ldg(ts), ts_u = __ldg(ts + 1);
  for (int u = u0; u < u1; u += UB) {
    const int ub = u1 - u < UB ? u1 - u : UB;
    float acc[UB][NT][4];
#pragma unroll
    for (int k = 0; k < UB; ++k)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) acc[k][nt][0] = acc[k][nt][1] = acc[k][nt][2] = acc[k][nt][3] = 0.f;
    const uint8_t* st[UB];
#pragma unroll
    for (int k = 0; k < UB; ++k) {
      const int slot = (it + k) % p.nstage;
      if (k < ub && ok) ok = wait_full(p, slot, (uint32_t)((it + k) / p.nstage) & 1u);
      st[k] = p.stages + slot * p.stage_bytes;
    }
    if (ok) {
      // code line `warp` of row g: [warp][g][128 B], chunk c at c ^ g; scale
      // line g: the warp's 16 blocks are chunk `warp`, at warp ^ g, of which
      // this thread's columns use word q
      const int qoff = (warp * 8 + g) * 128;
      const int soff = f4::GU_SF + g * f4::GU_SFROW + ((warp ^ g) * 16) + 4 * q;
#pragma unroll
      for (int m = 0; m < 2; ++m) {
#pragma unroll
        for (int k = 0; k < UB; ++k) {
          if (k >= ub) continue;
          const uint8_t* ql = st[k] + qoff + (((2 * q + m) ^ g) * 16);
          const uint4 clo = *reinterpret_cast<const uint4*>(ql);
          const uint4 chi = *reinterpret_cast<const uint4*>(ql + f4::GU_UPQ);
          const uint32_t wl = *reinterpret_cast<const uint32_t*>(st[k] + soff);
          const uint32_t wh = *reinterpret_cast<const uint32_t*>(st[k] + soff + 8 * f4::GU_SFROW);
          const uint32_t cl[4] = {clo.x, clo.y, clo.z, clo.w};
          const uint32_t ch[4] = {chi.x, chi.y, chi.z, chi.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            // block of step (m, i) = 4q + 2m + i/2 of the warp's 16: byte
            // 2m + i/2 of word q
            const int sh_bits = 8 * (2 * m + (i >> 1));
            const uint32_t scl = e4m3_bcast_f16x2((wl >> sh_bits) & 0xffu);
            const uint32_t sch = e4m3_bcast_f16x2((wh >> sh_bits) & 0xffu);
            uint32_t l0, l1, l2, l3, h0, h1, h2, h3;
            e2m1x8_to_f16x2(cl[i], l0, l1, l2, l3);
            e2m1x8_to_f16x2(ch[i], h0, h1, h2, h3);
            l0 = hmul2(l0, scl); l1 = hmul2(l1, scl); l2 = hmul2(l2, scl); l3 = hmul2(l3, scl);
            h0 = hmul2(h0, sch); h1 = hmul2(h1, sch); h2 = hmul2(h2, sch); h3 = hmul2(h3, sch);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
              const uint4 b = bfr[nt][m][i];
              mma_f16(acc[k][nt], l0, h0, l1, h1, b.x, b.y);
              mma_f16(acc[k][nt], l2, h2, l3, h3, b.z, b.w);
            }
          }
        }
      }
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < UB; ++k)
      if (k < ub && lane == 0) mbar_arrive(empty_bar(p, (it + k) % p.nstage));
    it += ub;
#pragma unroll
    for (int k = 0; k < UB; ++k) {
      float* rw = red + ((k * f4::CWARPS + warp) * 16) * NC;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const int col = nt * 8 + 2 * q;
        rw[g * NC + col] = acc[k][nt][0];
        rw[g * NC + col + 1] = acc[k][nt][1];
        rw[(g + 8) * NC + col] = acc[k][nt][2];
        rw[(g + 8) * NC + col + 1] = acc[k][nt][3];
      }
    }
    named_sync(1, f4::CWARPS * 32);
    {
      // 8 adjacent lanes = the 8 rows of one (unit k, token j): they store the
      // token's h block together
      static_assert(f4::CWARPS * 32 / 8 >= UB * NC, "one 8-lane group per (unit, token)");
      const int G = threadIdx.x >> 3;
      const int r = threadIdx.x & 7;
      const int k = G / NC, j = G % NC;
      const bool valid = k < ub && j < n;
      const int kr = valid ? k : 0, jr = valid ? j : 0;
      float gs = 0.f, us = 0.f;
#pragma unroll
      for (int w = 0; w < f4::CWARPS; ++w) {
        gs += red[((kr * f4::CWARPS + w) * 16 + r) * NC + jr];
        us += red[((kr * f4::CWARPS + w) * 16 + r + 8) * NC + jr];
      }
      const int blk = (u + kr) & (f4::UNITS - 1);
      // h beyond the f16 pair's range would reach the down kernel as infinities
      if (store_h_block8_nv(a.ws.h, (size_t)(pair0 + jr), blk, silu_mul(gs * ts_g, us * ts_u),
                            valid && ok))
        set_error(a.ws.hdr, DEV_BAD_INPUT);
    }
    named_sync(1, f4::CWARPS * 32);
  }
}

// Tensor maps of the gate/up codes and scales (routed and shared expert
// stacks): codes as (128 bytes, row, 8 column blocks) with strides (1 B,
// 1 KiB, 128 B), scales as (128 bytes, row); boxes of 8 rows; 128-byte swizzle.
struct GuMaps {
  CUtensorMap q, sq, sf, ssf;
};

__device__ __forceinline__ void tma_3d(uint32_t dst, const CUtensorMap* map, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
      "l"(map), "r"(0), "r"(c1), "r"(0), "r"(bar), "l"(l2_evict_first())
      : "memory");
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(0), "r"(c1), "r"(bar), "l"(l2_evict_first())
      : "memory");
}

__device__ __forceinline__ void gu_produce(const Pipe& p, const GuMaps& maps, const int4* groups,
                                           int n, uint32_t* claim, uint32_t* done,
                                           int2* s_chunk) {
  produce_claimed<GU_CLAIM_ALIGN>(p, n, GU_CLAIM_MIN, claim, done, s_chunk, [&](int u, int slot) {
    const int4 grp = groups[u / f4::UNITS];
    const int blk = u & (f4::UNITS - 1);
    const bool routed = grp.x < E;
    const int e = routed ? grp.x : grp.x - E;
    const CUtensorMap* mq = routed ? &maps.q : &maps.sq;
    const CUtensorMap* ms = routed ? &maps.sf : &maps.ssf;
    const int gate_row = e * (2 * I) + blk * 8, up_row = gate_row + I;
    mbar_expect_tx(full_bar(p, slot), f4::GU_STAGE);
    const uint32_t dst = p.stages_addr + slot * p.stage_bytes;
    tma_3d(dst, mq, gate_row, full_bar(p, slot));
    tma_3d(dst + f4::GU_UPQ, mq, up_row, full_bar(p, slot));
    tma_2d(dst + f4::GU_SF, ms, gate_row, full_bar(p, slot));
    tma_2d(dst + f4::GU_UPSF, ms, up_row, full_bar(p, slot));
  });
}

}  // namespace

__global__ void __launch_bounds__(f4::THREADS, 1)
    gateup_nvfp4_kernel(ExpertArgs a, const __grid_constant__ GuMaps maps) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + f4::GU_ALIGN - 1) & ~uint32_t(f4::GU_ALIGN - 1)) - raw_addr);
  __shared__ int s_abort;
  __shared__ LocalSelectSmem s_sel;
  __shared__ int2 s_chunk[f4::GU_NSTAGE];  // claimed chunk starting at each stage
  float* red = reinterpret_cast<float*>(smem + f4::GU_NSTAGE * f4::GU_STAGE);
  MetaSmem& meta = *reinterpret_cast<MetaSmem*>(reinterpret_cast<uint8_t*>(red) + f4::GU_BUF);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(&meta) + sizeof(MetaSmem));
  Pipe p;
  init_pipe(p, smem, f4::GU_STAGE, f4::GU_NSTAGE, bars, f4::GU_NSTAGE, &s_abort, a.ws.hdr);
  __syncthreads();
  p.deadline = wait_deadline(a.ws.hdr);
  pdl_wait();     // the router's logits / routing
  if ((threadIdx.x >> 5) == f4::CWARPS) {
    named_sync(2, ALL_THREADS);  // routing metadata is in shared memory
    if ((threadIdx.x & 31) == 0)
      gu_produce(p, maps, meta.groups, meta.n_groups * f4::UNITS, &a.ws.hdr->gu_claim,
                 &a.ws.hdr->gu_done, s_chunk);
    return;
  }
  fill_meta(a, a.local_select != 0, meta, nullptr, red, &s_sel);
  pdl_trigger();
  named_sync(2, ALL_THREADS);
  int it = 0;
  bool ok = true;
  const int n_units = meta.n_groups * f4::UNITS;
  const bool claimed = claims_used(n_units, GU_CLAIM_MIN);
  int2 ch = make_int2(static_begin(n_units, blockIdx.x),
                      static_begin(n_units, blockIdx.x + 1) - static_begin(n_units, blockIdx.x));
  while (ok) {  // the CTA's share, or the producer's chunks in its order
    if (claimed) {
      const int slot = it % p.nstage;
      if (!wait_full(p, slot, (uint32_t)(it / p.nstage) & 1u)) break;
      ch = s_chunk[slot];
      if (ch.x < 0) break;
    }
    int u = ch.x;
    const int u_end = ch.x + ch.y;
    while (ok && u < u_end) {
      const int gi = u / f4::UNITS;
      const int4 grp = meta.groups[gi];
      const int u1 = min(u_end, (gi + 1) * f4::UNITS);
      switch ((grp.z + 7) >> 3) {
        case 1: gu_segment<1>(p, a, meta.pair_tok, red, u, u1, grp.x, grp.y, grp.z, it, ok); break;
        case 2: gu_segment<2>(p, a, meta.pair_tok, red, u, u1, grp.x, grp.y, grp.z, it, ok); break;
        default: gu_segment<3>(p, a, meta.pair_tok, red, u, u1, grp.x, grp.y, grp.z, it, ok); break;
      }
      u = u1;
    }
    if (!claimed) break;
  }
}

// Map of `rows` rows of `row_bytes` bytes at `base`, as (128 bytes, row) or,
// for code rows (1 KiB), as (128 bytes, row, 8 column blocks); boxes of 8 rows.
static cudaError_t encode_gu(CUtensorMap* m, const uint8_t* base, size_t rows, int row_bytes) {
  const EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return cudaErrorNotSupported;
  const bool codes = row_bytes == f4::GU_QROW;
  const cuuint64_t dims[3] = {128, (cuuint64_t)rows, (cuuint64_t)(row_bytes / 128)};
  const cuuint64_t strides[2] = {(cuuint64_t)row_bytes, 128};  // bytes, for dims 1 and 2
  const cuuint32_t box[3] = {128, 8, (cuuint32_t)(row_bytes / 128)};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes ? 3 : 2,
                         const_cast<uint8_t*>(base), dims, strides, box, elem,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gateup_nvfp4(const ExpertArgs& a, cudaStream_t stream, int num_sms) {
  GuMaps maps;
  cudaError_t em = encode_gu(&maps.q, a.w.w13_q, (size_t)E * 2 * I, f4::GU_QROW);
  if (em == cudaSuccess) em = encode_gu(&maps.sq, a.w.ws13_q, (size_t)S * 2 * I, f4::GU_QROW);
  if (em == cudaSuccess) em = encode_gu(&maps.sf, a.w.w13_sf, (size_t)E * 2 * I, f4::GU_SFROW);
  if (em == cudaSuccess) em = encode_gu(&maps.ssf, a.w.ws13_sf, (size_t)S * 2 * I, f4::GU_SFROW);
  if (em != cudaSuccess) return em;
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t es = set_smem_limit_once(gateup_nvfp4_kernel, (int)f4::GU_SMEM, smem_set);
  if (es != cudaSuccess) return es;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms, 1, 1);
  cfg.blockDim = dim3(f4::THREADS, 1, 1);
  cfg.dynamicSmemBytes = f4::GU_SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gateup_nvfp4_kernel, a, maps);
}

// ---------------------------------------------------------------- down
//
// Split-combine: a unit is (group, block of 128 output rows): the block's
// 128 x 256 code bytes (32 KiB) and 128 x 32 scale bytes (4 KiB), plus the
// group's f16 h rows, arrive as three bulk copies into one stage; the units
// are split evenly over one CTA per SM, so each SM streams a few large units
// instead of walking every group.  Warp w computes rows 16w .. 16w + 15 of the
// block over all 512 columns: lane (g, q) takes, at MMA step s, columns
// 128q + 4s .. +3 of rows g and g + 8, so its 64 code bytes and 8 scale bytes
// per row are loaded once per unit and dequantised from registers; h follows
// the same order (h_off_nv).  Each warp writes its rows' partial sums,
// already weighted by the routing weight and the tensor scale, to y[pair][row].
// A second kernel, chained after this one, adds for each token its SLOTS rows
// of y in ascending pair order to the residual -- a fixed order, so the result
// is bitwise reproducible.  The kernel boundary orders every y store before
// the combine: no fence, ticket or barrier per unit (those cost ~1 us per unit
// while the copies stream, measured).

namespace f4 {
constexpr int DN_RB = 128;                      // output rows per unit
constexpr int DN_UNITS = H / DN_RB;             // units per group
constexpr int DN_QROW = I / 2;                  // code bytes per row
constexpr int DN_SFROW = I / 16;                // scale bytes per row
constexpr int DN_QB = DN_RB * DN_QROW;          // 32 KiB
constexpr int DN_SB = DN_RB * DN_SFROW;         // 4 KiB
constexpr int DN_HROW = I * 4;                  // one h row (f16 hi + lo pairs)
constexpr int DN_MAX_STAGES = 4;
constexpr int SMEM_CAP = 232448 - 1024;
__host__ __device__ inline int dn_stage(int B) {
  return DN_QB + DN_SB + (B < GROUP_MAX ? B : GROUP_MAX) * DN_HROW;
}
__host__ __device__ inline int dn_fixed() { return (int)sizeof(MetaSmem) + 2 * DN_MAX_STAGES * 8; }
__host__ __device__ inline int dn_nstages(int B) {
  const int n = (SMEM_CAP - dn_fixed()) / dn_stage(B);
  return n > DN_MAX_STAGES ? DN_MAX_STAGES : n;
}
__host__ __device__ inline int dn_smem(int B) { return dn_nstages(B) * dn_stage(B) + dn_fixed(); }
static_assert(DN_QB + DN_SB + GROUP_MAX * DN_HROW + (int)sizeof(MetaSmem) + 2 * DN_MAX_STAGES * 8 <=
                  SMEM_CAP,
              "a stage of the largest group fits");
}  // namespace f4

namespace {

// One warp, one unit: rows 16w .. 16w + 15 of the block, NT token tiles.
// Lane (g, q): rows g and g + 8, columns 128q + 4s .. +3 at step s.
template <int NT>
__device__ __forceinline__ void dn_unit(const ExpertArgs& a, const uint8_t* st, int expert,
                                        int pair0, int n, int rb, float* y) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const uint8_t* cr = st + (16 * warp + g) * f4::DN_QROW + 64 * q;
  uint4 c0[4], c1[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    c0[i] = *reinterpret_cast<const uint4*>(cr + 16 * i);
    c1[i] = *reinterpret_cast<const uint4*>(cr + 8 * f4::DN_QROW + 16 * i);
  }
  const uint8_t* sr = st + f4::DN_QB + (16 * warp + g) * f4::DN_SFROW + 8 * q;
  const uint2 s0 = *reinterpret_cast<const uint2*>(sr);
  const uint2 s1 = *reinterpret_cast<const uint2*>(sr + 8 * f4::DN_SFROW);
  // Token columns past n read token 0's h row: their sums are never used.
  const uint8_t* hrow[NT];
  int hx[NT];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int slot = nt * 8 + g < n ? nt * 8 + g : 0;
    hrow[nt] = st + f4::DN_QB + f4::DN_SB + slot * f4::DN_HROW + q * 32;
    hx[nt] = ((pair0 + slot) & 1) * 16;
  }
  float acc[NT][2][4];  // [tile][even, odd step][fragment]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) acc[nt][c][0] = acc[nt][c][1] = acc[nt][c][2] = acc[nt][c][3] = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {  // two MMA steps: one code word and one h block per row
    const uint4 v0 = c0[j >> 2], v1 = c1[j >> 2];
    const uint32_t w0 = (j & 3) == 0 ? v0.x : (j & 3) == 1 ? v0.y : (j & 3) == 2 ? v0.z : v0.w;
    const uint32_t w1 = (j & 3) == 0 ? v1.x : (j & 3) == 1 ? v1.y : (j & 3) == 2 ? v1.z : v1.w;
    // 16 columns per scale: steps 4m .. 4m + 3 share scale m
    const uint32_t sb0 = (j >> 1) < 4 ? s0.x : s0.y, sb1 = (j >> 1) < 4 ? s1.x : s1.y;
    const int sh = 8 * ((j >> 1) & 3);
    const uint32_t sc0 = e4m3_bcast_f16x2((sb0 >> sh) & 0xffu);
    const uint32_t sc1 = e4m3_bcast_f16x2((sb1 >> sh) & 0xffu);
    uint32_t l0, l1, l2, l3, u0, u1, u2, u3;
    e2m1x8_to_f16x2(w0, l0, l1, l2, l3);
    e2m1x8_to_f16x2(w1, u0, u1, u2, u3);
    l0 = hmul2(l0, sc0); l1 = hmul2(l1, sc0); l2 = hmul2(l2, sc0); l3 = hmul2(l3, sc0);
    u0 = hmul2(u0, sc1); u1 = hmul2(u1, sc1); u2 = hmul2(u2, sc1); u3 = hmul2(u3, sc1);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // block 16q + j of the token's row (h_off_nv): hi and lo halves
      const uint8_t* hb8 = hrow[nt] + j * 128;
      const uint4 hh = *reinterpret_cast<const uint4*>(hb8 + hx[nt]);
      const uint4 hl = *reinterpret_cast<const uint4*>(hb8 + (16 - hx[nt]));
      mma_f16(acc[nt][0], l0, u0, l1, u1, hh.x, hh.y);
      mma_f16(acc[nt][1], l2, u2, l3, u3, hh.z, hh.w);
      mma_f16(acc[nt][0], l0, u0, l1, u1, hl.x, hl.y);
      mma_f16(acc[nt][1], l2, u2, l3, u3, hl.z, hl.w);
    }
  }
  // h was stored scaled by NV_H_SCALE (a power of two): undone here, exactly
  const float ts = (expert < E ? __ldg(a.w.w2_ts + expert) : __ldg(a.w.ws2_ts + (expert - E))) *
                   (1.0f / NV_H_SCALE);
  const int row = rb * f4::DN_RB + 16 * warp + g;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int col = nt * 8 + 2 * q + e;
      if (col < n) {
        const int pr = pair0 + col;
        const float wt = __ldg(a.ws.pair_w + pr) * ts;
        const float d0 = acc[nt][0][e] + acc[nt][1][e];
        const float d1 = acc[nt][0][2 + e] + acc[nt][1][2 + e];
        y[(size_t)pr * H + row] = wt * d0;
        y[(size_t)pr * H + row + 8] = wt * d1;
      }
    }
  }
}

__device__ __forceinline__ void dn_produce(const Pipe& p, const ExpertArgs& a, const int4* groups,
                                           int n, int2* s_chunk) {
  produce_claimed<1>(p, n, DN_CLAIM_MIN, &a.ws.hdr->dn_claim, &a.ws.hdr->dn_done, s_chunk,
                  [&](int u, int slot) {
    const int4 grp = groups[u / f4::DN_UNITS];
    const int rb = u % f4::DN_UNITS;
    const bool routed = grp.x < E;
    const int e = routed ? grp.x : grp.x - E;
    const size_t row0 = (size_t)e * H + (size_t)rb * f4::DN_RB;
    const uint8_t* qb = (routed ? a.w.w2_q : a.w.ws2_q) + row0 * f4::DN_QROW;
    const uint8_t* sb = (routed ? a.w.w2_sf : a.w.ws2_sf) + row0 * f4::DN_SFROW;
    mbar_expect_tx(full_bar(p, slot), f4::DN_QB + f4::DN_SB + grp.z * f4::DN_HROW);
    const uint32_t dst = p.stages_addr + slot * p.stage_bytes;
    bulk_g2s_stream(dst, qb, f4::DN_QB, full_bar(p, slot));
    bulk_g2s_stream(dst + f4::DN_QB, sb, f4::DN_SB, full_bar(p, slot));
    bulk_g2s(dst + f4::DN_QB + f4::DN_SB,
             reinterpret_cast<const uint8_t*>(a.ws.h) + (size_t)grp.y * f4::DN_HROW,
             grp.z * f4::DN_HROW, full_bar(p, slot));
  });
}

}  // namespace

__global__ void __launch_bounds__(f4::THREADS, 1) down_nvfp4_kernel(ExpertArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ int s_abort;
  __shared__ int2 s_chunk[f4::DN_MAX_STAGES];  // claimed chunk starting at each stage
  const int B = a.B;
  const int nstage = f4::dn_nstages(B), stage = f4::dn_stage(B);
  MetaSmem& meta = *reinterpret_cast<MetaSmem*>(smem + nstage * stage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(&meta) + sizeof(MetaSmem));
  Pipe p;
  init_pipe(p, smem, stage, nstage, bars, f4::DN_MAX_STAGES, &s_abort, a.ws.hdr);
  __syncthreads();
  p.deadline = wait_deadline(a.ws.hdr);
  pdl_wait();  // h, the group table and the pairs come from the preceding kernels
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == f4::CWARPS) {
    named_sync(2, ALL_THREADS);  // routing metadata is in shared memory
    if (lane == 0) dn_produce(p, a, meta.groups, meta.n_groups * f4::DN_UNITS, s_chunk);
    return;
  }
  fill_meta(a, false, meta, nullptr, nullptr, nullptr);
  pdl_trigger();
  named_sync(2, ALL_THREADS);
  float* y = ws_y(a.ws, B);
  bool ok = true;
  int it = 0;
  const int n_units = meta.n_groups * f4::DN_UNITS;
  const bool claimed = claims_used(n_units, DN_CLAIM_MIN);
  int2 ch = make_int2(static_begin(n_units, blockIdx.x),
                      static_begin(n_units, blockIdx.x + 1) - static_begin(n_units, blockIdx.x));
  while (ok) {  // the CTA's share, or the producer's chunks in its order
    if (claimed) {
      if (!wait_full(p, it % p.nstage, (uint32_t)(it / p.nstage) & 1u)) break;
      ch = s_chunk[it % p.nstage];
      if (ch.x < 0) break;
    }
    for (int u = ch.x; u < ch.x + ch.y; ++u, ++it) {
      const int4 grp = meta.groups[u / f4::DN_UNITS];
      const int rb = u % f4::DN_UNITS;
      const int slot = it % p.nstage;
      if (ok) ok = wait_full(p, slot, (uint32_t)(it / p.nstage) & 1u);
      if (ok) {
        const uint8_t* st = p.stages + slot * p.stage_bytes;
        switch ((grp.z + 7) >> 3) {
          case 1: dn_unit<1>(a, st, grp.x, grp.y, grp.z, rb, y); break;
          case 2: dn_unit<2>(a, st, grp.x, grp.y, grp.z, rb, y); break;
          default: dn_unit<3>(a, st, grp.x, grp.y, grp.z, rb, y); break;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty_bar(p, slot));
      if (!ok) break;  // a failed wait set the abort flag: the producer stops too
    }
    if (!claimed) break;
  }
}

// out[t][r] = residual[t][r] + the token's SLOTS rows of y at r, added in
// ascending pair order.  Block (x, t): token t, rows 256x .. 256x + 255; warp 0
// lists the token's pairs (ballots over pair_tok) before the sums.
__global__ void __launch_bounds__(256) combine_y_kernel(ExpertArgs a) {
  __shared__ int s_pairs[SLOTS];
  __shared__ int s_ok;
  pdl_wait();  // y and the pair table come from the preceding kernels
  pdl_trigger();  // a following router may start loading its rows
  const int t = blockIdx.y, lane = threadIdx.x & 31;
  if (threadIdx.x < 32) {
    const int np = a.B * SLOTS;
    int cnt = 0;
    for (int base = 0; base < np; base += 32) {
      const int pr = base + lane;
      const bool mine = pr < np && __ldcg(a.ws.pair_tok + pr) == t;
      const uint32_t m = __ballot_sync(0xffffffffu, mine);
      const int k = cnt + __popc(m & ((1u << lane) - 1u));
      if (mine && k < SLOTS) s_pairs[k] = pr;
      cnt += __popc(m);
    }
    if (lane == 0) {
      s_ok = cnt == SLOTS;
      // every token has SLOTS pairs; without them nothing is combined
      if (cnt != SLOTS && blockIdx.x == 0) set_error(a.ws.hdr, DEV_BAD_ROUTING);
    }
  }
  __syncthreads();
  if (!s_ok) return;
  const float* y = ws_y(a.ws, a.B);
  const int r = blockIdx.x * 256 + threadIdx.x;
  float yv[SLOTS];
#pragma unroll
  for (int j = 0; j < SLOTS; ++j) yv[j] = __ldcg(y + (size_t)s_pairs[j] * H + r);
  float v = 0.f;
#pragma unroll
  for (int j = 0; j < SLOTS; ++j) v += yv[j];
  const size_t o = (size_t)t * H + r;
  a.out[o] = f2bf(bf_lo((uint32_t)a.residual[o]) + v);
}

cudaError_t launch_down_nvfp4(const ExpertArgs& a, cudaStream_t stream, int num_sms) {
  static std::atomic<uint64_t> smem_set{0};
  const cudaError_t es = set_smem_limit_once(down_nvfp4_kernel, f4::SMEM_CAP, smem_set);
  if (es != cudaSuccess) return es;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms, 1, 1);
  cfg.blockDim = dim3(f4::THREADS, 1, 1);
  cfg.dynamicSmemBytes = f4::dn_smem(a.B);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, down_nvfp4_kernel, a);
}

cudaError_t launch_combine_y(const ExpertArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(H / 256, a.B, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_y_kernel, a);
}

}  // namespace flint
