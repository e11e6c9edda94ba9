// common.cuh — shapes, workspace layout and sm_103a PTX helpers shared by the
// Flint decode-MoE kernels.  Device code only uses what is defined here and in
// the CUDA runtime headers.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace flint {

// ---- the specialised layer shape ------------------------------------------
constexpr int H = 2048;   // hidden
constexpr int E = 256;    // routed experts
constexpr int TOPK = 6;   // experts per token
constexpr int I = 512;    // expert intermediate size
constexpr int S = 1;      // shared experts
constexpr int MAX_B = 256;
constexpr int SLOTS = TOPK + S;          // h rows per token
constexpr int GROUP_MAX = 24;            // tokens per (expert, token-range) group
// Groups: each distinct expert contributes ceil(cnt/G) <= cnt/G + 1 groups,
// so routed groups <= TOPK*B/G + min(E, TOPK*B); plus S*ceil(B/G) shared.
constexpr int MAX_GROUPS = TOPK * MAX_B / GROUP_MAX + E + S * (MAX_B / GROUP_MAX + 1);

// Device error codes written to the workspace error word.
constexpr uint32_t DEV_OK = 0;
constexpr uint32_t DEV_BAD_ROUTING = 1;  // bucketing got an index outside [0,E) or a repeat
constexpr uint32_t DEV_BAD_INPUT = 1;    // an NVFP4 activation beyond its f16 operand's range
                                         // (|x| >= 65520, or |h| >= 65520 / NV_H_SCALE)
constexpr uint32_t DEV_TIMEOUT = 5;

// ---- workspace layout ------------------------------------------------------
// [ header | logits fp32 [MAX_B,E] | topk_idx i32 [MAX_B,K] | topk_w f32 [MAX_B,K] |
//   pair_tok i32 [MAX_B*SLOTS] | pair_w f32 [MAX_B*SLOTS] | groups int4 [MAX_GROUPS] |
//   tagged logits u64 [SMALL_B,E] | tagged h u64 [SMALL_B*SLOTS, I] |
//   tagged y u64 [SMALL_B*SLOTS, H] |
//   h [max_batch*SLOTS, I] x 4 bytes | y fp32 [max_batch*SLOTS, H] ]
// The tagged regions belong to the persistent small-batch kernels: each 8-byte
// word holds a 32-bit value and the call's tag (see call_tag), so a reader on
// another SM knows from the word itself whether it was written in this call.
// h holds the three-kernel paths' hi + lo pairs: the BF16 gate/up kernel's
// bf16 ones (see h_chunk) or the NVFP4 one's f16 ones (h_off_nv).
// Every array but the last two is sized for MAX_B (or the small-batch bound),
// so the offsets do not depend on the batch a workspace was sized for; h and y
// grow with max_batch, and a call with batch B finds y right after the first
// B * SLOTS h rows.
constexpr int SMALL_B = 8;  // largest batch of the persistent small-batch kernels
// Counters of the small-batch kernels, one per 128-byte line: polled by many
// SMs and bumped by many more, they must not share an L2 line (a shared line
// turns the polling into a hot spot that slows every access mapped there).
struct alignas(128) SyncLine {
  uint32_t v;
  uint32_t pad[31];
};
constexpr int SYNC_GROUPS = 64;               // completion counters per call
constexpr int SYNC_UNIT = SYNC_GROUPS;        // next unclaimed unit
constexpr int SYNC_ARRIVE = SYNC_GROUPS + 1;  // CTAs whose logits are stored
constexpr int SYNC_LINES = SYNC_GROUPS + 2;
struct WsHeader {
  uint32_t error;            // DEV_OK or an error code (first writer wins)
  uint32_t epoch;            // small-batch kernels: calls completed on this workspace
  uint64_t wait_limit_ns;    // bound of every device-side wait
  // ---- everything from here on may be cleared between calls ----
  uint32_t tiles_done;       // router: token tiles whose top-k is final
  uint32_t n_groups;         // number of (expert, token range) groups
  uint32_t n_uniq;           // distinct routed experts
  uint32_t stall_armed;      // test hook: one-shot wait on stall_release
  uint32_t stall_release;    // never written by the library
  uint32_t gu_claim;         // chained gate/up kernels: next unit to claim (reset by the last CTA)
  uint32_t gu_done;          // chained gate/up kernels: CTAs done claiming
  uint32_t dn_claim;         // NVFP4 down kernel: next unit to claim (reset by the last CTA)
  uint32_t dn_done;          // NVFP4 down kernel: CTAs done claiming
  uint32_t pad0[19];
  uint32_t tile_ctas_done[MAX_B / 8];  // router: finished CTAs per token tile
  uint32_t pad2[16];
  uint32_t pad1[176];
  // small-batch kernels, by epoch parity: completion counters of the groups,
  // the unit queue and the logits arrivals
  SyncLine sync[2][SYNC_LINES];
};
static_assert(sizeof(WsHeader) == 1024 + 2 * SYNC_LINES * 128, "header layout");
constexpr size_t WS_HDR_KEEP = 16;  // error, epoch, wait limit: not cleared between calls
static_assert(offsetof(WsHeader, tiles_done) == WS_HDR_KEEP, "clearable part starts at 16");
static_assert(offsetof(WsHeader, sync) == 1024, "counter lines start at 1 KiB");

__host__ __device__ constexpr size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

struct WsLayout {
  static constexpr size_t logits = sizeof(WsHeader);
  static constexpr size_t topk_idx = align256(logits + sizeof(float) * (size_t)MAX_B * E);
  static constexpr size_t topk_w = align256(topk_idx + sizeof(int) * (size_t)MAX_B * TOPK);
  static constexpr size_t pair_tok = align256(topk_w + sizeof(float) * (size_t)MAX_B * TOPK);
  static constexpr size_t pair_w = align256(pair_tok + sizeof(int) * (size_t)MAX_B * SLOTS);
  static constexpr size_t groups = align256(pair_w + sizeof(float) * (size_t)MAX_B * SLOTS);
  static constexpr size_t tlogits = align256(groups + 16 * (size_t)MAX_GROUPS);
  static constexpr size_t th = align256(tlogits + 8 * (size_t)SMALL_B * E);
  static constexpr size_t ty = align256(th + 8 * (size_t)SMALL_B * SLOTS * I);
  static constexpr size_t h = align256(ty + 8 * (size_t)SMALL_B * SLOTS * H);
  static constexpr size_t total(int max_b) {
    return align256(h + sizeof(float) * (size_t)max_b * SLOTS * (I + H));
  }
};

// Pointers into one workspace (built on the host, passed by value).
struct Ws {
  WsHeader* hdr;
  float* logits;
  uint64_t* tlogits;  // [SMALL_B][E] tagged
  uint64_t* th;       // [SMALL_B * SLOTS][I] tagged
  uint64_t* ty;       // [SMALL_B * SLOTS][H] tagged per-pair down projections
  int* topk_idx;
  float* topk_w;
  int* pair_tok;
  float* pair_w;
  int4* groups;   // {expert (E.. for shared), first pair, pair count, 0}
  float* h;
};
// Per-pair partial down projections of the NVFP4 path, [B * SLOTS][H] fp32,
// for a call with batch B.
__host__ __device__ inline float* ws_y(const Ws& w, int B) { return w.h + (size_t)B * SLOTS * I; }

inline Ws ws_view(void* base) {
  char* b = static_cast<char*>(base);
  Ws w;
  w.hdr = reinterpret_cast<WsHeader*>(b);
  w.logits = reinterpret_cast<float*>(b + WsLayout::logits);
  w.tlogits = reinterpret_cast<uint64_t*>(b + WsLayout::tlogits);
  w.th = reinterpret_cast<uint64_t*>(b + WsLayout::th);
  w.ty = reinterpret_cast<uint64_t*>(b + WsLayout::ty);
  w.topk_idx = reinterpret_cast<int*>(b + WsLayout::topk_idx);
  w.topk_w = reinterpret_cast<float*>(b + WsLayout::topk_w);
  w.pair_tok = reinterpret_cast<int*>(b + WsLayout::pair_tok);
  w.pair_w = reinterpret_cast<float*>(b + WsLayout::pair_w);
  w.groups = reinterpret_cast<int4*>(b + WsLayout::groups);
  w.h = reinterpret_cast<float*>(b + WsLayout::h);
  return w;
}

// ---- host: launch attributes -------------------------------------------------
// A kernel's dynamic shared-memory limit belongs to the current device's
// context, so it is set once per device (bit d of `done` for device d < 64;
// devices beyond that set it on every call), safely from any host thread.
template <class Kernel>
inline cudaError_t set_smem_limit_once(Kernel kernel, int bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev >= 0 && dev < 64 ? (uint64_t{1} << dev) : uint64_t{0};
  if (bit != 0u && (done.load(std::memory_order_acquire) & bit) != 0u) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// ---- small device helpers ---------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: wait for the preceding grid's completion and
// memory flush / allow the next grid to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
// try_wait that may suspend the thread for up to `ns` nanoseconds; the thread
// resumes when the phase completes, so a waiting warp leaves its scheduler's
// issue slots to the warps that compute instead of spinning.
constexpr uint32_t MBAR_SUSPEND_NS = 0;
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return done != 0;
}
// Bounded wait for the phase with the given parity; false if the deadline passed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t deadline) {
  if (mbar_try_wait(bar, parity)) return true;
  while (true) {
    if (MBAR_SUSPEND_NS > 0 ? mbar_try_wait_suspend(bar, parity, MBAR_SUSPEND_NS)
                            : mbar_try_wait(bar, parity))
      return true;
    if (globaltimer_ns() > deadline) return false;
  }
}

// 1-D bulk copy global -> shared (TMA engine); completion counted on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// L2 policy for the weight streams: evict first.  Every weight byte is read
// once per layer, so keeping it buys nothing, while the kernels' code, the
// activations, h and the routing tables -- reused within and across layers --
// would otherwise be pushed out of L2 by the stream.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// bulk_g2s for weight bytes (L2 evict-first).
__device__ __forceinline__ void bulk_g2s_stream(uint32_t dst, const void* src, uint32_t bytes,
                                                uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(l2_evict_first())
      : "memory");
}

// Bulk prefetch of global memory into L2 (no shared-memory destination).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Named barrier over the first `nthreads` threads (multiple of 32).
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// bf16 pair (one 32-bit word, low half first) -> two fp32.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// fp32 -> bf16 bits, round to nearest even.
__device__ __forceinline__ uint16_t f2bf(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
// Two fp32 -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  return (uint32_t)f2bf(lo) | ((uint32_t)f2bf(hi) << 16);
}

// (a, b) = hi + lo with hi = bf16(a, b) and lo = bf16 of the remainders; the
// pair carries ~16 significant bits of each fp32 value.
__device__ __forceinline__ void split_bf2(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf2(a, b);
  lo = pack_bf2(a - bf_lo(hi), b - bf_hi(hi));
}

// Split h rows.  Column k belongs to block b = k / 8; the row is 16 lines of
// 128 bytes, and block b lives in line kc = 2 (b / 8) + b % 2 at chunk pair
// q = (b % 8) / 2: its 8 hi = bf16(h) values in 16-byte chunk 2q and its 8
// lo = bf16(h - hi) values in chunk 2q + 1, both XOR-permuted by the row's
// pair index mod 8.  hi + lo keeps ~16 significant bits of the fp32 h, the
// parts are ready-made bf16 MMA operands, and a reader whose lane q takes
// block 8 (kc / 2) + 2q + kc % 2 at step kc finds the 8 lanes of each
// 128-bit load phase (two consecutive rows) in distinct banks.
__host__ __device__ __forceinline__ int h_chunk(size_t pair, int blk, int part) {
  const int line = 2 * (blk >> 3) + (blk & 1);
  const int q = (blk & 7) >> 1;
  return line * 128 + (((2 * q + part) ^ (int)(pair & 7)) * 16);
}

// One element.
__device__ __forceinline__ void store_h_split(float* h, size_t pair, int k, float v) {
  uint8_t* row = reinterpret_cast<uint8_t*>(h + pair * I);
  const uint16_t hi = f2bf(v);
  *reinterpret_cast<uint16_t*>(row + h_chunk(pair, k >> 3, 0) + (k & 7) * 2) = hi;
  *reinterpret_cast<uint16_t*>(row + h_chunk(pair, k >> 3, 1) + (k & 7) * 2) =
      f2bf(v - bf_lo((uint32_t)hi));
}

// A whole block at once: called by all 32 lanes of a warp, lanes 8m..8m+7
// holding elements 0..7 of one block (v); the first lane of each 8-lane group
// stores the two chunks when `store` is true (uniform within the group).
__device__ __forceinline__ void store_h_block8(float* h, size_t pair, int blk, float v,
                                               bool store) {
  const uint32_t hi = f2bf(v);
  const uint32_t lo = f2bf(v - bf_lo(hi));
  const uint32_t hw = hi | (__shfl_down_sync(0xffffffffu, hi, 1) << 16);
  const uint32_t lw = lo | (__shfl_down_sync(0xffffffffu, lo, 1) << 16);
  const uint4 hv = make_uint4(hw, __shfl_down_sync(0xffffffffu, hw, 2),
                              __shfl_down_sync(0xffffffffu, hw, 4),
                              __shfl_down_sync(0xffffffffu, hw, 6));
  const uint4 lv = make_uint4(lw, __shfl_down_sync(0xffffffffu, lw, 2),
                              __shfl_down_sync(0xffffffffu, lw, 4),
                              __shfl_down_sync(0xffffffffu, lw, 6));
  if ((threadIdx.x & 7) == 0 && store) {
    uint8_t* row = reinterpret_cast<uint8_t*>(h + pair * I);
    *reinterpret_cast<uint4*>(row + h_chunk(pair, blk, 0)) = hv;
    *reinterpret_cast<uint4*>(row + h_chunk(pair, blk, 1)) = lv;
  }
}

// The NVFP4 path's h: each value scaled by NV_H_SCALE (a power of two) as an
// f16 pair hi + lo -- ~22 significant bits, and the operand type of the down
// kernel's f16 MMAs, whose dequantised weights are exact in f16 -- for |h| <
// 65520 / NV_H_SCALE (~1.7e7; beyond that the gate/up kernel reports
// DEV_BAD_INPUT); one 2 KiB row per pair (pair p at byte 2048 p of the h
// region).  The
// 32-byte block b (columns 8b .. 8b + 7: 8 hi values, then 8 lo values) sits
// in 128-byte line b % 16 at slot b / 16 -- the order in which the NVFP4 down
// kernel's lanes take K (lane q: columns 128q .. 128q + 127, blocks 16q ..
// 16q + 15 in turn) -- with the two halves swapped in odd pairs, so that two
// consecutive rows read at the same step land in opposite 16-byte halves.
__host__ __device__ __forceinline__ int h_off_nv(size_t pair, int blk, int part) {
  return (blk & 15) * 128 + (blk >> 4) * 32 + ((part ^ (int)(pair & 1)) * 16);
}
constexpr float NV_H_SCALE = 1.0f / 256.0f;

// One block at once: called by all 32 lanes of a warp, lanes 8m..8m+7
// holding elements 0..7 of one block (v); the first lane of each 8-lane group
// stores the block when `store` is true (uniform within the group).  Returns
// true on a lane whose stored value is beyond the f16 range.
__device__ __forceinline__ bool store_h_block8_nv(float* h, size_t pair, int blk, float v,
                                                  bool store) {
  const float vs = v * NV_H_SCALE;
  const __half hh = __float2half_rn(vs);
  const __half hl = __float2half_rn(vs - __half2float(hh));
  const uint32_t hi = __half_as_ushort(hh);
  const uint32_t lo = __half_as_ushort(hl);
  const uint32_t hw = hi | (__shfl_down_sync(0xffffffffu, hi, 1) << 16);
  const uint32_t lw = lo | (__shfl_down_sync(0xffffffffu, lo, 1) << 16);
  const uint4 hv = make_uint4(hw, __shfl_down_sync(0xffffffffu, hw, 2),
                              __shfl_down_sync(0xffffffffu, hw, 4),
                              __shfl_down_sync(0xffffffffu, hw, 6));
  const uint4 lv = make_uint4(lw, __shfl_down_sync(0xffffffffu, lw, 2),
                              __shfl_down_sync(0xffffffffu, lw, 4),
                              __shfl_down_sync(0xffffffffu, lw, 6));
  if ((threadIdx.x & 7) == 0 && store) {
    uint8_t* row = reinterpret_cast<uint8_t*>(h) + pair * (I * 4);
    *reinterpret_cast<uint4*>(row + h_off_nv(pair, blk, 0)) = hv;
    *reinterpret_cast<uint4*>(row + h_off_nv(pair, blk, 1)) = lv;
  }
  return store && !(fabsf(vs) < 65520.0f);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Record a device error (first writer wins).
__device__ __forceinline__ void set_error(WsHeader* hdr, uint32_t code) {
  atomicCAS(&hdr->error, DEV_OK, code);
}

__device__ __forceinline__ uint64_t wait_deadline(const WsHeader* hdr) {
  uint64_t lim = *reinterpret_cast<const volatile uint64_t*>(&hdr->wait_limit_ns);
  return globaltimer_ns() + lim;
}

// silu(g) * u with silu(g) = g / (1 + exp(-g))
// ("SiLU-and-mul": Flint on Intel Arc Pro B70, "norm.py: Triton kernels that assumed CUDA").
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// ---- tagged words (cross-CTA publication without fences) ----------------------
// The persistent small-batch kernels publish values to other SMs as 8-byte
// words {value bits, tag} written by one 64-bit store: a reader that finds the
// call's tag in a word has that call's value, with no fence between writer and
// reader (a GPU-scope fence waits for the SM's outstanding memory traffic and
// costs microseconds while weight copies stream).  The tag is derived from the
// workspace's call counter (epoch, taken modulo 2^31) and never equals a
// zero-filled word; every call stamps all words of the tagged regions (the
// ones it does not use with a dead value), so a stale word always carries the
// previous call's tag, which differs from the current one.  Counters that
// announce completion are only hints: the reader confirms every word's tag and
// re-reads the ones that have not landed.
__host__ __device__ __forceinline__ uint32_t call_tag(uint32_t epoch) {
  return 0x80000000u | (epoch & 0x7fffffffu);
}
__device__ __forceinline__ void st_tagged(uint64_t* p, float v, uint32_t tag) {
  const uint64_t w = ((uint64_t)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged(const uint64_t* p) {
  uint64_t w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void red_add_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A tagged word's value if it carries `tag`; otherwise re-reads it from global
// memory until it does (bounded by `deadline`; false if the wait ran out).
__device__ __forceinline__ bool settle_tagged(uint64_t& w, const uint64_t* src, uint32_t tag,
                                              uint64_t deadline) {
  while ((uint32_t)(w >> 32) != tag) {
    if (globaltimer_ns() > deadline) return false;
    w = ld_tagged(src);
  }
  return true;
}

}  // namespace flint
