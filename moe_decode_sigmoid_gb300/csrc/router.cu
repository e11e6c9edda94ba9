// router.cu — router GEMV, sigmoid top-k with renormalisation, and token-to-
// expert bucketing for the Flint decode MoE layer.
//
// "256 experts, employing a sigmoid top-6 selection mechanism plus a shared
// expert" [vLLM Day-0 Support for Recursive's Flint, "Flint Model
// Architecture"]; the router reads its 1 MiB matrix once per batch and the
// experts downstream read only the selected experts' weights ("Small-batch MoE
// Kernels", same page, "Optimization Strategies").
//
// grid (E/2, ceil(B/8)), 256 threads: each CTA dots two router rows with an
// 8-token tile (fp32 accumulation; warp w owns expert 2*bx + w/4 and the
// K-quarter w%4; all loads of the tile are issued at once, so the tile costs
// one memory round trip; the quarter sums meet in shared memory).
// Then, without any device-side wait:
//   - logits-only mode (the batch <= 8 decode chain): done; every expert-kernel
//     CTA ranks and buckets the tokens itself from the logits;
//   - otherwise the last CTA to finish a token tile (atomic ticket after a
//     fence) ranks that tile's tokens, one warp per token; with a single tile
//     it buckets the batch right away from shared memory, else the last tile
//     to finish buckets it.  Tickets are reset by their last user, so the
//     workspace is ready for the next call.
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace flint {

namespace {

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

struct SyncCta {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

__device__ __forceinline__ BucketDst ws_dst(const Ws& ws) {
  BucketDst d;
  d.pair_tok = ws.pair_tok;
  d.pair_w = ws.pair_w;
  d.groups = ws.groups;
  d.n_groups = reinterpret_cast<int*>(&ws.hdr->n_groups);
  d.n_uniq = reinterpret_cast<int*>(&ws.hdr->n_uniq);
  return d;
}

// After a CTA's logits of token tile blockIdx.y (TT tokens from t0, nt of
// them real): the last CTA to finish the tile (atomic ticket after a fence)
// ranks its tokens, one warp per token; with a single tile it buckets the
// batch right away from shared memory, else the last tile to finish buckets
// it.  Tickets are reset by their last user.
template <int TT>
__device__ __forceinline__ void route_tail(const RouterArgs& a, int t0, int nt) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  WsHeader* hdr = a.ws.hdr;
  __shared__ uint32_t s_ticket;
  __shared__ int s_idx[TT * TOPK];
  __shared__ float s_w[TT * TOPK];
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_ticket = atomicAdd(&hdr->tile_ctas_done[blockIdx.y], 1u);
  }
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  if (threadIdx.x == 0) hdr->tile_ctas_done[blockIdx.y] = 0u;
  for (int j = warp; j < nt; j += 8) {
    const int t = t0 + j;
    int ix;
    float wt;
    topk_warp<true>(a.ws.logits + (size_t)t * E, a.bias, a.bias_select_only != 0, ix, wt);
    if (lane < TOPK) {
      a.ws.topk_idx[t * TOPK + lane] = ix;
      a.ws.topk_w[t * TOPK + lane] = wt;
      if (a.user_idx) a.user_idx[t * TOPK + lane] = ix;
      if (a.user_w) a.user_w[t * TOPK + lane] = wt;
      s_idx[j * TOPK + lane] = ix;
      s_w[j * TOPK + lane] = wt;
    }
  }
  if (!a.do_bucket) return;
  __syncthreads();
  bool bad = false;
  if (gridDim.y == 1) {  // one token tile: the routing is already in shared memory
    __shared__ BucketScratch<1> sc1;
    bucket_cta<1, false>(a.B, s_idx, s_w, ws_dst(a.ws), a.bucket, sc1, bad, SyncCta());
  } else {
    if (threadIdx.x == 0) {
      __threadfence();
      s_ticket = atomicAdd(&hdr->tiles_done, 1u);
    }
    __syncthreads();
    if (s_ticket != gridDim.y - 1) return;
    __threadfence();
    if (threadIdx.x == 0) hdr->tiles_done = 0u;
    __shared__ BucketScratch<MAX_B / 32> sc8;
    bucket_cta<MAX_B / 32, true>(a.B, a.ws.topk_idx, a.ws.topk_w, ws_dst(a.ws), a.bucket, sc8, bad,
                                 SyncCta());
  }
  if (bad) set_error(hdr, DEV_BAD_ROUTING);
}

}  // namespace

__global__ void __launch_bounds__(256) router_kernel(RouterArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int el = warp >> 2, qk = warp & 3;
  const int e = blockIdx.x * 2 + el;
  const int c0 = qk * 64 + lane, c1 = c0 + 32;  // 16-byte chunks of the 4 KiB row
  const uint4* wrow = reinterpret_cast<const uint4*>(a.wr + (size_t)e * H);
  // The router rows are weights, which no kernel writes: their loads start
  // before the wait, so they overlap the end of the preceding kernel.
  const uint4 w0 = ldg_stream(wrow + c0), w1 = ldg_stream(wrow + c1);
  pdl_wait();     // x may come from the preceding kernel in the stream
  pdl_trigger();  // the expert kernels may start their prologue
  const int t0 = blockIdx.y * 8;
  const int nt = min(8, a.B - t0);
  WsHeader* hdr = a.ws.hdr;

  if (a.stall_check && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 &&
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

  uint4 xv[8][2];
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    if (t < nt) {
      const uint4* xrow = reinterpret_cast<const uint4*>(a.x + (size_t)(t0 + t) * H);
      xv[t][0] = __ldg(xrow + c0);
      xv[t][1] = __ldg(xrow + c1);
    } else {
      xv[t][0] = xv[t][1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  float acc[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t] = dot8(w1, xv[t][1], dot8(w0, xv[t][0], 0.f));
#pragma unroll
  for (int t = 0; t < 8; ++t) acc[t] = warp_sum(acc[t]);
  __shared__ float s_part[2][4][8];
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < 8; ++t) s_part[el][qk][t] = acc[t];
  }
  __syncthreads();
  if (threadIdx.x < 16) {
    const int le = threadIdx.x >> 3, t = threadIdx.x & 7;
    if (t < nt) {
      const int ee = blockIdx.x * 2 + le;
      a.ws.logits[(size_t)(t0 + t) * E + ee] =  // the router score; offsets join at ranking
          (s_part[le][0][t] + s_part[le][1][t]) + (s_part[le][2][t] + s_part[le][3][t]);
    }
  }
  if (a.logits_only) return;

  route_tail<8>(a, t0, nt);
}

__global__ void __launch_bounds__(256) bucket_kernel(Ws ws, int B, BucketOut user) {
  pdl_wait();
  pdl_trigger();
  __shared__ BucketScratch<MAX_B / 32> sc;
  bool bad = false;
  bucket_cta<MAX_B / 32, true>(B, ws.topk_idx, ws.topk_w, ws_dst(ws), user, sc, bad, SyncCta());
  if (bad) set_error(ws.hdr, DEV_BAD_ROUTING);
}

// Batches above 8: the router product [B, H] x [H, E] on tensor cores.
// grid (E/8, ceil(B/16)), 256 threads: each CTA takes 8 experts (the MMA's N)
// and a 16-token tile (its M; tokens past B read nothing and stay zero); warp
// w takes the 256-column K-slice w, thread q of a quad the 8 columns
// 32b + 8q .. +7 of block b for both K-steps of the block, on both operands
// (one 16-byte load each, from L2), so every dot product is complete.  The 8
// warps' partial tiles meet in shared memory in a fixed order.  Then the same
// ranking / bucketing tail as router_kernel, with 16-token tiles.  Against
// 8-token tiles of 2 experts, x is re-read 4x less often from L2.
__global__ void __launch_bounds__(256) router_mma_kernel(RouterArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int e0 = blockIdx.x * 8, t0 = blockIdx.y * 16;
  const uint4* wrow = reinterpret_cast<const uint4*>(a.wr + (size_t)(e0 + g) * H);
  uint4 wv[8];
#pragma unroll
  for (int b = 0; b < 8; ++b) wv[b] = ldg_stream(wrow + warp * 32 + b * 4 + q);  // before the wait, as above
  pdl_wait();     // x may come from the preceding kernel in the stream
  pdl_trigger();  // the expert kernels may start their prologue
  const int nt = min(16, a.B - t0);
  WsHeader* hdr = a.ws.hdr;
  if (a.stall_check && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 &&
      *reinterpret_cast<volatile uint32_t*>(&hdr->stall_armed)) {
    // Test hook: as in router_kernel.
    const uint64_t deadline = wait_deadline(hdr);
    while (!*reinterpret_cast<volatile uint32_t*>(&hdr->stall_release)) {
      if (globaltimer_ns() > deadline) {
        set_error(hdr, DEV_TIMEOUT);
        break;
      }
    }
    hdr->stall_armed = 0;
  }
  const bool lo_in = g < nt, hi_in = g + 8 < nt;
  const uint4* xlo = reinterpret_cast<const uint4*>(a.x + (size_t)(t0 + (lo_in ? g : 0)) * H);
  const uint4* xhi = reinterpret_cast<const uint4*>(a.x + (size_t)(t0 + (hi_in ? g + 8 : 0)) * H);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 xl[8], xh[8];
#pragma unroll
  for (int b = 0; b < 8; ++b) {  // all loads of the slice in flight at once
    const int c = warp * 32 + b * 4 + q;  // 16-byte chunk: columns 256w + 32b + 8q
    xl[b] = lo_in ? __ldg(xlo + c) : zero;
    xh[b] = hi_in ? __ldg(xhi + c) : zero;
  }
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int b = 0; b < 8; ++b) {
    mma_bf16(acc[b & 1], xl[b].x, xh[b].x, xl[b].y, xh[b].y, wv[b].x, wv[b].y);
    mma_bf16(acc[b & 1], xl[b].z, xh[b].z, xl[b].w, xh[b].w, wv[b].z, wv[b].w);
  }
  // acc: (token g, expert 2q), (g, 2q+1), (g+8, 2q), (g+8, 2q+1)
  __shared__ float s_red[8][16][8];
  s_red[warp][g][2 * q] = acc[0][0] + acc[1][0];
  s_red[warp][g][2 * q + 1] = acc[0][1] + acc[1][1];
  s_red[warp][g + 8][2 * q] = acc[0][2] + acc[1][2];
  s_red[warp][g + 8][2 * q + 1] = acc[0][3] + acc[1][3];
  __syncthreads();
  if (threadIdx.x < 128) {
    const int t = threadIdx.x >> 3, e = threadIdx.x & 7;
    if (t < nt) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += s_red[w][t][e];
      a.ws.logits[(size_t)(t0 + t) * E + e0 + e] = v;  // the router score; offsets join at ranking
    }
  }
  route_tail<16>(a, t0, nt);
}

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  const bool mma = a.B > 8 && !a.logits_only;
  cfg.gridDim = mma ? dim3(E / 8, (a.B + 15) / 16, 1) : dim3(E / 2, (a.B + 7) / 8, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return mma ? cudaLaunchKernelEx(&cfg, router_mma_kernel, a)
             : cudaLaunchKernelEx(&cfg, router_kernel, a);
}

cudaError_t launch_bucket(const Ws& ws, int B, const BucketOut& user, cudaStream_t stream) {
  bucket_kernel<<<1, 256, 0, stream>>>(ws, B, user);
  return cudaGetLastError();
}

}  // namespace flint
