// router.cu — router GEMV, sigmoid top-k with renormalisation, and token-to-
// expert bucketing for the Flint decode MoE layer.
//
// "256 experts, employing a sigmoid top-6 selection mechanism plus a shared
// expert" [vLLM Day-0 Support for Recursive's Flint, "Flint Model
// Architecture"]; the router reads its 1 MiB matrix once per batch and the
// experts downstream read only the selected experts' weights ("Small-batch MoE
// Kernels", same page, "Optimization Strategies").
//
// One launch does all three steps without any device-side wait:
//   grid (E/2, ceil(B/8)), 256 threads: each CTA dots two router rows with an
//   8-token tile (fp32 accumulation, warp-shuffle and shared-memory sums).
//   The last CTA to finish a token tile (atomic ticket after a fence) ranks
//   that tile's tokens, one warp per token; with a single tile it buckets the
//   batch right away from shared memory, otherwise the last tile to finish
//   buckets it.  Tickets are reset by their last user, so the workspace is
//   ready for the next call.
#include "common.cuh"
#include "kernels.h"

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

// Order-preserving map of fp32 onto uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f2key(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Top-k of one token's E logits by one warp.  Lane l holds experts l + 32 j.
// Each round takes the largest remaining logit; among equal logits the lowest
// expert index wins (ties resolved first within a lane by ascending j, then
// across lanes by the minimum index).  Weights: sigmoid of the selected
// logits divided by their sum.
__device__ void topk_token(const float* logits_row, int* idx_out, float* w_out,
                           int* user_idx, float* user_w, int* s_idx, float* s_w) {
  const int lane = threadIdx.x & 31;
  float v[E / 32];
#pragma unroll
  for (int j = 0; j < E / 32; ++j) v[j] = __ldcg(logits_row + lane + 32 * j);
  uint32_t taken = 0;
  int sel_e[TOPK];
  float sel_v[TOPK];
#pragma unroll
  for (int r = 0; r < TOPK; ++r) {
    uint32_t best_key = 0;
    uint32_t best_e = 0xffffffffu;
#pragma unroll
    for (int j = 0; j < E / 32; ++j) {
      const uint32_t k = f2key(v[j]);
      const bool free_j = !((taken >> j) & 1u);
      if (free_j && (best_e == 0xffffffffu || k > best_key)) {
        best_key = k;
        best_e = (uint32_t)(lane + 32 * j);
      }
    }
    const uint32_t top = __reduce_max_sync(0xffffffffu, best_key);
    const uint32_t win = __reduce_min_sync(0xffffffffu, best_key == top ? best_e : 0xffffffffu);
    if ((int)(win & 31u) == lane) taken |= 1u << (win >> 5);
    sel_e[r] = (int)win;
    sel_v[r] = key2f(top);
  }
  float s[TOPK], ssum = 0.f;
#pragma unroll
  for (int r = 0; r < TOPK; ++r) {
    s[r] = 1.0f / (1.0f + expf(-sel_v[r]));
    ssum += s[r];
  }
  if (lane < TOPK) {
    float wl = 0.f;
    int el = 0;
#pragma unroll
    for (int r = 0; r < TOPK; ++r)
      if (r == lane) { wl = s[r] / ssum; el = sel_e[r]; }
    idx_out[lane] = el;
    w_out[lane] = wl;
    if (user_idx) user_idx[lane] = el;
    if (user_w) user_w[lane] = wl;
    s_idx[lane] = el;
    s_w[lane] = wl;
  }
}

// Block-wide exclusive scan of one int per thread (256 threads).
__device__ int block_excl_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    int c = s_warp[w];
    if (w < warp) base += c;
    tot += c;
  }
  __syncthreads();
  *total = tot;
  return base + incl - v;
}

}  // namespace

// Buckets the batch's (token, slot) pairs by expert.  Called by one 256-thread
// CTA after every token's top-k is final.  Produces, in the workspace:
//   pair_tok/pair_w: routed pairs ordered by (expert, token), then the shared
//                    experts' pairs (token order, weight 1);
//   groups:          (expert, first pair, count <= GROUP_MAX) in that order,
//                    routed groups first, shared groups last;
//   n_groups, n_uniq in the header.
// Optionally also the plain bucket description (distinct experts ascending,
// their first pair, and the pairs encoded token*8 + slot).
template <bool SMEM_SRC>
__device__ __forceinline__ int ld_idx(const int* p) { return SMEM_SRC ? *p : __ldcg(p); }
template <bool SMEM_SRC>
__device__ __forceinline__ float ld_w(const float* p) { return SMEM_SRC ? *p : __ldcg(p); }

template <bool SMEM_SRC>
__device__ void bucket_batch(const Ws& ws, int B, BucketOut user, const int* src_idx,
                             const float* src_w) {
  constexpr int MW = MAX_B / 32;
  __shared__ uint32_t s_mask[E][MW];  // token bitmask per expert
  __shared__ int s_off[E];            // first pair of each expert
  __shared__ int s_warp[8];
  const int tid = threadIdx.x;
  for (int i = tid; i < E * MW; i += 256) (&s_mask[0][0])[i] = 0u;
  __syncthreads();
  const int npairs = B * TOPK;
  for (int p = tid; p < npairs; p += 256) {
    const int e = ld_idx<SMEM_SRC>(src_idx + p);
    const int t = p / TOPK;
    if (e < 0 || e >= E) {
      set_error(ws.hdr, DEV_BAD_ROUTING);
      continue;
    }
    const uint32_t bit = 1u << (t & 31);
    if (atomicOr(&s_mask[e][t >> 5], bit) & bit) set_error(ws.hdr, DEV_BAD_ROUTING);
  }
  __syncthreads();
  const int e = tid;  // one expert per thread (E == 256 == blockDim.x)
  int cnt = 0;
#pragma unroll
  for (int w = 0; w < MW; ++w) cnt += __popc(s_mask[e][w]);
  const int ng = (cnt + GROUP_MAX - 1) / GROUP_MAX;
  int tot_pairs, tot_groups, n_uniq;
  const int off = block_excl_scan(cnt, s_warp, &tot_pairs);
  const int goff = block_excl_scan(ng, s_warp, &tot_groups);
  const int urank = block_excl_scan(cnt > 0 ? 1 : 0, s_warp, &n_uniq);
  s_off[e] = off;
  for (int gi = 0; gi < ng; ++gi) {
    const int c = min(GROUP_MAX, cnt - gi * GROUP_MAX);
    ws.groups[goff + gi] = make_int4(e, off + gi * GROUP_MAX, c, 0);
  }
  if (user.uniq && cnt > 0) {
    user.uniq[urank] = e;
    user.offsets[urank] = off;
  }
  __syncthreads();
  // Each pair goes to its expert's first slot plus its rank among the expert's
  // tokens (the set bits of the expert's mask below the token).
  for (int p = tid; p < npairs; p += 256) {
    const int ex = ld_idx<SMEM_SRC>(src_idx + p);
    const int t = p / TOPK;
    if (ex < 0 || ex >= E) continue;
    const int wd = t >> 5;
    int rank = __popc(s_mask[ex][wd] & ((1u << (t & 31)) - 1u));
    for (int w = 0; w < wd; ++w) rank += __popc(s_mask[ex][w]);
    const int pos = s_off[ex] + rank;
    ws.pair_tok[pos] = t;
    ws.pair_w[pos] = ld_w<SMEM_SRC>(src_w + p);
    if (user.pairs) user.pairs[pos] = t * 8 + (p - t * TOPK);
  }
  // Shared experts: every token, weight 1, after the routed pairs.
  const int nsg = (B + GROUP_MAX - 1) / GROUP_MAX;
  for (int i = tid; i < S * B; i += 256) {
    ws.pair_tok[npairs + i] = i % B;
    ws.pair_w[npairs + i] = 1.0f;
  }
  for (int i = tid; i < S * nsg; i += 256) {
    const int s = i / nsg, gi = i % nsg;
    ws.groups[tot_groups + i] =
        make_int4(E + s, npairs + s * B + gi * GROUP_MAX, min(GROUP_MAX, B - gi * GROUP_MAX), 0);
  }
  if (tid == 0) {
    ws.hdr->n_groups = (uint32_t)(tot_groups + S * nsg);
    ws.hdr->n_uniq = (uint32_t)n_uniq;
    if (user.offsets) user.offsets[n_uniq] = npairs;
    if (user.n_uniq) *user.n_uniq = n_uniq;
  }
}

// grid (E/2, ceil(B/8)), 256 threads.  Warp w of CTA (bx, by) owns expert
// 2*bx + w/4 and the K-quarter w%4; each lane holds two 16-byte chunks of the
// router row and issues all 16 activation loads of the 8-token tile at once,
// so the whole tile costs one memory round trip.  The four quarter sums are
// combined in shared memory.
__global__ void __launch_bounds__(256) router_kernel(RouterArgs a) {
  pdl_wait();     // x may come from the preceding kernel in the stream
  pdl_trigger();  // the expert kernels may start their prologue
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int el = warp >> 2, qk = warp & 3;
  const int e = blockIdx.x * 2 + el;
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

  const int c0 = qk * 64 + lane, c1 = c0 + 32;  // 16-byte chunks of the 4 KiB row
  const uint4* wrow = reinterpret_cast<const uint4*>(a.wr + (size_t)e * H);
  const uint4 w0 = ldg_stream(wrow + c0), w1 = ldg_stream(wrow + c1);
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
      const float v = (s_part[le][0][t] + s_part[le][1][t]) + (s_part[le][2][t] + s_part[le][3][t]) +
                      (a.bias ? __ldg(a.bias + ee) : 0.0f);
      a.ws.logits[(size_t)(t0 + t) * E + ee] = v;
    }
  }

  // The last CTA to finish this token tile ranks its tokens.
  __shared__ uint32_t s_ticket;
  __shared__ int s_idx[8 * TOPK];
  __shared__ float s_w[8 * TOPK];
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_ticket = atomicAdd(&hdr->tile_ctas_done[blockIdx.y], 1u);
  }
  __syncthreads();
  if (s_ticket != gridDim.x - 1) return;
  __threadfence();
  if (threadIdx.x == 0) hdr->tile_ctas_done[blockIdx.y] = 0u;
  if (warp < nt) {
    const int t = t0 + warp;
    topk_token(a.ws.logits + (size_t)t * E, a.ws.topk_idx + (size_t)t * TOPK,
               a.ws.topk_w + (size_t)t * TOPK,
               a.user_idx ? a.user_idx + (size_t)t * TOPK : nullptr,
               a.user_w ? a.user_w + (size_t)t * TOPK : nullptr, s_idx + warp * TOPK,
               s_w + warp * TOPK);
  }
  if (!a.do_bucket) return;
  __syncthreads();
  if (gridDim.y == 1) {  // one token tile: the routing is already in shared memory
    bucket_batch<true>(a.ws, a.B, a.bucket, s_idx, s_w);
    return;
  }
  if (threadIdx.x == 0) {
    __threadfence();
    s_ticket = atomicAdd(&hdr->tiles_done, 1u);
  }
  __syncthreads();
  if (s_ticket != gridDim.y - 1) return;
  __threadfence();
  if (threadIdx.x == 0) hdr->tiles_done = 0u;
  bucket_batch<false>(a.ws, a.B, a.bucket, a.ws.topk_idx, a.ws.topk_w);
}

__global__ void __launch_bounds__(256) bucket_kernel(Ws ws, int B, BucketOut user) {
  pdl_wait();
  pdl_trigger();
  bucket_batch<false>(ws, B, user, ws.topk_idx, ws.topk_w);
}

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(E / 2, (a.B + 7) / 8, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, router_kernel, a);
}

cudaError_t launch_bucket(const Ws& ws, int B, const BucketOut& user, cudaStream_t stream) {
  bucket_kernel<<<1, 256, 0, stream>>>(ws, B, user);
  return cudaGetLastError();
}

}  // namespace flint
