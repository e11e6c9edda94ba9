// expert_common.cuh — routing metadata the expert kernels keep in shared
// memory for their whole launch, and the prologue that fills it.
//
// The group table and the pairs' tokens (and, for the down kernels, weights)
// are read once per CTA -- one memory round trip -- instead of once per group
// on the critical path.  For batches of at most LOCAL_SELECT_MAX_B tokens the
// gate/up kernels do not wait for a routing pass at all: every CTA ranks the
// batch's tokens from the router's logits and buckets them in shared memory
// (a few hundred cycles), and CTA 0 publishes the result to the workspace for
// the down kernel and the caller.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace flint {

// Barrier 1: the 8 consumer warps.  Barrier 2: consumers + producer warp.
constexpr int CONSUMER_THREADS = 256;
constexpr int ALL_THREADS = CONSUMER_THREADS + 32;

struct MetaSmem {
  int4 groups[MAX_GROUPS];
  int pair_tok[MAX_B * SLOTS];
  int n_groups;
  int pad[3];
};

struct LocalSelectSmem {
  BucketScratch<1> sc;
  int idx[LOCAL_SELECT_MAX_B * TOPK];
  float w[LOCAL_SELECT_MAX_B * TOPK];
  float pair_w[LOCAL_SELECT_MAX_B * SLOTS];
};

// Buckets the batch's (token, slot) pairs by expert for B <= 8 tokens, by
// NTHREADS threads (>= LANES * LOCAL_SELECT_MAX_B * TOPK): with at most 8 tokens
// every distinct expert forms one group (GROUP_MAX is larger), so pair p is
// ranked directly against all pairs -- its position is the number of pairs
// with a smaller expert plus those of the same expert from lower tokens --
// and one counting barrier gives the number of distinct experts.  The result is the group table and
// pair order of bucket_cta: routed groups by expert ascending (tokens
// ascending inside), then the shared expert's group of all tokens.
template <int NTHREADS, int LANES>
__device__ __forceinline__ void bucket_small(int B, const int* idx, const float* w, int* pair_tok,
                                             float* pair_w, int4* groups, int* n_groups,
                                             int* opener) {
  static_assert(LANES == 1 || LANES == 2 || LANES == 4, "lanes per pair divide a warp");
  static_assert(NTHREADS >= LANES * LOCAL_SELECT_MAX_B * TOPK, "LANES threads per pair");
  if constexpr (LANES == 1) {
    const int tid = threadIdx.x;
    const int np = B * TOPK;
    int e = 0, pos = 0, cnt = 0;
    bool first = false;
    if (tid < np) {
      e = idx[tid];
      int less = 0, before = 0;
      for (int q = 0; q < np; ++q) {
        const int eq = idx[q];
        less += eq < e ? 1 : 0;
        cnt += eq == e ? 1 : 0;
        before += (eq == e && q < tid) ? 1 : 0;
      }
      pos = less + before;
      first = before == 0;
      pair_tok[pos] = tid / TOPK;
      pair_w[pos] = w[tid];
      opener[tid] = first ? e : 0x7fffffff;  // experts whose first pair this is
    }
    if (tid < S * B) {
      pair_tok[np + tid] = tid % B;
      pair_w[np + tid] = 1.0f;
    }
    uint32_t n_uniq;
    asm volatile("{ .reg .pred p; setp.ne.u32 p, %1, 0; bar.red.popc.u32 %0, 1, %2, p; }"
                 : "=r"(n_uniq)
                 : "r"((tid < np && first) ? 1u : 0u), "n"(NTHREADS)
                 : "memory");
    if (tid < np && first) {
      int g = 0;
      for (int q = 0; q < np; ++q) g += opener[q] < e ? 1 : 0;
      groups[g] = make_int4(e, pos, cnt, 0);
    }
    if (tid == 0) {
      groups[n_uniq] = make_int4(E, np, B, 0);
      *n_groups = (int)n_uniq + S;
    }
  } else {
    const int tid = threadIdx.x;
    const int np = B * TOPK;
    // LANES adjacent lanes per pair p: each compares against every LANES-th
    // pair, then shuffles add their counts (fewer serial loads per thread).
    const int p = tid / LANES, part = tid % LANES;
    const bool act = p < np;
    const int e = act ? idx[p] : 0;
    int less = 0, cnt = 0, before = 0;
    if (act) {
      for (int q = part; q < np; q += LANES) {
        const int eq = idx[q];
        less += eq < e ? 1 : 0;
        cnt += eq == e ? 1 : 0;
        before += (eq == e && q < p) ? 1 : 0;
      }
    }
#pragma unroll
    for (int o = 1; o < LANES; o <<= 1) {
      less += __shfl_xor_sync(0xffffffffu, less, o);
      cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      before += __shfl_xor_sync(0xffffffffu, before, o);
    }
    const int pos = less + before;
    const bool first = act && before == 0;
    if (act && part == 0) {
      pair_tok[pos] = p / TOPK;
      pair_w[pos] = w[p];
      opener[p] = first ? e : 0x7fffffff;  // experts whose first pair this is
    }
    if (tid < S * B) {
      pair_tok[np + tid] = tid % B;
      pair_w[np + tid] = 1.0f;
    }
    uint32_t n_uniq;
    asm volatile("{ .reg .pred p; setp.ne.u32 p, %1, 0; bar.red.popc.u32 %0, 1, %2, p; }"
                 : "=r"(n_uniq)
                 : "r"((first && part == 0) ? 1u : 0u), "n"(NTHREADS)
                 : "memory");
    int g = 0;
    if (first) {
      for (int q = part; q < np; q += LANES) g += opener[q] < e ? 1 : 0;
    }
#pragma unroll
    for (int o = 1; o < LANES; o <<= 1) g += __shfl_xor_sync(0xffffffffu, g, o);
    if (first && part == 0) groups[g] = make_int4(e, pos, cnt, 0);
    if (tid == 0) {
      groups[n_uniq] = make_int4(E, np, B, 0);
      *n_groups = (int)n_uniq + S;
    }
  }
}

// Run by the 256 consumer threads after the grid dependency is satisfied.
// logits_buf: >= LOCAL_SELECT_MAX_B * E floats of shared memory, free here.
// pair_w: shared array for the pairs' weights, or null if not needed.
__device__ __forceinline__ void fill_meta(const ExpertArgs& a, bool local, MetaSmem& m,
                                          float* pair_w, float* logits_buf, LocalSelectSmem* ls) {
  const int tid = threadIdx.x;
  const int B = a.B;
  if (local) {
    // thread e loads expert e's logit of every token (all loads in flight at once)
    float lv[LOCAL_SELECT_MAX_B];
#pragma unroll
    for (int t = 0; t < LOCAL_SELECT_MAX_B; ++t)
      lv[t] = t < B ? __ldcg(a.ws.logits + (size_t)t * E + tid) : 0.f;
#pragma unroll
    for (int t = 0; t < LOCAL_SELECT_MAX_B; ++t)
      if (t < B) logits_buf[t * E + tid] = lv[t];
    named_sync(1, CONSUMER_THREADS);
    const int warp = tid >> 5, lane = tid & 31;
    if (warp < B) {
      int ix;
      float wt;
      topk_warp<false>(logits_buf + warp * E, a.bias, a.bias_select_only != 0, ix, wt);
      if (lane < TOPK) {
        const int p = warp * TOPK + lane;
        ls->idx[p] = ix;
        ls->w[p] = wt;
        if (blockIdx.x == 0) {
          a.ws.topk_idx[p] = ix;
          a.ws.topk_w[p] = wt;
          if (a.user_idx) a.user_idx[p] = ix;
          if (a.user_w) a.user_w[p] = wt;
        }
      }
    }
    named_sync(1, CONSUMER_THREADS);
    // indices come from topk_warp: always valid
    // one lane per pair here: these kernels measured faster with it
    bucket_small<CONSUMER_THREADS, 1>(B, ls->idx, ls->w, m.pair_tok, ls->pair_w, m.groups,
                                      &m.n_groups, ls->sc.off);
    named_sync(1, CONSUMER_THREADS);
    if (pair_w)
      for (int i = tid; i < B * SLOTS; i += CONSUMER_THREADS) pair_w[i] = ls->pair_w[i];
    if (blockIdx.x == 0) {  // the down kernel and the caller read the routing here
      const int n = m.n_groups;
      for (int i = tid; i < n; i += CONSUMER_THREADS) a.ws.groups[i] = m.groups[i];
      for (int i = tid; i < B * SLOTS; i += CONSUMER_THREADS) {
        a.ws.pair_tok[i] = m.pair_tok[i];
        a.ws.pair_w[i] = ls->pair_w[i];
      }
      if (tid == 0) a.ws.hdr->n_groups = (uint32_t)n;
    }
  } else {
    // Loads first, stores after, so the round trips overlap (the loop bounds
    // are at most MAX_GROUPS and MAX_B * SLOTS).
    const int n = (int)__ldcg(&a.ws.hdr->n_groups);
    constexpr int GR = (MAX_GROUPS + CONSUMER_THREADS - 1) / CONSUMER_THREADS;
    constexpr int PR = (MAX_B * SLOTS + CONSUMER_THREADS - 1) / CONSUMER_THREADS;
    int4 gv[GR];
    int tv[PR];
    float wv[PR];
#pragma unroll
    for (int k = 0; k < GR; ++k) {
      const int i = tid + k * CONSUMER_THREADS;
      gv[k] = i < n ? __ldcg(a.ws.groups + i) : make_int4(0, 0, 0, 0);
    }
#pragma unroll
    for (int k = 0; k < PR; ++k) {
      const int i = tid + k * CONSUMER_THREADS;
      const bool in = i < B * SLOTS;
      tv[k] = in ? __ldcg(a.ws.pair_tok + i) : 0;
      wv[k] = in && pair_w ? __ldcg(a.ws.pair_w + i) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < GR; ++k) {
      const int i = tid + k * CONSUMER_THREADS;
      if (i < n) m.groups[i] = gv[k];
    }
#pragma unroll
    for (int k = 0; k < PR; ++k) {
      const int i = tid + k * CONSUMER_THREADS;
      if (i < B * SLOTS) {
        m.pair_tok[i] = tv[k];
        if (pair_w) pair_w[i] = wv[k];
      }
    }
    if (tid == 0) m.n_groups = n;
  }
  named_sync(1, CONSUMER_THREADS);
}

}  // namespace flint
