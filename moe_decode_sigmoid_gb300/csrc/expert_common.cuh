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

struct ConsumerSync {
  __device__ __forceinline__ void operator()() const { named_sync(1, CONSUMER_THREADS); }
};

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
      topk_warp<false>(logits_buf + warp * E, ix, wt);
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
    BucketDst d;
    d.pair_tok = m.pair_tok;
    d.pair_w = ls->pair_w;
    d.groups = m.groups;
    d.n_groups = &m.n_groups;
    d.n_uniq = nullptr;
    BucketOut none = {nullptr, nullptr, nullptr, nullptr};
    bool bad = false;  // indices come from topk_warp: always valid
    bucket_cta<1, false>(B, ls->idx, ls->w, d, none, ls->sc, bad, ConsumerSync());
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
