// select.cuh — sigmoid top-k selection and token-to-expert bucketing, used by
// the router kernel and, for small batches, inside the expert kernels.
//
// "256 experts, employing a sigmoid top-6 selection mechanism plus a shared
// expert" (vLLM Day-0 Support for Recursive's Flint, "Flint Model
// Architecture").  Experts are ranked by (logit descending, index ascending);
// the weights are the selected sigmoids divided by their sum.
#pragma once

#include "common.cuh"

namespace flint {

// Order-preserving map of fp32 onto uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f2key(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Compare-exchange of a sorting network: (key descending, expert ascending).
__device__ __forceinline__ void topk_cas(uint32_t (&k)[E / 32], uint32_t (&e)[E / 32], int i, int j) {
  const bool swap = k[j] > k[i] || (k[j] == k[i] && e[j] < e[i]);
  const uint32_t ki = k[i], ei = e[i];
  k[i] = swap ? k[j] : ki;
  e[i] = swap ? e[j] : ei;
  k[j] = swap ? ki : k[j];
  e[j] = swap ? ei : e[j];
}

// Top-k of one token's E router scores by one warp.  The ranking key of
// expert e is its score plus its logit offset (bias, may be null); lane l
// holds experts l + 32 j and first sorts its 8 (key, expert) pairs -- key
// descending, expert ascending -- with a 19-comparator sorting network
// (Batcher's odd-even merge sort).  Each round then takes the largest lane
// head; among equal keys the lowest expert index wins (a lane's head is its
// lowest index for that key, and across lanes the minimum index is taken).
// Each kept expert's weight is the sigmoid of its key -- or, with
// select_only, of its score without the offset -- divided by the sum over the
// kept experts.  Lanes 0..k-1 return slot `lane`'s expert and weight.
template <bool GLOBAL_SRC>
__device__ __forceinline__ void topk_warp(const float* logits_row, const float* bias,
                                          bool select_only, int& idx_out, float& w_out) {
  static_assert(E / 32 == 8, "the sorting network is written for 8 values per lane");
  const int lane = threadIdx.x & 31;
  uint32_t k[8], e[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float score =
        GLOBAL_SRC ? __ldcg(logits_row + lane + 32 * j) : logits_row[lane + 32 * j];
    k[j] = f2key(bias ? score + __ldg(bias + lane + 32 * j) : score);
    e[j] = (uint32_t)(lane + 32 * j);
  }
  topk_cas(k, e, 0, 1); topk_cas(k, e, 2, 3); topk_cas(k, e, 4, 5); topk_cas(k, e, 6, 7);
  topk_cas(k, e, 0, 2); topk_cas(k, e, 1, 3); topk_cas(k, e, 4, 6); topk_cas(k, e, 5, 7);
  topk_cas(k, e, 1, 2); topk_cas(k, e, 5, 6);
  topk_cas(k, e, 0, 4); topk_cas(k, e, 1, 5); topk_cas(k, e, 2, 6); topk_cas(k, e, 3, 7);
  topk_cas(k, e, 2, 4); topk_cas(k, e, 3, 5);
  topk_cas(k, e, 1, 2); topk_cas(k, e, 3, 4); topk_cas(k, e, 5, 6);
  int sel_e[TOPK];
  float sel_v[TOPK];
#pragma unroll
  for (int r = 0; r < TOPK; ++r) {
    const uint32_t top = __reduce_max_sync(0xffffffffu, k[0]);
    const uint32_t m = __ballot_sync(0xffffffffu, k[0] == top);
    uint32_t win;
    if ((m & (m - 1u)) == 0u)  // one lane holds the maximum (the usual case)
      win = __shfl_sync(0xffffffffu, e[0], __ffs(m) - 1);
    else
      win = __reduce_min_sync(0xffffffffu, k[0] == top ? e[0] : 0xffffffffu);
    if ((int)(win & 31u) == lane) {  // the winner pops its head
#pragma unroll
      for (int j = 0; j < 7; ++j) {
        k[j] = k[j + 1];
        e[j] = e[j + 1];
      }
      k[7] = 0u;
      e[7] = 0xffffffffu;
    }
    sel_e[r] = (int)win;
    sel_v[r] = key2f(top);
  }
  // Lane r < k computes sigmoid r; every lane then sums the k values in rank
  // order (the same order and rounding in every lane).
  float sv = 0.f, mine = 0.f;
#pragma unroll
  for (int r = 0; r < TOPK; ++r)
    if (r == lane) {
      mine = sel_v[r];
      idx_out = sel_e[r];
    }
  if (lane >= TOPK) idx_out = 0;
  if (select_only && bias && lane < TOPK)  // the sigmoid of the score itself
    mine = GLOBAL_SRC ? __ldcg(logits_row + idx_out) : logits_row[idx_out];
  sv = 1.0f / (1.0f + expf(-mine));
  float ssum = 0.f;
#pragma unroll
  for (int r = 0; r < TOPK; ++r) ssum += __shfl_sync(0xffffffffu, sv, r);
  w_out = lane < TOPK ? sv / ssum : 0.f;
}

// Optional plain description of the buckets (flint_moe_bucket).
struct BucketOut {
  int* uniq;     // [E]   distinct experts, ascending (first n_uniq valid)
  int* offsets;  // [E+1] first pair of each, then B*TOPK
  int* pairs;    // [B*TOPK] token*8 + slot, ordered by (expert, token)
  int* n_uniq;   // [1]
};

// Where the buckets go: pairs (routed ones ordered by (expert, token), then
// the shared experts' pairs in token order with weight 1) and the group table
// (expert, first pair, count <= GROUP_MAX), routed groups first.
struct BucketDst {
  int* pair_tok;
  float* pair_w;   // may be null
  int4* groups;
  int* n_groups;   // [1]
  int* n_uniq;     // [1] or null
};

// Scratch for bucket_cta, MW = 32-bit words of token mask per expert.
template <int MW>
struct BucketScratch {
  uint32_t mask[E][MW];
  int off[E];
  int warp_tot[8];
};

// Exclusive scan of one int per thread over 256 threads; `sync` is the
// barrier all 256 threads take.
template <typename Sync>
__device__ __forceinline__ int scan256(int v, int* warp_tot, int* total, Sync sync) {
  const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) & 7;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) warp_tot[warp] = incl;
  sync();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const int c = warp_tot[w];
    if (w < warp) base += c;
    tot += c;
  }
  sync();
  *total = tot;
  return base + incl - v;
}

// Buckets a batch's (token, slot) pairs by expert, by 256 threads (thread e
// owns expert e).  The routing is read from src_idx / src_w ([B, TOPK], shared
// or global memory).  Each pair's position is its expert's offset plus the
// number of the expert's tokens below it (popcount of the token mask), so the
// order is deterministic.  Indices outside [0, E) or repeated within a token
// are reported through `bad` and skipped.
template <int MW, bool GLOBAL_SRC, typename Sync>
__device__ void bucket_cta(int B, const int* src_idx, const float* src_w, BucketDst dst,
                           BucketOut user, BucketScratch<MW>& sc, bool& bad, Sync sync) {
  const int tid = threadIdx.x & 255;
  // The thread's pairs tid, tid + 256, ...: loaded once, all in flight
  // together, and kept for both passes.
  constexpr int PPT = (MW * 32 * TOPK + 255) / 256;
  const int npairs = B * TOPK;
  int ev[PPT];
  float wv[PPT];
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int p = tid + 256 * k;
    ev[k] = p < npairs ? (GLOBAL_SRC ? __ldcg(src_idx + p) : src_idx[p]) : -1;
    wv[k] = p < npairs && dst.pair_w ? (GLOBAL_SRC ? __ldcg(src_w + p) : src_w[p]) : 0.f;
  }
  for (int i = tid; i < E * MW; i += 256) (&sc.mask[0][0])[i] = 0u;
  sync();
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int p = tid + 256 * k;
    if (p < npairs) {
      const int e = ev[k];
      const int t = p / TOPK;
      if (e < 0 || e >= E) {
        bad = true;
      } else {
        const uint32_t bit = 1u << (t & 31);
        if (atomicOr(&sc.mask[e][t >> 5], bit) & bit) bad = true;
      }
    }
  }
  sync();
  const int e = tid;
  int cnt = 0;
#pragma unroll
  for (int w = 0; w < MW; ++w) cnt += __popc(sc.mask[e][w]);
  const int ng = (cnt + GROUP_MAX - 1) / GROUP_MAX;
  int tot_pairs, tot_groups, n_uniq;
  const int off = scan256(cnt, sc.warp_tot, &tot_pairs, sync);
  const int goff = scan256(ng, sc.warp_tot, &tot_groups, sync);
  const int urank = scan256(cnt > 0 ? 1 : 0, sc.warp_tot, &n_uniq, sync);
  sc.off[e] = off;
  for (int gi = 0; gi < ng; ++gi)
    dst.groups[goff + gi] = make_int4(e, off + gi * GROUP_MAX, min(GROUP_MAX, cnt - gi * GROUP_MAX), 0);
  if (user.uniq && cnt > 0) {
    user.uniq[urank] = e;
    user.offsets[urank] = off;
  }
  sync();
#pragma unroll
  for (int k = 0; k < PPT; ++k) {
    const int p = tid + 256 * k;
    const int ex = ev[k];
    if (p >= npairs || ex < 0 || ex >= E) continue;
    const int t = p / TOPK;
    const int wd = t >> 5;
    int rank = __popc(sc.mask[ex][wd] & ((1u << (t & 31)) - 1u));
    for (int w = 0; w < wd; ++w) rank += __popc(sc.mask[ex][w]);
    const int pos = sc.off[ex] + rank;
    dst.pair_tok[pos] = t;
    if (dst.pair_w) dst.pair_w[pos] = wv[k];
    if (user.pairs) user.pairs[pos] = t * 8 + (p - t * TOPK);
  }
  const int nsg = (B + GROUP_MAX - 1) / GROUP_MAX;
  for (int i = tid; i < S * B; i += 256) {
    dst.pair_tok[npairs + i] = i % B;
    if (dst.pair_w) dst.pair_w[npairs + i] = 1.0f;
  }
  for (int i = tid; i < S * nsg; i += 256) {
    const int s = i / nsg, gi = i % nsg;
    dst.groups[tot_groups + i] =
        make_int4(E + s, npairs + s * B + gi * GROUP_MAX, min(GROUP_MAX, B - gi * GROUP_MAX), 0);
  }
  if (tid == 0) {
    *dst.n_groups = tot_groups + S * nsg;
    if (dst.n_uniq) *dst.n_uniq = n_uniq;
    if (user.offsets) user.offsets[n_uniq] = npairs;
    if (user.n_uniq) *user.n_uniq = n_uniq;
  }
}

}  // namespace flint
