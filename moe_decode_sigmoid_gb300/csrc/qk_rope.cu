// qk_rope.cu — the attention side of a decode step: per-head Q/K RMSNorm,
// rotary position embedding and the bf16 KV-cache write, in one kernel.
//
// The pages fuse "Q/K norm, RoPE, and KV-cache write into a single kernel"
// (vLLM Day-0 Support for Recursive's Flint, "Optimization Strategies",
// "Fused Kernels"); the attention they belong to has GQA with 32 query and 4
// KV heads, per-head Q/K RMSNorm, RoPE on the sliding-window layers and no
// positional encoding on the full-attention layers, and a bf16 KV cache
// (same page, "Flint Model Architecture").  Head size 128: 14 full-attention
// layers keep 28 KiB of KV per token, i.e. 2 KiB per layer = K and V of 4
// heads x 128 values x 2 bytes.
//
// Per token t at position pos[t], with its projection row
// qkv[t] = [q_0 .. q_31 | k_0 .. k_3 | v_0 .. v_3] (128 values per head):
//   q, k heads: n[i] = x[i] / sqrt(mean x^2 + eps) * g[i] (g = q_norm or
//               k_norm), then, if theta > 0, each pair (i, i + 64) turns by
//               pos * theta^(-2i/128) (rotate-half pairing);
//   q heads go to q_out[t], k heads to k_cache[slot[t]], v heads unchanged to
//   v_cache[slot[t]]; a slot outside [0, cache_slots) writes nothing (a
//   negative slot marks a padding token).
//
// One CTA per token: 64 threads first take the token's 64 rotation angles in
// fp64 -- a position of 2^18 times a frequency near 1 would leave an fp32
// angle ~0.03 rad off -- from frequencies the host computed in fp64, reduce
// them to [-pi, pi] (Cody and Waite's additive reduction, with 2 pi held as
// two doubles) and keep the fp32 cos / sin in shared memory; then warp w takes heads
// w, w + 8, ... (40 heads), lane l holding elements 2l, 2l + 1 and their
// partners 64 + 2l, 65 + 2l, so the head's sum of squares is one warp sum
// and each pair turns in one lane.  fp32 arithmetic, one bf16 rounding.
#include "common.cuh"
#include "qk_rope.h"

namespace flint {
namespace {

__device__ __forceinline__ uint32_t ld_u32(const uint16_t* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}
__device__ __forceinline__ void st_u32(uint16_t* p, uint32_t v) {
  *reinterpret_cast<uint32_t*>(p) = v;
}

}  // namespace

__global__ void __launch_bounds__(256) qk_norm_rope_kernel(QkArgs a) {
  __shared__ float s_cos[qk::HD / 2], s_sin[qk::HD / 2];
  pdl_wait();  // the projection rows come from the preceding kernel
  pdl_trigger();
  const int t = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint16_t* row = a.qkv + (size_t)t * qk::ROW;
  const int i0 = 2 * lane, i1 = qk::HD / 2 + 2 * lane;  // this lane's two element pairs
  // All of this warp's heads (w, w + 8, ...) are loaded first, so their round
  // trips overlap each other and the angle computation.
  constexpr int HPW = (qk::NQ + 2 * qk::NKV + 7) / 8;  // heads per warp
  uint32_t lo[HPW], hi[HPW];
#pragma unroll
  for (int j = 0; j < HPW; ++j) {
    const int h = warp + 8 * j;
    if (h < qk::NQ + 2 * qk::NKV) {
      lo[j] = ld_u32(row + (size_t)h * qk::HD + i0);
      hi[j] = ld_u32(row + (size_t)h * qk::HD + i1);
    }
  }
  const bool rope = a.rope != 0;
  if (rope && tid < qk::HD / 2) {
    constexpr double INV_TWO_PI = 0.15915494309189535;      // 1 / (2 pi)
    constexpr double TWO_PI_HI = 6.283185307179586;         // 2 pi = HI + LO
    constexpr double TWO_PI_LO = 2.4492935982947064e-16;
    const double ang = (double)a.pos[t] * a.inv_freq[tid];
    const double k = rint(ang * INV_TWO_PI);
    const double r = fma(-k, TWO_PI_LO, fma(-k, TWO_PI_HI, ang));
    float s, c;
    sincosf((float)r, &s, &c);
    s_cos[tid] = c;
    s_sin[tid] = s;
  }
  const int slot = a.slots[t];
  const bool write_kv = slot >= 0 && (long long)slot < a.cache_slots;
  __syncthreads();
#pragma unroll
  for (int j = 0; j < HPW; ++j) {
    const int h = warp + 8 * j;
    if (h >= qk::NQ + 2 * qk::NKV) break;
    if (h >= qk::NQ + qk::NKV) {  // v head: unchanged into the cache
      if (write_kv) {
        uint16_t* dst = a.v_cache + ((size_t)slot * qk::NKV + (h - qk::NQ - qk::NKV)) * qk::HD;
        st_u32(dst + i0, lo[j]);
        st_u32(dst + i1, hi[j]);
      }
      continue;
    }
    const bool is_q = h < qk::NQ;
    const uint16_t* g = is_q ? a.q_norm : a.k_norm;
    const uint32_t glo = ld_u32(g + i0), ghi = ld_u32(g + i1);
    const float x0 = bf_lo(lo[j]), x1 = bf_hi(lo[j]), x2 = bf_lo(hi[j]), x3 = bf_hi(hi[j]);
    const float ss = warp_sum(fmaf(x0, x0, fmaf(x1, x1, fmaf(x2, x2, x3 * x3))));
    const float inv = 1.0f / sqrtf(ss / (float)qk::HD + a.eps);
    float n0 = x0 * inv * bf_lo(glo), n1 = x1 * inv * bf_hi(glo);  // elements 2l, 2l + 1
    float n2 = x2 * inv * bf_lo(ghi), n3 = x3 * inv * bf_hi(ghi);  // elements 64 + 2l, 65 + 2l
    if (rope) {
      const float c0 = s_cos[i0], s0 = s_sin[i0], c1 = s_cos[i0 + 1], s1 = s_sin[i0 + 1];
      const float r0 = n0 * c0 - n2 * s0, r2 = n2 * c0 + n0 * s0;
      const float r1 = n1 * c1 - n3 * s1, r3 = n3 * c1 + n1 * s1;
      n0 = r0;
      n1 = r1;
      n2 = r2;
      n3 = r3;
    }
    uint16_t* dst;
    if (is_q) {
      dst = a.q_out + ((size_t)t * qk::NQ + h) * qk::HD;
    } else {
      if (!write_kv) continue;
      dst = a.k_cache + ((size_t)slot * qk::NKV + (h - qk::NQ)) * qk::HD;
    }
    st_u32(dst + i0, pack_bf2(n0, n1));
    st_u32(dst + i1, pack_bf2(n2, n3));
  }
}

cudaError_t launch_qk_norm_rope(const QkArgs& a, int B, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, qk_norm_rope_kernel, a);
}

}  // namespace flint
