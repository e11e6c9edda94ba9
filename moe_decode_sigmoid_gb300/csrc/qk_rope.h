// qk_rope.h — the attention side of a decode step (qk_rope.cu): per-head
// Q/K RMSNorm + RoPE + bf16 KV-cache write in one kernel.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace flint {
namespace qk {
constexpr int NQ = 32, NKV = 4, HD = 128;  // query heads, KV heads, head size
constexpr int ROW = (NQ + 2 * NKV) * HD;   // projection row of one token
}  // namespace qk

struct QkArgs {
  const uint16_t* qkv;       // [B, ROW] bf16
  const uint16_t* q_norm;    // [HD] bf16
  const uint16_t* k_norm;    // [HD] bf16
  const int32_t* pos;        // [B]
  const int32_t* slots;      // [B]
  int rope;                  // 0: no rotation (layers without positional encoding)
  double inv_freq[qk::HD / 2];  // theta^(-2i/HD), i < HD/2, in fp64
  float eps;
  uint16_t* q_out;           // [B, NQ, HD] bf16
  uint16_t* k_cache;         // [cache_slots, NKV, HD] bf16
  uint16_t* v_cache;         // [cache_slots, NKV, HD] bf16
  long long cache_slots;
};

cudaError_t launch_qk_norm_rope(const QkArgs& a, int B, cudaStream_t stream);

}  // namespace flint
