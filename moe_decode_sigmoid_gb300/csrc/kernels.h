// kernels.h — argument blocks and host launch wrappers of the Flint decode-MoE
// kernels (one translation unit per kernel family; the C ABI in api.cu calls
// these wrappers).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "common.cuh"
#include "flint_moe.h"
#include "select.cuh"

namespace flint {

struct RouterArgs {
  const uint16_t* x;   // [B,H] bf16
  const uint16_t* wr;  // [E,H] bf16
  const float* bias;   // [E] logit offsets or null
  int bias_select_only;  // the offsets steer the ranking only (not the weights)
  int B;
  Ws ws;
  int* user_idx;       // [B,TOPK] or null
  float* user_w;       // [B,TOPK] or null
  int do_bucket;       // build pairs/groups for the expert kernels
  int logits_only;     // write logits only: the expert kernels select (batch <= 8)
  int stall_check;     // honour the workspace's one-shot stall hook
  BucketOut bucket;    // optional plain bucket outputs (all null to skip)
};

// Expert weights of one layer in one of the two storage formats.
struct ExpertW {
  // bf16
  const uint16_t* w13;   // [E,2I,H]
  const uint16_t* w2;    // [E,H,I]
  const uint16_t* ws13;  // [S,2I,H]
  const uint16_t* ws2;   // [S,H,I]
  // nvfp4
  const uint8_t *w13_q, *w13_sf, *w2_q, *w2_sf;
  const float *w13_ts, *w2_ts;
  const uint8_t *ws13_q, *ws13_sf, *ws2_q, *ws2_sf;
  const float *ws13_ts, *ws2_ts;
};

struct ExpertArgs {
  const uint16_t* x;         // [B,H] bf16
  const uint16_t* residual;  // [B,H] bf16 (down kernel)
  uint16_t* out;             // [B,H] bf16 (down kernel)
  ExpertW w;
  int B;
  Ws ws;
  int early_shared;  // gate/up: start the shared expert before the router finishes
  int local_select;  // gate/up: rank and bucket the batch in every CTA (batch <= 8)
  const float* bias;     // logit offsets (local selection) or null
  int bias_select_only;  // as RouterArgs
  int* user_idx;     // gate/up with local_select: optional routing copies
  float* user_w;
  // Persistent kernel (BF16): the rows at x are the pre-norm activations, and
  // the kernel (its prenorm instance) takes bf16(x / sqrt(mean(x^2) + norm_eps))
  // (unit gain) in their place.
  int prenorm;
  float norm_eps;
};

// Largest batch whose routing the expert kernels compute themselves.
constexpr int LOCAL_SELECT_MAX_B = SMALL_B;
// Largest batch whose input RMSNorm the persistent kernel takes itself (the
// prenorm call); above it the standalone RMSNorm kernel runs first.  Measured
// per layer in the 47-layer stack on GB300, folded against RMSNorm kernel +
// persistent kernel: -1.2, -0.7, -0.6, -0.3 us at 1..4 tokens, +0.3, +0.35,
// +0.5 us at 5, 6, 8.
constexpr int PRENORM_FUSED_MAX_B = 4;

cudaError_t launch_router(const RouterArgs& a, cudaStream_t stream, bool pdl);
cudaError_t launch_bucket(const Ws& ws, int B, const BucketOut& user, cudaStream_t stream);
cudaError_t launch_gateup_bf16(const ExpertArgs& a, cudaStream_t stream, int num_sms);
cudaError_t launch_down_bf16(const ExpertArgs& a, cudaStream_t stream);
// The whole BF16 layer in one persistent cooperative kernel (batch <= 8), for
// grids of num_sms CTAs where small_supported(num_sms).
bool small_supported(int num_sms);
cudaError_t launch_small_bf16(const ExpertArgs& a, const RouterArgs& r, cudaStream_t stream,
                              int num_sms);
cudaError_t launch_gateup_nvfp4(const ExpertArgs& a, cudaStream_t stream, int num_sms);
cudaError_t launch_down_nvfp4(const ExpertArgs& a, cudaStream_t stream, int num_sms);
// out = residual + each token's SLOTS rows of y (after launch_down_nvfp4).
cudaError_t launch_combine_y(const ExpertArgs& a, cudaStream_t stream);
cudaError_t launch_rmsnorm(const uint16_t* in, uint16_t* out, int B, float eps,
                           cudaStream_t stream);
cudaError_t launch_ws_init(WsHeader* hdr, uint64_t wait_limit_ns, cudaStream_t stream);

// The host-side argument checks of flint_moe_decode_bf16 (everything but the
// launch), for entry points that must reject bad arguments before their own
// set-up.
flint_status decode_bf16_checks(const flint_moe_dims* dims, int32_t batch, const void* x,
                                const void* residual, const void* wr, const float* bias,
                                const void* w13, const void* w2, const void* ws13,
                                const void* ws2, void* out, int32_t* idx_out, float* w_out,
                                void* ws, size_t ws_bytes);

}  // namespace flint
