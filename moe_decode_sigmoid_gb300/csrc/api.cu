// api.cu — the C ABI (include/flint_moe.h): argument validation, workspace
// views and launch sequencing.  Every check runs on the host before the first
// launch; the kernels of one call are chained on the caller's stream with
// programmatic dependent launch, so each kernel's prologue overlaps the
// previous kernel's tail.  Nothing here allocates memory or synchronises,
// except flint_moe_get_device_status.
#include <cstdint>
#include <cstring>

#include <cmath>

#include "flint_moe.h"
#include "kernels.h"
#include "qk_rope.h"

using namespace flint;

namespace {

constexpr uint64_t DEFAULT_WAIT_NS = 1000000000ull;  // 1 s

bool dims_supported(const flint_moe_dims* d) {
  return d->hidden == H && d->n_experts == E && d->top_k == TOPK && d->inter == I &&
         d->n_shared == S &&
         (d->offset_mode == FLINT_OFFSET_LOGIT || d->offset_mode == FLINT_OFFSET_SELECT);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Required pointer: non-null and 16-byte aligned.
bool req(const void* p) { return p != nullptr && aligned16(p); }
// Small fp32 / int32 vectors (offsets, routing outputs): 4-byte alignment.
bool req4(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool opt4(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

flint_status check_common(const flint_moe_dims* dims, int32_t batch, void* ws, size_t ws_bytes) {
  if (dims == nullptr) return FLINT_ERR_INVALID_ARG;
  if (!dims_supported(dims)) return FLINT_ERR_UNSUPPORTED;
  if (batch < 1 || batch > MAX_B) return FLINT_ERR_INVALID_ARG;
  if (ws == nullptr || !aligned16(ws) || ws_bytes < WsLayout::total(batch))
    return FLINT_ERR_WORKSPACE;
  return FLINT_OK;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

flint_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FLINT_OK;
  (void)cudaGetLastError();  // clear a non-sticky launch error
  return FLINT_ERR_CUDA;
}

// Output / input aliasing rule of the decode calls.
bool aliasing_ok(int32_t batch, const void* x, const void* residual, const void* out,
                 const void* ws, size_t ws_bytes) {
  const size_t act = (size_t)batch * H * 2;
  if (overlap(out, act, x, act)) return false;
  if (out != residual && overlap(out, act, residual, act)) return false;
  if (overlap(out, act, ws, ws_bytes)) return false;
  return true;
}

flint_status decode_checks(const flint_moe_dims* dims, int32_t batch, const void* x,
                           const void* residual, const void* wr, const float* bias, void* out,
                           int32_t* idx_out, float* w_out, void* ws, size_t ws_bytes) {
  flint_status st = check_common(dims, batch, ws, ws_bytes);
  if (st != FLINT_OK) return st;
  if (!req(x) || !req(residual) || !req(wr) || !opt4(bias) || !req(out) || !opt4(idx_out) ||
      !opt4(w_out))
    return FLINT_ERR_INVALID_ARG;
  if (!aliasing_ok(batch, x, residual, out, ws, ws_bytes)) return FLINT_ERR_INVALID_ARG;
  return FLINT_OK;
}

}  // namespace

namespace flint {
flint_status decode_bf16_checks(const flint_moe_dims* dims, int32_t batch, const void* x,
                                const void* residual, const void* wr, const float* bias,
                                const void* w13, const void* w2, const void* ws13,
                                const void* ws2, void* out, int32_t* idx_out, float* w_out,
                                void* ws, size_t ws_bytes) {
  const flint_status st =
      decode_checks(dims, batch, x, residual, wr, bias, out, idx_out, w_out, ws, ws_bytes);
  if (st != FLINT_OK) return st;
  if (!req(w13) || !req(w2) || !req(ws13) || !req(ws2)) return FLINT_ERR_INVALID_ARG;
  return FLINT_OK;
}
}  // namespace flint

extern "C" {

const char* flint_status_string(flint_status status) {
  switch (status) {
    case FLINT_OK: return "FLINT_OK";
    case FLINT_ERR_INVALID_ARG: return "FLINT_ERR_INVALID_ARG";
    case FLINT_ERR_UNSUPPORTED: return "FLINT_ERR_UNSUPPORTED";
    case FLINT_ERR_WORKSPACE: return "FLINT_ERR_WORKSPACE";
    case FLINT_ERR_CUDA: return "FLINT_ERR_CUDA";
    case FLINT_ERR_DEVICE_TIMEOUT: return "FLINT_ERR_DEVICE_TIMEOUT";
  }
  return "FLINT_ERR_UNKNOWN";
}

size_t flint_moe_workspace_bytes(const flint_moe_dims* dims, int32_t max_batch) {
  if (dims == nullptr || !dims_supported(dims)) return 0;
  if (max_batch < 1 || max_batch > MAX_B) return 0;
  return WsLayout::total(max_batch);
}

flint_status flint_moe_workspace_init(void* workspace, size_t ws_bytes, uint64_t wait_limit_ns,
                                      cudaStream_t stream) {
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < WsLayout::total(1))
    return FLINT_ERR_WORKSPACE;
  cudaError_t e = cudaMemsetAsync(workspace, 0, ws_bytes, stream);
  if (e != cudaSuccess) return cuda_status(e);
  Ws w = ws_view(workspace);
  return cuda_status(launch_ws_init(w.hdr, wait_limit_ns ? wait_limit_ns : DEFAULT_WAIT_NS, stream));
}

flint_status flint_moe_get_device_status(const void* workspace, cudaStream_t stream) {
  if (workspace == nullptr || !aligned16(workspace)) return FLINT_ERR_WORKSPACE;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_status(e);
  uint32_t word = 0;
  e = cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  switch (word) {
    case DEV_OK: return FLINT_OK;
    case DEV_BAD_ROUTING: return FLINT_ERR_INVALID_ARG;
    case DEV_TIMEOUT: return FLINT_ERR_DEVICE_TIMEOUT;
    default: return FLINT_ERR_CUDA;
  }
}

flint_status flint_moe_debug_arm_stall(void* workspace, size_t ws_bytes, cudaStream_t stream) {
  if (workspace == nullptr || !aligned16(workspace) || ws_bytes < WsLayout::total(1))
    return FLINT_ERR_WORKSPACE;
  WsHeader* hdr = ws_view(workspace).hdr;
  return cuda_status(cudaMemsetAsync(&hdr->stall_armed, 1, sizeof(uint32_t), stream));
}

flint_status flint_moe_route(const flint_moe_dims* dims, int32_t batch, const void* x_bf16,
                             const void* w_router_bf16, const float* logit_bias, int32_t* topk_idx,
                             float* topk_w, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  flint_status st = check_common(dims, batch, workspace, ws_bytes);
  if (st != FLINT_OK) return st;
  if (!req(x_bf16) || !req(w_router_bf16) || !opt4(logit_bias) || !req4(topk_idx) || !req4(topk_w))
    return FLINT_ERR_INVALID_ARG;
  RouterArgs a = {};
  a.x = static_cast<const uint16_t*>(x_bf16);
  a.wr = static_cast<const uint16_t*>(w_router_bf16);
  a.bias = logit_bias;
  a.bias_select_only = dims->offset_mode == FLINT_OFFSET_SELECT;
  a.B = batch;
  a.ws = ws_view(workspace);
  a.user_idx = topk_idx;
  a.user_w = topk_w;
  a.do_bucket = 1;
  a.stall_check = 1;
  return cuda_status(launch_router(a, stream, true));
}

flint_status flint_moe_bucket(const flint_moe_dims* dims, int32_t batch, const int32_t* topk_idx,
                              int32_t* uniq, int32_t* offsets, int32_t* pairs, int32_t* n_uniq,
                              void* workspace, size_t ws_bytes, cudaStream_t stream) {
  flint_status st = check_common(dims, batch, workspace, ws_bytes);
  if (st != FLINT_OK) return st;
  if (!req4(topk_idx) || !req4(uniq) || !req4(offsets) || !req4(pairs) || !req4(n_uniq))
    return FLINT_ERR_INVALID_ARG;
  Ws w = ws_view(workspace);
  cudaError_t e = cudaMemcpyAsync(w.topk_idx, topk_idx, sizeof(int32_t) * (size_t)batch * TOPK,
                                  cudaMemcpyDeviceToDevice, stream);
  if (e != cudaSuccess) return cuda_status(e);
  BucketOut bo = {uniq, offsets, pairs, n_uniq};
  return cuda_status(launch_bucket(w, batch, bo, stream));
}

// norm_eps >= 0: x is not given; the layer input is RMSNorm(residual), taken
// by the persistent kernel itself (batch <= PRENORM_FUSED_MAX_B) or written
// into the workspace first by the RMSNorm kernel (the NVFP4 path's y rows,
// which the BF16 kernels do not use).
static flint_status run_layer(bool nvfp4, const flint_moe_dims* dims, int32_t batch,
                              const void* x, const void* residual,
                              const void* wr, const float* bias, const ExpertW& w, void* out,
                              int32_t* idx_out, float* w_out, void* workspace,
                              cudaStream_t stream, float norm_eps = -1.0f) {
  const int sms = num_sms();
  if (sms <= 0) return FLINT_ERR_CUDA;
  const bool fused =
      !nvfp4 && batch <= LOCAL_SELECT_MAX_B && small_supported(sms);
  const bool prenorm = norm_eps >= 0.0f;
  const bool fold = prenorm && fused && batch <= PRENORM_FUSED_MAX_B;
  if (prenorm) {
    if (fold) {
      x = residual;  // the kernel normalises the rows as it stages them
    } else {
      uint16_t* xn = reinterpret_cast<uint16_t*>(ws_y(ws_view(workspace), batch));
      const cudaError_t e = launch_rmsnorm(static_cast<const uint16_t*>(residual), xn, batch,
                                           norm_eps, stream);
      if (e != cudaSuccess) return cuda_status(e);
      x = xn;
    }
  }
  RouterArgs r = {};
  r.x = static_cast<const uint16_t*>(x);
  r.wr = static_cast<const uint16_t*>(wr);
  r.bias = bias;
  r.bias_select_only = dims->offset_mode == FLINT_OFFSET_SELECT;
  r.B = batch;
  r.ws = ws_view(workspace);
  r.user_idx = idx_out;
  r.user_w = w_out;
  r.do_bucket = 1;
  r.stall_check = 1;
  // Small batches: the router only writes logits and every gate/up CTA ranks
  // and buckets the tokens itself, which takes the router's serial tail off
  // the critical path.
  r.logits_only = batch <= LOCAL_SELECT_MAX_B ? 1 : 0;
  ExpertArgs a = {};
  a.x = r.x;
  a.residual = static_cast<const uint16_t*>(residual);
  a.out = static_cast<uint16_t*>(out);
  a.w = w;
  a.B = batch;
  a.ws = r.ws;
  // The router starts only after everything before it on the stream is done,
  // and lets the gate/up kernel launch early: the shared expert, which does not
  // depend on routing, is then computed while the router runs.
  a.early_shared = 1;
  a.local_select = r.logits_only;
  a.bias = bias;
  a.bias_select_only = r.bias_select_only;
  a.user_idx = idx_out;
  a.user_w = w_out;
  a.prenorm = fold;
  a.norm_eps = norm_eps;
  // BF16: one persistent kernel for small batches.  NVFP4 always takes the
  // chained kernels, whose gate/up and down kernels spread each group's
  // dequantisation over all SMs: measured faster at every batch on GB300 (1
  // token: 16.8 us against 18.6 us for an NVFP4 instance of the persistent
  // kernel; 2 tokens: 20.7 against 25.0 us).
  if (fused) return cuda_status(launch_small_bf16(a, r, stream, sms));
  cudaError_t e = launch_router(r, stream, true);
  if (e != cudaSuccess) return cuda_status(e);
  e = nvfp4 ? launch_gateup_nvfp4(a, stream, sms) : launch_gateup_bf16(a, stream, sms);
  if (e != cudaSuccess) return cuda_status(e);
  if (!nvfp4) return cuda_status(launch_down_bf16(a, stream));
  e = launch_down_nvfp4(a, stream, sms);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_combine_y(a, stream));
}

flint_status flint_moe_decode_bf16(const flint_moe_dims* dims, int32_t batch, const void* x_bf16,
                                   const void* residual_bf16, const void* w_router_bf16,
                                   const float* logit_bias, const void* w13_bf16,
                                   const void* w2_bf16, const void* ws13_bf16,
                                   const void* ws2_bf16, void* out_bf16, int32_t* topk_idx_out,
                                   float* topk_w_out, void* workspace, size_t ws_bytes,
                                   cudaStream_t stream) {
  const flint_status st =
      flint::decode_bf16_checks(dims, batch, x_bf16, residual_bf16, w_router_bf16, logit_bias,
                                w13_bf16, w2_bf16, ws13_bf16, ws2_bf16, out_bf16, topk_idx_out,
                                topk_w_out, workspace, ws_bytes);
  if (st != FLINT_OK) return st;
  ExpertW w = {};
  w.w13 = static_cast<const uint16_t*>(w13_bf16);
  w.w2 = static_cast<const uint16_t*>(w2_bf16);
  w.ws13 = static_cast<const uint16_t*>(ws13_bf16);
  w.ws2 = static_cast<const uint16_t*>(ws2_bf16);
  return run_layer(false, dims, batch, x_bf16, residual_bf16, w_router_bf16, logit_bias, w,
                   out_bf16, topk_idx_out, topk_w_out, workspace, stream);
}

flint_status flint_moe_decode_bf16_prenorm(const flint_moe_dims* dims, int32_t batch,
                                           const void* residual_bf16, float norm_eps,
                                           const void* w_router_bf16, const float* logit_bias,
                                           const void* w13_bf16, const void* w2_bf16,
                                           const void* ws13_bf16, const void* ws2_bf16,
                                           void* out_bf16, int32_t* topk_idx_out,
                                           float* topk_w_out, void* workspace, size_t ws_bytes,
                                           cudaStream_t stream) {
  flint_status st = check_common(dims, batch, workspace, ws_bytes);
  if (st != FLINT_OK) return st;
  if (!req(residual_bf16) || !req(w_router_bf16) || !opt4(logit_bias) || !req(w13_bf16) ||
      !req(w2_bf16) || !req(ws13_bf16) || !req(ws2_bf16) || !req(out_bf16) ||
      !opt4(topk_idx_out) || !opt4(topk_w_out) || !(norm_eps >= 0.0f))
    return FLINT_ERR_INVALID_ARG;
  const size_t act = (size_t)batch * H * 2;
  if (out_bf16 != residual_bf16 && overlap(out_bf16, act, residual_bf16, act))
    return FLINT_ERR_INVALID_ARG;
  if (overlap(out_bf16, act, workspace, ws_bytes) ||
      overlap(residual_bf16, act, workspace, ws_bytes))
    return FLINT_ERR_INVALID_ARG;
  ExpertW w = {};
  w.w13 = static_cast<const uint16_t*>(w13_bf16);
  w.w2 = static_cast<const uint16_t*>(w2_bf16);
  w.ws13 = static_cast<const uint16_t*>(ws13_bf16);
  w.ws2 = static_cast<const uint16_t*>(ws2_bf16);
  return run_layer(false, dims, batch, nullptr, residual_bf16, w_router_bf16, logit_bias, w,
                   out_bf16, topk_idx_out, topk_w_out, workspace, stream, norm_eps);
}

flint_status flint_moe_gateup_bf16(const flint_moe_dims* dims, int32_t batch, const void* x_bf16,
                                   const void* w13_bf16, const void* ws13_bf16, void* workspace,
                                   size_t ws_bytes, cudaStream_t stream) {
  flint_status st = check_common(dims, batch, workspace, ws_bytes);
  if (st != FLINT_OK) return st;
  if (!req(x_bf16) || !req(w13_bf16) || !req(ws13_bf16)) return FLINT_ERR_INVALID_ARG;
  const int sms = num_sms();
  if (sms <= 0) return FLINT_ERR_CUDA;
  ExpertArgs a = {};
  a.x = static_cast<const uint16_t*>(x_bf16);
  a.w.w13 = static_cast<const uint16_t*>(w13_bf16);
  a.w.ws13 = static_cast<const uint16_t*>(ws13_bf16);
  a.B = batch;
  a.ws = ws_view(workspace);
  return cuda_status(launch_gateup_bf16(a, stream, sms));
}

flint_status flint_moe_down_bf16(const flint_moe_dims* dims, int32_t batch,
                                 const void* residual_bf16, const void* w2_bf16,
                                 const void* ws2_bf16, void* out_bf16, void* workspace,
                                 size_t ws_bytes, cudaStream_t stream) {
  flint_status st = check_common(dims, batch, workspace, ws_bytes);
  if (st != FLINT_OK) return st;
  if (!req(residual_bf16) || !req(w2_bf16) || !req(ws2_bf16) || !req(out_bf16))
    return FLINT_ERR_INVALID_ARG;
  const size_t act = (size_t)batch * H * 2;
  if (out_bf16 != residual_bf16 && overlap(out_bf16, act, residual_bf16, act))
    return FLINT_ERR_INVALID_ARG;
  if (overlap(out_bf16, act, workspace, ws_bytes)) return FLINT_ERR_INVALID_ARG;
  ExpertArgs a = {};
  a.residual = static_cast<const uint16_t*>(residual_bf16);
  a.out = static_cast<uint16_t*>(out_bf16);
  a.w.w2 = static_cast<const uint16_t*>(w2_bf16);
  a.w.ws2 = static_cast<const uint16_t*>(ws2_bf16);
  a.B = batch;
  a.ws = ws_view(workspace);
  return cuda_status(launch_down_bf16(a, stream));
}

flint_status flint_moe_decode_nvfp4_w4a16(
    const flint_moe_dims* dims, int32_t batch, const void* x_bf16, const void* residual_bf16,
    const void* w_router_bf16, const float* logit_bias, const uint8_t* w13_q,
    const uint8_t* w13_sf, const float* w13_ts, const uint8_t* w2_q, const uint8_t* w2_sf,
    const float* w2_ts, const uint8_t* ws13_q, const uint8_t* ws13_sf, const float* ws13_ts,
    const uint8_t* ws2_q, const uint8_t* ws2_sf, const float* ws2_ts, void* out_bf16,
    int32_t* topk_idx_out, float* topk_w_out, void* workspace, size_t ws_bytes,
    cudaStream_t stream) {
  flint_status st = decode_checks(dims, batch, x_bf16, residual_bf16, w_router_bf16, logit_bias,
                                  out_bf16, topk_idx_out, topk_w_out, workspace, ws_bytes);
  if (st != FLINT_OK) return st;
  if (!req(w13_q) || !req(w13_sf) || !req4(w13_ts) || !req(w2_q) || !req(w2_sf) || !req4(w2_ts) ||
      !req(ws13_q) || !req(ws13_sf) || !req4(ws13_ts) || !req(ws2_q) || !req(ws2_sf) ||
      !req4(ws2_ts))
    return FLINT_ERR_INVALID_ARG;
  ExpertW w = {};
  w.w13_q = w13_q; w.w13_sf = w13_sf; w.w13_ts = w13_ts;
  w.w2_q = w2_q; w.w2_sf = w2_sf; w.w2_ts = w2_ts;
  w.ws13_q = ws13_q; w.ws13_sf = ws13_sf; w.ws13_ts = ws13_ts;
  w.ws2_q = ws2_q; w.ws2_sf = ws2_sf; w.ws2_ts = ws2_ts;
  return run_layer(true, dims, batch, x_bf16, residual_bf16, w_router_bf16, logit_bias, w,
                   out_bf16, topk_idx_out, topk_w_out, workspace, stream);
}

flint_status flint_qk_norm_rope_kv_bf16(const flint_attn_dims* dims, int32_t batch,
                                        const void* qkv_bf16, const void* q_norm_bf16,
                                        const void* k_norm_bf16, const int32_t* positions,
                                        const int32_t* slot_mapping, float rope_theta, float eps,
                                        void* q_out_bf16, void* k_cache_bf16, void* v_cache_bf16,
                                        int64_t cache_slots, cudaStream_t stream) {
  if (dims == nullptr) return FLINT_ERR_INVALID_ARG;
  if (dims->n_q_heads != qk::NQ || dims->n_kv_heads != qk::NKV || dims->head_dim != qk::HD)
    return FLINT_ERR_UNSUPPORTED;
  if (batch < 1 || batch > MAX_B || cache_slots < 1 || !req(qkv_bf16) || !req(q_norm_bf16) ||
      !req(k_norm_bf16) || !req4(positions) || !req4(slot_mapping) || !req(q_out_bf16) ||
      !req(k_cache_bf16) || !req(v_cache_bf16))
    return FLINT_ERR_INVALID_ARG;
  if (!(rope_theta >= 0.0f) || rope_theta > 3.0e38f || !(eps >= 0.0f) || eps > 3.0e38f)
    return FLINT_ERR_INVALID_ARG;
  const size_t in_b = (size_t)batch * qk::ROW * 2, q_b = (size_t)batch * qk::NQ * qk::HD * 2;
  const size_t c_b = (size_t)cache_slots * qk::NKV * qk::HD * 2;
  if (overlap(q_out_bf16, q_b, qkv_bf16, in_b) || overlap(k_cache_bf16, c_b, qkv_bf16, in_b) ||
      overlap(v_cache_bf16, c_b, qkv_bf16, in_b) || overlap(k_cache_bf16, c_b, q_out_bf16, q_b) ||
      overlap(v_cache_bf16, c_b, q_out_bf16, q_b) || overlap(k_cache_bf16, c_b, v_cache_bf16, c_b))
    return FLINT_ERR_INVALID_ARG;
  QkArgs a;
  a.qkv = static_cast<const uint16_t*>(qkv_bf16);
  a.q_norm = static_cast<const uint16_t*>(q_norm_bf16);
  a.k_norm = static_cast<const uint16_t*>(k_norm_bf16);
  a.pos = positions;
  a.slots = slot_mapping;
  a.rope = rope_theta > 0.0f;
  for (int i = 0; i < qk::HD / 2; ++i)
    a.inv_freq[i] = a.rope ? std::pow((double)rope_theta, -2.0 * i / qk::HD) : 0.0;
  a.eps = eps;
  a.q_out = static_cast<uint16_t*>(q_out_bf16);
  a.k_cache = static_cast<uint16_t*>(k_cache_bf16);
  a.v_cache = static_cast<uint16_t*>(v_cache_bf16);
  a.cache_slots = (long long)cache_slots;
  return cuda_status(launch_qk_norm_rope(a, batch, stream));
}

flint_status flint_moe_rmsnorm_bf16(const flint_moe_dims* dims, int32_t batch, const void* in_bf16,
                                    void* out_bf16, float eps, cudaStream_t stream) {
  if (dims == nullptr) return FLINT_ERR_INVALID_ARG;
  if (dims->hidden != H) return FLINT_ERR_UNSUPPORTED;
  if (batch < 1 || batch > MAX_B || !req(in_bf16) || !req(out_bf16) || !(eps >= 0.0f))
    return FLINT_ERR_INVALID_ARG;
  const size_t act = (size_t)batch * H * 2;
  if (overlap(in_bf16, act, out_bf16, act)) return FLINT_ERR_INVALID_ARG;
  return cuda_status(launch_rmsnorm(static_cast<const uint16_t*>(in_bf16),
                                    static_cast<uint16_t*>(out_bf16), batch, eps, stream));
}

}  // extern "C"
