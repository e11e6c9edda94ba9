// noalloc.cu — flint_moe_decode_bf16_noalloc: the BF16 decode layer for
// callers that cannot allocate device memory at all.
//
// Some hosts own every byte of device memory themselves: a serving engine that
// carves the GPU into fixed pools at start-up and forbids plugins from calling
// cudaMalloc, an embedded or safety-certified runtime whose memory budget is
// fixed when it is built, or a real-time step loop that must never take the
// allocator's locks or latency.  Such a caller cannot create the workspace the
// other entry points take.  This entry point needs none: its scratch is one
// file-scope device array, sized for batches of up to
// FLINT_MOE_NOALLOC_MAX_BATCH tokens, that the CUDA module holds on every GPU
// that loads the library until the process exits.
//
// The call runs exactly the same kernels as flint_moe_decode_bf16 (it calls
// it, with the array as the workspace), so it produces the same outputs.
// Because every call shares the one array, two calls whose GPU work overlaps
// in time (different streams, or different host threads, on one device) race
// and corrupt each other's results; the caller must order them.
#include <cstddef>
#include <mutex>

#include "common.cuh"
#include "flint_moe.h"
#include "kernels.h"

namespace {

using flint::WsHeader;
using flint::WsLayout;

// The device status word is copied out as a flint_status: the codes agree.
static_assert(flint::DEV_OK == (uint32_t)FLINT_OK, "device and host codes agree");
static_assert(flint::DEV_BAD_ROUTING == (uint32_t)FLINT_ERR_INVALID_ARG, "device and host codes agree");
static_assert(flint::DEV_TIMEOUT == (uint32_t)FLINT_ERR_DEVICE_TIMEOUT, "device and host codes agree");

constexpr size_t kScratchBytes = WsLayout::total(FLINT_MOE_NOALLOC_MAX_BATCH);

// The only storage this entry point uses.  In host code the name stands for a
// host-side shadow, never a device address: the kernels get the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_scratch_dev[kMaxDevices] = {};  // per device: the array's address
bool g_scratch_ready[kMaxDevices] = {};  // per device: header initialised

// Device address of g_scratch on the current device (a lookup, no GPU work).
flint_status scratch_address(int* dev_out, void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FLINT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_dev[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return FLINT_ERR_CUDA;
    g_scratch_dev[dev] = p;
  }
  *dev_out = dev;
  *out = g_scratch_dev[dev];
  return FLINT_OK;
}

// On the first call for a device: zero-fills the array, writes its header
// (wait limit) and waits for that to finish.
flint_status scratch_setup(int dev, void* p, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (g_scratch_ready[dev]) return FLINT_OK;
  // Set-up enqueues work and synchronises `stream`: it must not run while
  // the stream is being captured.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return FLINT_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return FLINT_ERR_CUDA;
  const flint_status st = flint_moe_workspace_init(p, kScratchBytes, 0, stream);
  if (st != FLINT_OK) return st;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return FLINT_ERR_CUDA;
  g_scratch_ready[dev] = true;
  return FLINT_OK;
}

}  // namespace

extern "C" flint_status flint_moe_decode_bf16_noalloc(
    const flint_moe_dims* dims, int32_t batch, const void* x_bf16, const void* residual_bf16,
    const void* w_router_bf16, const float* logit_bias, const void* w13_bf16,
    const void* w2_bf16, const void* ws13_bf16, const void* ws2_bf16, void* out_bf16,
    int32_t* topk_idx_out, float* topk_w_out, int32_t* device_status_out, cudaStream_t stream) {
  if (batch < 1 || batch > FLINT_MOE_NOALLOC_MAX_BATCH) return FLINT_ERR_INVALID_ARG;
  if (device_status_out != nullptr && (reinterpret_cast<uintptr_t>(device_status_out) & 3u) != 0)
    return FLINT_ERR_INVALID_ARG;
  int dev = -1;
  void* ws = nullptr;
  flint_status st = scratch_address(&dev, &ws);
  if (st != FLINT_OK) return st;
  // Every argument is checked before anything is enqueued.
  st = flint::decode_bf16_checks(dims, batch, x_bf16, residual_bf16, w_router_bf16, logit_bias,
                                 w13_bf16, w2_bf16, ws13_bf16, ws2_bf16, out_bf16, topk_idx_out,
                                 topk_w_out, ws, kScratchBytes);
  if (st != FLINT_OK) return st;
  st = scratch_setup(dev, ws, stream);
  if (st != FLINT_OK) return st;
  // The array keeps whatever the previous call left.  Everything the layer
  // reads is written earlier in the same call (the small-batch kernel tells
  // this call's words from older ones by the header's call counter), except
  // the header: its error word and counters must start at zero (a call that
  // ran out of time may have left them set).  The call counter and the wait
  // limit are kept.
  char* hdr = static_cast<char*>(ws);
  if (cudaMemsetAsync(hdr, 0, sizeof(uint32_t), stream) != cudaSuccess) return FLINT_ERR_CUDA;
  if (cudaMemsetAsync(hdr + flint::WS_HDR_KEEP, 0, sizeof(WsHeader) - flint::WS_HDR_KEEP,
                      stream) != cudaSuccess)
    return FLINT_ERR_CUDA;
  st = flint_moe_decode_bf16(dims, batch, x_bf16, residual_bf16, w_router_bf16, logit_bias,
                             w13_bf16, w2_bf16, ws13_bf16, ws2_bf16, out_bf16, topk_idx_out,
                             topk_w_out, ws, kScratchBytes, stream);
  if (st != FLINT_OK) return st;
  if (device_status_out != nullptr &&
      cudaMemcpyAsync(device_status_out, hdr, sizeof(int32_t), cudaMemcpyDeviceToDevice,
                      stream) != cudaSuccess)
    return FLINT_ERR_CUDA;
  return FLINT_OK;
}
