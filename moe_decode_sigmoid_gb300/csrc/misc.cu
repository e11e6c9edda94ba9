// misc.cu — inter-layer RMSNorm and workspace initialisation.
//
// Pre-norm between stacked MoE layers ("49-layer pre-norm MoE architecture":
// vLLM Day-0 Support for Recursive's Flint, "Flint Model Architecture"):
//   out[t] = bf16( in[t] / sqrt(mean(in[t]^2) + eps) ), unit gain.
#include "common.cuh"
#include "kernels.h"

namespace flint {

// One CTA per token, 256 threads x 8 elements; fp32 sum of squares.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const uint16_t* in, uint16_t* out, float eps) {
  pdl_wait();
  pdl_trigger();
  __shared__ float s_part[8];
  const int t = blockIdx.x, tid = threadIdx.x;
  const uint4 v = reinterpret_cast<const uint4*>(in + (size_t)t * H)[tid];
  const float f[8] = {bf_lo(v.x), bf_hi(v.x), bf_lo(v.y), bf_hi(v.y),
                      bf_lo(v.z), bf_hi(v.z), bf_lo(v.w), bf_hi(v.w)};
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) ss = fmaf(f[i], f[i], ss);
  ss = warp_sum(ss);
  if ((tid & 31) == 0) s_part[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += s_part[w];
  const float inv = rsqrtf(tot / (float)H + eps);
  uint4 o;
  o.x = pack_bf2(f[0] * inv, f[1] * inv);
  o.y = pack_bf2(f[2] * inv, f[3] * inv);
  o.z = pack_bf2(f[4] * inv, f[5] * inv);
  o.w = pack_bf2(f[6] * inv, f[7] * inv);
  reinterpret_cast<uint4*>(out + (size_t)t * H)[tid] = o;
}

cudaError_t launch_rmsnorm(const uint16_t* in, uint16_t* out, int B, float eps, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(B, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rmsnorm_kernel, in, out, eps);
}

__global__ void ws_init_kernel(WsHeader* hdr, uint64_t wait_limit_ns) {
  hdr->wait_limit_ns = wait_limit_ns;
}

cudaError_t launch_ws_init(WsHeader* hdr, uint64_t wait_limit_ns, cudaStream_t stream) {
  ws_init_kernel<<<1, 1, 0, stream>>>(hdr, wait_limit_ns);
  return cudaGetLastError();
}

}  // namespace flint
