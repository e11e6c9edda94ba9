// down.cu — the BF16 weight format of the large-batch down kernel
// (down_ring.cuh holds the kernel; the fused kernel covers batches of at most
// 8 tokens).
//
// A group's 16-row Wd slice (16 KiB) arrives through one 3-D tensor copy
// (TMA) with a 128-byte swizzle: the map views a Wd stack as (64 columns,
// row, 8 column blocks) with strides (2 bytes, 1 KiB, 128 bytes), so a
// (64, 16, 8) box lands as 8 column blocks of 16 rows x 128 bytes with each
// row's 16-byte chunks XOR-permuted by row mod 8.  Lane q takes, at step kk of
// K half kh (kc = 8 kh + kk), K block 8 (kc / 2) + 2q + kc % 2: the two rows of
// every 8-lane phase of a 128-bit load then fall in opposite chunk parities,
// so the fragment loads are free of bank conflicts.  The gate/up kernel
// writes h with the same block order (h_chunk).  The odd warp of a pair hands
// its tiles over in the half of the slice that only it reads.
#include "down_ring.cuh"
#include "tmap.h"

namespace flint {
namespace {

struct Bf16Wd {
  static constexpr int WBYTES = dring::RS * I * 2;  // 16 KiB
  static constexpr int WCOPY = WBYTES;
  static constexpr int XCH = WBYTES / 2;
  static constexpr int NDESC = 16;
  struct Maps {
    CUtensorMap w2;
    CUtensorMap ws2;
  };
  struct Frag {};
  __device__ static void issue(const Maps& maps, const ExpertArgs&, uint32_t dst, int4 grp, int r0,
                               uint32_t bar) {
    if (grp.x < E)
      dring::tma_load_3d(dst, &maps.w2, 0, grp.x * H + r0, 0, bar);
    else
      dring::tma_load_3d(dst, &maps.ws2, 0, (grp.x - E) * H + r0, 0, bar);
  }
  __device__ static void load(const uint8_t*, int, int, int, Frag&) {}
  // Wd (row r, column k) sits at line (k / 64) * 16 + r, chunk ((k / 8) % 8) ^ (r % 8).
  __device__ static void a(const uint8_t* st, const Frag&, int gq, int q, int khalf, int kk,
                           uint4& alo, uint4& ahi) {
    const int kc = khalf * (I / 64) + kk;
    const uint8_t* wl = st + gq * 128 + (kc >> 1) * (16 * 128) + (((2 * q + (kc & 1)) ^ gq) * 16);
    alo = *reinterpret_cast<const uint4*>(wl);
    ahi = *reinterpret_cast<const uint4*>(wl + 8 * 128);
  }
  __device__ static void mma(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                             uint32_t b0, uint32_t b1) {
    mma_bf16(d, a0, a1, a2, a3, b0, b1);
  }
  __device__ static float scale(const ExpertArgs&, int) { return 1.f; }
};

// Map of a Wd stack of `experts` matrices [H][I] (bf16, rows contiguous).
cudaError_t encode_wd(CUtensorMap* m, const uint16_t* w, int experts) {
  const EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {64, (cuuint64_t)experts * H, I / 64};
  const cuuint64_t strides[2] = {(cuuint64_t)I * 2, 128};  // bytes, for dims 1 and 2
  const cuuint32_t box[3] = {64, dring::RS, I / 64};
  const cuuint32_t elem[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint16_t*>(w), dims,
                         strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_down_bf16(const ExpertArgs& a, cudaStream_t stream) {
  Bf16Wd::Maps maps;
  cudaError_t e = encode_wd(&maps.w2, a.w.w2, E);
  if (e == cudaSuccess) e = encode_wd(&maps.ws2, a.w.ws2, S);
  if (e != cudaSuccess) return e;
  return dring::launch_down_ring<Bf16Wd>(a, maps, stream);
}

}  // namespace flint
