// FP8 block-scaled weights: quantization of a bf16 [rows, cols] matrix into
// E4M3 codes with one power-of-two scale per 128 x 128 block.  The dense-block
// page counts the checkpoint's tensors "FP8 block scales excluded": the
// weights are stored in FP8 with one scale per block.  Block size and scale
// format are not printed; here: 128 x 128 blocks, scale 2^k with the smallest
// k such that amax(block) <= 448 * 2^k (448 = the largest finite E4M3 value),
// code = E4M3 round-to-nearest-even (saturating) of w / 2^k.  The stored
// weight q * 2^k is then exact in bfloat16, so dequantization adds no
// rounding of its own.  Codes are stored block-major (each 128 x 128 block
// 16 KB contiguous, row-major inside, rows past the matrix zero), so that a
// tile of rows of one 128-wide K slice is one contiguous read.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace mla {

namespace {

constexpr int kQBlock = 128;

// One CTA (256 threads) per 128 x 128 block: thread tid holds row tid / 2,
// columns (tid & 1) * 64 .. + 63 of the block.
__global__ void __launch_bounds__(256) fp8_quantize_kernel(const __nv_bfloat16* __restrict__ w, int rows, int cols,
                                                           uint8_t* __restrict__ codes, float* __restrict__ scales,
                                                           int nb_c) {
  pdl_launch_dependents();
  pdl_wait();
  const int bi = blockIdx.y, bj = blockIdx.x;
  const int r0 = bi * kQBlock, c0 = bj * kQBlock;
  const int tid = threadIdx.x;
  // thread tid: row r0 + tid / 2, columns c0 + (tid & 1) * 64 .. + 63
  const int r = r0 + (tid >> 1);
  const int cb = c0 + (tid & 1) * 64;
  float v[64];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const int c = cb + i;
    v[i] = (r < rows && c < cols) ? __bfloat162float(w[(size_t)r * cols + c]) : 0.f;
    amax = fmaxf(amax, fabsf(v[i]));
  }
  __shared__ float red[8];
  amax = warp_max(amax);
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  float a = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
  // smallest k with a <= 448 * 2^k: a = m 2^e (m in [0.5, 1)), 448 = 0.875 2^9
  int k = 0;
  if (a > 0.f) {
    int e;
    const float m = frexpf(a, &e);
    k = m <= 0.875f ? e - 9 : e - 8;
  }
  if (tid == 0) scales[(size_t)bi * nb_c + bj] = ldexpf(1.f, k);
  // this thread's 64 codes: bytes (tid / 2) * 128 + (tid & 1) * 64 .. of the block
  uint8_t* dst = codes + ((size_t)bi * nb_c + bj) * (kQBlock * kQBlock) + (size_t)(tid >> 1) * kQBlock + (tid & 1) * 64;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t word = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = 16 * j + 4 * q + e;
        const uint32_t code =
            (r < rows) ? (uint32_t)__nv_cvt_float_to_fp8(ldexpf(v[i], -k), __NV_SATFINITE, __NV_E4M3) : 0u;
        word |= code << (8 * e);
      }
      w[q] = word;
    }
    reinterpret_cast<uint4*>(dst)[j] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace

cudaError_t launch_fp8_quantize(const __nv_bfloat16* w, int rows, int cols, uint8_t* codes, float* scales,
                                cudaStream_t stream) {
  if (cols % kQBlock) return cudaErrorInvalidValue;
  const int nb_r = (rows + kQBlock - 1) / kQBlock, nb_c = cols / kQBlock;
  return launch_pdl(fp8_quantize_kernel, dim3(nb_c, nb_r), dim3(256), 0, stream, w, rows, cols, codes, scales, nb_c);
}

}  // namespace mla
