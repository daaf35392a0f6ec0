// Row-wise kernels of the MLA path (HBM-bound, one pass over each row):
//   * input RMSNorm x_attn = g * x / sqrt(mean(x^2) + eps) (dense-block page,
//     first equation), float32 math, one bf16 rounding;
//   * split of the A-projection output into c^Q, c^KV and k^pe, with the
//     q_a / kv_a latent RMSNorms and RoPE on the shared rotary key
//     (key-value compression page: split after the product, only the
//     512-wide latent normalised), plus the optional latent-cache write and
//     the RoPE table R_t: (cos, sin)(t * theta_i), theta_i = base^(-2i/64)
//     (dense-block page: "R [T positions, 32 pairs]"), the angle reduced
//     modulo 2 pi in double precision so that large positions keep float
//     accuracy.
#include "common.cuh"
#include "internal.h"

namespace mla {

namespace {

// One CTA of 128 threads per row of 7168 (= 128 threads x 7 uint4).
__global__ void __launch_bounds__(128) rmsnorm_7168_kernel(const __nv_bfloat16* __restrict__ x,
                                                           const __nv_bfloat16* __restrict__ g,
                                                           __nv_bfloat16* __restrict__ y, float eps) {
  constexpr int kVec = 7;  // 7168 / 8 / 128
  pdl_launch_dependents();
  pdl_wait();
  const size_t row = blockIdx.x;
  const uint4* xr = reinterpret_cast<const uint4*>(x + row * 7168);
  uint4 v[kVec];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < kVec; ++j) {
    v[j] = xr[threadIdx.x + j * 128];
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float2 f = unpack_bf16x2(w[q]);
      ss += f.x * f.x + f.y * f.y;
    }
  }
  __shared__ float red[4];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  const float tot = red[0] + red[1] + red[2] + red[3];
  const float rstd = rsqrtf(tot * (1.0f / 7168.0f) + eps);
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  uint4* yr = reinterpret_cast<uint4*>(y + row * 7168);
#pragma unroll
  for (int j = 0; j < kVec; ++j) {
    const uint4 gv = gr[threadIdx.x + j * 128];
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
    const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float2 f = unpack_bf16x2(w[q]);
      float2 gg = unpack_bf16x2(gw[q]);
      o[q] = pack_bf16x2(gg.x * (f.x * rstd), gg.y * (f.y * rstd));
    }
    yr[threadIdx.x + j * 128] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// One warp per row of ca [rows, 2112] (float32) = [c^Q 1536 | c^KV 512 | k^pe 64].
__device__ __forceinline__ void norm_store(const float4* src, int n4, const __nv_bfloat16* g, float eps,
                                           __nv_bfloat16* dst, __nv_bfloat16* dst2, int lane) {
  // n4 float4 per lane (n4 * 4 * 32 values in the row)
  float4 v[12];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < 12; ++j) {
    if (j < n4) {
      v[j] = src[lane + 32 * j];
      ss += v[j].x * v[j].x + v[j].y * v[j].y + v[j].z * v[j].z + v[j].w * v[j].w;
    }
  }
  const float rstd = rsqrtf(warp_sum(ss) / (float)(n4 * 128) + eps);
  const uint2* gp = reinterpret_cast<const uint2*>(g);
  uint2* dp = reinterpret_cast<uint2*>(dst);
  uint2* dp2 = reinterpret_cast<uint2*>(dst2);
#pragma unroll
  for (int j = 0; j < 12; ++j) {
    if (j < n4) {
      const uint2 gv = gp[lane + 32 * j];
      const float2 g0 = unpack_bf16x2(gv.x), g1 = unpack_bf16x2(gv.y);
      const uint2 o = make_uint2(pack_bf16x2(g0.x * (v[j].x * rstd), g0.y * (v[j].y * rstd)),
                                 pack_bf16x2(g1.x * (v[j].z * rstd), g1.y * (v[j].w * rstd)));
      dp[lane + 32 * j] = o;
      if (dst2) dp2[lane + 32 * j] = o;
    }
  }
}

__global__ void __launch_bounds__(256) latent_split_kernel(const LatentArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= a.rows) return;
  const size_t row = warp;
  const float* src = a.ca + row * 2112;
  const int b = (int)(row / a.t_mod);
  const int t = a.t_off + (int)(row % a.t_mod);
  // c^Q-hat = RMSNorm(c^Q): 1536 values = 12 float4 per lane
  norm_store(reinterpret_cast<const float4*>(src), 12, a.g_qa, a.eps, a.cq + row * 1536, nullptr, lane);
  // c^KV-hat = RMSNorm(c^KV): 512 values = 4 float4 per lane; also the latent cache row
  __nv_bfloat16* dcache = a.ckv_cache ? a.ckv_cache + ((size_t)b * a.cap + t) * 512 : nullptr;
  norm_store(reinterpret_cast<const float4*>(src + 1536), 4, a.g_kva, a.eps, a.ckv + row * 512, dcache, lane);
  // R_t: angle (pos0 + t) * theta_i formed and reduced modulo 2 pi in double
  // precision (Cody-Waite style, 2 pi split in two doubles), then a float
  // sincos of the reduced angle
  const int tm = (int)(row % a.t_mod);
  const double ang = (double)(a.pos0 + tm) * a.inv_freq[lane];
  const double kq = rint(ang * 0.15915494309189535);  // 1 / (2 pi)
  const double red = fma(-kq, 6.283185307179586, ang) - kq * 2.4492935982947064e-16;
  float sn, cn;
  sincosf((float)red, &sn, &cn);
  const float2 cs = make_float2(cn, sn);
  if (b == 0) a.cs[(size_t)tm * 32 + lane] = cs;
  // k^R = RoPE(k^pe, t): lane i rotates pair (i, i + 32); k^pe is not normalised
  const float x1 = src[2048 + lane];
  const float x2 = src[2048 + 32 + lane];
  const __nv_bfloat16 y1 = __float2bfloat16_rn(x1 * cs.x - x2 * cs.y);
  const __nv_bfloat16 y2 = __float2bfloat16_rn(x2 * cs.x + x1 * cs.y);
  __nv_bfloat16* d = a.kpe + row * 64;
  d[lane] = y1;
  d[lane + 32] = y2;
  if (a.kpe_cache) {
    __nv_bfloat16* dc = a.kpe_cache + ((size_t)b * a.cap + t) * 64;
    dc[lane] = y1;
    dc[lane + 32] = y2;
  }
}

__global__ void copy_qpe_kernel(const __nv_bfloat16* __restrict__ q, __nv_bfloat16* __restrict__ qlat, int B) {
  pdl_launch_dependents();
  pdl_wait();
  // one thread per (b, h, 16-byte chunk of the 64 pe values): 8 chunks
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= B * 64 * 8) return;
  const int c = idx & 7;
  const int bh = idx >> 3;
  const int b = bh >> 6, h = bh & 63;
  const uint4* s = reinterpret_cast<const uint4*>(q + (size_t)b * 12288 + h * 192 + 128);
  uint4* d = reinterpret_cast<uint4*>(qlat + ((size_t)b * 64 + h) * 576 + 512);
  d[c] = s[c];
}

}  // namespace

cudaError_t launch_rmsnorm_rows(const __nv_bfloat16* x, const __nv_bfloat16* g, __nv_bfloat16* y, int rows,
                                float eps, cudaStream_t stream) {
  return launch_pdl(rmsnorm_7168_kernel, dim3(rows), dim3(128), 0, stream, x, g, y, eps);
}

cudaError_t launch_latent_split(const LatentArgs& a, cudaStream_t stream) {
  const int warps_per_block = 8;
  return launch_pdl(latent_split_kernel, dim3((a.rows + warps_per_block - 1) / warps_per_block),
                    dim3(32 * warps_per_block), 0, stream, a);
}

cudaError_t launch_copy_qpe(const __nv_bfloat16* q, __nv_bfloat16* qlat, int B, cudaStream_t stream) {
  const int n = B * 64 * 8;
  return launch_pdl(copy_qpe_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, q, qlat, B);
}

}  // namespace mla
