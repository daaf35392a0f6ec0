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
  const uint4* gr = reinterpret_cast<const uint4*>(g);
  uint4 gvs[kVec];  // gains fetched before the reduction (its latency overlaps the loads')
#pragma unroll
  for (int j = 0; j < kVec; ++j) gvs[j] = gr[threadIdx.x + j * 128];
  __shared__ float red[4];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  const float tot = red[0] + red[1] + red[2] + red[3];
  const float rstd = rsqrtf(tot * (1.0f / 7168.0f) + eps);
  uint4* yr = reinterpret_cast<uint4*>(y + row * 7168);
#pragma unroll
  for (int j = 0; j < kVec; ++j) {
    const uint4 gv = gvs[j];
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

// One CTA of 128 threads per row of ca [rows, 2112] (float32) =
// [c^Q 1536 | c^KV 512 | k^pe 64]; every load (row and gains) is issued
// before the two reductions.
__device__ __forceinline__ uint2 scale_pack4(const float4 v, const uint2 gv, float rstd) {
  const float2 g0 = unpack_bf16x2(gv.x), g1 = unpack_bf16x2(gv.y);
  return make_uint2(pack_bf16x2(g0.x * (v.x * rstd), g0.y * (v.y * rstd)),
                    pack_bf16x2(g1.x * (v.z * rstd), g1.y * (v.w * rstd)));
}

__global__ void __launch_bounds__(128) latent_split_kernel(const LatentArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int row = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* src = a.ca + (size_t)row * 2112;
  const float4* src4 = reinterpret_cast<const float4*>(src);
  float4 q[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) q[j] = src4[tid + 128 * j];  // c^Q: 384 float4
  const float4 kv = src4[384 + tid];                       // c^KV: 128 float4
  float x1 = 0.f, x2 = 0.f;
  if (tid < 32) {  // k^pe pair (tid, tid + 32)
    x1 = src[2048 + tid];
    x2 = src[2048 + 32 + tid];
  }
  uint2 gq[3];
#pragma unroll
  for (int j = 0; j < 3; ++j) gq[j] = reinterpret_cast<const uint2*>(a.g_qa)[tid + 128 * j];
  const uint2 gk = reinterpret_cast<const uint2*>(a.g_kva)[tid];
  float ssq = 0.f;
#pragma unroll
  for (int j = 0; j < 3; ++j) ssq += q[j].x * q[j].x + q[j].y * q[j].y + q[j].z * q[j].z + q[j].w * q[j].w;
  float ssk = kv.x * kv.x + kv.y * kv.y + kv.z * kv.z + kv.w * kv.w;
  __shared__ float red[2][4];
  ssq = warp_sum(ssq);
  ssk = warp_sum(ssk);
  if (lane == 0) {
    red[0][warp] = ssq;
    red[1][warp] = ssk;
  }
  __syncthreads();
  const int b = row / a.t_mod;
  const int tm = row - b * a.t_mod;
  // position of this row: pos0 + tm (prefill, uniform decode) or its own
  // (decode with per-sequence lengths, t_mod = 1)
  int pos_row = a.pos0 + tm, t = a.t_off + tm;
  if (a.pos) {
    const int p = a.pos[row];
    if ((p < 0 || p > a.pos_max) && tid == 0 && a.status) atomicOr(a.status, kStatusBadLength);
    pos_row = t = clamp_pos(p, a.pos_max);
  }
  // c^Q-hat = RMSNorm(c^Q); c^KV-hat = RMSNorm(c^KV) (also the latent cache row)
  const float rq = rsqrtf(((red[0][0] + red[0][1]) + (red[0][2] + red[0][3])) * (1.0f / 1536.0f) + a.eps);
  const float rk = rsqrtf(((red[1][0] + red[1][1]) + (red[1][2] + red[1][3])) * (1.0f / 512.0f) + a.eps);
  uint2* dq = reinterpret_cast<uint2*>(a.cq + (size_t)row * 1536);
#pragma unroll
  for (int j = 0; j < 3; ++j) dq[tid + 128 * j] = scale_pack4(q[j], gq[j], rq);
  const uint2 ok = scale_pack4(kv, gk, rk);
  reinterpret_cast<uint2*>(a.ckv + (size_t)row * 512)[tid] = ok;
  if (a.ckv_cache) reinterpret_cast<uint2*>(a.ckv_cache + ((size_t)b * a.cap + t) * 512)[tid] = ok;
  if (tid < 32) {
    // R_t: angle (pos0 + t) * theta_i formed and reduced modulo 2 pi in double
    // precision (Cody-Waite style, 2 pi split in two doubles), then a float
    // sincos of the reduced angle
    const double ang = (double)pos_row * a.inv_freq[lane];
    const double kq = rint(ang * 0.15915494309189535);  // 1 / (2 pi)
    const double red2 = fma(-kq, 6.283185307179586, ang) - kq * 2.4492935982947064e-16;
    float sn, cn;
    sincosf((float)red2, &sn, &cn);
    const float2 cs = make_float2(cn, sn);
    if (a.pos)
      a.cs[(size_t)row * 32 + lane] = cs;  // one table row per token
    else if (b == 0)
      a.cs[(size_t)tm * 32 + lane] = cs;
    // k^R = RoPE(k^pe, t): lane i rotates pair (i, i + 32); k^pe is not normalised
    const __nv_bfloat16 y1 = __float2bfloat16_rn(x1 * cs.x - x2 * cs.y);
    const __nv_bfloat16 y2 = __float2bfloat16_rn(x2 * cs.x + x1 * cs.y);
    __nv_bfloat16* d = a.kpe + (size_t)row * 64;
    d[lane] = y1;
    d[lane + 32] = y2;
    if (a.kpe_cache) {
      __nv_bfloat16* dc = a.kpe_cache + ((size_t)b * a.cap + t) * 64;
      dc[lane] = y1;
      dc[lane + 32] = y2;
    }
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

// pos[i] = p0 + i % t: the position of each token of a chunk (rows ordered
// by sequence, then token)
__global__ void chunk_positions_kernel(int* __restrict__ pos, int n, int t, int p0) {
  pdl_launch_dependents();
  pdl_wait();  // the previous call may still read the array
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) pos[i] = p0 + i % t;
}

}  // namespace

cudaError_t launch_chunk_positions(int* pos, int n, int t, int p0, cudaStream_t stream) {
  if (n < 1 || t < 1) return cudaErrorInvalidValue;
  return launch_pdl(chunk_positions_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, pos, n, t, p0);
}

cudaError_t launch_rmsnorm_rows(const __nv_bfloat16* x, const __nv_bfloat16* g, __nv_bfloat16* y, int rows,
                                float eps, cudaStream_t stream) {
  return launch_pdl(rmsnorm_7168_kernel, dim3(rows), dim3(128), 0, stream, x, g, y, eps);
}

cudaError_t launch_latent_split(const LatentArgs& a, cudaStream_t stream) {
  return launch_pdl(latent_split_kernel, dim3(a.rows), dim3(128), 0, stream, a);
}

cudaError_t launch_copy_qpe(const __nv_bfloat16* q, __nv_bfloat16* qlat, int B, cudaStream_t stream) {
  const int n = B * 64 * 8;
  return launch_pdl(copy_qpe_kernel, dim3((n + 255) / 256), dim3(256), 0, stream, q, qlat, B);
}

}  // namespace mla
