// Causal prefill attention for MLA heads (qk = 192, v = 128).
//
// "Mix and project" page, code excerpt: scores = Q K^T * softmax_scale plus
// the causal mask, softmax in float32, then P V.  This kernel computes it in
// the flash form (online softmax over key tiles; the probabilities never
// reach global memory) on the CUDA cores, in float32.
//
// Layout: q [B*T, 64*192] (token-major, head h at columns h*192), k/v caches
// [B, 64, cap, 192|128], o [B*T, 64*128].
// CTA = (64-query block, head, batch); 256 threads; thread (qi, sub) owns
// query qi, keys sub + 4j of each 64-key tile and output dims sub*32..+31.
#include "common.cuh"
#include "internal.h"

namespace mla {

namespace {

constexpr int kQB = 64;                 // queries per CTA
constexpr int kKB = 64;                 // keys per tile
constexpr int kKStride = 196;           // bf16 per K row in smem (192 + 4 pad)
constexpr int kVStride = 136;           // bf16 per V row in smem (128 + 8 pad)
constexpr int kQStride = 196;

struct __align__(16) PrefillSmem {
  __nv_bfloat16 q[kQB * kQStride];
  __nv_bfloat16 k[kKB * kKStride];
  __nv_bfloat16 v[kKB * kVStride];
  float p[kQB][kKB + 1];
};

__global__ void __launch_bounds__(256) prefill_attn_cuda_core(const PrefillAttnArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  PrefillSmem& sm = *reinterpret_cast<PrefillSmem*>(smem_raw);
  const int nqb = (a.T + kQB - 1) / kQB;
  const int qb = nqb - 1 - (int)blockIdx.x;  // heaviest blocks first
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x;
  const int qi = tid >> 2;
  const int sub = tid & 3;
  const int q0 = qb * kQB;
  const float sl2 = a.scale * 1.4426950408889634f;  // scores in log2 units

  // load the Q block (zero rows beyond T)
  for (int i = tid; i < kQB * 24; i += 256) {
    const int r = i / 24, c = i % 24;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (q0 + r < a.T)
      val = *reinterpret_cast<const uint4*>(a.q + ((size_t)b * a.T + q0 + r) * 12288 + h * 192 + c * 8);
    *reinterpret_cast<uint2*>(&sm.q[r * kQStride + c * 8]) = make_uint2(val.x, val.y);
    *reinterpret_cast<uint2*>(&sm.q[r * kQStride + c * 8 + 4]) = make_uint2(val.z, val.w);
  }

  float o[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) o[i] = 0.f;
  float m_run = -INFINITY, l_run = 0.f;
  const int qpos = q0 + qi;
  const size_t kv_base = ((size_t)b * 64 + h) * a.cap;
  const int n_tiles = min(qb + 1, (a.T + kKB - 1) / kKB);

  for (int kt = 0; kt < n_tiles; ++kt) {
    const int k0 = kt * kKB;
    __syncthreads();
    for (int i = tid; i < kKB * 24; i += 256) {
      const int r = i / 24, c = i % 24;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (k0 + r < a.T) val = *reinterpret_cast<const uint4*>(a.k + (kv_base + k0 + r) * 192 + c * 8);
      *reinterpret_cast<uint2*>(&sm.k[r * kKStride + c * 8]) = make_uint2(val.x, val.y);
      *reinterpret_cast<uint2*>(&sm.k[r * kKStride + c * 8 + 4]) = make_uint2(val.z, val.w);
    }
    for (int i = tid; i < kKB * 16; i += 256) {
      const int r = i / 16, c = i % 16;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (k0 + r < a.T) val = *reinterpret_cast<const uint4*>(a.v + (kv_base + k0 + r) * 128 + c * 8);
      *reinterpret_cast<uint4*>(&sm.v[r * kVStride + c * 8]) = val;
    }
    __syncthreads();

    float s[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) s[j] = 0.f;
    const __nv_bfloat162* qrow = reinterpret_cast<const __nv_bfloat162*>(&sm.q[qi * kQStride]);
#pragma unroll 4
    for (int d2 = 0; d2 < 96; ++d2) {
      const float2 qv = __bfloat1622float2(qrow[d2]);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const float2 kv = __bfloat1622float2(
            reinterpret_cast<const __nv_bfloat162*>(&sm.k[(sub + 4 * j) * kKStride])[d2]);
        s[j] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, s[j]));
      }
    }
    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int key = k0 + sub + 4 * j;
      s[j] = (key <= qpos && key < a.T) ? s[j] * sl2 : -INFINITY;
      mt = fmaxf(mt, s[j]);
    }
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const float m_new = fmaxf(m_run, mt);
    // rows beyond T see only masked keys: keep them finite
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = exp2f(m_run - m_use);
    float ls = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float p = exp2f(s[j] - m_use);
      ls += p;
      sm.p[qi][sub + 4 * j] = p;
    }
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    l_run = l_run * alpha + ls;
    m_run = m_new;
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] *= alpha;
    __syncwarp();
#pragma unroll 2
    for (int kj = 0; kj < kKB; ++kj) {
      const float p = sm.p[qi][kj];
      const __nv_bfloat162* vr = reinterpret_cast<const __nv_bfloat162*>(&sm.v[kj * kVStride + sub * 32]);
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 vv = __bfloat1622float2(vr[e]);
        o[2 * e] = fmaf(p, vv.x, o[2 * e]);
        o[2 * e + 1] = fmaf(p, vv.y, o[2 * e + 1]);
      }
    }
  }
  if (qpos < a.T) {
    const float inv = 1.f / l_run;
    uint32_t packed[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) packed[e] = pack_bf16x2(o[2 * e] * inv, o[2 * e + 1] * inv);
    uint4* dst = reinterpret_cast<uint4*>(a.o + ((size_t)b * a.T + qpos) * 8192 + h * 128 + sub * 32);
#pragma unroll
    for (int j = 0; j < 4; ++j) dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
  }
}

}  // namespace

cudaError_t launch_prefill_attention(const PrefillAttnArgs& a, const DevStatusHost& st, int num_sms,
                                     cudaStream_t stream) {
  (void)st;
  (void)num_sms;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(prefill_attn_cuda_core, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(PrefillSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((a.T + kQB - 1) / kQB, 64, a.B);
  prefill_attn_cuda_core<<<grid, 256, sizeof(PrefillSmem), stream>>>(a);
  return cudaGetLastError();
}

}  // namespace mla
