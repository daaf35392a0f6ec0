// Decode attention: one new query per sequence against L = P + 1 keys.
//
// (1) Rebuilt per-head cache ("Mix and project" page, decode at P = 1,000:
//     A [B, 64, 1, 1001], V [B, 64, 1001, 128]).  Pure HBM streaming: each
//     (sequence, head) reads its contiguous K rows (384 B) and V rows (256 B)
//     once.  CTA = (batch, head, split); one thread issues cp.async.bulk
//     copies of 32-key chunks into a 4-deep shared-memory ring, four warps
//     compute the 32 scores (8 lanes per key, 16-byte loads), an online
//     softmax and P.V.  Splits of the key range are merged by a combine
//     kernel (log-sum-exp weights).
// (2) Latent cache (576 values per position, key-value compression page):
//     scores s_j = (q_lat . c_j + q_pe . k^R_j) * scale with q_lat = W_UK^T
//     q_nope already formed by a GEMM, o_lat = sum_j p_j c_j; W_UV is applied
//     afterwards by a GEMM.  CUDA-core version, one CTA per (batch, split).
#include "common.cuh"
#include "internal.h"

namespace mla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// rebuilt-cache decode
// ---------------------------------------------------------------------------
constexpr int kDecChunk = 32;
constexpr int kDecStages = 4;

struct __align__(128) DecodeSmem {
  __nv_bfloat16 k[kDecStages][kDecChunk * 192];
  __nv_bfloat16 v[kDecStages][kDecChunk * 128];
  float s[kDecChunk];
  float ohalf[128];
  uint64_t full[kDecStages];
};

__global__ void __launch_bounds__(128) decode_attn_kernel(const DecodeAttnArgs a, const DevStatus st,
                                                          int chunk_len) {
  extern __shared__ __align__(128) uint8_t dec_smem_raw[];
  DecodeSmem& sm = *reinterpret_cast<DecodeSmem*>(dec_smem_raw);
  const int split = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int key_begin = split * chunk_len;
  const int key_end = min(a.L, key_begin + chunk_len);
  const int nchunks = (key_end - key_begin + kDecChunk - 1) / kDecChunk;
  const size_t slot0 = ((size_t)b * 64 + h) * a.cap;
  const __nv_bfloat16* kbase = a.k + slot0 * 192;
  const __nv_bfloat16* vbase = a.v + slot0 * 128;

  if (tid == 0) {
    for (int i = 0; i < kDecStages; ++i) mbar_init(&sm.full[i], 1);
    fence_barrier_init();
  }
  __syncthreads();

  auto issue = [&](int c) {
    const int stg = c % kDecStages;
    const int k0 = key_begin + c * kDecChunk;
    const int n = min(kDecChunk, key_end - k0);
    mbar_arrive_expect_tx(&sm.full[stg], n * 640);
    bulk_load(sm.k[stg], kbase + (size_t)k0 * 192, n * 384, &sm.full[stg]);
    bulk_load(sm.v[stg], vbase + (size_t)k0 * 128, n * 256, &sm.full[stg]);
  };
  if (tid == 0)
    for (int c = 0; c < kDecStages && c < nchunks; ++c) issue(c);

  // query slice held by this lane for the score step: dims part*8 + 64j + e
  const int part = lane & 7;
  float qr[24];
  {
    const __nv_bfloat16* q = a.q + (size_t)b * 12288 + h * 192;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const uint4 u = *reinterpret_cast<const uint4*>(q + part * 8 + 64 * j);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack_bf16x2(w[e]);
        qr[8 * j + 2 * e] = f.x;
        qr[8 * j + 2 * e + 1] = f.y;
      }
    }
  }
  const float sl2 = a.scale * kLog2e;
  float m_run = -INFINITY, l_run = 0.f;
  float o0 = 0.f, o1 = 0.f;
  const int dp = tid & 63;   // output dims 2dp, 2dp+1
  const int kh = tid >> 6;   // key half of each chunk
  int c_fail = -1;

  for (int c = 0; c < nchunks; ++c) {
    const int stg = c % kDecStages;
    const int k0 = key_begin + c * kDecChunk;
    const int n = min(kDecChunk, key_end - k0);
    const bool got = mbar_wait(&sm.full[stg], (c / kDecStages) & 1, st, nullptr, 20);
    if (!__syncthreads_and(got)) {
      c_fail = c;
      break;
    }
    // scores: warp w -> keys 8w .. 8w+7, 4 keys per round, 8 lanes per key
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int key = warp * 8 + r * 4 + (lane >> 3);
      const __nv_bfloat16* kr = sm.k[stg] + key * 192 + part * 8;
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        const uint4 u = *reinterpret_cast<const uint4*>(kr + 64 * j);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack_bf16x2(w[e]);
          acc = fmaf(qr[8 * j + 2 * e], f.x, acc);
          acc = fmaf(qr[8 * j + 2 * e + 1], f.y, acc);
        }
      }
      acc += __shfl_xor_sync(0xffffffffu, acc, 1);
      acc += __shfl_xor_sync(0xffffffffu, acc, 2);
      acc += __shfl_xor_sync(0xffffffffu, acc, 4);
      if (part == 0) sm.s[key] = key < n ? acc * sl2 : -INFINITY;
    }
    __syncthreads();
    // online softmax (every warp holds the same 32 probabilities, lane = key)
    const float s = sm.s[lane];
    const float m_new = fmaxf(m_run, warp_max(s));
    const float alpha = exp2f(m_run - m_new);
    const float p = exp2f(s - m_new);
    l_run = l_run * alpha + warp_sum(p);
    m_run = m_new;
    o0 *= alpha;
    o1 *= alpha;
    const __nv_bfloat162* vr = reinterpret_cast<const __nv_bfloat162*>(sm.v[stg]) + dp;
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      const int key = kh * 16 + kk;
      const float pk = __shfl_sync(0xffffffffu, p, key);
      if (key < n) {
        const float2 vv = __bfloat1622float2(vr[key * 64]);
        o0 = fmaf(pk, vv.x, o0);
        o1 = fmaf(pk, vv.y, o1);
      }
    }
    __syncthreads();
    if (tid == 0 && c + kDecStages < nchunks) issue(c + kDecStages);
  }
  if (c_fail >= 0) {
    // chunks c_fail .. c_fail + stages - 1 may still be in flight: wait (bounded)
    if (tid == 0)
      for (int c = c_fail; c < nchunks && c < c_fail + kDecStages; ++c)
        mbar_wait(&sm.full[c % kDecStages], (c / kDecStages) & 1, st, nullptr, 21);
    return;
  }
  // merge the two key halves
  if (kh == 1) {
    sm.ohalf[2 * dp] = o0;
    sm.ohalf[2 * dp + 1] = o1;
  }
  __syncthreads();
  if (kh == 0) {
    o0 += sm.ohalf[2 * dp];
    o1 += sm.ohalf[2 * dp + 1];
    if (a.splits == 1) {
      const float inv = 1.f / l_run;
      reinterpret_cast<uint32_t*>(a.o + (size_t)b * 8192 + h * 128)[dp] = pack_bf16x2(o0 * inv, o1 * inv);
    } else {
      const size_t pi = ((size_t)b * 64 + h) * a.splits + split;
      reinterpret_cast<float2*>(a.part_o + pi * 128)[dp] = make_float2(o0, o1);
      if (tid == 0) a.part_ml[pi] = make_float2(m_run, l_run);
    }
  }
}

// out[row, 0:width] = sum_s w_s part_o[row, s] / sum_s w_s l_s,  w_s = 2^(m_s - max m)
__global__ void combine_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                               __nv_bfloat16* __restrict__ out, int splits, int width) {
  const size_t row = blockIdx.x;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, part_ml[row * splits + s].x);
  float den = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float2 ml = part_ml[row * splits + s];
    den += exp2f(ml.x - mx) * ml.y;
  }
  const float inv = 1.f / den;
  for (int d = threadIdx.x; d < width; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s)
      acc += exp2f(part_ml[row * splits + s].x - mx) * part_o[(row * splits + s) * width + d];
    out[row * width + d] = __float2bfloat16_rn(acc * inv);
  }
}

// ---------------------------------------------------------------------------
// latent-cache decode (CUDA cores)
// ---------------------------------------------------------------------------
constexpr int kLatChunk = 16;
constexpr int kLatStages = 2;
constexpr int kQStride = 584;  // bf16 per q_lat row in smem (576 + 8 pad)

struct __align__(128) LatentSmem {
  __nv_bfloat16 ckv[kLatStages][kLatChunk * 512];
  __nv_bfloat16 kpe[kLatStages][kLatChunk * 64];
  __nv_bfloat16 q[64 * kQStride];
  uint64_t full[kLatStages];
};

__global__ void __launch_bounds__(256) latent_attn_cuda_core(const LatentAttnArgs a, const DevStatus st,
                                                             int chunk_len) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  LatentSmem& sm = *reinterpret_cast<LatentSmem*>(smem_raw);
  const int split = blockIdx.x;
  const int b = blockIdx.y;
  const int tid = threadIdx.x;
  const int h = tid >> 2;     // head of this thread
  const int sub = tid & 3;    // key phase (scores) and latent quarter (P.V)
  const int key_begin = split * chunk_len;
  const int key_end = min(a.L, key_begin + chunk_len);
  const int nchunks = (key_end - key_begin + kLatChunk - 1) / kLatChunk;
  const __nv_bfloat16* cbase = a.ckv + (size_t)b * a.cap * 512;
  const __nv_bfloat16* rbase = a.kpe + (size_t)b * a.cap * 64;

  if (tid == 0) {
    for (int i = 0; i < kLatStages; ++i) mbar_init(&sm.full[i], 1);
    fence_barrier_init();
  }
  for (int i = tid; i < 64 * 72; i += 256) {
    const int r = i / 72, c = i % 72;
    *reinterpret_cast<uint4*>(&sm.q[r * kQStride + c * 8]) =
        *reinterpret_cast<const uint4*>(a.qlat + ((size_t)b * 64 + r) * 576 + c * 8);
  }
  __syncthreads();
  auto issue = [&](int c) {
    const int stg = c % kLatStages;
    const int k0 = key_begin + c * kLatChunk;
    const int n = min(kLatChunk, key_end - k0);
    mbar_arrive_expect_tx(&sm.full[stg], n * 1152);
    bulk_load(sm.ckv[stg], cbase + (size_t)k0 * 512, n * 1024, &sm.full[stg]);
    bulk_load(sm.kpe[stg], rbase + (size_t)k0 * 64, n * 128, &sm.full[stg]);
  };
  if (tid == 0)
    for (int c = 0; c < kLatStages && c < nchunks; ++c) issue(c);

  const float sl2 = a.scale * kLog2e;
  float m_run = -INFINITY, l_run = 0.f;
  float o[128];
#pragma unroll
  for (int i = 0; i < 128; ++i) o[i] = 0.f;
  int c_fail = -1;
  const __nv_bfloat162* qrow = reinterpret_cast<const __nv_bfloat162*>(&sm.q[h * kQStride]);

  for (int c = 0; c < nchunks; ++c) {
    const int stg = c % kLatStages;
    const int k0 = key_begin + c * kLatChunk;
    const int n = min(kLatChunk, key_end - k0);
    const bool got = mbar_wait(&sm.full[stg], (c / kLatStages) & 1, st, nullptr, 30);
    if (!__syncthreads_and(got)) {
      c_fail = c;
      break;
    }
    // scores for keys sub + 4i, i = 0..3
    float s[4] = {0.f, 0.f, 0.f, 0.f};
    const __nv_bfloat162* cr = reinterpret_cast<const __nv_bfloat162*>(sm.ckv[stg]);
    const __nv_bfloat162* rr = reinterpret_cast<const __nv_bfloat162*>(sm.kpe[stg]);
#pragma unroll 4
    for (int d2 = 0; d2 < 256; ++d2) {
      const float2 qv = __bfloat1622float2(qrow[d2]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 kv = __bfloat1622float2(cr[(sub + 4 * i) * 256 + d2]);
        s[i] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, s[i]));
      }
    }
#pragma unroll 4
    for (int d2 = 0; d2 < 32; ++d2) {
      const float2 qv = __bfloat1622float2(qrow[256 + d2]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 kv = __bfloat1622float2(rr[(sub + 4 * i) * 32 + d2]);
        s[i] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, s[i]));
      }
    }
    float mt = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      s[i] = (sub + 4 * i < n) ? s[i] * sl2 : -INFINITY;
      mt = fmaxf(mt, s[i]);
    }
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 1));
    mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, 2));
    const float m_new = fmaxf(m_run, mt);
    const float alpha = exp2f(m_run - m_new);
    float p[4], ls = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      p[i] = exp2f(s[i] - m_new);
      ls += p[i];
    }
    ls += __shfl_xor_sync(0xffffffffu, ls, 1);
    ls += __shfl_xor_sync(0xffffffffu, ls, 2);
    l_run = l_run * alpha + ls;
    m_run = m_new;
#pragma unroll
    for (int i = 0; i < 128; ++i) o[i] *= alpha;
    // P.V over latent dims sub*128 .. +127
    const int lane_base = (threadIdx.x & 31) & ~3;
#pragma unroll 1
    for (int j = 0; j < kLatChunk; ++j) {
      const int pi = j >> 2;
      const float psel = pi == 0 ? p[0] : pi == 1 ? p[1] : pi == 2 ? p[2] : p[3];
      const float pj = __shfl_sync(0xffffffffu, psel, lane_base + (j & 3));
      if (j < n) {
        const __nv_bfloat162* vr = cr + j * 256 + sub * 64;
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          const float2 vv = __bfloat1622float2(vr[e]);
          o[2 * e] = fmaf(pj, vv.x, o[2 * e]);
          o[2 * e + 1] = fmaf(pj, vv.y, o[2 * e + 1]);
        }
      }
    }
    __syncthreads();
    if (tid == 0 && c + kLatStages < nchunks) issue(c + kLatStages);
  }
  if (c_fail >= 0) {
    if (tid == 0)
      for (int c = c_fail; c < nchunks && c < c_fail + kLatStages; ++c)
        mbar_wait(&sm.full[c % kLatStages], (c / kLatStages) & 1, st, nullptr, 31);
    return;
  }
  if (a.splits == 1) {
    const float inv = 1.f / l_run;
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.olat + ((size_t)b * 64 + h) * 512 + sub * 128);
#pragma unroll
    for (int e = 0; e < 64; ++e) dst[e] = pack_bf16x2(o[2 * e] * inv, o[2 * e + 1] * inv);
  } else {
    const size_t pi = ((size_t)b * a.splits + split) * 64 + h;
    float4* dst = reinterpret_cast<float4*>(a.part_o + pi * 512 + sub * 128);
#pragma unroll
    for (int e = 0; e < 32; ++e) dst[e] = make_float4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
    if (sub == 0) a.part_ml[pi] = make_float2(m_run, l_run);
  }
}

// latent partials are laid out [(b*splits + s), 64, 512]; the generic combine
// expects [(row*splits + s), width] with row = (b, h): regroup here.
__global__ void latent_combine_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                                      __nv_bfloat16* __restrict__ out, int splits) {
  const int h = blockIdx.x, b = blockIdx.y;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, part_ml[((size_t)b * splits + s) * 64 + h].x);
  float den = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float2 ml = part_ml[((size_t)b * splits + s) * 64 + h];
    den += exp2f(ml.x - mx) * ml.y;
  }
  const float inv = 1.f / den;
  for (int d = threadIdx.x; d < 512; d += blockDim.x) {
    float acc = 0.f;
    for (int s = 0; s < splits; ++s) {
      const size_t pi = ((size_t)b * splits + s) * 64 + h;
      acc += exp2f(part_ml[pi].x - mx) * part_o[pi * 512 + d];
    }
    out[((size_t)b * 64 + h) * 512 + d] = __float2bfloat16_rn(acc * inv);
  }
}

int chunk_len_for(int L, int splits, int granule) {
  int c = (L + splits - 1) / splits;
  return (c + granule - 1) / granule * granule;
}

}  // namespace

int decode_splits(int B, int L, int num_sms) {
  const int pairs = B * 64;
  const int want = 4 * num_sms;  // about 2 waves of 2 resident CTAs per SM
  int s = (want + pairs - 1) / pairs;
  const int max_s = (L + 127) / 128;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  // re-derive so that every split holds at least one key
  const int cl = chunk_len_for(L, s, kDecChunk);
  return (L + cl - 1) / cl;
}

cudaError_t launch_decode_attention(const DecodeAttnArgs& a, const DevStatusHost& st, cudaStream_t stream,
                                    int* launches) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(decode_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(DecodeSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int cl = chunk_len_for(a.L, a.splits, kDecChunk);
  DevStatus dst{st.word, st.wait_limit_ns};
  dim3 grid(a.splits, 64, a.B);
  decode_attn_kernel<<<grid, 128, sizeof(DecodeSmem), stream>>>(a, dst, cl);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
  if (a.splits > 1) {
    combine_kernel<<<a.B * 64, 64, 0, stream>>>(a.part_o, a.part_ml, a.o, a.splits, 128);
    e = cudaGetLastError();
    ++*launches;
  }
  return e;
}

int latent_splits(int B, int L, int num_sms) {
  int s = (2 * num_sms + B - 1) / B;
  const int max_s = (L + 63) / 64;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  const int cl = chunk_len_for(L, s, kLatChunk);
  return (L + cl - 1) / cl;
}

cudaError_t launch_latent_attention(const LatentAttnArgs& a, const DevStatusHost& st, cudaStream_t stream,
                                    int* launches) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(latent_attn_cuda_core, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(LatentSmem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int cl = chunk_len_for(a.L, a.splits, kLatChunk);
  DevStatus dst{st.word, st.wait_limit_ns};
  dim3 grid(a.splits, a.B);
  latent_attn_cuda_core<<<grid, 256, sizeof(LatentSmem), stream>>>(a, dst, cl);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  ++*launches;
  if (a.splits > 1) {
    latent_combine_kernel<<<dim3(64, a.B), 128, 0, stream>>>(a.part_o, a.part_ml, a.olat, a.splits);
    e = cudaGetLastError();
    ++*launches;
  }
  return e;
}

}  // namespace mla
