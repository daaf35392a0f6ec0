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
//     afterwards by a GEMM.  Tensor cores (tcgen05), one CTA per (batch, split).
#include "common.cuh"
#include "internal.h"

namespace mla {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThresholdLatent = 8.0f;  // log2 units

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
  pdl_launch_dependents();
  pdl_wait();

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
  pdl_launch_dependents();
  pdl_wait();
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
// latent-cache decode on tcgen05
//
// CTA = (sequence b, split of the key range), 192 threads:
//   warp 0     TMA: q_lat [64 heads x 576] once; per 64-key tile the latent
//              rows c_j [64 x 512] (8 boxes) and rotary keys k^R_j [64 x 64]
//              into a 2-stage ring (3D tensor maps bound positions to L, so
//              rows >= L read as zeros)
//   warp 1     TMEM allocation; one lane issues
//                S_j   = q_lat . [c_j ; k^R_j]^T      M=64 (heads) N=64 K=576
//                O^T  += c_j^T . P_j^T               M=128 (latent, 4 blocks)
//                                                    N=64 (heads) K=64 keys
//              (O is kept transposed so the 512-wide latent output takes 256
//              TMEM columns; c_j serves as the K-major B operand of S and the
//              MN-major A operand of O^T without a copy)
//   warps 2..5 softmax: head h = 16*(warp%4) + lane (lanes 0..15; an M=64
//              accumulator row r lives in TMEM lane 32*(r/16) + r%16), lazy
//              rescaling (O^T columns rescaled only when a head's max grows by
//              more than 2^8), P_j [64 heads x 64 keys] bf16 to shared memory;
//              at the end every thread writes the latent rows it holds.
// ---------------------------------------------------------------------------
constexpr int kLatTile = 64;
constexpr uint32_t kLatBox = 64 * 128;                       // 64 rows x 64 bf16
constexpr uint32_t kLatQOff = 0;                             // 9 boxes
constexpr uint32_t kLatCOff = 9 * kLatBox;                   // 2 stages x 8 boxes
constexpr uint32_t kLatROff = kLatCOff + 16 * kLatBox;       // 2 stages x 1 box
constexpr uint32_t kLatPOff = kLatROff + 2 * kLatBox;        // 1 box
constexpr uint32_t kLatBarOff = kLatPOff + kLatBox;
constexpr uint32_t kLatSmemBytes = kLatBarOff + 1536 + 1024;

struct LatBars {
  uint64_t q_full;
  uint64_t c_full[2], c_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, pv_done, drain;
  uint32_t tmem_slot;
  int abort;
  int need[2][4];
  float alpha[2][64];
  float m[64], l[64];
};

__device__ __forceinline__ void named_sync_128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__global__ void __launch_bounds__(192, 1)
    latent_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmR, const LatentAttnArgs a, const DevStatus st,
                   int chunk_len) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  LatBars* bar = reinterpret_cast<LatBars*>(smem + kLatBarOff);
  volatile int* abort_flag = &bar->abort;
  const int split = blockIdx.x;
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int key_begin = split * chunk_len;
  const int key_end = min(a.L, key_begin + chunk_len);
  const int n_tiles = (key_end - key_begin + kLatTile - 1) / kLatTile;

  if (threadIdx.x == 0) {
    mbar_init(&bar->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->c_full[i], 1);
      mbar_init(&bar->c_empty[i], 1);
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->s_free[i], 128);
    }
    mbar_init(&bar->p_full, 128);
    mbar_init(&bar->pv_done, 1);
    mbar_init(&bar->drain, 1);
    bar->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bar->tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmC);
      tma_prefetch_desc(&tmR);
      mbar_arrive_expect_tx(&bar->q_full, 9 * kLatBox);
      for (int c = 0; c < 9; ++c) tma_load_2d(smem + kLatQOff + c * kLatBox, &tmQ, &bar->q_full, 64 * c, b * 64);
      int issued[2] = {0, 0};
      for (int j = 0; j < n_tiles; ++j) {
        const int stg = j & 1;
        if (!mbar_wait(&bar->c_empty[stg], ((j >> 1) & 1) ^ 1, st, abort_flag, 60)) break;
        const int k0 = key_begin + j * kLatTile;
        mbar_arrive_expect_tx(&bar->c_full[stg], 9 * kLatBox);
        for (int c = 0; c < 8; ++c)
          tma_load_3d(smem + kLatCOff + (stg * 8 + c) * kLatBox, &tmC, &bar->c_full[stg], 64 * c, k0, b);
        tma_load_3d(smem + kLatROff + stg * kLatBox, &tmR, &bar->c_full[stg], 0, k0, b);
        issued[stg]++;
      }
      mbar_wait(&bar->q_full, 0, st, nullptr, 61);
      for (int i = 0; i < 2; ++i)
        if (issued[i]) mbar_wait(&bar->c_full[i], (issued[i] - 1) & 1, st, nullptr, 61);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16(64, 64, false, false);
      constexpr uint32_t idesc_o = idesc_bf16(128, 64, true, false);
      const uint32_t q_addr = smem_u32(smem + kLatQOff);
      const uint32_t c_addr = smem_u32(smem + kLatCOff);
      const uint32_t r_addr = smem_u32(smem + kLatROff);
      const uint32_t p_addr = smem_u32(smem + kLatPOff);
      bool ok = mbar_wait(&bar->q_full, 0, st, abort_flag, 62);
      tc_fence_after();
      // Event loop: S_j needs its latent tile and a free score buffer; P.V_j
      // needs P_j.  Issue whichever is ready (S at most two tiles ahead), so
      // that a P.V never waits behind the load of a later tile.
      int next_s = 0, next_pv = 0;
      Watchdog wd;
      wd.reset();
      while (ok && next_pv < n_tiles) {
        bool progress = false;
        if (next_s < n_tiles && next_s <= next_pv + 1) {
          const int stg = next_s & 1;
          const uint32_t ph = (next_s >> 1) & 1;
          if (mbar_test(&bar->c_full[stg], ph) && mbar_test(&bar->s_free[stg], ph ^ 1)) {
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 36; ++kk) {
              const int box = kk >> 2;
              const uint32_t koff = (kk & 3) * 32;
              const uint32_t bb = (box < 8 ? c_addr + (stg * 8 + box) * kLatBox : r_addr + stg * kLatBox) + koff;
              umma_bf16(tmem + stg * 64, sdesc_sw128(q_addr + box * kLatBox + koff, 16, 1024),
                        sdesc_sw128(bb, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
            }
            umma_commit(&bar->s_full[stg]);
            ++next_s;
            progress = true;
          }
        }
        if (next_pv < next_s && mbar_test(&bar->p_full, next_pv & 1)) {
          tc_fence_after();
          const uint32_t cb = c_addr + (next_pv & 1) * 8 * kLatBox;
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = sdesc_sw128(cb + 2 * mb * kLatBox + kk * 2048, kLatBox, 1024);
              const uint64_t bdesc = sdesc_sw128(p_addr + kk * 32, 16, 1024);
              umma_bf16(tmem + 128 + mb * 64, adesc, bdesc, idesc_o, (next_pv > 0 || kk > 0) ? 1u : 0u);
            }
          }
          umma_commit(&bar->pv_done);
          umma_commit(&bar->c_empty[next_pv & 1]);
          ++next_pv;
          progress = true;
        }
        if (progress) {
          wd.reset();
        } else {
          if (wd.expired(st, abort_flag, 63)) break;
          __nanosleep(32);
        }
      }
      umma_commit(&bar->drain);
      mbar_wait(&bar->drain, 0, st, nullptr, 66);
    }
  } else {
    const int quarter = warp & 3;
    const int tid = threadIdx.x - 64;
    const bool valid = lane < 16;
    const int h = quarter * 16 + (lane & 15);
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    uint8_t* pbuf = smem + kLatPOff;
    const float sl2 = a.scale * kLog2e;
    float m = -INFINITY, l = 0.f;
    // Every softmax warp runs every iteration and reaches every named barrier
    // (bar.sync has no time limit); after a failed wait (ok == false) the
    // work of the remaining iterations is skipped, the barriers are not.
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int stg = j & 1;
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&bar->s_full[stg], (j >> 1) & 1, st, abort_flag, 67));
      uint32_t s[64];
      if (ok) {
        tc_fence_after();
        uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
        uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
        tmem_ld32(tmem + lane_addr + stg * 64, s0);
        tmem_ld32(tmem + lane_addr + stg * 64 + 32, s1);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar->s_free[stg]);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) s[c] = 0u;
      }
      const int k0 = key_begin + j * kLatTile;
      float mx = -INFINITY;
      if (k0 + kLatTile > key_end) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (k0 + c >= key_end) s[c] = __float_as_uint(-INFINITY);
      }
      {
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = __uint_as_float(s[i]);
#pragma unroll
        for (int c = 8; c < 64; ++c) mp[c & 7] = fmaxf(mp[c & 7], __uint_as_float(s[c]));
        mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])), fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      }
      mx *= sl2;  // log2 units (the scale is positive)
      const bool need = valid && mx > m + kRescaleThresholdLatent;
      const float m_new = need ? mx : m;
      const float alpha = need ? ex2_approx(m - m_new) : 1.f;
      float sp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p = ex2_approx(fmaf(__uint_as_float(s[c]), sl2, -m_new));
        s[c] = __float_as_uint(p);
        sp[c & 7] += p;
      }
      const float sum = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
      l = l * alpha + sum;
      m = m_new;
      if (valid) bar->alpha[stg][h] = alpha;
      const bool warp_need = __any_sync(0xffffffffu, need);
      if (lane == 0) bar->need[stg][quarter] = warp_need ? 1 : 0;
      named_sync_128();
      const bool any_need = bar->need[stg][0] | bar->need[stg][1] | bar->need[stg][2] | bar->need[stg][3];
      if (j > 0) ok = ok && __all_sync(0xffffffffu, mbar_wait(&bar->pv_done, (j - 1) & 1, st, abort_flag, 68));
      if (!ok) continue;
      if (j > 0) {
        tc_fence_after();
        if (any_need) {
#pragma unroll 1
          for (int mb = 0; mb < 4; ++mb) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t r[32];
              const uint32_t ta = tmem + lane_addr + 128 + mb * 64 + half * 32;
              tmem_ld32(ta, r);
              tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                r[i] = __float_as_uint(__uint_as_float(r[i]) * bar->alpha[stg][half * 32 + i]);
              tmem_st32(ta, r);
            }
          }
          tmem_wait_st();
        }
      }
      if (valid) {
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          const int k = c8 * 8;
          const uint4 v = make_uint4(pack_bf16x2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])),
                                     pack_bf16x2(__uint_as_float(s[k + 2]), __uint_as_float(s[k + 3])),
                                     pack_bf16x2(__uint_as_float(s[k + 4]), __uint_as_float(s[k + 5])),
                                     pack_bf16x2(__uint_as_float(s[k + 6]), __uint_as_float(s[k + 7])));
          *reinterpret_cast<uint4*>(pbuf + h * 128 + ((c8 ^ (h & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar->p_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&bar->pv_done, (n_tiles - 1) & 1, st, abort_flag, 69));
    if (valid) {
      bar->m[h] = m;
      bar->l[h] = l;
    }
    named_sync_128();
    if (ok) {
      tc_fence_after();
      const size_t prow = (size_t)b * a.splits + split;
#pragma unroll 1
      for (int mb = 0; mb < 4; ++mb) {
        const int latent = mb * 128 + quarter * 32 + lane;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_addr + 128 + mb * 64 + half * 32, r);
          tmem_wait_ld();
          if (a.splits == 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int hh = half * 32 + i;
              a.olat[((size_t)b * 64 + hh) * 512 + latent] = __float2bfloat16_rn(__uint_as_float(r[i]) / bar->l[hh]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int hh = half * 32 + i;
              a.part_o[(prow * 64 + hh) * 512 + latent] = __uint_as_float(r[i]);
            }
          }
        }
      }
      if (a.splits > 1 && tid < 64) a.part_ml[prow * 64 + tid] = make_float2(bar->m[tid], bar->l[tid]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// latent partials are laid out [(b*splits + s), 64, 512]; the generic combine
// expects [(row*splits + s), width] with row = (b, h): regroup here.
__global__ void latent_combine_kernel(const float* __restrict__ part_o, const float2* __restrict__ part_ml,
                                      __nv_bfloat16* __restrict__ out, int splits) {
  pdl_launch_dependents();
  pdl_wait();
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
  cudaError_t e = launch_pdl(decode_attn_kernel, grid, dim3(128), sizeof(DecodeSmem), stream, a, dst, cl);
  if (e != cudaSuccess) return e;
  ++*launches;
  if (a.splits > 1) {
    e = launch_pdl(combine_kernel, dim3(a.B * 64), dim3(64), 0, stream, (const float*)a.part_o,
                   (const float2*)a.part_ml, a.o, a.splits, 128);
    ++*launches;
  }
  return e;
}

int latent_splits(int B, int L, int num_sms) {
  // one wave of CTAs: about one (sequence, split) per SM; the split partials
  // cost 128 KB per (sequence, split), so large batches use few splits
  int s = (num_sms + B / 2) / B;
  const int max_s = (L + 255) / 256;
  if (s > max_s) s = max_s;
  if (s < 1) s = 1;
  const int cl = chunk_len_for(L, s, kLatTile);
  return (L + cl - 1) / cl;
}

cudaError_t launch_latent_attention(const LatentAttnArgs& a, const DevStatusHost& st, cudaStream_t stream,
                                    int* launches) {
  CUtensorMap tq, tc, tr;
  if (!make_tmap_bf16_2d(&tq, a.qlat, (uint64_t)a.B * 64, 576, 576, 64, 64) ||
      !make_tmap_bf16_3d(&tc, a.ckv, 512, a.L, a.B, 1024, (uint64_t)a.cap * 1024, 64, 64) ||
      !make_tmap_bf16_3d(&tr, a.kpe, 64, a.L, a.B, 128, (uint64_t)a.cap * 128, 64, 64))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(latent_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kLatSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int cl = chunk_len_for(a.L, a.splits, kLatTile);
  DevStatus dst{st.word, st.wait_limit_ns};
  dim3 grid(a.splits, a.B);
  cudaError_t e = launch_pdl(latent_attn_tc, grid, dim3(192), kLatSmemBytes, stream, tq, tc, tr, a, dst, cl);
  if (e != cudaSuccess) return e;
  ++*launches;
  if (a.splits > 1) {
    e = launch_pdl(latent_combine_kernel, dim3(64, a.B), dim3(128), 0, stream, (const float*)a.part_o,
                   (const float2*)a.part_ml, a.olat, a.splits);
    ++*launches;
  }
  return e;
}

}  // namespace mla
