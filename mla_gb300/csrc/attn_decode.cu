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
  // keys of this sequence: L, or P_b + 1 with per-sequence lengths (a split
  // beyond them has no keys and leaves an empty partial: m = -inf, l = 0)
  const int Lb = a.lens_pos ? clamp_pos(a.lens_pos[b], a.L - 1) + 1 : a.L;
  const int key_begin = split * chunk_len;
  const int key_end = min(Lb, key_begin + chunk_len);
  const int nchunks = key_end > key_begin ? (key_end - key_begin + kDecChunk - 1) / kDecChunk : 0;

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
// Work: the B sequences' 64-key tiles, flattened in (sequence, tile) order,
// are cut into G contiguous, equal ranges, one per CTA (G = the SM count, or
// fewer for small problems).  A range covers the end of one sequence, whole
// sequences and the start of another; each piece ("segment") is attended
// with its own online softmax.  A segment that is a whole sequence writes
// o_lat directly; the pieces of a sequence cut between CTAs are written as
// unnormalised partials (two slots per CTA: its first and its last segment)
// and merged by latent_combine_kernel.
//
// CTA, 224 threads:
//   warp 0     TMA: q_lat [64 heads x 576] per segment; per tile the rotary
//              keys k^R_j [64 x 64] (one box) and the latent rows c_j
//              [64 x 512] (eight 64x64 boxes) into a 2-stage ring (3D tensor
//              maps bound positions to L, so rows >= L read as zeros)
//   warp 1     TMEM allocation; one lane issues S_j = q_lat . [k^R_j ; c_j]^T
//              (M=64 heads, N=64 keys, K=576), rotary box first: that box is
//              released as soon as its MMAs are done
//   warp 6     one lane issues O^T += c_j^T . P_j^T (M=128 latent rows in 4
//              blocks, N=64 heads, K=64 keys); its completion releases the
//              latent boxes and tells the softmax that P may be rewritten
//              (O is kept transposed so the 512-wide latent output takes 256
//              TMEM columns; c_j serves as the K-major B operand of S and the
//              MN-major A operand of O^T without a copy).  Two issuing
//              threads keep the tensor pipe fed while either one waits.
//   warps 2..5 softmax: head h = 16*(warp%4) + lane%16 (an M=64
//              accumulator row r lives in TMEM lane 32*(r/16) + r%16), lanes
//              i and i+16 each take 32 of the head's 64 keys (16x32bx2 loads);
//              lazy rescaling (O^T columns rescaled only when a head's max
//              grows by more than 2^8), P_j [64 heads x 64 keys] bf16 to shared
//              memory; at the end of a segment every thread writes the latent
//              rows it holds.
// ---------------------------------------------------------------------------
constexpr int kLatTile = 64;
constexpr uint32_t kLatBox = 64 * 128;                       // 64 rows x 64 bf16
constexpr uint32_t kLatQOff = 0;                             // 9 boxes
constexpr uint32_t kLatCOff = 9 * kLatBox;                   // 2 stages x 9 boxes (box 8 = rotary keys)
constexpr uint32_t kLatPOff = kLatCOff + 18 * kLatBox;       // 1 box
constexpr uint32_t kLatBarOff = kLatPOff + kLatBox;
constexpr uint32_t kLatSmemBytes = kLatBarOff + 1536 + 1024;
constexpr int kLatThreads = 224;

struct LatBars {
  uint64_t q_full, q_free;
  uint64_t kpe_full[2], kpe_empty[2], ckv_full[2], ckv_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, drain_s, drain_pv;
  uint32_t tmem_slot;
  int abort;
  int need[2][4];
  float alpha[2][64];
  float m[64], l[64];
};
static_assert(sizeof(LatBars) <= 1536, "barrier block");

// First flattened tile of CTA g's range (ranges are [start(g), start(g+1))).
__device__ __forceinline__ long long lat_range_start(int g, long long total, int G) {
  return (long long)g * total / G;
}

__device__ __forceinline__ void named_sync_128() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Walk over a CTA's range of (sequence, tile) work.  Every sequence has
// L = p_max + 1 keys, or P_b + 1 with per-sequence lengths (read when the
// walk enters the sequence).
struct SeqWalk {
  const int* pos;
  int p_max, B;
  int b, t, len, nt;  // current sequence, tile within it, its keys and tiles
  __device__ __forceinline__ void enter(int s) {
    b = s;
    len = !pos ? p_max + 1 : (s < B ? clamp_pos(pos[s], p_max) + 1 : 1);
    nt = (len + kLatTile - 1) / kLatTile;
  }
  __device__ __forceinline__ void start(int first_seq, int first_t) {
    enter(first_seq);
    t = first_t - 1;
  }
  __device__ __forceinline__ void next() {
    if (++t == nt) {
      t = 0;
      enter(b + 1);
    }
  }
};

// The work plan for per-sequence lengths (one CTA of 1024 threads):
// flattened tile offsets of the sequences, then each persistent CTA's first
// sequence, first tile and tile count (the same equal cut of the total as
// the uniform case).
__global__ void __launch_bounds__(1024) latent_plan_kernel(const int* __restrict__ pos, int B, int p_max, int G,
                                                           int* __restrict__ plan) {
  __shared__ int part[1024];
  pdl_launch_dependents();
  pdl_wait();
  const int tid = threadIdx.x;
  const int per = (B + 1023) / 1024;
  const int s0 = min(B, tid * per), s1 = min(B, s0 + per);
  int sum = 0;
  for (int s = s0; s < s1; ++s) sum += (clamp_pos(pos[s], p_max) + kLatTile) / kLatTile;
  part[tid] = sum;
  __syncthreads();
  // inclusive scan of the 1024 chunk sums (Hillis-Steele)
  for (int o = 1; o < 1024; o <<= 1) {
    const int v = tid >= o ? part[tid - o] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int off = part[tid] - sum;
  for (int s = s0; s < s1; ++s) {
    plan[s] = off;
    off += (clamp_pos(pos[s], p_max) + kLatTile) / kLatTile;
  }
  const long long total = part[1023];
  if (tid == 0) plan[B] = (int)total;
  __syncthreads();
  for (int g = tid; g < G; g += 1024) {
    const long long x0 = lat_range_start(g, total, G);
    const int R = (int)(lat_range_start(g + 1, total, G) - x0);
    int lo = 0, hi = B - 1;  // the last sequence whose first tile is <= x0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (plan[mid] <= x0) lo = mid; else hi = mid - 1;
    }
    int* r = plan + B + 1 + 3 * g;
    r[0] = lo;
    r[1] = (int)(x0 - plan[lo]);
    r[2] = R;
  }
}

__global__ void __launch_bounds__(kLatThreads, 1)
    latent_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmC,
                   const __grid_constant__ CUtensorMap tmR, const LatentAttnArgs a, const DevStatus st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  LatBars* bar = reinterpret_cast<LatBars*>(smem + kLatBarOff);
  volatile int* abort_flag = &bar->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nt = (a.L + kLatTile - 1) / kLatTile;  // tiles per sequence (uniform lengths)
  const int g = blockIdx.x;

  if (threadIdx.x == 0) {
    mbar_init(&bar->q_full, 1);
    mbar_init(&bar->q_free, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->kpe_full[i], 1);
      mbar_init(&bar->kpe_empty[i], 1);
      mbar_init(&bar->ckv_full[i], 1);
      mbar_init(&bar->ckv_empty[i], 1);
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->s_free[i], 128);
    }
    mbar_init(&bar->p_full, 128);
    mbar_init(&bar->drain_s, 1);
    mbar_init(&bar->drain_pv, 1);
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
  // this CTA's range of flattened (sequence, tile) work
  int R, first_seq, first_t;
  if (a.plan) {
    const int* r = a.plan + a.B + 1 + 3 * g;
    first_seq = r[0];
    first_t = r[1];
    R = r[2];
  } else {
    const long long total = (long long)a.B * nt;
    const long long x0 = lat_range_start(g, total, a.ctas);
    R = (int)(lat_range_start(g + 1, total, a.ctas) - x0);
    first_seq = (int)(x0 / nt);
    first_t = (int)(x0 - (long long)first_seq * nt);  // tile index of x0 within its sequence
  }
  SeqWalk walk{a.pos, a.L - 1, a.B, 0, 0, 0, 0};
  if (R > 0) walk.start(first_seq, first_t);

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmC);
      tma_prefetch_desc(&tmR);
      int seg = 0;
      int kpe_used[2] = {0, 0}, ckv_used[2] = {0, 0};  // loads issued per stage
      for (int i = 0; i < R; ++i) {
        walk.next();
        const int b = walk.b, t = walk.t;
        const int stg = i & 1;
        const uint32_t eph = ((i >> 1) & 1) ^ 1;
        const int k0 = t * kLatTile;
        const int plane = a.kv_div == 1 ? b : b / a.kv_div;  // the cache plane this sequence reads
        uint8_t* cbase = smem + kLatCOff + stg * 9 * kLatBox;
        // the rotary box first: it frees earliest and S starts with it
        if (!mbar_wait(&bar->kpe_empty[stg], eph, st, abort_flag, 61)) break;
        mbar_arrive_expect_tx(&bar->kpe_full[stg], kLatBox);
        tma_load_3d(cbase + 8 * kLatBox, &tmR, &bar->kpe_full[stg], 0, k0, plane);
        kpe_used[stg]++;
        if (!mbar_wait(&bar->ckv_empty[stg], eph, st, abort_flag, 62)) break;
        mbar_arrive_expect_tx(&bar->ckv_full[stg], 8 * kLatBox);
        for (int c = 0; c < 8; ++c) tma_load_3d(cbase + c * kLatBox, &tmC, &bar->ckv_full[stg], 64 * c, k0, plane);
        ckv_used[stg]++;
        if (i == 0 || t == 0) {
          // a new segment: reload q_lat once every S of the previous one is done
          if (seg > 0 && !mbar_wait(&bar->q_free, (seg - 1) & 1, st, abort_flag, 60)) break;
          mbar_arrive_expect_tx(&bar->q_full, 9 * kLatBox);
          for (int c = 0; c < 9; ++c) tma_load_2d(smem + kLatQOff + c * kLatBox, &tmQ, &bar->q_full, 64 * c, b * 64);
          ++seg;
        }
      }
      // never leave with copies in flight (matters only after a failed wait)
      if (seg > 0) mbar_wait(&bar->q_full, (seg - 1) & 1, st, nullptr, 64);
      for (int sg = 0; sg < 2; ++sg) {
        if (kpe_used[sg]) mbar_wait(&bar->kpe_full[sg], (kpe_used[sg] - 1) & 1, st, nullptr, 65);
        if (ckv_used[sg]) mbar_wait(&bar->ckv_full[sg], (ckv_used[sg] - 1) & 1, st, nullptr, 65);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // S issuer
      constexpr uint32_t idesc_s = idesc_bf16(64, 64, false, false);
      const uint32_t q_addr = smem_u32(smem + kLatQOff);
      const uint32_t c_addr = smem_u32(smem + kLatCOff);
      int seg = 0;
      for (int i = 0; i < R; ++i) {
        walk.next();
        const int t = walk.t;
        const bool seg_first = i == 0 || t == 0;
        const bool seg_last = i == R - 1 || t == walk.nt - 1;
        const int stg = i & 1;
        const uint32_t ph = (i >> 1) & 1;
        if (!mbar_wait(&bar->s_free[stg], ph ^ 1, st, abort_flag, 70)) break;
        if (seg_first && !mbar_wait(&bar->q_full, seg & 1, st, abort_flag, 71)) break;
        if (!mbar_wait(&bar->kpe_full[stg], ph, st, abort_flag, 72)) break;
        tc_fence_after();
        const uint32_t cb = c_addr + stg * 9 * kLatBox;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16(tmem + stg * 64, sdesc_sw128(q_addr + 8 * kLatBox + kk * 32, 16, 1024),
                    sdesc_sw128(cb + 8 * kLatBox + kk * 32, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
        umma_commit(&bar->kpe_empty[stg]);
        if (!mbar_wait(&bar->ckv_full[stg], ph, st, abort_flag, 73)) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 32; ++kk) {
          const uint32_t off = (kk >> 2) * kLatBox + (kk & 3) * 32;
          umma_bf16(tmem + stg * 64, sdesc_sw128(q_addr + off, 16, 1024), sdesc_sw128(cb + off, 16, 1024), idesc_s,
                    1u);
        }
        umma_commit(&bar->s_full[stg]);
        if (seg_last) {
          umma_commit(&bar->q_free);
          ++seg;
        }
      }
      umma_commit(&bar->drain_s);
      mbar_wait(&bar->drain_s, 0, st, nullptr, 66);
    }
  } else if (warp == 6) {
    if (lane == 0) {
      // P.V issuer
      constexpr uint32_t idesc_o = idesc_bf16(128, 64, true, false);
      const uint32_t c_addr = smem_u32(smem + kLatCOff);
      const uint32_t p_addr = smem_u32(smem + kLatPOff);
      for (int i = 0; i < R; ++i) {
        walk.next();
        const bool seg_first = i == 0 || walk.t == 0;
        const int stg = i & 1;
        if (!mbar_wait(&bar->p_full, i & 1, st, abort_flag, 74)) break;
        tc_fence_after();
        const uint32_t cb = c_addr + stg * 9 * kLatBox;
#pragma unroll
        for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t adesc = sdesc_sw128(cb + 2 * mb * kLatBox + kk * 2048, kLatBox, 1024);
            const uint64_t bdesc = sdesc_sw128(p_addr + kk * 32, 16, 1024);
            umma_bf16(tmem + 128 + mb * 64, adesc, bdesc, idesc_o, (!seg_first || kk > 0) ? 1u : 0u);
          }
        }
        umma_commit(&bar->ckv_empty[stg]);
      }
      umma_commit(&bar->drain_pv);
      mbar_wait(&bar->drain_pv, 0, st, nullptr, 66);
    }
  } else {
    const int quarter = warp & 3;
    const int tid = threadIdx.x - 64;
    // head h = 16 * quarter + lane % 16 (an M=64 accumulator row r lives in
    // TMEM lane 32*(r/16) + r%16); lanes i and i + 16 take keys 0..31 and
    // 32..63 of the head's 64 scores
    const int h = quarter * 16 + (lane & 15);
    const int kh = lane >> 4;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    uint8_t* pbuf = smem + kLatPOff;
    const float sl2 = a.scale * kLog2e;
    float m = -INFINITY, l = 0.f;  // l: this thread's half of the head's sum
    // Every softmax warp runs every iteration and reaches every named barrier
    // (bar.sync has no time limit); after a failed wait (ok == false) the
    // work of the remaining iterations is skipped, the barriers are not.
    bool ok = true;
    for (int i = 0; i < R; ++i) {
      walk.next();
      const int b = walk.b, t = walk.t;
      const int Lb = walk.len;
      const bool seg_first = i == 0 || t == 0;
      const bool seg_last = i == R - 1 || t == walk.nt - 1;
      const int stg = i & 1;
      if (seg_first) {
        m = -INFINITY;
        l = 0.f;
      }
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&bar->s_full[stg], (i >> 1) & 1, st, abort_flag, 67));
      uint32_t s[32];
      if (ok) {
        tc_fence_after();
        tmem_ld16x2_32<32>(tmem + lane_addr + stg * 64, s);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bar->s_free[stg]);
      } else {
#pragma unroll
        for (int c = 0; c < 32; ++c) s[c] = 0u;
      }
      const int k0 = t * kLatTile + kh * 32;  // first key of this thread's half
      if (k0 + 32 > Lb) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (k0 + c >= Lb) s[c] = __float_as_uint(-INFINITY);
      }
      float mx;
      {
        // three-input maxima and two-lane float32 FMA / add (as the prefill
        // softmax): fewer instructions on the per-tile chain
        float mp[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) mp[c] = fmaxf(__uint_as_float(s[c]), __uint_as_float(s[c + 8]));
#pragma unroll
        for (int c = 0; c < 8; ++c) mp[c] = fmax3(mp[c], __uint_as_float(s[16 + c]), __uint_as_float(s[24 + c]));
        mx = fmaxf(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], fmax3(mp[5], mp[6], mp[7])));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));  // the head's other half
      }
      mx *= sl2;  // log2 units (the scale is positive)
      const bool need = mx > m + kRescaleThresholdLatent;
      const float m_new = need ? mx : m;
      const float alpha = need ? ex2_approx(m - m_new) : 1.f;
      float sp[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float x0, x1;
        fma_x2(x0, x1, __uint_as_float(s[c]), __uint_as_float(s[c + 1]), sl2, sl2, -m_new, -m_new);
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        s[c] = __float_as_uint(p0);
        s[c + 1] = __float_as_uint(p1);
        add_x2(sp[c & 3], sp[(c & 3) + 1], sp[c & 3], sp[(c & 3) + 1], p0, p1);
      }
      l = l * alpha + ((sp[0] + sp[1]) + (sp[2] + sp[3]));
      m = m_new;
      if (kh == 0) bar->alpha[stg][h] = alpha;
      const bool warp_need = __any_sync(0xffffffffu, need);
      if (lane == 0) bar->need[stg][quarter] = warp_need ? 1 : 0;
      named_sync_128();
      // O^T is rescaled only between two P.V of the same segment
      const bool any_need =
          !seg_first && (bar->need[stg][0] | bar->need[stg][1] | bar->need[stg][2] | bar->need[stg][3]);
      // P.V of the previous tile must be done: it reads the P buffer and writes O^T
      if (i > 0)
        ok = ok && __all_sync(0xffffffffu,
                              mbar_wait(&bar->ckv_empty[(i - 1) & 1], ((i - 1) >> 1) & 1, st, abort_flag, 68));
      if (ok && any_need) {
        tc_fence_after();
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            const uint32_t ta = tmem + lane_addr + 128 + mb * 64 + half * 32;
            tmem_ld32(ta, r);
            tmem_wait_ld();
#pragma unroll
            for (int c = 0; c < 32; ++c)
              r[c] = __float_as_uint(__uint_as_float(r[c]) * bar->alpha[stg][half * 32 + c]);
            tmem_st32(ta, r);
          }
        }
        tmem_wait_st();
      }
      if (ok) {
        // this thread's 32 keys of row h: 16-byte chunks kh*4 .. kh*4+3 (128-byte swizzle)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int k = j * 8;
          const uint4 v = make_uint4(pack_bf16x2(__uint_as_float(s[k]), __uint_as_float(s[k + 1])),
                                     pack_bf16x2(__uint_as_float(s[k + 2]), __uint_as_float(s[k + 3])),
                                     pack_bf16x2(__uint_as_float(s[k + 4]), __uint_as_float(s[k + 5])),
                                     pack_bf16x2(__uint_as_float(s[k + 6]), __uint_as_float(s[k + 7])));
          *reinterpret_cast<uint4*>(pbuf + h * 128 + (((kh * 4 + j) ^ (h & 7)) << 4)) = v;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bar->p_full);
      if (!seg_last) continue;

      // end of a segment: O^T complete after this tile's P.V
      ok = ok && __all_sync(0xffffffffu, mbar_wait(&bar->ckv_empty[stg], (i >> 1) & 1, st, abort_flag, 69));
      const float l_head = l + __shfl_xor_sync(0xffffffffu, l, 16);
      if (kh == 0) {
        bar->m[h] = m;
        bar->l[h] = l_head;
      }
      named_sync_128();
      const bool whole = t == walk.nt - 1 && i >= t;  // the sequence's tile 0 is in this CTA too
      const int slot = (b == first_seq) ? 2 * g : 2 * g + 1;
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int mb = 0; mb < 4; ++mb) {
          const int latent = mb * 128 + quarter * 32 + lane;
#pragma unroll 1
          for (int half = 0; half < 2; ++half) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_addr + 128 + mb * 64 + half * 32, r);
            tmem_wait_ld();
            if (whole) {
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const int hh = half * 32 + c;
                a.olat[((size_t)b * 64 + hh) * 512 + latent] =
                    __float2bfloat16_rn(__uint_as_float(r[c]) / bar->l[hh]);
              }
            } else {
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const int hh = half * 32 + c;
                a.part_o[((size_t)slot * 64 + hh) * 512 + latent] = __uint_as_float(r[c]);
              }
            }
          }
        }
        if (!whole && tid < 64) a.part_ml[(size_t)slot * 64 + tid] = make_float2(bar->m[tid], bar->l[tid]);
      }
      tc_fence_before();
      named_sync_128();  // m/l are rewritten by the next segment's end
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Merge the partials of the sequences cut between CTAs (the others were
// written by latent_attn_tc directly).  Block = (group of 8 heads, sequence),
// one warp per head, 16 latent columns per lane.  The pieces are taken four
// at a time: their (m, l) pairs and partial rows are all requested before
// any is used (one memory round trip per group of four), then folded into
// a running maximum, denominator and sum.
constexpr int kLatMaxCtas = 1024;
constexpr int kCombineHeads = 8;

__global__ void __launch_bounds__(32 * kCombineHeads) latent_combine_kernel(const float* __restrict__ part_o,
                                                                             const float2* __restrict__ part_ml,
                                                                             __nv_bfloat16* __restrict__ out, int L,
                                                                             int B, int G,
                                                                             const int* __restrict__ plan) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x * kCombineHeads + (threadIdx.x >> 5), b = blockIdx.y;
  const int nt = (L + kLatTile - 1) / kLatTile;
  // the sequence's first and last flattened tile (per-sequence lengths: from the plan)
  const long long total = plan ? (long long)plan[B] : (long long)B * nt;
  const long long xa = plan ? (long long)plan[b] : (long long)b * nt;
  const long long xb = plan ? (long long)plan[b + 1] - 1 : xa + nt - 1;
  // CTA holding flattened tile x: the largest g with start(g) <= x
  const int g0 = (int)(((xa + 1) * G - 1) / total);
  const int g1 = (int)(((xb + 1) * G - 1) / total);
  if (g0 == g1) return;  // whole sequence in one CTA: written directly
  const int n = g1 - g0 + 1;
  float m_run = -INFINITY, l_run = 0.f;
  float4 acc[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) acc[j] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < n; k0 += 4) {
    float2 ml[4];
    float4 v[4][4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const int gg = g0 + k0 + kk;
      int slot = -1;
      if (k0 + kk < n && !(plan && plan[B + 1 + 3 * gg + 2] == 0)) {  // a CTA with no tiles wrote nothing
        const int gseq = plan ? plan[B + 1 + 3 * gg] : (int)(lat_range_start(gg, total, G) / nt);
        slot = (b == gseq) ? 2 * gg : 2 * gg + 1;
      }
      if (slot >= 0) {
        ml[kk] = part_ml[(size_t)slot * 64 + h];
        const float* row = part_o + ((size_t)slot * 64 + h) * 512;
#pragma unroll
        for (int j = 0; j < 4; ++j) v[kk][j] = *reinterpret_cast<const float4*>(row + j * 128 + lane * 4);
      } else {
        ml[kk] = make_float2(-INFINITY, 0.f);
#pragma unroll
        for (int j = 0; j < 4; ++j) v[kk][j] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float m_new = m_run;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) m_new = fmaxf(m_new, ml[kk].x);
    // the first piece of a sequence always holds keys, so m_new is finite
    const float sc = exp2f(m_run - m_new);
    l_run *= sc;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[j].x *= sc;
      acc[j].y *= sc;
      acc[j].z *= sc;
      acc[j].w *= sc;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float w = exp2f(ml[kk].x - m_new);
      l_run = fmaf(w, ml[kk].y, l_run);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        acc[j].x = fmaf(w, v[kk][j].x, acc[j].x);
        acc[j].y = fmaf(w, v[kk][j].y, acc[j].y);
        acc[j].z = fmaf(w, v[kk][j].z, acc[j].z);
        acc[j].w = fmaf(w, v[kk][j].w, acc[j].w);
      }
    }
    m_run = m_new;
  }
  const float inv = 1.f / l_run;
  __nv_bfloat16* o = out + ((size_t)b * 64 + h) * 512;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint2 w;
    w.x = pack_bf16x2(acc[j].x * inv, acc[j].y * inv);
    w.y = pack_bf16x2(acc[j].z * inv, acc[j].w * inv);
    *reinterpret_cast<uint2*>(o + j * 128 + lane * 4) = w;
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

int latent_ctas(int B, int L, int num_sms) {
  // one CTA per SM (persistent over its range of tiles), at least two tiles each
  const long long total = (long long)B * ((L + kLatTile - 1) / kLatTile);
  long long g = total / 2;
  if (g > num_sms) g = num_sms;
  if (g > kLatMaxCtas) g = kLatMaxCtas;  // bounds the partial slots and the plan
  if (g < 1) g = 1;
  return (int)g;
}

cudaError_t launch_latent_attention(const LatentAttnArgs& a, const DevStatusHost& st, cudaStream_t stream,
                                    int* launches) {
  CUtensorMap tq, tc, tr;
  if (a.kv_div < 1 || a.B % a.kv_div) return cudaErrorInvalidValue;
  const uint64_t planes = (uint64_t)(a.B / a.kv_div);
  if (!make_tmap_bf16_2d(&tq, a.qlat, (uint64_t)a.B * 64, 576, 576, 64, 64) ||
      !make_tmap_bf16_3d(&tc, a.ckv, 512, a.L, planes, 1024, (uint64_t)a.cap * 1024, 64, 64) ||
      !make_tmap_bf16_3d(&tr, a.kpe, 64, a.L, planes, 128, (uint64_t)a.cap * 128, 64, 64))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(latent_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kLatSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  DevStatus dst{st.word, st.wait_limit_ns};
  cudaError_t e;
  LatentAttnArgs la = a;
  if (a.pos) {
    if (!a.plan) return cudaErrorInvalidValue;
    e = launch_pdl(latent_plan_kernel, dim3(1), dim3(1024), 0, stream, a.pos, a.B, a.L - 1, a.ctas, a.plan);
    if (e != cudaSuccess) return e;
    ++*launches;
  } else {
    la.plan = nullptr;
  }
  e = launch_pdl(latent_attn_tc, dim3(a.ctas), dim3(kLatThreads), kLatSmemBytes, stream, tq, tc, tr, la, dst);
  if (e != cudaSuccess) return e;
  ++*launches;
  if (a.ctas > 1) {
    e = launch_pdl(latent_combine_kernel, dim3(64 / kCombineHeads, a.B), dim3(32 * kCombineHeads), 0, stream,
                   (const float*)a.part_o,
                   (const float2*)a.part_ml, a.olat, a.L, a.B, a.ctas, (const int*)la.plan);
    ++*launches;
  }
  return e;
}

}  // namespace mla
