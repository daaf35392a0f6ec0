// Persistent tcgen05 GEMM for the MLA projections, sm_103a.
//
// D[m, n] = sum_k A[m, k] B[n, k] with bf16 operands staged by TMA (128-byte
// swizzle) and an f32 accumulator in tensor memory; the epilogue reads the
// accumulator with tcgen05.ld and applies the step-specific output transform:
//   kStoreBf16  plain bf16 store (latent absorption)
//   kStoreF32   plain float32 store (A-projection: its columns are normalised
//               or rotated before they are rounded once to bf16)
//   kQRope      q_b_proj: RoPE on the 64 "pe" columns of each 192-column
//               head (dense-block page: Q^R_t = RoPE(Q^pe_t, R_t)); tiles of
//               half a head, a head, or 256 columns
//   kKVCache    kv_b_proj: one head (256 columns) per tile, writes k_nope and
//               v into the per-head caches and appends the shared rotary key
//               (dense-block page: K_i = [K^C_i ; k^R])
//   kResidual   o_proj: out = x + Delta_attn, one bf16 rounding
//
// Warp roles (192 threads): warp 0 issues TMA loads into a STAGES-deep ring,
// warp 1 allocates tensor memory and one lane issues the MMAs, warps 2..5 run
// the epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).  The accumulator is
// double buffered in TMEM so the epilogue of one tile overlaps the main loop
// of the next.  Every wait is bounded (see common.cuh).
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

#include <cudaTypedefs.h>

#include <mutex>

namespace mla {

namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;
constexpr int kBK = 64;

__host__ __device__ constexpr uint32_t pow2_cols(uint32_t n) {
  return n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : n <= 256 ? 256 : 512;
}

// One pipeline stage holds KSUB consecutive 64-wide K blocks of A and of B,
// so that each weight row is fetched in runs of KSUB * 128 bytes.
template <int BM, int BN, int STAGES, int KSUB, bool TMA_ST = false, bool PAIR = false>
struct GemmSmem {
  static constexpr uint32_t kA1 = BM * kBK * 2;  // one 64-wide K block of A
  static constexpr uint32_t kB1 = (PAIR ? BN / 2 : BN) * kBK * 2;  // CTA pair: half of the B rows each
  static constexpr uint32_t kA = KSUB * kA1;
  static constexpr uint32_t kB = KSUB * kB1;
  static constexpr uint32_t kStage = kA + kB;
  static constexpr uint32_t kStagingOff = STAGES * kStage;              // 4 warps x 2 x 4 KB
  static constexpr uint32_t kBarOff = kStagingOff + (TMA_ST ? 32768 : 0);
  static constexpr uint32_t kBytes = kBarOff + 256 + 1024;  // barriers + alignment slack
};

__device__ __forceinline__ void store32_bf16(__nv_bfloat16* dst, const uint32_t (&r)[32]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    d[j] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * j + 0]), __uint_as_float(r[8 * j + 1])),
                      pack_bf16x2(__uint_as_float(r[8 * j + 2]), __uint_as_float(r[8 * j + 3])),
                      pack_bf16x2(__uint_as_float(r[8 * j + 4]), __uint_as_float(r[8 * j + 5])),
                      pack_bf16x2(__uint_as_float(r[8 * j + 6]), __uint_as_float(r[8 * j + 7])));
  }
}

// h = SiLU(g) u = g u / (1 + e^-g) on 32 columns, in place in g (float32;
// e^-g = 2^(-g log2 e); for g far below zero the reciprocal of the infinite
// denominator is 0 and h = 0).
__device__ __forceinline__ void swiglu32(uint32_t (&g)[32], const uint32_t (&u)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float gv = __uint_as_float(g[i]);
    const float e = ex2_approx(-1.4426950408889634f * gv);
    g[i] = __float_as_uint(gv * __frcp_rn(1.f + e) * __uint_as_float(u[i]));
  }
}

// Accumulator sources for the epilogue: the tile in tensor memory, or (after
// a split-K reduction) the float32 partial slots in global memory.
struct TmemSrc {
  uint32_t taddr;
  __device__ __forceinline__ void operator()(int c, uint32_t (&r)[32]) const {
    tmem_ld32(taddr + c, r);
    tmem_wait_ld();
  }
};

// Split-K partial slots.  A slot holds one K slice's BM x BN fp32 tile,
// stored per warp quarter column by column: element (row r of quarter q,
// column c) at (q * BN + c) * (BM / 4) + r, so that the quarter's threads
// (one row each) write and read each column as one contiguous run.
template <int BM, int BN>
__device__ __forceinline__ float* part_slot(float* part, int slot, int quarter, int lq) {
  return part + (size_t)slot * BM * BN + (size_t)quarter * BN * (BM / 4) + lq;
}

template <int RPQ>
struct PartSrc {
  const float* base;    // this thread's element of column 0 in slot 0
  size_t slot_stride;   // floats between slots
  int slots;
  bool ok;
  __device__ __forceinline__ void operator()(int c, uint32_t (&r)[32]) const {
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.f;
    if (ok) {
      const float* p = base + (size_t)c * RPQ;
      int sl = 0;
      for (; sl + 2 <= slots; sl += 2) {  // two slots (64 loads) in flight
        float v[64];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int j = 0; j < 32; ++j) v[32 * u + j] = __ldcg(p + (sl + u) * slot_stride + j * RPQ);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] += v[j] + v[32 + j];
      }
      for (; sl < slots; ++sl) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __ldcg(p + sl * slot_stride + j * RPQ);
#pragma unroll
        for (int j = 0; j < 32; ++j) acc[j] += v[j];
      }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(acc[i]);
  }
};

template <int BN, Epi EPI, class Src>
__device__ __forceinline__ void run_epilogue(const EpiArgs& ea, const Src& ld, int batch, int row, int n0,
                                             bool row_ok) {
  if constexpr (EPI == Epi::kStoreBf16) {
    __nv_bfloat16* dst = ea.out + (size_t)row * ea.ldo + ea.c_col0 + batch * ea.c_col_step + n0;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ld(c, r);
      if (row_ok) store32_bf16(dst + c, r);
    }
  } else if constexpr (EPI == Epi::kStoreF32) {
    float* dst = ea.out_f32 + (size_t)row * ea.ldo + n0;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ld(c, r);
      if (row_ok) {
        float4* d = reinterpret_cast<float4*>(dst + c);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          d[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]), __uint_as_float(r[4 * j + 2]),
                             __uint_as_float(r[4 * j + 3]));
      }
    }
  } else if constexpr (EPI == Epi::kQRope) {
    // 192-column heads [128 nope | 64 pe], RoPE pairs (128+i, 160+i); a
    // tile (half a head, a head, or 256 columns) never splits a pe block
    static_assert(BN == 192 || BN == 96 || BN == 256, "q_b epilogue tile width");
    const int o0 = n0 % 192;
    __nv_bfloat16* dst = ea.out + (size_t)row * ea.ldo + n0;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int o = (o0 + c) % 192;
      if (o < 128) {
        uint32_t r[32];
        ld(c, r);
        if (row_ok) store32_bf16(dst + c, r);
        continue;
      }
      // o == 128: the pe block of head (n0 + c) / 192
      uint32_t x1[32], x2[32];
      ld(c, x1);
      ld(c + 32, x2);
      if (row_ok) {
        const float2* cs = ea.cs + (size_t)(row % ea.t_mod) * 32;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float2 t = cs[i];
          float a = __uint_as_float(x1[i]), b = __uint_as_float(x2[i]);
          x1[i] = __float_as_uint(a * t.x - b * t.y);
          x2[i] = __float_as_uint(b * t.x + a * t.y);
        }
        store32_bf16(dst + c, x1);
        store32_bf16(dst + c + 32, x2);
        if (ea.qpe_out) {  // latent decode: the rotated q^pe is also q_lat[row, head, 512:576]
          __nv_bfloat16* qd = ea.qpe_out + ((size_t)row * 64 + (n0 + c) / 192) * 576 + 512;
          store32_bf16(qd, x1);
          store32_bf16(qd + 32, x2);
        }
      }
      c += 32;
    }
  } else if constexpr (EPI == Epi::kKVCache) {
    // the tile covers columns o0 .. o0+BN-1 of one 256-wide head [128 k_nope | 128 v]
    static_assert(BN == 256 || BN == 128, "kv_b epilogue works on whole or half heads");
    const int h = n0 / 256;
    const int o0 = n0 % 256;
    const int b = row_ok ? row / ea.t_mod : 0;
    const int t = ea.pos ? (row_ok ? clamp_pos(ea.pos[b], ea.pos_max) : 0) : ea.t_off + (row_ok ? row % ea.t_mod : 0);
    const size_t slot = ((size_t)b * 64 + h) * ea.cap + t;
    __nv_bfloat16* krow = ea.kc + slot * 192;
    __nv_bfloat16* vrow = ea.vc + slot * 128;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ld(c, r);
      const int col = o0 + c;
      if (row_ok) store32_bf16(col < 128 ? krow + col : vrow + (col - 128), r);
    }
    if (row_ok && o0 == 0) {
      const uint4* src = reinterpret_cast<const uint4*>(ea.kpe + (size_t)row * 64);
      uint4* dst = reinterpret_cast<uint4*>(krow + 128);
#pragma unroll
      for (int j = 0; j < 8; ++j) dst[j] = src[j];
    }
  } else if constexpr (EPI == Epi::kSwiGLU) {
    // columns [0, BN/2) gate, [BN/2, BN) up, both of intermediate j0 + c
    __nv_bfloat16* dst = ea.out + (size_t)row * ea.ldo + n0 / 2;
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 32) {
      uint32_t g[32], u[32];
      ld(c, g);
      ld(BN / 2 + c, u);
      swiglu32(g, u);
      if (row_ok) store32_bf16(dst + c, g);
    }
  } else {  // kResidual
    const size_t base = (size_t)row * ea.ldo + n0;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      uint32_t r[32];
      ld(c, r);
      if (row_ok) {
        if (ea.delta) {
          float4* dd = reinterpret_cast<float4*>(ea.delta + base + c);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            dd[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
        }
        const uint4* xs = reinterpret_cast<const uint4*>(ea.x + base + c);
        uint32_t o[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          uint4 xv = xs[j];
          uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float2 xf = unpack_bf16x2(xw[q]);
            o[8 * j + 2 * q] = __float_as_uint(xf.x + __uint_as_float(r[8 * j + 2 * q]));
            o[8 * j + 2 * q + 1] = __float_as_uint(xf.y + __uint_as_float(r[8 * j + 2 * q + 1]));
          }
        }
        store32_bf16(ea.out + base + c, o);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Epilogue through shared memory and TMA stores (BM = 128, one tile per
// pass): each epilogue warp converts a 32-row x 32-column chunk into one of
// its two 4 KB staging buffers (swizzled so that the 32 row-writes of a
// chunk hit distinct banks) and one lane stores it with cp.async.bulk.tensor,
// so global writes leave the SM as whole rows.  Rows at or beyond the
// tensor's row extent are clipped by the TMA unit.
// ---------------------------------------------------------------------------
struct StoreStage {
  uint8_t* base;  // this warp's two buffers
  int n;          // chunks issued so far
  __device__ __forceinline__ uint8_t* next(int lane) {
    uint8_t* buf = base + (n & 1) * 4096;
    if (n >= 2) {
      if (lane == 0) bulk_wait_read<1>();
      __syncwarp();
    }
    return buf;
  }
  __device__ __forceinline__ void issue2(const CUtensorMap* m, uint8_t* buf, int c0, int c1, int lane) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(m, buf, c0, c1);
      bulk_commit();
    }
    ++n;
  }
  __device__ __forceinline__ void issue3(const CUtensorMap* m, uint8_t* buf, int c0, int c1, int c2, int lane) {
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(m, buf, c0, c1, c2);
      bulk_commit();
    }
    ++n;
  }
};

// row `lane` of a 32 x 32 bf16 chunk: 64 bytes, 64-byte swizzle
__device__ __forceinline__ void stage_bf16(uint8_t* buf, int lane, const uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int phys = c ^ ((lane >> 1) & 3);
    *reinterpret_cast<uint4*>(buf + lane * 64 + phys * 16) =
        make_uint4(pack_bf16x2(__uint_as_float(r[8 * c + 0]), __uint_as_float(r[8 * c + 1])),
                   pack_bf16x2(__uint_as_float(r[8 * c + 2]), __uint_as_float(r[8 * c + 3])),
                   pack_bf16x2(__uint_as_float(r[8 * c + 4]), __uint_as_float(r[8 * c + 5])),
                   pack_bf16x2(__uint_as_float(r[8 * c + 6]), __uint_as_float(r[8 * c + 7])));
  }
}

// row `lane` of a 32 x 64 bf16 chunk (columns 0-31 from a, 32-63 from b):
// 128 bytes, 128-byte swizzle
__device__ __forceinline__ void stage_bf16_64(uint8_t* buf, int lane, const uint32_t (&a)[32],
                                              const uint32_t (&b)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t* r = c < 4 ? &a[8 * c] : &b[8 * (c - 4)];
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((c ^ (lane & 7)) * 16)) =
        make_uint4(pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1])),
                   pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3])),
                   pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5])),
                   pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7])));
  }
}

// row `lane` of a 32 x 64 bf16 chunk from 8 packed uint4 (already bf16)
__device__ __forceinline__ void stage_bf16_raw_64(uint8_t* buf, int lane, const uint4 (&v)[8]) {
#pragma unroll
  for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(buf + lane * 128 + ((c ^ (lane & 7)) * 16)) = v[c];
}

// row `lane` of a 32 x 32 bf16 chunk from 4 packed uint4 (already bf16)
__device__ __forceinline__ void stage_bf16_raw(uint8_t* buf, int lane, const uint4 (&v)[4]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) *reinterpret_cast<uint4*>(buf + lane * 64 + ((c ^ ((lane >> 1) & 3)) * 16)) = v[c];
}

// row `lane` of a 32 x 32 float32 chunk: 128 bytes, 128-byte swizzle
__device__ __forceinline__ void stage_f32(uint8_t* buf, int lane, const uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((c ^ (lane & 7)) * 16)) =
        make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]);
}

template <int BN, Epi EPI>
__device__ __forceinline__ void run_epilogue_tma(const EpiArgs& ea, const TmemSrc& src, StoreStage& ss,
                                                 const CUtensorMap* m0, const CUtensorMap* m1, int batch,
                                                 int row0, int row, int n0, bool row_ok, int lane, int M) {
  const uint32_t taddr = src.taddr;
  if constexpr (EPI == Epi::kStoreF32) {
    tmem_chunk_loop(taddr, 0, BN, [&](int c, uint32_t (&r)[32]) {
      uint8_t* buf = ss.next(lane);
      stage_f32(buf, lane, r);
      ss.issue2(m0, buf, n0 + c, row0, lane);
    });
  } else if constexpr (EPI == Epi::kStoreBf16) {
    const int col0 = ea.c_col0 + batch * ea.c_col_step + n0;
    tmem_chunk_loop(taddr, 0, BN, [&](int c, uint32_t (&r)[32]) {
      uint8_t* buf = ss.next(lane);
      stage_bf16(buf, lane, r);
      ss.issue2(m0, buf, col0 + c, row0, lane);
    });
  } else if constexpr (EPI == Epi::kQRope) {
    // Heads are 192 columns: 128 "nope" then the 64 "pe" columns RoPE
    // rotates in pairs (i, i + 32).  A tile is a half head, a head, or 256
    // columns; a pe block never straddles a 256-column boundary
    // (256 k - 192 h never lies strictly between 128 and 192).
    static_assert(BN == 192 || BN == 96 || BN == 256, "q_b epilogue tile width");
    const int o0 = n0 % 192;
    // the RoPE table row of this token, fetched while the "nope" chunks are stored
    float2 cs[32];
    const bool has_pe = (128 - o0 + 192) % 192 < BN;
    if (has_pe) {
      const float4* csr = reinterpret_cast<const float4*>(ea.cs + (size_t)(row % ea.t_mod) * 32);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float4 v = csr[i];
        cs[2 * i] = make_float2(v.x, v.y);
        cs[2 * i + 1] = make_float2(v.z, v.w);
      }
    }
    int c = 0;
#pragma unroll 1
    while (c < BN) {
      const int o = (o0 + c) % 192;
      if (o < 128) {  // a run of nope columns
        const int run = (128 - o) < (BN - c) ? (128 - o) : (BN - c);
        tmem_chunk_loop(taddr, c, c + run, [&](int cc, uint32_t (&r)[32]) {
          uint8_t* buf = ss.next(lane);
          stage_bf16(buf, lane, r);
          ss.issue2(m0, buf, n0 + cc, row0, lane);
        });
        c += run;
        continue;
      }
      // o == 128: a whole pe block
      uint32_t x1[32], x2[32];
      tmem_ld32(taddr + c, x1);
      tmem_ld32(taddr + c + 32, x2);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float2 t = cs[i];
        const float a = __uint_as_float(x1[i]), b = __uint_as_float(x2[i]);
        x1[i] = __float_as_uint(a * t.x - b * t.y);
        x2[i] = __float_as_uint(b * t.x + a * t.y);
      }
      uint8_t* buf = ss.next(lane);
      stage_bf16(buf, lane, x1);
      ss.issue2(m0, buf, n0 + c, row0, lane);
      buf = ss.next(lane);
      stage_bf16(buf, lane, x2);
      ss.issue2(m0, buf, n0 + c + 32, row0, lane);
      c += 64;
    }
  } else if constexpr (EPI == Epi::kKVCache) {
    // the 32 rows of this warp are consecutive positions of one sequence
    // (the host uses this path only when t_mod is a multiple of 32)
    static_assert(BN == 256 || BN == 128, "kv_b epilogue works on whole or half heads");
    const int h = n0 / 256;
    const int o0 = n0 % 256;
    const bool warp_ok = row0 < M;
    const int b = row0 / ea.t_mod;
    const int t0 = ea.t_off + row0 % ea.t_mod;
    const int plane = b * 64 + h;
    // the shared rotary key of this row (K columns 128..191), loaded first so
    // that its latency overlaps the accumulator chunks
    uint4 kv4[8];
    if (o0 == 0) {
      const uint4* kp = reinterpret_cast<const uint4*>(ea.kpe + (size_t)row * 64);
#pragma unroll
      for (int j = 0; j < 8; ++j) kv4[j] = row_ok ? kp[j] : make_uint4(0, 0, 0, 0);
    }
    // 64-column chunks (32 rows x 128 bytes, the store maps' box): each row
    // piece is a whole 128-byte line of a K (384-byte) or V (256-byte) row
    if (warp_ok) {
#pragma unroll 1
      for (int c = 0; c < BN; c += 64) {
        uint32_t ra[32], rb[32];
        tmem_ld32(taddr + c, ra);
        tmem_ld32(taddr + c + 32, rb);
        tmem_wait_ld();
        const int col = o0 + c;
        uint8_t* buf = ss.next(lane);
        stage_bf16_64(buf, lane, ra, rb);
        if (col < 128)
          ss.issue3(m0, buf, col, t0, plane, lane);
        else
          ss.issue3(m1, buf, col - 128, t0, plane, lane);
      }
    }
    if (warp_ok && o0 == 0) {
      uint8_t* buf = ss.next(lane);
      stage_bf16_raw_64(buf, lane, kv4);
      ss.issue3(m0, buf, 128, t0, plane, lane);
    }
  } else if constexpr (EPI == Epi::kSwiGLU) {
#pragma unroll 1
    for (int c = 0; c < BN / 2; c += 32) {
      uint32_t g[32], u[32];
      tmem_ld32(taddr + c, g);
      tmem_ld32(taddr + BN / 2 + c, u);
      tmem_wait_ld();
      swiglu32(g, u);
      uint8_t* buf = ss.next(lane);
      stage_bf16(buf, lane, g);
      ss.issue2(m0, buf, n0 / 2 + c, row0, lane);
    }
  } else {  // kResidual
    const size_t base = (size_t)row * ea.ldo + n0;
    tmem_chunk_loop(taddr, 0, BN, [&](int c, uint32_t (&r)[32]) {
      if (row_ok && ea.delta) {
        float4* dd = reinterpret_cast<float4*>(ea.delta + base + c);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dd[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                              __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
      }
      if (row_ok) {
        const uint4* xs = reinterpret_cast<const uint4*>(ea.x + base + c);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 xv = xs[j];
          const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 xf = unpack_bf16x2(xw[q]);
            r[8 * j + 2 * q] = __float_as_uint(xf.x + __uint_as_float(r[8 * j + 2 * q]));
            r[8 * j + 2 * q + 1] = __float_as_uint(xf.y + __uint_as_float(r[8 * j + 2 * q + 1]));
          }
        }
      }
      uint8_t* buf = ss.next(lane);
      stage_bf16(buf, lane, r);
      ss.issue2(m0, buf, n0 + c, row0, lane);
    });
  }
}

// Tile index -> (batch, row block, column block).  Tiles walk groups of g row
// blocks; inside a group the row block changes fastest, so one wave of CTAs
// shares a few column blocks of B and a few row blocks of A (g = 1: column
// block fastest, every row block of A read once while all of B is reused).
__device__ __forceinline__ void tile_coords(int tile, int m_tiles, int n_tiles, int g, int& batch, int& m_blk,
                                            int& n_blk) {
  const int per_batch = m_tiles * n_tiles;
  batch = tile / per_batch;
  const int t = tile % per_batch;
  const int group_tiles = g * n_tiles;
  const int grp = t / group_tiles;
  const int gm = (m_tiles - grp * g) < g ? (m_tiles - grp * g) : g;  // rows in this (last) group
  const int r = t % group_tiles;
  m_blk = grp * g + r % gm;
  n_blk = r / gm;
}

// BM = 128: accumulator row r in TMEM lane r.  BM = 64 (few rows, decode):
// row r in lane 32*(r/16) + r%16, so each epilogue warp holds 16 rows.
template <int BM, int BN, int STAGES, int KSUB, Epi EPI, bool B_MN, bool TMA_ST, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
                const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO0,
                const __grid_constant__ CUtensorMap tmO1, const GemmShape s, const EpiArgs ea,
                const DevStatus st) {
  static_assert(!TMA_ST || BM == 128, "TMA-store epilogue needs 32 rows per warp");
  static_assert(!PAIR || (!B_MN && KSUB == 1 && BM == 128), "pair mode: K-major B, one K block per stage");
  using L = GemmSmem<BM, BN, STAGES, KSUB, TMA_ST, PAIR>;
  constexpr bool kSwi = EPI == Epi::kSwiGLU;  // B rows: gate half then up half of each tile
  static_assert(!kSwi || (!B_MN && BN % 64 == 0), "SwiGLU tiles: K-major B, 32-column halves");
  constexpr uint32_t kTmemCols = pow2_cols(2 * BN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* empty_bar = full_bar + STAGES;
  uint64_t* tfull_bar = empty_bar + STAGES;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tiles = (s.M + BM - 1) / BM;
  const int n_tiles = TMA_ST ? (s.N + BN - 1) / BN : s.N / BN;  // TMA stores clip columns >= N
  // Pair mode (cta_group::2): the two CTAs of a cluster compute one 256-row
  // tile, row blocks 2p (even CTA) and 2p + 1 (odd CTA) of one column block;
  // each stages its own 128 rows of A and half of the B rows, so every SM
  // reads half of B from shared memory per MMA.  The even CTA issues the
  // MMAs; both run the epilogue of their own rows (the host guarantees an
  // even m_tiles).
  const uint32_t crank = PAIR ? cluster_ctarank() : 0;
  const bool leader = crank == 0;
  const int m_units = PAIR ? m_tiles / 2 : m_tiles;
  const int num_tiles = s.batches * m_units * n_tiles;
  const int kblocks = s.K / (kBK * KSUB);  // stages of KSUB K blocks
  const int ksplit = s.ksplit;
  const int num_units = num_tiles * ksplit;
  const int unit0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int ustep = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      // pair: one cluster-scope arrival per epilogue warp of both CTAs (in
      // place of one per thread); single CTA: every epilogue thread
      mbar_init(&tempty_bar[i], PAIR ? 8 : 128);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    if (s.n_split < s.N) tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();
  // The producer waits for the preceding kernel itself, after it has issued
  // the weight (B) half of its first stages: the weights are read-only for
  // the whole step, so their first loads overlap the preceding kernel's tail.
  if (warp != 0) pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued[STAGES];
#pragma unroll
      for (int i = 0; i < STAGES; ++i) issued[i] = 0;
      bool ok = true;
      int pre = 0;  // stages of the first unit whose B half is already in flight
      if constexpr (!PAIR) {
        if (unit0 < num_units) {
          const int tile = unit0 / ksplit;
          const int kb0 = (unit0 % ksplit) * s.kb_per;
          const int kb1 = min(kblocks, kb0 + s.kb_per);
          int batch, m_blk, n_blk;
          tile_coords(tile, m_units, n_tiles, s.raster_g, batch, m_blk, n_blk);
          const int n0 = n_blk * BN;
          const int b_row = s.b_row0 + batch * s.b_row_step;
          const CUtensorMap* mb = (n0 < s.n_split) ? &tmB0 : &tmB1;
          const int nb = (n0 < s.n_split) ? n0 : n0 - s.n_split;
          pre = min(STAGES, kb1 - kb0);
          for (int i = 0; i < pre; ++i) {  // fresh ring: every stage is free
            uint8_t* sb = smem + i * L::kStage + L::kA;
            mbar_arrive_expect_tx(&full_bar[i], L::kStage);
            issued[i] = 1;  // counted now: the exit wait covers these copies even after an abort
#pragma unroll
            for (int u = 0; u < KSUB; ++u) {
              const int k0 = ((kb0 + i) * KSUB + u) * kBK;
              if constexpr (kSwi) {
                tma_load_2d(sb + u * L::kB1, &tmB0, &full_bar[i], k0, b_row + n0 / 2);
                tma_load_2d(sb + u * L::kB1 + (BN / 2) * 128, &tmB1, &full_bar[i], k0, b_row + n0 / 2);
              } else if constexpr (B_MN) {
#pragma unroll
                for (int j = 0; j < BN / 64; ++j)
                  tma_load_2d(sb + u * L::kB1 + j * (64 * 128), mb, &full_bar[i], nb + j * 64, b_row + k0);
              } else {
                tma_load_2d(sb + u * L::kB1, mb, &full_bar[i], k0, b_row + nb);
              }
            }
          }
        }
      }
      pdl_wait();
      for (int unit = unit0; unit < num_units && ok; unit += ustep) {
        const int tile = unit / ksplit;
        const int kb0 = (unit % ksplit) * s.kb_per;
        const int kb1 = min(kblocks, kb0 + s.kb_per);
        int batch, m_blk, n_blk;
        tile_coords(tile, m_units, n_tiles, s.raster_g, batch, m_blk, n_blk);
        if (PAIR) m_blk = 2 * m_blk + (int)crank;
        const int n0 = n_blk * BN;
        const int a_col = s.a_col0 + batch * s.a_col_step;
        const int b_row = s.b_row0 + batch * s.b_row_step;
        const CUtensorMap* mb = (n0 < s.n_split) ? &tmB0 : &tmB1;
        const int nb = (n0 < s.n_split) ? n0 : n0 - s.n_split;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_t<PAIR>(&empty_bar[stage], phase ^ 1, st, abort_flag, 1)) {
            ok = false;
            break;
          }
          uint8_t* sa = smem + stage * L::kStage;
          uint8_t* sb = sa + L::kA;
          if constexpr (PAIR) {
            // both CTAs' halves complete on the even CTA's barrier
            if (leader) mbar_arrive_expect_tx(&full_bar[stage], 2 * L::kStage);
            const uint32_t fb = mapa_rank(smem_u32(&full_bar[stage]), 0);
            const int k0 = kb * kBK;
            tma_load_2d_pair(sa, &tmA, fb, a_col + k0, m_blk * BM);
            if constexpr (kSwi)  // even CTA: gate rows, odd CTA: up rows of the same j
              tma_load_2d_pair(sb, crank ? &tmB1 : &tmB0, fb, k0, b_row + n0 / 2);
            else
              tma_load_2d_pair(sb, mb, fb, k0, b_row + nb + (int)crank * (BN / 2));
            issued[stage]++;
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1;
            }
            continue;
          }
          const bool b_done = unit == unit0 && kb - kb0 < pre;  // B half issued before the wait
          if (!b_done) mbar_arrive_expect_tx(&full_bar[stage], L::kStage);
#pragma unroll
          for (int u = 0; u < KSUB; ++u) {
            const int k0 = (kb * KSUB + u) * kBK;
            tma_load_2d(sa + u * L::kA1, &tmA, &full_bar[stage], a_col + k0, m_blk * BM);
            if (b_done) continue;
            if constexpr (kSwi) {
              tma_load_2d(sb + u * L::kB1, &tmB0, &full_bar[stage], k0, b_row + n0 / 2);
              tma_load_2d(sb + u * L::kB1 + (BN / 2) * 128, &tmB1, &full_bar[stage], k0, b_row + n0 / 2);
            } else if constexpr (B_MN) {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j)
                tma_load_2d(sb + u * L::kB1 + j * (64 * 128), mb, &full_bar[stage], nb + j * 64, b_row + k0);
            } else {
              tma_load_2d(sb + u * L::kB1, mb, &full_bar[stage], k0, b_row + nb);
            }
          }
          if (!b_done) issued[stage]++;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // make sure no copy into this CTA's shared memory is still in flight
      // (pair mode: the odd CTA's copies complete on the even CTA's barriers;
      // it waits until the MMAs released its last use of every stage)
#pragma unroll
      for (int i = 0; i < STAGES; ++i) {
        if (!issued[i]) continue;
        if (!PAIR || leader)
          mbar_wait_t<PAIR>(&full_bar[i], (issued[i] - 1) & 1, st, nullptr, 2);
        else
          mbar_wait_t<PAIR>(&empty_bar[i], (issued[i] - 1) & 1, st, nullptr, 2);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && (!PAIR || leader)) {
      // ---------------- MMA issuer (pair mode: the even CTA) ----------------
      constexpr uint32_t idesc = idesc_bf16(PAIR ? 2 * BM : BM, BN, false, B_MN);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int unit = unit0; unit < num_units && ok; unit += ustep) {
        const int kb0 = (unit % ksplit) * s.kb_per;
        const int kb1 = min(kblocks, kb0 + s.kb_per);
        if (!mbar_wait_t<PAIR>(&tempty_bar[acc], acc_phase ^ 1, st, abort_flag, 3)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_t<PAIR>(&full_bar[stage], phase, st, abort_flag, 4)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * L::kStage);
          const uint32_t b_base = a_base + L::kA;
#pragma unroll
          for (int u = 0; u < KSUB; ++u) {
            const uint32_t a_addr = a_base + u * L::kA1;
            const uint32_t b_addr = b_base + u * L::kB1;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint64_t adesc = sdesc_sw128(a_addr + k * 32, 16, 1024);
              uint64_t bdesc;
              if constexpr (B_MN)
                bdesc = sdesc_sw128(b_addr + k * 2048, 64 * 128, 1024);
              else
                bdesc = sdesc_sw128(b_addr + k * 32, 16, 1024);
              if constexpr (PAIR)
                umma_bf16_pair(d_tmem, adesc, bdesc, idesc, (kb != kb0 || u != 0 || k != 0) ? 1u : 0u);
              else
                umma_bf16(d_tmem, adesc, bdesc, idesc, (kb != kb0 || u != 0 || k != 0) ? 1u : 0u);
            }
          }
          if constexpr (PAIR)
            umma_commit_pair(&empty_bar[stage], (uint16_t)0x3);  // frees the stage in both CTAs
          else
            umma_commit(&empty_bar[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (PAIR)
          umma_commit_pair(&tfull_bar[acc], (uint16_t)0x3);
        else
          umma_commit(&tfull_bar[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // all MMAs issued by this thread have finished before TMEM is freed
      if constexpr (PAIR)
        umma_commit_pair(drain_bar, (uint16_t)0x1);
      else
        umma_commit(drain_bar);
      mbar_wait_t<PAIR>(drain_bar, 0, st, nullptr, 5);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;
    StoreStage ss{smem + L::kStagingOff + quarter * 8192, 0};
    const bool lane_ok = (BM == 128) || lane < 16;
    const int rit = (BM == 128) ? quarter * 32 + lane : quarter * 16 + (lane & 15);  // row within the tile
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int unit = unit0; unit < num_units; unit += ustep) {
      const int tile = unit / ksplit;
      const int ks = unit % ksplit;
      int batch, m_blk, n_blk;
      tile_coords(tile, m_units, n_tiles, s.raster_g, batch, m_blk, n_blk);
      if (PAIR) m_blk = 2 * m_blk + (int)crank;
      bool ok = mbar_wait_t<PAIR>(&tfull_bar[acc], acc_phase, st, abort_flag, 6);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int row = m_blk * BM + rit;
      const bool row_ok = lane_ok && row < s.M;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (ksplit == 1) {
        if constexpr (TMA_ST) {
          run_epilogue_tma<BN, EPI>(ea, TmemSrc{taddr}, ss, &tmO0, &tmO1, batch, m_blk * BM + quarter * 32, row,
                                    n_blk * BN, row_ok, lane, s.M);
        } else {
          run_epilogue<BN, EPI>(ea, TmemSrc{taddr}, batch, row, n_blk * BN, row_ok);
        }
        tc_fence_before();
        if constexpr (PAIR) {
          __syncwarp();  // the warp's accumulator reads are done
          if (lane == 0) mbar_arrive_cluster(mapa_rank(smem_u32(&tempty_bar[acc]), 0));  // the even CTA's barrier
        } else {
          mbar_arrive(&tempty_bar[acc]);
        }
      } else {
        // this K slice's partial -> its slot; the last warp of the quarter reduces
        const int lq = rit - quarter * (BM / 4);  // row within the quarter
        float* slot = part_slot<BM, BN>(ea.part, tile * ksplit + ks, quarter, lq);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + c, r);
          tmem_wait_ld();
          if (row_ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j) slot[(c + j) * (BM / 4)] = __uint_as_float(r[j]);
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty_bar[acc]);
        __threadfence();
        __syncwarp();
        int prev = 0;
        if (lane == 0) prev = atomicAdd(&ea.counters[tile * 4 + quarter], 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == ksplit - 1) {
          __threadfence();
          const PartSrc<BM / 4> src{part_slot<BM, BN>(ea.part, tile * ksplit, quarter, lq), (size_t)BM * BN, ksplit,
                                    row_ok};
          run_epilogue<BN, EPI>(ea, src, batch, row, n_blk * BN, row_ok);
          if (lane == 0) ea.counters[tile * 4 + quarter] = 0;  // ready for the next GEMM
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if constexpr (TMA_ST) {
      if (lane == 0) bulk_wait_all();
      __syncwarp();
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) {
    // every MMA of the pair has finished (the even CTA drained them) and no
    // remote arrive or copy is still in flight before the collective free
    cluster_sync();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc_pair(tmem_base, kTmemCols);
    }
  } else {
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tmem_base, kTmemCols);
    }
  }
}

template <int BM, int BN, int STAGES, Epi EPI, bool B_MN, int KSUB = 1, bool TMA_ST = false, bool PAIR = false>
cudaError_t launch_impl(const GemmShape& s, const GemmOperands& op, const EpiArgs& ea, const DevStatusHost& st,
                        int num_sms, cudaStream_t stream) {
  using L = GemmSmem<BM, BN, STAGES, KSUB, TMA_ST, PAIR>;
  if (s.K % (kBK * KSUB)) return cudaErrorInvalidValue;
  static_assert(L::kBytes <= 232448, "shared memory budget");
  CUtensorMap ta, tb0, tb1;
  if (!make_tmap_bf16_2d(&ta, op.A, op.a_rows, (uint64_t)op.lda, op.lda, BM, kBK))
    return cudaErrorInvalidValue;
  if (B_MN) {
    if (!make_tmap_bf16_2d(&tb0, op.B0, op.b0_rows, op.ldb0, op.ldb0, 64, 64)) return cudaErrorInvalidValue;
  } else {
    // pair mode: each CTA loads half the rows; SwiGLU: half the rows from each matrix
    constexpr uint32_t box_rows = (PAIR || EPI == Epi::kSwiGLU) ? BN / 2 : BN;
    if (!make_tmap_bf16_2d(&tb0, op.B0, op.b0_rows, op.ldb0, op.ldb0, box_rows, kBK)) return cudaErrorInvalidValue;
  }
  tb1 = tb0;
  if (op.B1 && !make_tmap_bf16_2d(&tb1, op.B1, op.b1_rows, op.ldb1, op.ldb1,
                                  (PAIR || EPI == Epi::kSwiGLU) ? BN / 2 : BN, kBK))
    return cudaErrorInvalidValue;
  CUtensorMap to0 = ta, to1 = ta;
  if constexpr (TMA_ST) {
    bool ok = true;
    if constexpr (EPI == Epi::kStoreF32) {
      ok = make_tmap_store_f32_2d(&to0, ea.out_f32, s.M, ea.ldo, ea.ldo);
    } else if constexpr (EPI == Epi::kKVCache) {
      ok = make_tmap_store_bf16_3d(&to0, ea.kc, 192, ea.cap, (uint64_t)ea.B * 64, 384, (uint64_t)ea.cap * 384) &&
           make_tmap_store_bf16_3d(&to1, ea.vc, 128, ea.cap, (uint64_t)ea.B * 64, 256, (uint64_t)ea.cap * 256);
    } else {
      ok = make_tmap_store_bf16_2d(&to0, ea.out, s.M, ea.ldo, ea.ldo);
    }
    if (!ok) return cudaErrorInvalidValue;
  }
  auto kern = gemm_kernel<BM, BN, STAGES, KSUB, EPI, B_MN, TMA_ST, PAIR>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;  // pair mode: clusters of 2 that fit at once
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
    if (attr_err == cudaSuccess && PAIR) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * num_sms);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = L::kBytes;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = 2;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
      if (attr_err == cudaSuccess && max_clusters < 1) attr_err = cudaErrorInvalidConfiguration;
    }
  });
  if (attr_err != cudaSuccess) return attr_err;
  GemmShape sh = s;
  if (sh.raster_g < 1) sh.raster_g = 1;
  const int m_tiles = (s.M + BM - 1) / BM;
  const int tiles = s.batches * m_tiles * (TMA_ST ? (s.N + BN - 1) / BN : s.N / BN);
  const int kblocks = s.K / (kBK * KSUB);
  sh.ksplit = 1;
  sh.kb_per = kblocks;
  if (!PAIR && ea.part && ea.counters && m_tiles == 1 && tiles * 2 <= num_sms && kblocks >= 2 &&
      tiles * 4 <= kMaxSplitCounters) {
    int ks = num_sms / tiles;
    if (ks > 4) ks = 4;  // the reduction reads every slice: keep it short
    if (ks > kMaxSplitUnits / tiles) ks = kMaxSplitUnits / tiles;
    if (ks > kblocks) ks = kblocks;
    const int kb_per = (kblocks + ks - 1) / ks;
    ks = (kblocks + kb_per - 1) / kb_per;
    const size_t need = (size_t)tiles * ks * BM * BN * sizeof(float);
    if (ks > 1 && need <= ea.part_bytes) {
      sh.ksplit = ks;
      sh.kb_per = kb_per;
    }
  }
  DevStatus dst{st.word, st.wait_limit_ns};
  if constexpr (PAIR) {
    if (m_tiles % 2 || sh.ksplit != 1) return cudaErrorInvalidValue;
    const int pairs = tiles / 2;
    const int clusters = pairs < max_clusters ? pairs : max_clusters;
    return launch_pdl_cluster2(kern, dim3(2 * clusters), dim3(kThreads), L::kBytes, stream, ta, tb0, tb1, to0, to1,
                               sh, ea, dst);
  } else {
    const int units = tiles * sh.ksplit;
    const int grid = units < num_sms ? units : num_sms;
    return launch_pdl(kern, dim3(grid), dim3(kThreads), L::kBytes, stream, ta, tb0, tb1, to0, to1, sh, ea, dst);
  }
}

// ---------------------------------------------------------------------------
// CTA-pair GEMM for a short K (at most kResKb 64-wide blocks) over many rows:
// the kv_b projection of a long prefill (K = 512).  Each CTA keeps its half
// of a 256-row B tile for the whole K resident in shared memory while the
// pair runs a group of row tiles against it, so per tile the SM receives only
// its 128 rows of A (128 KB at K = 512) and sends 64 KB of cache rows, where
// the streaming GEMM above also receives its 128 KB half of B again: the
// tensor-copy engine, which carries both directions, is what bounds this
// product (about 42 B per cycle per SM measured, against 64 that a 256-wide
// MMA stream asks for).  Warp roles as gemm_kernel (192 threads): warp 0
// copies B once per unit and A stage by stage, warp 1 (even CTA) issues the
// MMAs, warps 2..5 run the TMA-store epilogue of their CTA's 128 rows.
// ---------------------------------------------------------------------------
constexpr int kResKb = 8;
constexpr int kResStages = 4;

struct ResSmem {
  static constexpr uint32_t kBlk = 128 * kBK * 2;          // 128 rows x 64 bf16 (A stage, or a B block)
  static constexpr uint32_t kBOff = 0;                     // kResKb resident B blocks
  static constexpr uint32_t kAOff = kResKb * kBlk;         // kResStages A stages
  static constexpr uint32_t kStagingOff = kAOff + kResStages * kBlk;
  static constexpr uint32_t kBarOff = kStagingOff + 32768;
  static constexpr uint32_t kBytes = kBarOff + 256 + 1024;
};
static_assert(ResSmem::kBytes <= 232448, "shared memory budget");

// unit u of a resident-B GEMM: column block u % n_tiles, row-pair tiles
// [g * G, min((g + 1) * G, m_pairs)) with g = u / n_tiles (the pairs that run
// at once share one group of A rows in L2), walked from a tile that depends
// on the column block: pairs that all read the same A tile at the same time
// left each SM waiting for its A stages (about 16 B per cycle arrived)
template <Epi EPI>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_resb_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmO0, const __grid_constant__ CUtensorMap tmO1,
                          const GemmShape s, int group, const EpiArgs ea, const DevStatus st) {
  constexpr int BN = 256;
  using L = ResSmem;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* a_empty = a_full + kResStages;
  uint64_t* b_full = a_empty + kResStages;
  uint64_t* b_empty = b_full + 1;
  uint64_t* tfull_bar = b_empty + 1;
  uint64_t* tempty_bar = tfull_bar + 2;
  uint64_t* drain_bar = tempty_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const bool leader = crank == 0;
  const int m_pairs = (s.M + 255) / 256;
  const int n_tiles = s.N / BN;
  const int kb_n = s.K / kBK;  // <= kResKb (host-checked)
  const int groups = (m_pairs + group - 1) / group;
  const int num_units = groups * n_tiles;
  const int unit0 = (int)(blockIdx.x >> 1), ustep = (int)(gridDim.x >> 1);
  // the i-th row-pair tile of unit u
  auto unit_tile = [&](int u, int i) {
    const int p0 = (u / n_tiles) * group;
    const int cnt = min(group, m_pairs - p0);
    return p0 + (i + u % n_tiles) % cnt;
  };
  auto unit_count = [&](int u) { return min(group, m_pairs - (u / n_tiles) * group); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kResStages; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    mbar_init(b_full, 1);
    mbar_init(b_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 8);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any remote signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0, nb = 0;
      uint32_t phase = 0;
      int a_issued[kResStages] = {};
      bool ok = true;
      for (int unit = unit0; unit < num_units && ok; unit += ustep, ++nb) {
        const int n0 = (unit % n_tiles) * BN;
        const int cnt = unit_count(unit);
        // the previous unit's MMAs have read the resident B
        if (nb > 0 && !mbar_wait_t<true>(b_empty, (nb - 1) & 1, st, abort_flag, 91)) break;
        const uint32_t bfb = mapa_rank(smem_u32(b_full), 0);
        if (leader) mbar_arrive_expect_tx(b_full, 2 * kb_n * L::kBlk);
        for (int kb = 0; kb < kb_n; ++kb)
          tma_load_2d_pair(smem + L::kBOff + kb * L::kBlk, &tmB, bfb, kb * kBK, n0 + (int)crank * (BN / 2));
        for (int i = 0; i < cnt && ok; ++i) {
          const int m_blk = 2 * unit_tile(unit, i) + (int)crank;
          for (int kb = 0; kb < kb_n; ++kb) {
            if (!mbar_wait_t<true>(&a_empty[stage], phase ^ 1, st, abort_flag, 92)) {
              ok = false;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&a_full[stage], 2 * L::kBlk);
            tma_load_2d_pair(smem + L::kAOff + stage * L::kBlk, &tmA, mapa_rank(smem_u32(&a_full[stage]), 0),
                             kb * kBK, m_blk * 128);
            a_issued[stage]++;
            if (++stage == kResStages) {
              stage = 0;
              phase ^= 1;
            }
          }
        }
      }
      // no copy into this CTA's shared memory may still be in flight: the
      // even CTA sees them complete on its own barriers, the odd CTA waits
      // until the MMAs released every buffer it filled
      for (int i = 0; i < kResStages; ++i) {
        if (!a_issued[i]) continue;
        if (leader)
          mbar_wait_t<true>(&a_full[i], (a_issued[i] - 1) & 1, st, nullptr, 93);
        else
          mbar_wait_t<true>(&a_empty[i], (a_issued[i] - 1) & 1, st, nullptr, 93);
      }
      if (nb > 0) {
        if (leader)
          mbar_wait_t<true>(b_full, (nb - 1) & 1, st, nullptr, 93);
        else
          mbar_wait_t<true>(b_empty, (nb - 1) & 1, st, nullptr, 93);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (the even CTA) ----------------
      constexpr uint32_t idesc = idesc_bf16(256, BN, false, false);
      int stage = 0, nb = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int unit = unit0; unit < num_units && ok; unit += ustep, ++nb) {
        const int cnt = unit_count(unit);
        if (!mbar_wait_t<true>(b_full, nb & 1, st, abort_flag, 94)) break;
        for (int i = 0; i < cnt; ++i) {
          if (!mbar_wait_t<true>(&tempty_bar[acc], acc_phase ^ 1, st, abort_flag, 95)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          for (int kb = 0; kb < kb_n; ++kb) {
            if (!mbar_wait_t<true>(&a_full[stage], phase, st, abort_flag, 96)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(smem + L::kAOff + stage * L::kBlk);
            const uint32_t b_addr = smem_u32(smem + L::kBOff + kb * L::kBlk);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              umma_bf16_pair(d_tmem, sdesc_sw128(a_addr + k * 32, 16, 1024), sdesc_sw128(b_addr + k * 32, 16, 1024),
                             idesc, (kb != 0 || k != 0) ? 1u : 0u);
            umma_commit_pair(&a_empty[stage], (uint16_t)0x3);  // frees the A stage in both CTAs
            if (++stage == kResStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          umma_commit_pair(&tfull_bar[acc], (uint16_t)0x3);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        }
        if (!ok) break;
        umma_commit_pair(b_empty, (uint16_t)0x3);  // the resident B may be replaced
      }
      umma_commit_pair(drain_bar, (uint16_t)0x1);
      mbar_wait_t<true>(drain_bar, 0, st, nullptr, 97);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;
    StoreStage ss{smem + L::kStagingOff + quarter * 8192, 0};
    const int rit = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int unit = unit0; unit < num_units && ok; unit += ustep) {
      const int n0 = (unit % n_tiles) * BN;
      const int cnt = unit_count(unit);
      for (int i = 0; i < cnt; ++i) {
        const int m_blk = 2 * unit_tile(unit, i) + (int)crank;
        ok = __all_sync(0xffffffffu, mbar_wait_t<true>(&tfull_bar[acc], acc_phase, st, abort_flag, 98));
        if (!ok) break;
        tc_fence_after();
        const int row = m_blk * 128 + rit;
        const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
        run_epilogue_tma<BN, EPI>(ea, TmemSrc{taddr}, ss, &tmO0, &tmO1, 0, m_blk * 128 + quarter * 32, row, n0,
                                  row < s.M, lane, s.M);
        tc_fence_before();
        __syncwarp();  // the warp's accumulator reads are done
        if (lane == 0) mbar_arrive_cluster(mapa_rank(smem_u32(&tempty_bar[acc]), 0));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  // every MMA of the pair has finished (the even CTA drained them) and no
  // remote arrive or copy is still in flight before the collective free
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

template <Epi EPI>
cudaError_t launch_resb_pair(const GemmShape& s, const GemmOperands& op, const EpiArgs& ea, const DevStatusHost& st,
                             int num_sms, cudaStream_t stream) {
  constexpr int BN = 256;
  using L = ResSmem;
  if (s.K % kBK || s.K / kBK > kResKb || s.N % BN || s.M % 256 || s.batches != 1 || op.b_mn_major)
    return cudaErrorInvalidValue;
  CUtensorMap ta, tb, to0, to1;
  if (!make_tmap_bf16_2d(&ta, op.A, op.a_rows, (uint64_t)op.lda, op.lda, 128, kBK) ||
      !make_tmap_bf16_2d(&tb, op.B0, op.b0_rows, op.ldb0, op.ldb0, BN / 2, kBK))
    return cudaErrorInvalidValue;
  to1 = to0 = ta;
  bool ok = true;
  if constexpr (EPI == Epi::kKVCache) {
    ok = make_tmap_store_bf16_3d(&to0, ea.kc, 192, ea.cap, (uint64_t)ea.B * 64, 384, (uint64_t)ea.cap * 384) &&
         make_tmap_store_bf16_3d(&to1, ea.vc, 128, ea.cap, (uint64_t)ea.B * 64, 256, (uint64_t)ea.cap * 256);
  } else {
    ok = make_tmap_store_bf16_2d(&to0, ea.out, s.M, ea.ldo, ea.ldo);
  }
  if (!ok) return cudaErrorInvalidValue;
  auto kern = gemm_resb_pair_kernel<EPI>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
    if (attr_err != cudaSuccess) return;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kBytes;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    attr_err = cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg);
    if (attr_err == cudaSuccess && max_clusters < 1) attr_err = cudaErrorInvalidConfiguration;
  });
  if (attr_err != cudaSuccess) return attr_err;
  // row-pair groups: about six units per cluster, at least 4 tiles per unit
  const int m_pairs = s.M / 256, n_tiles = s.N / BN;
  int group = (m_pairs * n_tiles) / (6 * max_clusters);
  if (group < 4) group = 4;
  if (group > m_pairs) group = m_pairs;
  const int units = ((m_pairs + group - 1) / group) * n_tiles;
  const int clusters = units < max_clusters ? units : max_clusters;
  DevStatus dst{st.word, st.wait_limit_ns};
  return launch_pdl_cluster2(kern, dim3(2 * clusters), dim3(kThreads), L::kBytes, stream, ta, tb, to0, to1, s,
                             group, ea, dst);
}

// ---------------------------------------------------------------------------
// GEMM with FP8 block-scaled B (decode-size M).  480 threads:
//   warp 0      code producer: E4M3 tiles of B (BN rows x 128 bytes per
//               128-wide K stage; the codes are stored block-major, so a
//               tile's stage is one or two contiguous bulk copies) into a
//               deep SF-slot ring, from before the wait on the preceding
//               kernel (weights are read-only)
//   warp 14     A producer: two 64-wide bf16 TMA boxes per stage into an
//               SA-slot ring (its own thread, so an A load never waits
//               behind the issue of a code copy)
//   warp 1      TMEM allocation; one lane issues the bf16 MMAs
//   warps 2..5  epilogue (as gemm_kernel: register stores, split-K fixup)
//   warps 6..13 dequantization: each E4M3 tile -> bf16 (x its block scale)
//               in the 128-byte-swizzled K-major layout of a 2-slot ring
//               that the MMAs read; a unit's block scales are read once
//               into a shared-memory table
// ---------------------------------------------------------------------------
constexpr int kW8Threads = 480;
constexpr int kW8Deq = 256;    // dequantization threads (warps 6..13)
constexpr int kW8MaxKb = 64;   // 128-wide K stages per unit whose scales fit the table

template <int BM, int BN, int SA, int SF>
struct W8Smem {
  static constexpr uint32_t kA1 = BM * 64 * 2;  // one 64-wide bf16 block of A
  static constexpr uint32_t kA = 2 * kA1;       // an A stage (128 K)
  static constexpr uint32_t kF = BN * 128;      // an E4M3 B stage (128 K)
  static constexpr uint32_t kB1 = BN * 64 * 2;  // one 64-wide bf16 block of B
  static constexpr uint32_t kB = 2 * kB1;
  static constexpr uint32_t kFOff = SA * kA;
  static constexpr uint32_t kBOff = kFOff + SF * kF;
  static constexpr uint32_t kBarOff = kBOff + 2 * kB;
  static constexpr uint32_t kScOff = kBarOff + 512;  // [2 row blocks][kW8MaxKb] scales
  static constexpr uint32_t kBytes = kScOff + 2 * kW8MaxKb * 4 + 1024;
};

// The (unit, 128-wide K stage) sequence of one persistent CTA.  With one
// row block every CTA reads the same A panel: each column block starts at a
// different K stage (as in gemm_kernel) so the CTAs spread over L2.
struct W8Cursor {
  int unit, i, nk, kb0, rot;
  int ustep, num_units, ksplit, kb_per, kstages, m_tiles, n_tiles, raster_g;
  __device__ __forceinline__ void range() {
    if (unit < num_units) {
      kb0 = (unit % ksplit) * kb_per;
      nk = min(kstages, kb0 + kb_per) - kb0;
      i = 0;
      rot = 0;
      if (m_tiles == 1 && nk > 1) {
        int bt, mb_, nb_;
        tile_coords(unit / ksplit, m_tiles, n_tiles, raster_g, bt, mb_, nb_);
        rot = (nb_ * 7) % nk;
      }
    }
  }
  __device__ __forceinline__ bool valid() const { return unit < num_units; }
  __device__ __forceinline__ int kb() const { return kb0 + (i + rot) % nk; }
  __device__ __forceinline__ void next() {
    if (++i == nk) {
      unit += ustep;
      range();
    }
  }
};

// Four E4M3 codes (one 32-bit word, code 0 in the low byte) -> four bf16
// values times s (a power of two), exactly, with integer and fp32 multiply
// instructions only.  A code c = [sign | 4-bit exponent E | 3-bit mantissa m]
// placed as the bf16 bits (c & 0x80) << 8 | (c & 0x7F) << 4 is a bf16 of the
// same sign whose exponent field is E and mantissa m / 8: for E > 0 that is
// 2^(E-127) (1 + m/8) = value * 2^-120, for E = 0 the bf16 subnormal
// m 2^-129 = value * 2^-120 too.  Widened to fp32 (exact, a shift) and
// multiplied by 2^120 and then by s (both exact: powers of two, the
// results normal), the product's upper half is the bf16 result.
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, float s, uint32_t& lo, uint32_t& hi) {
  // codes 0,1 -> high bytes of two 16-bit halves; codes 2,3 likewise
  const uint32_t v01 = __byte_perm(w, 0u, 0x1404);
  const uint32_t v23 = __byte_perm(w, 0u, 0x3424);
  const uint32_t b01 = ((v01 >> 4) & 0x07F007F0u) | (v01 & 0x80008000u);  // value * 2^-120 as bf16x2
  const uint32_t b23 = ((v23 >> 4) & 0x07F007F0u) | (v23 & 0x80008000u);
  const float f0 = (__uint_as_float(b01 << 16) * 0x1p120f) * s;
  const float f1 = (__uint_as_float(b01 & 0xFFFF0000u) * 0x1p120f) * s;
  const float f2 = (__uint_as_float(b23 << 16) * 0x1p120f) * s;
  const float f3 = (__uint_as_float(b23 & 0xFFFF0000u) * 0x1p120f) * s;
  lo = __byte_perm(__float_as_uint(f0), __float_as_uint(f1), 0x7632);
  hi = __byte_perm(__float_as_uint(f2), __float_as_uint(f3), 0x7632);
}

template <int BM, int BN, int SA, int SF, Epi EPI>
__global__ void __launch_bounds__(kW8Threads, 1)
    gemm_w8_kernel(const __grid_constant__ CUtensorMap tmA, const uint8_t* __restrict__ B0,
                   const uint8_t* __restrict__ B1, const float* __restrict__ s0, const float* __restrict__ s1,
                   const GemmShape s, const EpiArgs ea, const DevStatus st) {
  static_assert(SF >= SA && BN % 32 == 0 && BN <= 128, "W8 GEMM configuration");
  using L = W8Smem<BM, BN, SA, SF>;
  constexpr uint32_t kTmemCols = pow2_cols(2 * BN);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* a_full = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* a_empty = a_full + SA;
  uint64_t* f_full = a_empty + SA;
  uint64_t* f_empty = f_full + SF;
  uint64_t* b_full = f_empty + SF;
  uint64_t* b_empty = b_full + 2;
  uint64_t* tfull = b_empty + 2;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tiles = (s.M + BM - 1) / BM;
  const int n_tiles = s.N / BN;
  const int kstages = s.K / 128;
  const int num_units = m_tiles * n_tiles * s.ksplit;
  const int unit0 = (int)blockIdx.x, ustep = (int)gridDim.x;
  const int kb_per = s.kb_per;  // 128-wide stages per K slice
  auto cursor = [&]() {
    W8Cursor c{unit0, 0, 1, 0, 0, ustep, num_units, s.ksplit, kb_per, kstages, m_tiles, n_tiles, s.raster_g};
    c.range();
    return c;
  };
  // column block of a unit -> (B rows of the tile, which matrix)
  auto tile_n0 = [&](int unit, int& m_blk) {
    int batch, n_blk;
    tile_coords(unit / s.ksplit, m_tiles, n_tiles, s.raster_g, batch, m_blk, n_blk);
    return n_blk * BN;
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < SA; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < SF; ++i) {
      mbar_init(&f_full[i], 1);
      mbar_init(&f_empty[i], kW8Deq);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&b_full[i], kW8Deq);
      mbar_init(&b_empty[i], 1);
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], 128);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kW8Threads / 32 - 1 && lane == 0) tma_prefetch_desc(&tmA);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_launch_dependents();
  // the code producer and the dequantization warps touch only weights and
  // shared memory: only the MMA, epilogue and A-producer warps wait for the
  // preceding kernel
  if ((warp >= 1 && warp <= 5) || warp == kW8Threads / 32 - 1) pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      // E4M3 code tiles: weights only, so no wait on the preceding kernel
      W8Cursor cf = cursor();
      int nf = 0;
      for (; cf.valid(); cf.next(), ++nf) {
        const int slot = nf % SF;
        if (nf >= SF && !mbar_wait(&f_empty[slot], ((nf / SF) & 1) ^ 1, st, abort_flag, 81)) break;
        int m_blk;
        const int n0 = tile_n0(cf.unit, m_blk);
        const bool first_mat = n0 < s.n_split;
        const uint8_t* bm = first_mat ? B0 : B1;
        const int rb = first_mat ? n0 : n0 - s.n_split;
        uint8_t* dst = smem + L::kFOff + slot * L::kF;
        mbar_arrive_expect_tx(&f_full[slot], L::kF);
        // rows rb .. rb+BN-1 of K stage kb: contiguous within each 128-row block
        const int r_in = rb & 127;
        const int n1 = BN < 128 - r_in ? BN : 128 - r_in;
        bulk_load(dst, bm + (((size_t)(rb >> 7) * kstages + cf.kb()) * 128 + r_in) * 128, n1 * 128, &f_full[slot]);
        if (n1 < BN)
          bulk_load(dst + n1 * 128, bm + ((size_t)((rb >> 7) + 1) * kstages + cf.kb()) * 128 * 128, (BN - n1) * 128,
                    &f_full[slot]);
      }
      // no copy may still be in flight into this CTA's shared memory
      for (int i = 0; i < SF && i < nf; ++i) {
        const int uses = (nf - 1 - i) / SF + 1;
        mbar_wait(&f_full[i], (uses - 1) & 1, st, nullptr, 83);
      }
    }
  } else if (warp == kW8Threads / 32 - 1) {
    if (lane == 0) {
      // ---------------- A producer (its own warp: an A load never waits
      // behind the issue of a code copy) ----------------
      W8Cursor ca = cursor();
      int na = 0;
      for (; ca.valid(); ca.next(), ++na) {
        const int slot = na % SA;
        if (na >= SA && !mbar_wait(&a_empty[slot], ((na / SA) & 1) ^ 1, st, abort_flag, 82)) break;
        int m_blk;
        tile_n0(ca.unit, m_blk);
        mbar_arrive_expect_tx(&a_full[slot], L::kA);
        uint8_t* sa = smem + slot * L::kA;
        tma_load_2d(sa, &tmA, &a_full[slot], ca.kb() * 128, m_blk * BM);
        tma_load_2d(sa + L::kA1, &tmA, &a_full[slot], ca.kb() * 128 + 64, m_blk * BM);
      }
      for (int i = 0; i < SA && i < na; ++i) {
        const int uses = (na - 1 - i) / SA + 1;
        mbar_wait(&a_full[i], (uses - 1) & 1, st, nullptr, 83);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(BM, BN, false, false);
      W8Cursor c = cursor();
      int n = 0, acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      while (ok && c.valid()) {
        const int unit = c.unit;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, st, abort_flag, 84)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        bool first = true;
        for (; c.valid() && c.unit == unit; c.next(), ++n) {
          const int sa = n % SA, sb = n & 1;
          if (!mbar_wait(&a_full[sa], (n / SA) & 1, st, abort_flag, 85) ||
              !mbar_wait(&b_full[sb], (n >> 1) & 1, st, abort_flag, 86)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + sa * L::kA);
          const uint32_t b_base = smem_u32(smem + L::kBOff + sb * L::kB);
#pragma unroll
          for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_bf16(d_tmem, sdesc_sw128(a_base + u * L::kA1 + k * 32, 16, 1024),
                        sdesc_sw128(b_base + u * L::kB1 + k * 32, 16, 1024), idesc, (first && u == 0 && k == 0) ? 0u : 1u);
          first = false;
          umma_commit(&a_empty[sa]);
          umma_commit(&b_empty[sb]);
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      umma_commit(drain);
      mbar_wait(drain, 0, st, nullptr, 87);
    }
  } else if (warp >= 6) {
    // ---------------- dequantization (warps 6..13) ----------------
    const int tid = threadIdx.x - 192;
    const int sld = kstages;  // scale columns (K / 128)
    float* sc_tab = reinterpret_cast<float*>(smem + L::kScOff);
    W8Cursor c = cursor();
    int rb = 0, rb0 = 0;
    for (int n = 0; c.valid(); c.next(), ++n) {
      if (c.i == 0) {
        // a new unit: its rows' block scales for every K stage of its slice
        int m_blk;
        const int n0 = tile_n0(c.unit, m_blk);
        const bool first_mat = n0 < s.n_split;
        const float* sc = first_mat ? s0 : s1;
        rb = first_mat ? n0 : n0 - s.n_split;
        rb0 = rb >> 7;
        const int nrb = ((rb + BN - 1) >> 7) - rb0 + 1;  // 1 or 2 row blocks
        asm volatile("bar.sync 2, %0;" ::"n"(kW8Deq) : "memory");  // the previous unit's readers are done
        for (int e = tid; e < 2 * kW8MaxKb; e += kW8Deq) {
          const int j = e / kW8MaxKb, i = e % kW8MaxKb;
          if (j < nrb && i < c.nk) sc_tab[e] = __ldg(sc + (size_t)(rb0 + j) * sld + c.kb0 + i);
        }
        asm volatile("bar.sync 2, %0;" ::"n"(kW8Deq) : "memory");
      }
      const int fs = n % SF, bs = n & 1;
      bool ok = mbar_wait(&f_full[fs], (n / SF) & 1, st, abort_flag, 88);
      ok = ok && mbar_wait(&b_empty[bs], ((n >> 1) & 1) ^ 1, st, abort_flag, 89);
      // every dequantization thread reaches the next unit's named barriers:
      // after a failed wait the rest of the work is skipped, not the loop
      if (!__all_sync(0xffffffffu, ok)) continue;
      const int kcol = c.kb() - c.kb0;
      const uint8_t* fst = smem + L::kFOff + fs * L::kF;
      uint8_t* bst = smem + L::kBOff + bs * L::kB;
      constexpr int kChunks = BN * 8 / kW8Deq;  // 16-byte E4M3 chunks per thread
      static_assert(BN * 8 % kW8Deq == 0, "chunks per dequantization thread");
      uint4 f[kChunks];
      float sv[kChunks];
#pragma unroll
      for (int q = 0; q < kChunks; ++q) {  // every load first: independent chains
        const int ci = tid + q * kW8Deq, r = ci >> 3;
        f[q] = *reinterpret_cast<const uint4*>(fst + ci * 16);
        sv[q] = sc_tab[(((rb + r) >> 7) - rb0) * kW8MaxKb + kcol];
      }
#pragma unroll
      for (int q = 0; q < kChunks; ++q) {
        const int ci = tid + q * kW8Deq, r = ci >> 3;
        const int lk = ci & 7;  // 16-element K chunk of row r (the E4M3 stage is not swizzled)
        uint32_t o[8];
        e4m3x4_to_bf16x4(f[q].x, sv[q], o[0], o[1]);
        e4m3x4_to_bf16x4(f[q].y, sv[q], o[2], o[3]);
        e4m3x4_to_bf16x4(f[q].z, sv[q], o[4], o[5]);
        e4m3x4_to_bf16x4(f[q].w, sv[q], o[6], o[7]);
        // 16 bf16 = logical 16-byte chunks 2 (lk % 4) and 2 (lk % 4) + 1 of 64-wide block lk / 4
        uint8_t* row = bst + (lk >> 2) * L::kB1 + r * 128;
        const int j0 = (lk & 3) * 2;
        *reinterpret_cast<uint4*>(row + ((j0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(row + (((j0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_proxy_async_smem();  // generic-proxy writes -> the tensor core's reads
      mbar_arrive(&b_full[bs]);
      mbar_arrive(&f_empty[fs]);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quarter = warp & 3;
    const bool lane_ok = (BM == 128) || lane < 16;
    const int rit = (BM == 128) ? quarter * 32 + lane : quarter * 16 + (lane & 15);
    const int ksplit = s.ksplit;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int unit = unit0; unit < num_units; unit += ustep) {
      const int tile = unit / ksplit;
      const int ks = unit % ksplit;
      int m_blk;
      const int n0 = tile_n0(unit, m_blk);
      bool ok = mbar_wait(&tfull[acc], acc_phase, st, abort_flag, 90);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc_fence_after();
      const int row = m_blk * BM + rit;
      const bool row_ok = lane_ok && row < s.M;
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) + acc * BN;
      if (ksplit == 1) {
        run_epilogue<BN, EPI>(ea, TmemSrc{taddr}, 0, row, n0, row_ok);
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
      } else {
        const int lq = rit - quarter * (BM / 4);  // row within the quarter
        float* slot = part_slot<BM, BN>(ea.part, tile * ksplit + ks, quarter, lq);
#pragma unroll 1
        for (int cc = 0; cc < BN; cc += 32) {
          uint32_t r[32];
          tmem_ld32(taddr + cc, r);
          tmem_wait_ld();
          if (row_ok) {
#pragma unroll
            for (int j = 0; j < 32; ++j) slot[(cc + j) * (BM / 4)] = __uint_as_float(r[j]);
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[acc]);
        __threadfence();
        __syncwarp();
        int prev = 0;
        if (lane == 0) prev = atomicAdd(&ea.counters[tile * 4 + quarter], 1);
        prev = __shfl_sync(0xffffffffu, prev, 0);
        if (prev == ksplit - 1) {
          __threadfence();
          const PartSrc<BM / 4> src{part_slot<BM, BN>(ea.part, tile * ksplit, quarter, lq), (size_t)BM * BN, ksplit,
                                    row_ok};
          run_epilogue<BN, EPI>(ea, src, 0, row, n0, row_ok);
          if (lane == 0) ea.counters[tile * 4 + quarter] = 0;
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int BM, int BN, int SA, int SF, Epi EPI>
cudaError_t launch_w8_impl(const GemmShape& s, const GemmW8Operands& op, const EpiArgs& ea, const DevStatusHost& st,
                           int num_sms, cudaStream_t stream) {
  using L = W8Smem<BM, BN, SA, SF>;
  static_assert(L::kBytes <= 232448, "shared memory budget");
  if (s.K % 128 || s.N % BN || s.n_split % BN || s.batches != 1) return cudaErrorInvalidValue;
  if (s.K / 128 > kW8MaxKb) return cudaErrorInvalidValue;  // the per-unit scale table
  if (s.n_split > op.b0_rows || (s.n_split < s.N && (!op.B1 || s.N - s.n_split > op.b1_rows)))
    return cudaErrorInvalidValue;
  CUtensorMap ta;
  if (!make_tmap_bf16_2d(&ta, op.A, op.a_rows, (uint64_t)op.lda, op.lda, BM, 64)) return cudaErrorInvalidValue;
  auto kern = gemm_w8_kernel<BM, BN, SA, SF, EPI>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::kBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  GemmShape sh = s;
  if (sh.raster_g < 1) sh.raster_g = 1;
  const int m_tiles = (s.M + BM - 1) / BM;
  const int tiles = m_tiles * (s.N / BN);
  const int kstages = s.K / 128;
  sh.ksplit = 1;
  sh.kb_per = kstages;
  // split-K as the bf16 path: too few tiles for the GPU (one row block)
  if (ea.part && ea.counters && m_tiles == 1 && tiles * 2 <= num_sms && kstages >= 2 &&
      tiles * 4 <= kMaxSplitCounters) {
    int ks = num_sms / tiles;
    if (ks > 4) ks = 4;
    if (ks > kMaxSplitUnits / tiles) ks = kMaxSplitUnits / tiles;
    if (ks > kstages) ks = kstages;
    const int kb_per = (kstages + ks - 1) / ks;
    ks = (kstages + kb_per - 1) / kb_per;
    const size_t need = (size_t)tiles * ks * BM * BN * sizeof(float);
    if (ks > 1 && need <= ea.part_bytes) {
      sh.ksplit = ks;
      sh.kb_per = kb_per;
    }
  }
  DevStatus dst{st.word, st.wait_limit_ns};
  const int units = tiles * sh.ksplit;
  const int grid = units < num_sms ? units : num_sms;
  return launch_pdl(kern, dim3(grid), dim3(kW8Threads), L::kBytes, stream, ta, op.B0, op.B1, op.s0, op.s1, sh, ea,
                    dst);
}

template <Epi EPI, int BN>
cudaError_t launch_w8_bm(const GemmShape& s, const GemmW8Operands& op, const EpiArgs& ea, const DevStatusHost& st,
                         int num_sms, cudaStream_t stream) {
  // 64-96 KB of A stages, two bf16 B stages, and the E4M3 ring as deep as
  // the rest of shared memory allows (both latencies are several
  // microseconds here: the per-SM copy engine serves both rings)
  constexpr int kSA64 = BN == 128 ? 4 : 6, kSF64 = BN == 64 ? 12 : 6;
  constexpr int kSA128 = BN == 128 ? 2 : 3, kSF128 = BN == 64 ? 12 : 6;
  if (s.M <= 64) return launch_w8_impl<64, BN, kSA64, kSF64, EPI>(s, op, ea, st, num_sms, stream);
  return launch_w8_impl<128, BN, kSA128, kSF128, EPI>(s, op, ea, st, num_sms, stream);
}

}  // namespace

cudaError_t launch_gemm(const GemmShape& s, const GemmOperands& op, Epi epi, const EpiArgs& ea,
                        const DevStatusHost& st, int num_sms, cudaStream_t stream) {
  if (s.M <= 0 || s.K % kBK != 0 || s.batches <= 0) return cudaErrorInvalidValue;
  // Few rows (decode): narrower N tiles so that enough CTAs stream the
  // weights, and M = 64 tiles when M <= 64 so that shared memory holds more
  // weight bytes in flight; many rows (prefill): wide tiles.
  const bool tiny = s.M <= 64;
  const bool small = s.M <= kBM;
  const bool k256 = s.K % 256 == 0;
  // many rows: CTA pairs run 256-row MMAs (an even number of row blocks)
  const bool pairs = ((s.M + kBM - 1) / kBM) % 2 == 0 && s.M > 2 * kBM;
  switch (epi) {
    case Epi::kQRope:
      if (s.N % 192 || op.b_mn_major) return cudaErrorInvalidValue;
      if (tiny && k256) return launch_impl<64, 96, 5, Epi::kQRope, false, 2>(s, op, ea, st, num_sms, stream);
      if (small && k256) return launch_impl<128, 96, 3, Epi::kQRope, false, 2>(s, op, ea, st, num_sms, stream);
      if (small) return launch_impl<128, 96, 7, Epi::kQRope, false>(s, op, ea, st, num_sms, stream);
      // CTA pairs: 256-column tiles (as the A- and o-projections), whose
      // operand bytes per MMA cycle the TMA ring sustains; 192-column tiles
      // ask for 14% more
      if (pairs && s.N % 256 == 0)
        return launch_impl<128, 256, 6, Epi::kQRope, false, 1, true, true>(s, op, ea, st, num_sms, stream);
      if (pairs) return launch_impl<128, 192, 6, Epi::kQRope, false, 1, true, true>(s, op, ea, st, num_sms, stream);
      return launch_impl<128, 192, 4, Epi::kQRope, false, 1, true>(s, op, ea, st, num_sms, stream);
    case Epi::kKVCache:
      if (s.N % 256 || op.b_mn_major) return cudaErrorInvalidValue;
      if (tiny && k256) return launch_impl<64, 128, 4, Epi::kKVCache, false, 2>(s, op, ea, st, num_sms, stream);
      if (small && k256) return launch_impl<128, 128, 3, Epi::kKVCache, false, 2>(s, op, ea, st, num_sms, stream);
      if (small) return launch_impl<128, 128, 6, Epi::kKVCache, false>(s, op, ea, st, num_sms, stream);
      // many row pairs: the resident-B pair kernel (K = 512 fits shared memory)
      if (ea.t_mod % 32 == 0 && ea.B > 0 && !ea.pos && pairs && s.M % 256 == 0 && s.M >= 16 * 256 &&
          s.K <= kResKb * kBK && s.batches == 1)
        return launch_resb_pair<Epi::kKVCache>(s, op, ea, st, num_sms, stream);
      if (ea.t_mod % 32 == 0 && ea.B > 0 && !ea.pos && pairs)
        return launch_impl<128, 256, 6, Epi::kKVCache, false, 1, true, true>(s, op, ea, st, num_sms, stream);
      if (ea.t_mod % 32 == 0 && ea.B > 0 && !ea.pos)
        return launch_impl<128, 256, 4, Epi::kKVCache, false, 1, true>(s, op, ea, st, num_sms, stream);
      return launch_impl<128, 256, 4, Epi::kKVCache, false>(s, op, ea, st, num_sms, stream);
    case Epi::kResidual: {
      if (s.N % 256 || op.b_mn_major) return cudaErrorInvalidValue;
      // o_proj: W_o (117 MB) does not stay in L2 -> waves of 16 row blocks
      GemmShape g16 = s;
      g16.raster_g = 16;
      // long K (the MLP's down product, K = 18432): 128-wide tiles split in two
      // K halves stream the weights faster than 64-wide whole-K tiles
      if (tiny && k256 && s.K >= 16384)
        return launch_impl<64, 128, 4, Epi::kResidual, false, 2>(s, op, ea, st, num_sms, stream);
      if (tiny && k256) return launch_impl<64, 64, 3, Epi::kResidual, false, 4>(s, op, ea, st, num_sms, stream);
      if (small && k256) return launch_impl<128, 64, 4, Epi::kResidual, false, 2>(s, op, ea, st, num_sms, stream);
      if (small) return launch_impl<128, 64, 8, Epi::kResidual, false>(s, op, ea, st, num_sms, stream);
      if (pairs) {
        GemmShape g8 = s;
        g8.raster_g = 8;  // groups of 8 row-block pairs
        return launch_impl<128, 256, 6, Epi::kResidual, false, 1, true, true>(g8, op, ea, st, num_sms, stream);
      }
      return launch_impl<128, 256, 4, Epi::kResidual, false, 1, true>(g16, op, ea, st, num_sms, stream);
    }
    case Epi::kSwiGLU: {
      // N = 2 I output columns of [gate | up]; B0 = W_1, B1 = W_3, both [I, K]
      if (s.N % 256 || 2 * s.n_split != s.N || op.b_mn_major || !op.B1 || s.batches != 1)
        return cudaErrorInvalidValue;
      GemmShape g8 = s;
      g8.raster_g = 8;  // the gate/up weights do not stay in L2: walk groups of 8 row blocks (pairs)
      if (tiny && k256) return launch_impl<64, 128, 4, Epi::kSwiGLU, false, 2>(s, op, ea, st, num_sms, stream);
      if (small) return launch_impl<128, 128, 6, Epi::kSwiGLU, false>(s, op, ea, st, num_sms, stream);
      if (pairs) return launch_impl<128, 256, 6, Epi::kSwiGLU, false, 1, true, true>(g8, op, ea, st, num_sms, stream);
      return launch_impl<128, 256, 4, Epi::kSwiGLU, false, 1, true>(g8, op, ea, st, num_sms, stream);
    }
    case Epi::kStoreF32:
      if (s.N % 192 || s.n_split % 192 || op.b_mn_major) return cudaErrorInvalidValue;
      if (tiny && k256) return launch_impl<64, 64, 3, Epi::kStoreF32, false, 4>(s, op, ea, st, num_sms, stream);
      if (small && k256) return launch_impl<128, 64, 4, Epi::kStoreF32, false, 2>(s, op, ea, st, num_sms, stream);
      if (small) return launch_impl<128, 64, 8, Epi::kStoreF32, false>(s, op, ea, st, num_sms, stream);
      // 256-wide tiles (2112 = 8.25 x 256: 9 column tiles, the last one
      // clipped on store; the c^Q / c^KV split at 1536 is tile-aligned) read
      // the fewest operand bytes from L2 per MMA, and 16 row blocks make 144
      // tiles, one wave; 128-wide tiles when there are too few tiles for a wave.
      if (s.n_split % 256 == 0 && ((s.M + kBM - 1) / kBM) * 9 >= num_sms / 2) {
        if (pairs) return launch_impl<128, 256, 6, Epi::kStoreF32, false, 1, true, true>(s, op, ea, st, num_sms, stream);
        return launch_impl<128, 256, 4, Epi::kStoreF32, false, 1, true>(s, op, ea, st, num_sms, stream);
      }
      return launch_impl<128, 128, 6, Epi::kStoreF32, false, 1, true>(s, op, ea, st, num_sms, stream);
    case Epi::kStoreBf16:
    default:
      if (op.b_mn_major) {
        if (s.N % 128) return cudaErrorInvalidValue;
        if (tiny) return launch_impl<64, 128, 8, Epi::kStoreBf16, true>(s, op, ea, st, num_sms, stream);
        return launch_impl<128, 128, 6, Epi::kStoreBf16, true>(s, op, ea, st, num_sms, stream);
      }
      if (tiny && k256 && s.N % 64 == 0 && s.n_split % 64 == 0)
        return launch_impl<64, 64, 3, Epi::kStoreBf16, false, 4>(s, op, ea, st, num_sms, stream);
      if (small && s.N % 64 == 0 && s.n_split % 64 == 0)
        return launch_impl<128, 64, 8, Epi::kStoreBf16, false>(s, op, ea, st, num_sms, stream);
      if (s.N % 192 == 0 && s.n_split % 192 == 0)
        return launch_impl<128, 192, 5, Epi::kStoreBf16, false>(s, op, ea, st, num_sms, stream);
      if (s.N % 128 == 0 && s.n_split % 128 == 0)
        return launch_impl<128, 128, 6, Epi::kStoreBf16, false>(s, op, ea, st, num_sms, stream);
      return cudaErrorInvalidValue;
  }
}

// ---------------------------------------------------------------------------
// tensor maps (driver entry point looked up once through the runtime)
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                       uint32_t box_rows, uint32_t box_cols) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool encode(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base, const cuuint64_t* dims,
                   const cuuint64_t* strides, const cuuint32_t* box, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tmap_store_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 2};
  cuuint32_t box[2] = {32, 32};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_64B);
}

bool make_tmap_store_f32_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {ld * 4};
  cuuint32_t box[2] = {32, 32};
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_tmap_store_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
                             uint64_t mid_stride_bytes, uint64_t outer_stride_bytes) {
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {mid_stride_bytes, outer_stride_bytes};
  cuuint32_t box[3] = {64, 32, 1};  // 32 rows x 64 bf16, 128-byte swizzle
  return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
                       uint64_t mid_stride_bytes, uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_mid) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, mid, outer};
  cuuint64_t strides[2] = {mid_stride_bytes, outer_stride_bytes};
  cuuint32_t box[3] = {box_inner, box_mid, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_gemm_w8(const GemmShape& s, const GemmW8Operands& op, Epi epi, const EpiArgs& ea,
                           const DevStatusHost& st, int num_sms, cudaStream_t stream) {
  if (s.M <= 0 || s.K % 128 != 0) return cudaErrorInvalidValue;
  switch (epi) {
    case Epi::kStoreF32: return launch_w8_bm<Epi::kStoreF32, 64>(s, op, ea, st, num_sms, stream);
    case Epi::kQRope: return launch_w8_bm<Epi::kQRope, 96>(s, op, ea, st, num_sms, stream);
    case Epi::kKVCache: return launch_w8_bm<Epi::kKVCache, 128>(s, op, ea, st, num_sms, stream);
    // o_proj: 128-row code tiles (split-K 2 fills the GPU), half the activation
    // bytes per code byte of 64-row tiles: 55 -> 48 us at 64 rows (ncu)
    case Epi::kResidual: return launch_w8_bm<Epi::kResidual, 128>(s, op, ea, st, num_sms, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace mla
