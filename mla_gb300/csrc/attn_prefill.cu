// Causal prefill attention for MLA heads (qk = 192, v = 128) on tcgen05.
//
// "Mix and project" page, code excerpt: scores = Q K^T * softmax_scale plus
// the causal mask, softmax in float32, then P V.  Computed in the flash form
// (online softmax over 128-key tiles; scores and probabilities never reach
// global memory).
//
// Persistent: one CTA per SM takes work items (128-query tile, head,
// sequence) from an atomic counter, in the order (sequence, group of G
// heads, query tile from the last, heaviest, to the first, head within the
// group): the query tiles of a few heads run together and share their K/V
// tiles in L2, and within a group the heavy tiles of every head come first,
// so the dynamic grab ends on light tiles (G is chosen so that a group holds
// enough work for every SM to take one of its heaviest tiles early, and so
// that its heads' K/V fit comfortably in L2).  Each item's Q load and first
// scores overlap the previous item's last P.V and epilogue.
// Chunked prefill: the queries sit at positions past..past+T-1 and attend to
// keys 0..past+T-1 of the cache (the chunk's own keys written after the
// cached ones), the causal mask offset by past.
// Warp roles (256 threads):
//   warp 0   work scheduler (atomic counter -> a 4-slot ring of item
//            indices in shared memory that every role reads), then TMA: the
//            item's Q tile, then its K tiles into a 2-slot ring
//   warp 6   TMA: V tiles into a 2-slot ring (each K and V tile is requested
//            a whole tile ahead of the MMA that reads it)
//   warp 1   TMEM allocation; one lane issues S_j = Q K_j^T (M=128 N=128
//            K=192) into score buffer j & 1: the 128 "nope" dimensions of Q
//            read from tensor memory (the softmax warps copy them there
//            once), the 64 RoPE dimensions from one of two shared-memory
//            slots (alternating items), K from its TMA tile; a score buffer
//            is reused as soon as the softmax has read it
//   warp 7   one lane issues O += P_j V_j (M=128 N=128 K=128), P read from
//            its own tensor-memory buffer (row m in lane m, bf16 pairs
//            packed per column), V read MN-major from its TMA tile
//   (two issuing threads, each on blocking waits, keep the tensor pipe fed
//   while either one waits.  With P apart from the scores, the chain of a
//   score buffer is S -> softmax read -> next S; P waits only for the
//   previous P.V.  The tensor-memory columns this needs come from keeping
//   Q's RoPE dimensions in shared memory: 4 of the 12 K steps of S read A
//   from there, 16 KB of operand reads per key tile.)
//   warps 2..5  one thread per query row: copy the Q row into tensor memory;
//            read S_j from TMEM, scale, causal mask on the diagonal tile,
//            running max with lazy rescaling (O is rescaled in TMEM only when
//            the max grows by more than 2^8, so P stays <= 256), P_j as bf16
//            into the P buffer (once the previous P.V has read it), and at
//            the end O / l to global memory (after the next item's Q has
//            been copied, so its first scores overlap).
// Layout: Q [B*T, 64*192], K/V caches [B, 64, cap, 192|128] (TMA 3D views
// whose position extent is T, so keys >= T read as zeros), O [B*T, 64*128].
#include "common.cuh"
#include "internal.h"

namespace mla {

namespace {

constexpr int kThreads = 256;
constexpr uint32_t kAtom = 128 * 128;            // 128 rows x 64 bf16
constexpr uint32_t kQOff = 0;                    // Q dims 0-127: 2 atoms (staging)
constexpr uint32_t kQpeOff = 2 * kAtom;          // Q dims 128-191: 2 slots x 1 atom
constexpr uint32_t kKOff = 4 * kAtom;            // 2 slots x 3 atoms
constexpr uint32_t kVOff = 10 * kAtom;           // 2 slots x 2 atoms (vdim 0-63, 64-127)
constexpr uint32_t kBarOff = 14 * kAtom;
// tensor memory columns: S_0, S_1 (fp32), O (fp32), P (bf16 pairs, 128 keys),
// Q dims 0-127 (bf16 pairs)
constexpr uint32_t kTmS = 0, kTmO = 256, kTmP = 384, kTmQ = 448;
constexpr uint32_t kSmemBytes = kBarOff + 512 + 1024;
static_assert(kSmemBytes <= 232448, "prefill attention shared memory");
constexpr float kRescaleThreshold = 8.0f;        // log2 units

constexpr int kItemRing = 4;
constexpr int kItemReaders = 3 + 128;  // V producer, S issuer, P.V issuer, softmax threads

struct Bars {
  uint64_t q_full, q_tmem, qn_empty, qpe_empty[2];
  uint64_t item_full[kItemRing], item_empty[kItemRing];
  uint64_t k_full[2], k_empty[2];
  uint64_t v_full[2], v_empty[2];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, pv_done;
  uint64_t drain_s, drain_pv;
  uint32_t tmem_slot;
  int abort;
  int item[kItemRing];
};
static_assert(sizeof(Bars) <= 512, "barrier block");

// Work item w (the order described above) -> its query tile, head, sequence.
struct Item {
  int qt, h, b, q0, n_kv;
  __device__ __forceinline__ Item(int w, int n_qt, int T, int past, int G) {
    const int per_seq = 64 * n_qt;
    b = w / per_seq;
    const int r = w - b * per_seq;
    const int full = 64 / G;                       // groups of G heads, then one of 64 % G
    int g = r / (G * n_qt), within, gs;
    if (g < full) {
      within = r - g * G * n_qt;
      gs = G;
    } else {
      g = full;
      within = r - full * G * n_qt;
      gs = 64 - full * G;
    }
    const int level = within / gs;
    h = g * G + (within - level * gs);
    qt = n_qt - 1 - level;
    q0 = qt * 128;
    // keys 0 .. past + q0 + 127 (the tile's last query), at most past + T of them
    n_kv = min((past + q0 + 127) / 128 + 1, (past + T + 127) / 128);
  }
};

// Every role reads item `it` from the ring (bounded wait), then releases the slot.
__device__ __forceinline__ bool read_item(Bars* bar, int it, int& w, const DevStatus& st, volatile int* abort_flag) {
  const int slot = it % kItemRing;
  if (!mbar_wait(&bar->item_full[slot], (it / kItemRing) & 1, st, abort_flag, 39)) return false;
  w = *reinterpret_cast<volatile int*>(&bar->item[slot]);
  mbar_arrive(&bar->item_empty[slot]);
  return true;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_attn_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ o, int T, int n_qt,
                    int n_items, float sl2, int past, int head_group, int* __restrict__ work,
                    const DevStatus st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bar = reinterpret_cast<Bars*>(smem + kBarOff);
  volatile int* abort_flag = &bar->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bar->q_full, 1);
    mbar_init(&bar->q_tmem, 128);
    mbar_init(&bar->qn_empty, 128);
    mbar_init(&bar->qpe_empty[0], 1);
    mbar_init(&bar->qpe_empty[1], 1);
    mbar_init(&bar->p_full, 128);
    mbar_init(&bar->pv_done, 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&bar->item_full[i], 1);
      mbar_init(&bar->item_empty[i], kItemReaders);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar->k_full[i], 1);
      mbar_init(&bar->k_empty[i], 1);
      mbar_init(&bar->v_full[i], 1);
      mbar_init(&bar->v_empty[i], 1);
      mbar_init(&bar->s_full[i], 1);
      mbar_init(&bar->s_free[i], 128);
    }
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

  if (warp == 0) {
    if (lane == 0) {
      // ---- work scheduler, Q and K producer ----
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      int issued[2] = {0, 0};
      int q_loads = 0;
      int gt = 0;  // this CTA's K tiles so far (ring position)
      for (int it = 0;; ++it) {
        const int slot = it % kItemRing;
        if (it >= kItemRing && !mbar_wait(&bar->item_empty[slot], (it / kItemRing - 1) & 1, st, abort_flag, 38))
          break;
        int w = atomicAdd(work, 1);
        if (w >= n_items) w = -1;
        bar->item[slot] = w;
        mbar_arrive(&bar->item_full[slot]);  // release: the index is visible to every waiting role
        if (w < 0) break;
        const Item t(w, n_qt, T, past, head_group);
        // the Q tile: dims 0-127 into the staging atoms once the softmax threads
        // copied the previous item's into tensor memory, dims 128-191 into the
        // slot of this item's parity once the S of the item two back are done
        if (it > 0 && !mbar_wait(&bar->qn_empty, (it - 1) & 1, st, abort_flag, 37)) break;
        if (it > 1 && !mbar_wait(&bar->qpe_empty[it & 1], ((it - 2) >> 1) & 1, st, abort_flag, 36)) break;
        mbar_arrive_expect_tx(&bar->q_full, 3 * kAtom);
        for (int c = 0; c < 2; ++c)
          tma_load_3d(smem + kQOff + c * kAtom, &tmQ, &bar->q_full, t.h * 192 + 64 * c, t.q0, t.b);
        tma_load_3d(smem + kQpeOff + (it & 1) * kAtom, &tmQ, &bar->q_full, t.h * 192 + 128, t.q0, t.b);
        ++q_loads;
        const int kv_row = t.b * 64 + t.h;
        bool ok = true;
        for (int j = 0; j < t.n_kv; ++j, ++gt) {
          const int ks = gt & 1;
          if (!mbar_wait(&bar->k_empty[ks], ((gt >> 1) & 1) ^ 1, st, abort_flag, 40)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar->k_full[ks], 3 * kAtom);
          for (int c = 0; c < 3; ++c)
            tma_load_3d(smem + kKOff + (ks * 3 + c) * kAtom, &tmK, &bar->k_full[ks], 64 * c, j * 128, kv_row);
          issued[ks]++;
        }
        if (!ok) break;
      }
      // no copy may still be in flight into shared memory
      if (q_loads) mbar_wait(&bar->q_full, (q_loads - 1) & 1, st, nullptr, 41);
      for (int i = 0; i < 2; ++i)
        if (issued[i]) mbar_wait(&bar->k_full[i], (issued[i] - 1) & 1, st, nullptr, 41);
    }
  } else if (warp == 6) {
    if (lane == 0) {
      // ---- V producer ----
      tma_prefetch_desc(&tmV);
      int issued[2] = {0, 0};
      int gt = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        int w;
        if (!read_item(bar, it, w, st, abort_flag) || w < 0) break;
        const Item t(w, n_qt, T, past, head_group);
        const int kv_row = t.b * 64 + t.h;
        for (int j = 0; j < t.n_kv; ++j, ++gt) {
          const int vs = gt & 1;
          if (!mbar_wait(&bar->v_empty[vs], ((gt >> 1) & 1) ^ 1, st, abort_flag, 42)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar->v_full[vs], 2 * kAtom);
          for (int c = 0; c < 2; ++c)
            tma_load_3d(smem + kVOff + (vs * 2 + c) * kAtom, &tmV, &bar->v_full[vs], 64 * c, j * 128, kv_row);
          issued[vs]++;
        }
      }
      for (int i = 0; i < 2; ++i)
        if (issued[i]) mbar_wait(&bar->v_full[i], (issued[i] - 1) & 1, st, nullptr, 43);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- S issuer: S_j = Q K_j^T into score buffer gt & 1 ----
      constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
      const uint32_t k_addr = smem_u32(smem + kKOff);
      const uint32_t q_tm = tmem + kTmQ;
      int gt = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        int w;
        if (!read_item(bar, it, w, st, abort_flag) || w < 0) break;
        const Item t(w, n_qt, T, past, head_group);
        if (!mbar_wait(&bar->q_tmem, it & 1, st, abort_flag, 44)) break;  // this item's Q in tensor memory
        const uint32_t qpe_addr = smem_u32(smem + kQpeOff + (it & 1) * kAtom);
        for (int j = 0; j < t.n_kv; ++j, ++gt) {
          const int sb = gt & 1;
          if (!mbar_wait(&bar->k_full[sb], (gt >> 1) & 1, st, abort_flag, 45)) {
            ok = false;
            break;
          }
          // the softmax has read the buffer's previous scores (tile gt-2)
          if (gt > 1 && !mbar_wait(&bar->s_free[sb], ((gt - 2) >> 1) & 1, st, abort_flag, 46)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + kTmS + sb * 128;
          const uint32_t kb = k_addr + sb * 3 * kAtom;
          // Q dims 0-127 from tensor memory, dims 128-191 from this item's slot
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t off = (kk >> 2) * kAtom + (kk & 3) * 32;
            umma_bf16_ts(d, q_tm + kk * 8, sdesc_sw128(kb + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            umma_bf16(d, sdesc_sw128(qpe_addr + kk * 32, 16, 1024), sdesc_sw128(kb + 2 * kAtom + kk * 32, 16, 1024),
                      idesc_s, 1u);
          umma_commit(&bar->s_full[sb]);
          umma_commit(&bar->k_empty[sb]);
        }
        if (!ok) break;
        umma_commit(&bar->qpe_empty[it & 1]);  // this item's Q slot may be reloaded
      }
      umma_commit(&bar->drain_s);
      mbar_wait(&bar->drain_s, 0, st, nullptr, 49);
    }
  } else if (warp == 7) {
    if (lane == 0) {
      // ---- P.V issuer: O += P_j V_j ----
      constexpr uint32_t idesc_pv = idesc_bf16(128, 128, false, true);
      const uint32_t v_addr = smem_u32(smem + kVOff);
      int gt = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        int w;
        if (!read_item(bar, it, w, st, abort_flag) || w < 0) break;
        const Item t(w, n_qt, T, past, head_group);
        for (int j = 0; j < t.n_kv; ++j, ++gt) {
          const int sb = gt & 1;
          // P_j is written (and, for an item's first tile, the previous item's
          // O read out: the softmax threads do that before writing P)
          if (!mbar_wait(&bar->p_full, gt & 1, st, abort_flag, 47) ||
              !mbar_wait(&bar->v_full[sb], (gt >> 1) & 1, st, abort_flag, 48)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vb = v_addr + sb * 2 * kAtom;
          const uint32_t pa = tmem + kTmP;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bdesc = sdesc_sw128(vb + kk * 2048, kAtom, 1024);
            umma_bf16_ts(tmem + kTmO, pa + kk * 8, bdesc, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bar->pv_done);
          umma_commit(&bar->v_empty[sb]);
        }
      }
      umma_commit(&bar->drain_pv);
      mbar_wait(&bar->drain_pv, 0, st, nullptr, 49);
    }
  } else {
    // ---- softmax / correction / epilogue: warps 2..5, one thread per query row ----
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    bool ok = true;
    int gt = 0;
    // the previous item, whose O is written out once the next item's Q is in place
    int prev_qpos = -1, prev_h = 0, prev_b = 0, prev_last = -1;
    float prev_l = 1.f;
    for (int it = 0; ok; ++it) {
      int w = -1;
      ok = __all_sync(0xffffffffu, read_item(bar, it, w, st, abort_flag));
      if (!ok) break;
      if (w >= 0) {
        // this item's Q rows, dims 0-127 (two 128-byte-swizzled 64-column
        // atoms), into tensor memory as bf16 pairs, the A operand of the
        // first 8 K steps of every S_j; the previous item's S are all done
        // (its last s_full was consumed)
        ok = __all_sync(0xffffffffu, mbar_wait(&bar->q_full, it & 1, st, abort_flag, 54));
        if (!ok) break;
        const uint8_t* qrow = smem + kQOff + row * 128;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t v[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint4 x = *reinterpret_cast<const uint4*>(qrow + c * kAtom + ((q ^ (row & 7)) << 4));
            v[4 * q] = x.x;
            v[4 * q + 1] = x.y;
            v[4 * q + 2] = x.z;
            v[4 * q + 3] = x.w;
          }
          tmem_st32(tmem + lane_addr + kTmQ + c * 32, v);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bar->q_tmem);
        mbar_arrive(&bar->qn_empty);
      }
      if (prev_last >= 0) {
        // epilogue of the previous item: O / l once its last P.V is done
        ok = __all_sync(0xffffffffu, mbar_wait(&bar->pv_done, prev_last & 1, st, abort_flag, 52));
        if (!ok) break;
        tc_fence_after();
        const float inv = 1.f / prev_l;
        const uint32_t ta = tmem + lane_addr + kTmO;
        __nv_bfloat16* dst = o + ((size_t)prev_b * T + prev_qpos) * 8192 + prev_h * 128;
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
          uint32_t r[32];
          tmem_ld32(ta + c, r);
          tmem_wait_ld();
          if (prev_qpos < T) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              d4[q] = make_uint4(pack_bf16x2(__uint_as_float(r[8 * q]) * inv, __uint_as_float(r[8 * q + 1]) * inv),
                                 pack_bf16x2(__uint_as_float(r[8 * q + 2]) * inv, __uint_as_float(r[8 * q + 3]) * inv),
                                 pack_bf16x2(__uint_as_float(r[8 * q + 4]) * inv, __uint_as_float(r[8 * q + 5]) * inv),
                                 pack_bf16x2(__uint_as_float(r[8 * q + 6]) * inv, __uint_as_float(r[8 * q + 7]) * inv));
          }
        }
        prev_last = -1;
      }
      if (w < 0) break;
      const Item t(w, n_qt, T, past, head_group);
      const int qpos = t.q0 + row;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < t.n_kv; ++j, ++gt) {
        const int sb = gt & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar->s_full[sb], (gt >> 1) & 1, st, abort_flag, 50));
        if (!ok) break;
        tc_fence_after();
        uint32_t s[128];
        {
          uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
          uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
          uint32_t (&s2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[64]);
          uint32_t (&s3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[96]);
          const uint32_t ta = tmem + lane_addr + kTmS + sb * 128;
          tmem_ld32(ta, s0);
          tmem_ld32(ta + 32, s1);
          tmem_ld32(ta + 64, s2);
          tmem_ld32(ta + 96, s3);
          tmem_wait_ld();
        }
        tc_fence_before();
        mbar_arrive(&bar->s_free[sb]);  // the score buffer may take S_{j+2}
        const int k0 = j * 128;
        // max of the raw scores (the scale is positive), causal mask (key k
        // visible to query position past + qpos iff k <= past + qpos) on the
        // tiles that reach beyond the tile's first query
        if (k0 + 127 > past + t.q0) {
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (k0 + c > past + qpos) s[c] = __float_as_uint(-INFINITY);
        }
        // eight independent partial maxima / sums keep the reductions off a
        // single serial dependency chain; three-input maxima and two-lane
        // float32 FMA / add halve the instructions of the max, scale and sum
        // passes (the softmax threads are bound by instruction issue)
        float mp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mp[i] = fmaxf(__uint_as_float(s[i]), __uint_as_float(s[i + 8]));
#pragma unroll
        for (int c = 16; c < 128; c += 16)
#pragma unroll
          for (int i = 0; i < 8; ++i) mp[i] = fmax3(mp[i], __uint_as_float(s[c + i]), __uint_as_float(s[c + 8 + i]));
        float mx = fmaxf(fmax3(mp[0], mp[1], mp[2]), fmax3(mp[3], mp[4], fmax3(mp[5], mp[6], mp[7])));
        mx *= sl2;  // log2 units
        const bool need = mx > m + kRescaleThreshold;
        const float m_new = need ? mx : m;
        const float alpha = need ? ex2_approx(m - m_new) : 1.f;
        float sp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 128; c += 2) {
          float x0, x1;
          fma_x2(x0, x1, __uint_as_float(s[c]), __uint_as_float(s[c + 1]), sl2, sl2, -m_new, -m_new);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          s[c] = __float_as_uint(p0);
          s[c + 1] = __float_as_uint(p1);
          add_x2(sp[c & 7], sp[(c & 7) + 1], sp[c & 7], sp[(c & 7) + 1], p0, p1);
        }
        const float sum = ((sp[0] + sp[1]) + (sp[2] + sp[3])) + ((sp[4] + sp[5]) + (sp[6] + sp[7]));
        l = l * alpha + sum;
        m = m_new;
        // the previous P.V (this CTA's tile gt-1) has read P and added into O:
        // P may be rewritten and O rescaled
        if (gt > 0) {
          ok = __all_sync(0xffffffffu, mbar_wait(&bar->pv_done, (gt - 1) & 1, st, abort_flag, 53));
          if (!ok) break;
          tc_fence_after();  // P and O writes below come after that MMA's reads
        }
        if (j > 0 && __any_sync(0xffffffffu, need)) {
          const uint32_t ta = tmem + lane_addr + kTmO;
#pragma unroll 1
          for (int c = 0; c < 128; c += 32) {
            uint32_t r[32];
            tmem_ld32(ta + c, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
            tmem_st32(ta + c, r);
          }
          tmem_wait_st();
        }
        // P_j (bf16 pairs, low half = even key) into the P buffer
        {
          uint32_t pk[64];
#pragma unroll
          for (int c = 0; c < 64; ++c) pk[c] = pack_bf16x2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1]));
          const uint32_t tp = tmem + lane_addr + kTmP;
#pragma unroll
          for (int c = 0; c < 64; c += 16) tmem_st16(tp + c, &pk[c]);
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&bar->p_full);
      }
      prev_qpos = qpos;
      prev_h = t.h;
      prev_b = t.b;
      prev_l = l;
      prev_last = gt - 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}
}  // namespace

cudaError_t launch_prefill_attention(const PrefillAttnArgs& a, const DevStatusHost& st, int num_sms,
                                     cudaStream_t stream) {
  CUtensorMap tq, tk, tv;
  const uint64_t n_keys = (uint64_t)a.past + a.T;  // key positions beyond read as zeros
  if (!make_tmap_bf16_3d(&tq, a.q, 12288, a.T, a.B, 12288ull * 2, (uint64_t)a.T * 12288 * 2, 64, 128) ||
      !make_tmap_bf16_3d(&tk, a.k, 192, n_keys, (uint64_t)a.B * 64, 384, (uint64_t)a.cap * 384, 64, 128) ||
      !make_tmap_bf16_3d(&tv, a.v, 128, n_keys, (uint64_t)a.B * 64, 256, (uint64_t)a.cap * 256, 64, 128))
    return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(prefill_attn_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int n_qt = (a.T + 127) / 128;
  const long long items = (long long)n_qt * 64 * a.B;
  if (items > INT32_MAX || !st.word) return cudaErrorInvalidValue;
  const int n_items = (int)items;
  const int grid = n_items < num_sms ? n_items : num_sms;
  // head group G (a power of two, so the groups split the 64 heads evenly):
  // the smallest whose work (G heads' query tiles, in key tiles) is at least
  // 1.5x the CTA count times the heaviest item -- the heaviest tiles of the
  // last group then start early enough -- halved while its heads' K/V exceed
  // 16 MB (measured against 64, 32 and 8 MB caps: at B=8 T=4096 each halving
  // of the group down to 4 heads made the attention faster, 2.013 -> 1.977 ms,
  // as the heads in flight read their K/V from L2; at B=1 groups under 8
  // heads leave heavy tiles of the last groups for the end)
  const long long past_t = a.past / 128, heavy = past_t + n_qt + 1;
  const long long per_head = (long long)n_qt * past_t + (long long)n_qt * (n_qt + 1) / 2 + n_qt;
  const long long need = (3 * (long long)grid * heavy + 2 * per_head - 1) / (2 * per_head);
  const long long kv_head_bytes = ((long long)a.past + a.T) * (192 + 128) * 2;
  int G = 1;
  while (G < need && G < 64) G *= 2;
  while (G > 1 && (long long)G * kv_head_bytes > (16ll << 20)) G /= 2;
  // the work counter: an int of the status region (cleared before every call)
  int* work = reinterpret_cast<int*>(st.word) + kWorkCounterWord;
  DevStatus dst{st.word, st.wait_limit_ns};
  return launch_pdl(prefill_attn_tc, dim3(grid), dim3(kThreads), kSmemBytes, stream, tq, tk, tv, a.o, a.T, n_qt,
                    n_items, a.scale * 1.4426950408889634f, a.past, G, work, dst);
}

}  // namespace mla
