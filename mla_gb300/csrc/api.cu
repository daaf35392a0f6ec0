// C ABI of the MLA sublayer: argument checks, workspace layout and the
// launch sequence of each entry point.  Every compute step runs in the
// kernels of this library; nothing here touches tensor data on the host.
#include "common.cuh"
#include "internal.h"
#include "../../include/mla.h"

#include <math.h>
#include <string.h>

namespace mla {
namespace {

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kMaxSmsForSizing = 256;                     // workspace upper bound
constexpr int64_t kMaxTokens = 1 << 24;

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace carve-up.  Offsets are computed identically by the size query
// and by the entry points.
struct Layout {
  size_t status, cs, xn, ca, cq, ckv, kpe, q, o, kscr, vscr, qlat, olat, part_o, part_ml, split, h, plan, pos, total;
  size_t split_bytes;  // split-K partial slots (decode modes), 0 = none
};

// Status region: the device status word at byte 0, the prefill attention's
// work counter at word kWorkCounterWord, split-K counters from byte 256
// (kMaxSplitCounters ints); cleared at the start of every call.
constexpr size_t kStatusRegion = 256 + kMaxSplitCounters * sizeof(int);

Layout make_layout(int mode, int B, int t_or_p, int num_sms, int cap = 0) {
  Layout L{};
  const bool pre = mode == MLA_MODE_PREFILL || mode == MLA_MODE_CHUNK_LATENT;
  // absorbed chunk: one latent decode row per (sequence, new token)
  const bool absorbed = mode == MLA_MODE_CHUNK_ABSORBED;
  const size_t n = (pre || absorbed) ? (size_t)B * t_or_p : (size_t)B;
  const size_t npos = pre ? (size_t)t_or_p : 1;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  L.status = take(kStatusRegion);
  if (mode == MLA_MODE_FOLD) {  // the fold of W_UV into W_o: the status region only
    L.total = off;
    return L;
  }
  if (mode == MLA_MODE_FFN) {  // B * t_or_p rows: RMSNorm(x') and h
    const size_t rows = (size_t)B * t_or_p;
    L.xn = take(rows * MLA_D * 2);
    L.h = take(rows * MLA_FFN_INTER * 2);
    if (rows <= 128) {  // decode-size rows: split-K slots for the down product
      L.split_bytes = split_part_bytes((int)rows);
      L.split = take(L.split_bytes);
    }
    L.total = off;
    return L;
  }
  if (pre) L.cs = take(npos * 32 * sizeof(float2));
  L.xn = take(n * MLA_D * 2);
  L.ca = take(n * 2112 * 4);
  L.cq = take(n * MLA_Q_LORA * 2);
  L.ckv = take(n * MLA_KV_LORA * 2);
  L.kpe = take(n * MLA_QK_ROPE * 2);
  L.q = take(n * MLA_HEADS * MLA_QK * 2);
  L.o = take(n * MLA_HEADS * MLA_V * 2);
  // decode: the RoPE table (one row per sequence, 256 B, written by the
  // latent split and read by the q_b epilogue) lives in the attention output
  // region, which nothing writes before the attention
  if (!pre) L.cs = L.o;
  if (pre) {
    // K/V scratch: the chunk's positions (prefill without caches), or every
    // position up to cap rebuilt from the latent cache (latent chunk)
    const size_t pos = mode == MLA_MODE_CHUNK_LATENT ? (size_t)cap : (size_t)t_or_p;
    L.kscr = take((size_t)B * MLA_HEADS * pos * MLA_QK * 2);
    L.vscr = take((size_t)B * MLA_HEADS * pos * MLA_V * 2);
  } else if (mode == MLA_MODE_DECODE) {
    const int s = decode_splits(B, t_or_p + 1, num_sms);
    L.part_o = take((size_t)B * MLA_HEADS * s * MLA_V * sizeof(float));
    L.part_ml = take((size_t)B * MLA_HEADS * s * sizeof(float2));
  } else {
    // latent rows and the keys of the longest one (absorbed chunk: at most cap)
    const int rows = (int)n;
    const int keys = absorbed ? cap : t_or_p + 1;
    const int g = latent_ctas(rows, keys, num_sms);
    L.qlat = take(n * MLA_HEADS * 576 * 2);
    L.olat = take(n * MLA_HEADS * MLA_KV_LORA * 2);
    L.part_o = take((size_t)2 * g * MLA_HEADS * MLA_KV_LORA * sizeof(float));
    L.part_ml = take((size_t)2 * g * MLA_HEADS * sizeof(float2));
    L.plan = take(latent_plan_ints(rows, g) * sizeof(int));
    if (absorbed) L.pos = take(n * sizeof(int));
  }
  // split-K slots for the small-M projections: decode, and prefill of at
  // most 128 tokens (whose weight-streaming GEMMs have too few tiles to fill
  // the GPU otherwise)
  if (!pre || n <= 128) {
    L.split_bytes = split_part_bytes((int)n);
    L.split = take(L.split_bytes);
  }
  L.total = off;
  return L;
}

// Split-K scratch for the small-M (decode) GEMMs.
void set_split(EpiArgs& ea, void* ws, const Layout& L) {
  if (!L.split_bytes) return;
  ea.part = reinterpret_cast<float*>(static_cast<char*>(ws) + L.split);
  ea.part_bytes = L.split_bytes;
  ea.counters = reinterpret_cast<int*>(static_cast<char*>(ws) + L.status + 256);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int num_sms_of_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return n;
}

int check_weights(const mla_weights_t* w) {
  if (!w) return MLA_ERR_INVALID_ARG;
  const void* ps[] = {w->w_in_norm, w->w_q_a, w->w_q_a_norm, w->w_q_b,
                      w->w_kv_a,    w->w_kv_a_norm, w->w_kv_b, w->w_o};
  for (const void* p : ps) {
    if (!p) return MLA_ERR_INVALID_ARG;
    if (!aligned16(p)) return MLA_ERR_ALIGNMENT;
  }
  return MLA_OK;
}

// x/out may be the same buffer; any other overlap is rejected.
bool bad_overlap(const void* x, const void* out, size_t bytes) {
  if (x == out) return false;
  const char* a = static_cast<const char*>(x);
  const char* b = static_cast<const char*>(out);
  return a < b + bytes && b < a + bytes;
}

struct Params {
  float eps, base, scale;
  float* delta;
  mla_timing_t* timing;
};

Params resolve(const mla_params_t* p) {
  Params r{1e-6f, 10000.f, 1.0f / sqrtf(192.0f), nullptr, nullptr};
  if (p) {
    r.eps = p->eps;
    r.base = p->rope_base;
    r.scale = p->softmax_scale;
    r.delta = p->delta_out;
    r.timing = p->timing;
  }
  return r;
}

bool params_ok(const Params& p) {
  return p.eps >= 0.f && isfinite(p.eps) && p.base > 1.f && isfinite(p.base) && p.scale > 0.f &&
         isfinite(p.scale) && (p.delta == nullptr || aligned16(p.delta));
}

struct Stager {
  mla_timing_t* t;
  cudaStream_t s;
  void start(int id) {
    if (t && t->start[id]) cudaEventRecord(static_cast<cudaEvent_t>(t->start[id]), s);
  }
  void stop(int id) {
    if (t && t->stop[id]) cudaEventRecord(static_cast<cudaEvent_t>(t->stop[id]), s);
  }
};

#define MLA_TRY(expr)                            \
  do {                                           \
    cudaError_t e_ = (expr);                     \
    if (e_ != cudaSuccess) return MLA_ERR_CUDA;  \
  } while (0)

template <class T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// q_b over n_tok rows of c^Q with RoPE on the q^pe columns (RoPE table row
// r % t_mod, or row r with per-row positions); q^pe also into qpe_out if set.
int q_b_stage(const mla_weights_t* w, int n_tok, int t_mod, const int* pos, const mla_weights_fp8_t* f8,
              __nv_bfloat16* qpe_out, void* ws, const Layout& L, const DevStatusHost& st, int sms,
              cudaStream_t stream, int* launches) {
  GemmShape s{n_tok, MLA_HEADS * MLA_QK, MLA_Q_LORA, 1, 0, 0, 0, 0, MLA_HEADS * MLA_QK};
  GemmOperands op{at<__nv_bfloat16>(ws, L.cq), MLA_Q_LORA, n_tok,
                  static_cast<const __nv_bfloat16*>(w->w_q_b), MLA_Q_LORA, MLA_HEADS * MLA_QK,
                  nullptr, 0, 0, false};
  EpiArgs ea{};
  ea.out = at<__nv_bfloat16>(ws, L.q);
  ea.ldo = MLA_HEADS * MLA_QK;
  ea.cs = at<float2>(ws, L.cs);
  ea.t_mod = pos ? n_tok : t_mod;  // per-row positions: one RoPE table row per token
  ea.qpe_out = qpe_out;
  set_split(ea, ws, L);
  if (f8) {
    GemmW8Operands o8{at<__nv_bfloat16>(ws, L.cq), MLA_Q_LORA, n_tok, static_cast<const uint8_t*>(f8->w_q_b),
                      MLA_HEADS * MLA_QK, f8->s_q_b, nullptr, 0, nullptr};
    MLA_TRY(launch_gemm_w8(s, o8, Epi::kQRope, ea, st, sms, stream));
  } else {
    MLA_TRY(launch_gemm(s, op, Epi::kQRope, ea, st, sms, stream));
  }
  *launches += 1;
  return MLA_OK;
}

// Projection front end shared by the three entry points: input RMSNorm, RoPE
// table, A-projection, latent split (+ optional latent cache), q_b + RoPE.
int front_end(const mla_weights_t* w, const Params& p, const void* x, int n_tok, int n_pos, int pos0,
              int t_mod, int t_off, __nv_bfloat16* ckv_cache, __nv_bfloat16* kpe_cache, int cap, void* ws,
              const Layout& L, const DevStatusHost& st, int sms, cudaStream_t stream, Stager& sg,
              int* launches, bool with_q = true, const int* pos = nullptr, int pos_max = 0,
              const mla_weights_fp8_t* f8 = nullptr, __nv_bfloat16* qpe_out = nullptr) {
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);
  (void)n_pos;
  sg.start(MLA_STAGE_INPUT_NORM);
  MLA_TRY(launch_rmsnorm_rows(xb, static_cast<const __nv_bfloat16*>(w->w_in_norm), at<__nv_bfloat16>(ws, L.xn),
                              n_tok, p.eps, stream));
  *launches += 1;
  sg.stop(MLA_STAGE_INPUT_NORM);

  sg.start(MLA_STAGE_A_PROJ);
  {
    GemmShape s{n_tok, 2112, MLA_D, 1, 0, 0, 0, 0, MLA_Q_LORA};
    GemmOperands op{at<__nv_bfloat16>(ws, L.xn), MLA_D, n_tok,
                    static_cast<const __nv_bfloat16*>(w->w_q_a), MLA_D, MLA_Q_LORA,
                    static_cast<const __nv_bfloat16*>(w->w_kv_a), MLA_D, 576, false};
    EpiArgs ea{};
    ea.out_f32 = at<float>(ws, L.ca);
    ea.ldo = 2112;
    set_split(ea, ws, L);
    if (f8) {
      GemmW8Operands o8{at<__nv_bfloat16>(ws, L.xn), MLA_D, n_tok, static_cast<const uint8_t*>(f8->w_q_a),
                        MLA_Q_LORA, f8->s_q_a, static_cast<const uint8_t*>(f8->w_kv_a), 576, f8->s_kv_a};
      MLA_TRY(launch_gemm_w8(s, o8, Epi::kStoreF32, ea, st, sms, stream));
    } else {
      MLA_TRY(launch_gemm(s, op, Epi::kStoreF32, ea, st, sms, stream));
    }
    *launches += 1;
  }
  sg.stop(MLA_STAGE_A_PROJ);

  sg.start(MLA_STAGE_LATENT);
  {
    LatentArgs la{};
    la.ca = at<float>(ws, L.ca);
    la.g_qa = static_cast<const __nv_bfloat16*>(w->w_q_a_norm);
    la.g_kva = static_cast<const __nv_bfloat16*>(w->w_kv_a_norm);
    la.cs = at<float2>(ws, L.cs);
    for (int i = 0; i < 32; ++i) la.inv_freq[i] = pow((double)p.base, -2.0 * i / 64.0);
    la.pos0 = pos0;
    la.cq = at<__nv_bfloat16>(ws, L.cq);
    la.ckv = at<__nv_bfloat16>(ws, L.ckv);
    la.kpe = at<__nv_bfloat16>(ws, L.kpe);
    la.ckv_cache = ckv_cache;
    la.kpe_cache = kpe_cache;
    la.rows = n_tok;
    la.t_mod = t_mod;
    la.t_off = t_off;
    la.cap = cap;
    la.eps = p.eps;
    la.pos = pos;
    la.pos_max = pos_max;
    la.status = st.word;
    MLA_TRY(launch_latent_split(la, stream));
    *launches += 1;
  }
  sg.stop(MLA_STAGE_LATENT);
  if (!with_q) return MLA_OK;

  sg.start(MLA_STAGE_Q_B);
  const int rc = q_b_stage(w, n_tok, t_mod, pos, f8, qpe_out, ws, L, st, sms, stream, launches);
  sg.stop(MLA_STAGE_Q_B);
  return rc;
}

// kv_b over n_tok latent rows ckv [n_tok, 512] (rotary keys kpe [n_tok, 64]):
// K/V of row r at sequence r / t_mod, position t_off + r % t_mod.
int kv_b_rows(const mla_weights_t* w, const __nv_bfloat16* ckv, const __nv_bfloat16* kpe, int n_tok, int t_mod,
              int t_off, __nv_bfloat16* kc, __nv_bfloat16* vc, int cap, void* ws, const Layout& L,
              const DevStatusHost& st, int sms, cudaStream_t stream, int* launches, const int* pos = nullptr,
              int pos_max = 0, const mla_weights_fp8_t* f8 = nullptr, bool split_ok = true) {
  GemmShape s{n_tok, MLA_HEADS * 256, MLA_KV_LORA, 1, 0, 0, 0, 0, MLA_HEADS * 256};
  GemmOperands op{ckv, MLA_KV_LORA, n_tok,
                  static_cast<const __nv_bfloat16*>(w->w_kv_b), MLA_KV_LORA, MLA_HEADS * 256,
                  nullptr, 0, 0, false};
  EpiArgs ea{};
  ea.kc = kc;
  ea.vc = vc;
  ea.kpe = kpe;
  ea.B = (n_tok + t_mod - 1) / t_mod;
  ea.t_mod = t_mod;
  ea.t_off = t_off;
  ea.cap = cap;
  ea.pos = pos;
  ea.pos_max = pos_max;
  if (split_ok) set_split(ea, ws, L);
  if (f8) {
    GemmW8Operands o8{ckv, MLA_KV_LORA, n_tok, static_cast<const uint8_t*>(f8->w_kv_b), MLA_HEADS * 256,
                      f8->s_kv_b, nullptr, 0, nullptr};
    MLA_TRY(launch_gemm_w8(s, o8, Epi::kKVCache, ea, st, sms, stream));
  } else {
    MLA_TRY(launch_gemm(s, op, Epi::kKVCache, ea, st, sms, stream));
  }
  *launches += 1;
  return MLA_OK;
}

int kv_b_stage(const mla_weights_t* w, int n_tok, int t_mod, int t_off, __nv_bfloat16* kc, __nv_bfloat16* vc,
               int cap, void* ws, const Layout& L, const DevStatusHost& st, int sms, cudaStream_t stream,
               int* launches, const int* pos = nullptr, int pos_max = 0,
               const mla_weights_fp8_t* f8 = nullptr, bool split_ok = true) {
  return kv_b_rows(w, at<__nv_bfloat16>(ws, L.ckv), at<__nv_bfloat16>(ws, L.kpe), n_tok, t_mod, t_off, kc, vc, cap,
                   ws, L, st, sms, stream, launches, pos, pos_max, f8, split_ok);
}

// q_b and kv_b read different outputs of the latent split and neither reads
// the other's, so for up to kForkMaxRows rows kv_b runs on a second stream
// beside q_b: with few rows (decode, short prefill) each is a
// weight-streaming launch of 128 CTAs that leaves a sixth of the SMs idle;
// with a few thousand rows each ends on a partly filled last wave of tiles
// (q_b at 2048 rows: 384 CTA-pair tiles over 76 pairs), which the other's
// tiles fill.  Past that the waves are many and full.  One such stream and
// two events per host thread and device, created by the first call that
// uses them (never during a stream capture) and kept for the thread's
// lifetime.
constexpr int kForkMaxRows = 4096;

struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool failed = false;
  ~SideStream() {  // at thread exit (before the runtime's own teardown for the main thread)
    if (s) cudaStreamDestroy(s);
    if (fork) cudaEventDestroy(fork);
    if (join) cudaEventDestroy(join);
  }
};

SideStream* side_stream(cudaStream_t user) {
  constexpr int kMaxDevices = 64;
  thread_local SideStream per_device[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  SideStream& ss = per_device[dev];
  if (!ss.s && !ss.failed) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(user, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
      (void)cudaGetLastError();
      return nullptr;
    }
    if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess ||
        cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess) {
      (void)cudaGetLastError();
      ss.s = nullptr;
      ss.failed = true;  // one stream from then on
    }
  }
  return ss.s ? &ss : nullptr;
}

// kv_b on the side stream (or on `stream` itself when side is null),
// ordered after the work already queued on `stream`; join_side() makes
// `stream` wait for it.
int kv_b_beside(SideStream* side, const mla_weights_t* w, const Params& p, int n_tok, int t_mod, int t_off,
                __nv_bfloat16* kc, __nv_bfloat16* vc, int cap, void* ws, const Layout& L, const DevStatusHost& st,
                int sms, cudaStream_t stream, int* launches, const int* pos, int pos_max,
                const mla_weights_fp8_t* f8) {
  cudaStream_t kvs = stream;
  if (side) {
    MLA_TRY(cudaEventRecord(side->fork, stream));
    MLA_TRY(cudaStreamWaitEvent(side->s, side->fork, 0));
    kvs = side->s;
  }
  Stager sk{p.timing, kvs};
  sk.start(MLA_STAGE_KV_B);
  // no split-K: its partial slots and counters are those of the concurrent q_b
  const int rc = kv_b_stage(w, n_tok, t_mod, t_off, kc, vc, cap, ws, L, st, sms, kvs, launches, pos, pos_max, f8,
                            side == nullptr);
  if (rc) return rc;
  sk.stop(MLA_STAGE_KV_B);
  return MLA_OK;
}

int join_side(SideStream* side, cudaStream_t stream) {
  if (!side) return MLA_OK;
  MLA_TRY(cudaEventRecord(side->join, side->s));
  MLA_TRY(cudaStreamWaitEvent(stream, side->join, 0));
  return MLA_OK;
}

int o_proj_stage(const mla_weights_t* w, const Params& p, const void* x, void* out, int n_tok, void* ws,
                 const Layout& L, const DevStatusHost& st, int sms, cudaStream_t stream, int* launches,
                 const mla_weights_fp8_t* f8 = nullptr) {
  GemmShape s{n_tok, MLA_D, MLA_HEADS * MLA_V, 1, 0, 0, 0, 0, MLA_D};
  GemmOperands op{at<__nv_bfloat16>(ws, L.o), MLA_HEADS * MLA_V, n_tok,
                  static_cast<const __nv_bfloat16*>(w->w_o), MLA_HEADS * MLA_V, MLA_D, nullptr, 0, 0, false};
  EpiArgs ea{};
  ea.out = static_cast<__nv_bfloat16*>(out);
  ea.ldo = MLA_D;
  ea.x = static_cast<const __nv_bfloat16*>(x);
  ea.delta = p.delta;
  set_split(ea, ws, L);
  if (f8) {
    GemmW8Operands o8{at<__nv_bfloat16>(ws, L.o), MLA_HEADS * MLA_V, n_tok, static_cast<const uint8_t*>(f8->w_o),
                      MLA_D, f8->s_o, nullptr, 0, nullptr};
    MLA_TRY(launch_gemm_w8(s, o8, Epi::kResidual, ea, st, sms, stream));
  } else {
    MLA_TRY(launch_gemm(s, op, Epi::kResidual, ea, st, sms, stream));
  }
  *launches += 1;
  return MLA_OK;
}

int common_checks(const mla_weights_t* w, const Params& p, const void* x, const void* out, size_t n_tok,
                  void* ws, size_t ws_bytes, size_t need, bool out_optional = false) {
  int rc = check_weights(w);
  if (rc) return rc;
  if (!x || (!out && !out_optional)) return MLA_ERR_INVALID_ARG;
  if (!ws) return MLA_ERR_WORKSPACE;
  if (!params_ok(p)) return MLA_ERR_INVALID_ARG;
  if (!aligned16(x) || (out && !aligned16(out)) || !aligned16(ws)) return MLA_ERR_ALIGNMENT;
  if (out && bad_overlap(x, out, n_tok * MLA_D * 2)) return MLA_ERR_INVALID_ARG;
  if (ws_bytes < need) return MLA_ERR_WORKSPACE;
  return MLA_OK;
}

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

size_t mla_workspace_size(int mode, int B, int t_or_p, int cap) {
  if (B < 1) return 0;
  if (mode == MLA_MODE_PREFILL) {
    if (t_or_p < 1 || (int64_t)B * t_or_p > kMaxTokens) return 0;
  } else if (mode == MLA_MODE_CHUNK_LATENT) {
    if (t_or_p < 1 || (int64_t)B * t_or_p > kMaxTokens || cap < t_or_p || (int64_t)B * cap > (int64_t)1 << 26)
      return 0;
  } else if (mode == MLA_MODE_DECODE || mode == MLA_MODE_DECODE_LATENT) {
    if (t_or_p < 0 || B > kMaxTokens || t_or_p >= (1 << 24)) return 0;
  } else if (mode == MLA_MODE_FFN) {
    if (t_or_p < 1 || (int64_t)B * t_or_p > kMaxTokens) return 0;
  } else if (mode == MLA_MODE_CHUNK_ABSORBED) {
    if (t_or_p < 1 || (int64_t)B * t_or_p > kMaxTokens || cap < t_or_p || cap >= (1 << 24)) return 0;
  } else if (mode == MLA_MODE_FOLD) {
  } else {
    return 0;
  }
  return make_layout(mode, B, t_or_p, kMaxSmsForSizing, cap).total;
}

const char* mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "MLA_OK";
    case MLA_ERR_INVALID_ARG: return "MLA_ERR_INVALID_ARG: invalid argument";
    case MLA_ERR_ALIGNMENT: return "MLA_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case MLA_ERR_WORKSPACE: return "MLA_ERR_WORKSPACE: workspace missing or too small";
    case MLA_ERR_UNSUPPORTED: return "MLA_ERR_UNSUPPORTED: size or mode not supported";
    case MLA_ERR_CUDA: return "MLA_ERR_CUDA: CUDA call or kernel launch failed";
    case MLA_ERR_TIMEOUT: return "MLA_ERR_TIMEOUT: a bounded device wait gave up";
    default: return "unknown MLA status";
  }
}

int mla_device_status(const void* workspace, void* stream) {
  if (!workspace) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MLA_ERR_CUDA;
  if (word & kStatusTimeout) return MLA_ERR_TIMEOUT;
  return (word & kStatusBadLength) ? MLA_ERR_INVALID_ARG : MLA_OK;
}

}  // extern "C"

namespace {

// Prefill of T tokens per sequence at positions P0..P0+T-1; P0 > 0 (chunked
// prefill) attends to the P0 cached keys before the chunk's own.  With
// latent_past the past is the latent cache: after the chunk's latent rows
// are written there, keys and values of positions 0..P0+T-1 are rebuilt
// from it into workspace scratch (one kv_b product per sequence).
int prefill_impl(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T, int P0,
                 void* out, void* k_cache, void* v_cache, void* ckv_cache, void* kpe_cache, int cap,
                 void* workspace, size_t workspace_bytes, void* stream, bool latent_past = false) {
  const Params p = resolve(params);
  if (B < 1 || T < 1 || P0 < 0 || (int64_t)B * T > kMaxTokens) return MLA_ERR_INVALID_ARG;
  if ((k_cache == nullptr) != (v_cache == nullptr)) return MLA_ERR_INVALID_ARG;
  if ((ckv_cache == nullptr) != (kpe_cache == nullptr)) return MLA_ERR_INVALID_ARG;
  if ((k_cache || ckv_cache) && (int64_t)P0 + T > cap) return MLA_ERR_INVALID_ARG;
  if (latent_past && (k_cache || !ckv_cache || !out || (int64_t)B * cap > (int64_t)1 << 26))
    return MLA_ERR_INVALID_ARG;
  if (!latent_past && P0 > 0 && (!k_cache || !out)) return MLA_ERR_INVALID_ARG;
  const int mode = latent_past ? MLA_MODE_CHUNK_LATENT : MLA_MODE_PREFILL;
  for (const void* c : {(const void*)k_cache, (const void*)v_cache, (const void*)ckv_cache, (const void*)kpe_cache})
    if (c && !aligned16(c)) return MLA_ERR_ALIGNMENT;
  const size_t n_tok = (size_t)B * T;
  const bool cache_only = (out == nullptr);
  if (cache_only && !k_cache && !ckv_cache) return MLA_ERR_INVALID_ARG;
  int rc = common_checks(w, p, x, out, n_tok, workspace, workspace_bytes,
                         make_layout(mode, B, T, kMaxSmsForSizing, cap).total, true);
  if (rc) return rc;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MLA_ERR_CUDA;
  const Layout L = make_layout(mode, B, T, sms, cap);

  cudaStream_t stream_ = static_cast<cudaStream_t>(stream);
  const DevStatusHost st{at<uint32_t>(workspace, L.status), kDefaultWaitLimitNs};
  Stager sg{p.timing, stream_};
  int launches = 0;
  if (cudaMemsetAsync(st.word, 0, kStatusRegion, stream_) != cudaSuccess) return MLA_ERR_CUDA;

  SideStream* side = (n_tok <= (size_t)kForkMaxRows && !cache_only && !latent_past) ? side_stream(stream_) : nullptr;
  rc = front_end(w, p, x, (int)n_tok, T, P0, T, P0, static_cast<__nv_bfloat16*>(ckv_cache),
                 static_cast<__nv_bfloat16*>(kpe_cache), cap, workspace, L, st, sms, stream_, sg, &launches,
                 !cache_only && side == nullptr);
  if (rc) return rc;
  if (cache_only && !k_cache) {
    if (p.timing) p.timing->n_launches = launches;
    return MLA_OK;
  }

  __nv_bfloat16* kc = k_cache ? static_cast<__nv_bfloat16*>(k_cache) : at<__nv_bfloat16>(workspace, L.kscr);
  __nv_bfloat16* vc = v_cache ? static_cast<__nv_bfloat16*>(v_cache) : at<__nv_bfloat16>(workspace, L.vscr);
  const int kcap = (k_cache || latent_past) ? cap : T;
  if (side) {  // kv_b beside q_b
    rc = kv_b_beside(side, w, p, (int)n_tok, T, P0, kc, vc, kcap, workspace, L, st, sms, stream_, &launches,
                     nullptr, 0, nullptr);
    if (rc) return rc;
    sg.start(MLA_STAGE_Q_B);
    rc = q_b_stage(w, (int)n_tok, T, nullptr, nullptr, nullptr, workspace, L, st, sms, stream_, &launches);
    if (rc) return rc;
    sg.stop(MLA_STAGE_Q_B);
    rc = join_side(side, stream_);
    if (rc) return rc;
  } else {
    sg.start(MLA_STAGE_KV_B);
    if (latent_past) {
      const __nv_bfloat16* ckv = static_cast<const __nv_bfloat16*>(ckv_cache);
      const __nv_bfloat16* kpe = static_cast<const __nv_bfloat16*>(kpe_cache);
      for (int b = 0; b < B && rc == MLA_OK; ++b)
        rc = kv_b_rows(w, ckv + (size_t)b * cap * MLA_KV_LORA, kpe + (size_t)b * cap * MLA_QK_ROPE, P0 + T, P0 + T,
                       0, kc + (size_t)b * MLA_HEADS * cap * MLA_QK, vc + (size_t)b * MLA_HEADS * cap * MLA_V, cap,
                       workspace, L, st, sms, stream_, &launches);
    } else {
      rc = kv_b_stage(w, (int)n_tok, T, P0, kc, vc, kcap, workspace, L, st, sms, stream_, &launches);
    }
    if (rc) return rc;
    sg.stop(MLA_STAGE_KV_B);
  }
  if (cache_only) {
    if (p.timing) p.timing->n_launches = launches;
    return MLA_OK;
  }

  sg.start(MLA_STAGE_ATTN);
  {
    PrefillAttnArgs a{at<__nv_bfloat16>(workspace, L.q), kc, vc, at<__nv_bfloat16>(workspace, L.o), B, T, kcap,
                      p.scale, P0};
    if (launch_prefill_attention(a, st, sms, stream_) != cudaSuccess) return MLA_ERR_CUDA;
    launches += 1;
  }
  sg.stop(MLA_STAGE_ATTN);

  sg.start(MLA_STAGE_O_PROJ);
  rc = o_proj_stage(w, p, x, out, (int)n_tok, workspace, L, st, sms, stream_, &launches);
  if (rc) return rc;
  sg.stop(MLA_STAGE_O_PROJ);
  if (p.timing) p.timing->n_launches = launches;
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_prefill(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T, void* out,
                void* k_cache, void* v_cache, void* ckv_cache, void* kpe_cache, int cap, void* workspace,
                size_t workspace_bytes, void* stream) {
  return prefill_impl(w, params, x, B, T, 0, out, k_cache, v_cache, ckv_cache, kpe_cache, cap, workspace,
                      workspace_bytes, stream);
}

int mla_prefill_chunk(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T, int P0,
                      void* out, void* k_cache, void* v_cache, void* ckv_cache, void* kpe_cache, int cap,
                      void* workspace, size_t workspace_bytes, void* stream) {
  if (!k_cache || !v_cache || !out) return MLA_ERR_INVALID_ARG;
  return prefill_impl(w, params, x, B, T, P0, out, k_cache, v_cache, ckv_cache, kpe_cache, cap, workspace,
                      workspace_bytes, stream);
}

int mla_prefill_chunk_latent(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T,
                             int P0, void* out, void* ckv_cache, void* kpe_cache, int cap, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!ckv_cache || !kpe_cache || !out) return MLA_ERR_INVALID_ARG;
  return prefill_impl(w, params, x, B, T, P0, out, nullptr, nullptr, ckv_cache, kpe_cache, cap, workspace,
                      workspace_bytes, stream, true);
}

}  // extern "C"

namespace {

// One decode step, rebuilt cache.  pos = null: every sequence at position P;
// else sequence b at position pos[b] (device array), P = an upper bound.
int decode_impl(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int P, const int* pos,
                void* k_cache, void* v_cache, int cap, void* out, void* workspace, size_t workspace_bytes,
                void* stream, const mla_weights_fp8_t* f8 = nullptr) {
  const Params p = resolve(params);
  if (B < 1 || B > kMaxTokens || P < 0 || P >= (1 << 24)) return MLA_ERR_INVALID_ARG;
  if (!k_cache || !v_cache || cap < P + 1) return MLA_ERR_INVALID_ARG;
  if (pos && (reinterpret_cast<uintptr_t>(pos) & 3)) return MLA_ERR_ALIGNMENT;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return MLA_ERR_ALIGNMENT;
  int rc = common_checks(w, p, x, out, (size_t)B, workspace, workspace_bytes,
                         make_layout(MLA_MODE_DECODE, B, P, kMaxSmsForSizing).total);
  if (rc) return rc;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MLA_ERR_CUDA;
  const Layout L = make_layout(MLA_MODE_DECODE, B, P, sms);

  cudaStream_t stream_ = static_cast<cudaStream_t>(stream);
  const DevStatusHost st{at<uint32_t>(workspace, L.status), kDefaultWaitLimitNs};
  Stager sg{p.timing, stream_};
  int launches = 0;
  if (cudaMemsetAsync(st.word, 0, kStatusRegion, stream_) != cudaSuccess) return MLA_ERR_CUDA;
  SideStream* side = B <= kForkMaxRows ? side_stream(stream_) : nullptr;
  rc = front_end(w, p, x, B, 1, P, 1, P, nullptr, nullptr, cap, workspace, L, st, sms, stream_, sg, &launches,
                 side == nullptr, pos, P, f8);
  if (rc) return rc;

  __nv_bfloat16* kc = static_cast<__nv_bfloat16*>(k_cache);
  __nv_bfloat16* vc = static_cast<__nv_bfloat16*>(v_cache);
  if (side) {  // kv_b beside q_b
    rc = kv_b_beside(side, w, p, B, 1, P, kc, vc, cap, workspace, L, st, sms, stream_, &launches, pos, P, f8);
    if (rc) return rc;
    sg.start(MLA_STAGE_Q_B);
    rc = q_b_stage(w, B, 1, pos, f8, nullptr, workspace, L, st, sms, stream_, &launches);
    if (rc) return rc;
    sg.stop(MLA_STAGE_Q_B);
    rc = join_side(side, stream_);
    if (rc) return rc;
  } else {
    sg.start(MLA_STAGE_KV_B);
    rc = kv_b_stage(w, B, 1, P, kc, vc, cap, workspace, L, st, sms, stream_, &launches, pos, P, f8);
    if (rc) return rc;
    sg.stop(MLA_STAGE_KV_B);
  }

  sg.start(MLA_STAGE_ATTN);
  {
    DecodeAttnArgs a{};
    a.q = at<__nv_bfloat16>(workspace, L.q);
    a.k = kc;
    a.v = vc;
    a.o = at<__nv_bfloat16>(workspace, L.o);
    a.part_o = at<float>(workspace, L.part_o);
    a.part_ml = at<float2>(workspace, L.part_ml);
    a.B = B;
    a.L = P + 1;
    a.cap = cap;
    a.splits = decode_splits(B, P + 1, sms);
    a.scale = p.scale;
    a.lens_pos = pos;
    if (launch_decode_attention(a, st, stream_, &launches) != cudaSuccess) return MLA_ERR_CUDA;
  }
  sg.stop(MLA_STAGE_ATTN);

  sg.start(MLA_STAGE_O_PROJ);
  rc = o_proj_stage(w, p, x, out, B, workspace, L, st, sms, stream_, &launches, f8);
  if (rc) return rc;
  sg.stop(MLA_STAGE_O_PROJ);
  if (p.timing) p.timing->n_launches = launches;
  return MLA_OK;
}

// One decode step, latent cache; pos as decode_impl.
// W_UK absorption, latent attention, W_UV and o_proj for n latent rows whose
// RoPE'd queries front_end has written: row i attends to keys 0..pos[i] (or
// 0..P_max without pos) of cache plane i / kv_div.
int latent_tail(const mla_weights_t* w, const Params& p, const void* x, void* out, int n, int P_max, const int* pos,
                int kv_div, const __nv_bfloat16* ckv_cache, const __nv_bfloat16* kpe_cache, int cap, void* workspace,
                const Layout& L, const DevStatusHost& st, int sms, cudaStream_t stream_, Stager& sg, int* launches,
                bool qpe_in_epilogue, const __nv_bfloat16* w_fold = nullptr) {
  const __nv_bfloat16* wkvb = static_cast<const __nv_bfloat16*>(w->w_kv_b);
  sg.start(MLA_STAGE_ABSORB_Q);
  {
    // q_lat[i, h, 0:512] = sum_j q_nope[i, h, j] W_kv_b[h*256 + j, :]  (B operand [K=j, N=c], N contiguous)
    GemmShape s{n, MLA_KV_LORA, MLA_QK_NOPE, MLA_HEADS, 0, MLA_QK, 0, 256, MLA_KV_LORA};
    GemmOperands op{at<__nv_bfloat16>(workspace, L.q), MLA_HEADS * MLA_QK, n, wkvb, MLA_KV_LORA, MLA_HEADS * 256,
                    nullptr, 0, 0, true};
    EpiArgs ea{};
    ea.out = at<__nv_bfloat16>(workspace, L.qlat);
    ea.ldo = MLA_HEADS * 576;
    ea.c_col0 = 0;
    ea.c_col_step = 576;
    set_split(ea, workspace, L);
    MLA_TRY(launch_gemm(s, op, Epi::kStoreBf16, ea, st, sms, stream_));
    *launches += 1;
    if (!qpe_in_epilogue) {
      MLA_TRY(launch_copy_qpe(at<__nv_bfloat16>(workspace, L.q), at<__nv_bfloat16>(workspace, L.qlat), n, stream_));
      *launches += 1;
    }
  }
  sg.stop(MLA_STAGE_ABSORB_Q);

  sg.start(MLA_STAGE_ATTN);
  {
    LatentAttnArgs a{};
    a.qlat = at<__nv_bfloat16>(workspace, L.qlat);
    a.ckv = ckv_cache;
    a.kpe = kpe_cache;
    a.olat = at<__nv_bfloat16>(workspace, L.olat);
    a.part_o = at<float>(workspace, L.part_o);
    a.part_ml = at<float2>(workspace, L.part_ml);
    a.B = n;
    a.L = P_max + 1;
    a.cap = cap;
    a.ctas = latent_ctas(n, P_max + 1, sms);
    a.scale = p.scale;
    a.pos = pos;
    a.plan = at<int>(workspace, L.plan);
    a.kv_div = kv_div;
    if (launch_latent_attention(a, st, stream_, launches) != cudaSuccess) return MLA_ERR_CUDA;
  }
  sg.stop(MLA_STAGE_ATTN);

  if (w_fold) {
    // W_UV folded into o_proj: out = x + o_lat [n, 64*512] W_fold^T, one GEMM
    sg.start(MLA_STAGE_O_PROJ);
    GemmShape s{n, MLA_D, MLA_HEADS * MLA_KV_LORA, 1, 0, 0, 0, 0, MLA_D};
    GemmOperands op{at<__nv_bfloat16>(workspace, L.olat), MLA_HEADS * MLA_KV_LORA, n, w_fold,
                    MLA_HEADS * MLA_KV_LORA, MLA_D, nullptr, 0, 0, false};
    EpiArgs ea{};
    ea.out = static_cast<__nv_bfloat16*>(out);
    ea.ldo = MLA_D;
    ea.x = static_cast<const __nv_bfloat16*>(x);
    ea.delta = p.delta;
    set_split(ea, workspace, L);
    MLA_TRY(launch_gemm(s, op, Epi::kResidual, ea, st, sms, stream_));
    *launches += 1;
    sg.stop(MLA_STAGE_O_PROJ);
    return MLA_OK;
  }

  sg.start(MLA_STAGE_ABSORB_O);
  {
    // o[i, h*128 + d] = sum_c o_lat[i, h, c] W_kv_b[h*256 + 128 + d, c]
    GemmShape s{n, MLA_V, MLA_KV_LORA, MLA_HEADS, 0, MLA_KV_LORA, 128, 256, MLA_V};
    GemmOperands op{at<__nv_bfloat16>(workspace, L.olat), MLA_HEADS * MLA_KV_LORA, n, wkvb, MLA_KV_LORA,
                    MLA_HEADS * 256, nullptr, 0, 0, false};
    EpiArgs ea{};
    ea.out = at<__nv_bfloat16>(workspace, L.o);
    ea.ldo = MLA_HEADS * MLA_V;
    ea.c_col0 = 0;
    ea.c_col_step = MLA_V;
    set_split(ea, workspace, L);
    MLA_TRY(launch_gemm(s, op, Epi::kStoreBf16, ea, st, sms, stream_));
    *launches += 1;
  }
  sg.stop(MLA_STAGE_ABSORB_O);

  sg.start(MLA_STAGE_O_PROJ);
  int rc = o_proj_stage(w, p, x, out, n, workspace, L, st, sms, stream_, launches);
  if (rc) return rc;
  sg.stop(MLA_STAGE_O_PROJ);
  return MLA_OK;
}

int decode_latent_impl(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int P,
                       const int* pos, void* ckv_cache, void* kpe_cache, int cap, void* out, void* workspace,
                       size_t workspace_bytes, void* stream, const void* w_fold = nullptr) {
  const Params p = resolve(params);
  if (B < 1 || B > kMaxTokens || P < 0 || P >= (1 << 24)) return MLA_ERR_INVALID_ARG;
  if (!ckv_cache || !kpe_cache || cap < P + 1) return MLA_ERR_INVALID_ARG;
  if (pos && (reinterpret_cast<uintptr_t>(pos) & 3)) return MLA_ERR_ALIGNMENT;
  if (!aligned16(ckv_cache) || !aligned16(kpe_cache) || (w_fold && !aligned16(w_fold))) return MLA_ERR_ALIGNMENT;
  int rc = common_checks(w, p, x, out, (size_t)B, workspace, workspace_bytes,
                         make_layout(MLA_MODE_DECODE_LATENT, B, P, kMaxSmsForSizing).total);
  if (rc) return rc;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MLA_ERR_CUDA;
  const Layout L = make_layout(MLA_MODE_DECODE_LATENT, B, P, sms);

  cudaStream_t stream_ = static_cast<cudaStream_t>(stream);
  const DevStatusHost st{at<uint32_t>(workspace, L.status), kDefaultWaitLimitNs};
  Stager sg{p.timing, stream_};
  int launches = 0;
  if (cudaMemsetAsync(st.word, 0, kStatusRegion, stream_) != cudaSuccess) return MLA_ERR_CUDA;
  // up to 128 rows the q_b epilogue (register stores) also writes the rotated
  // q^pe into q_lat; more rows take the TMA-store epilogue and a copy kernel
  const bool qpe_in_epilogue = B <= 128;
  rc = front_end(w, p, x, B, 1, P, 1, P, static_cast<__nv_bfloat16*>(ckv_cache),
                 static_cast<__nv_bfloat16*>(kpe_cache), cap, workspace, L, st, sms, stream_, sg, &launches, true,
                 pos, P, nullptr, qpe_in_epilogue ? at<__nv_bfloat16>(workspace, L.qlat) : nullptr);
  if (rc) return rc;
  rc = latent_tail(w, p, x, out, B, P, pos, 1, static_cast<const __nv_bfloat16*>(ckv_cache),
                   static_cast<const __nv_bfloat16*>(kpe_cache), cap, workspace, L, st, sms, stream_, sg, &launches,
                   qpe_in_epilogue, static_cast<const __nv_bfloat16*>(w_fold));
  if (rc) return rc;
  if (p.timing) p.timing->n_launches = launches;
  return MLA_OK;
}

// Absorbed chunked prefill: the chunk's B*T tokens through the front end as
// a chunk (RoPE positions and latent cache rows P0 + t), then one latent
// decode row per token, row b*T + t reading plane b up to position P0 + t.
int chunk_absorbed_impl(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T, int P0,
                        void* out, void* ckv_cache, void* kpe_cache, int cap, void* workspace,
                        size_t workspace_bytes, void* stream) {
  const Params p = resolve(params);
  if (B < 1 || T < 1 || (int64_t)B * T > kMaxTokens || P0 < 0 || cap >= (1 << 24) || (int64_t)P0 + T > cap)
    return MLA_ERR_INVALID_ARG;
  if (!ckv_cache || !kpe_cache) return MLA_ERR_INVALID_ARG;
  if (!aligned16(ckv_cache) || !aligned16(kpe_cache)) return MLA_ERR_ALIGNMENT;
  const int n = B * T;
  int rc = common_checks(w, p, x, out, (size_t)n, workspace, workspace_bytes,
                         make_layout(MLA_MODE_CHUNK_ABSORBED, B, T, kMaxSmsForSizing, cap).total);
  if (rc) return rc;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MLA_ERR_CUDA;
  const Layout L = make_layout(MLA_MODE_CHUNK_ABSORBED, B, T, sms, cap);

  cudaStream_t stream_ = static_cast<cudaStream_t>(stream);
  const DevStatusHost st{at<uint32_t>(workspace, L.status), kDefaultWaitLimitNs};
  Stager sg{p.timing, stream_};
  int launches = 0;
  if (cudaMemsetAsync(st.word, 0, kStatusRegion, stream_) != cudaSuccess) return MLA_ERR_CUDA;
  int* pos = at<int>(workspace, L.pos);
  MLA_TRY(launch_chunk_positions(pos, n, T, P0, stream_));
  launches += 1;
  const bool qpe_in_epilogue = n <= 128;
  rc = front_end(w, p, x, n, T, P0, T, P0, static_cast<__nv_bfloat16*>(ckv_cache),
                 static_cast<__nv_bfloat16*>(kpe_cache), cap, workspace, L, st, sms, stream_, sg, &launches, true,
                 nullptr, 0, nullptr, qpe_in_epilogue ? at<__nv_bfloat16>(workspace, L.qlat) : nullptr);
  if (rc) return rc;
  rc = latent_tail(w, p, x, out, n, P0 + T - 1, pos, T, static_cast<const __nv_bfloat16*>(ckv_cache),
                   static_cast<const __nv_bfloat16*>(kpe_cache), cap, workspace, L, st, sms, stream_, sg, &launches,
                   qpe_in_epilogue);
  if (rc) return rc;
  if (p.timing) p.timing->n_launches = launches;
  return MLA_OK;
}

}  // namespace

extern "C" {

int mla_decode(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int P, void* k_cache,
               void* v_cache, int cap, void* out, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(w, params, x, B, P, nullptr, k_cache, v_cache, cap, out, workspace, workspace_bytes, stream);
}

int mla_decode_fp8(const mla_weights_fp8_t* w, const mla_params_t* params, const void* x, int B, int P,
                   void* k_cache, void* v_cache, int cap, void* out, void* workspace, size_t workspace_bytes,
                   void* stream) {
  if (!w) return MLA_ERR_INVALID_ARG;
  for (const void* q : {(const void*)w->s_q_a, (const void*)w->s_q_b, (const void*)w->s_kv_a, (const void*)w->s_kv_b,
                        (const void*)w->s_o}) {
    if (!q) return MLA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(q) & 3) return MLA_ERR_ALIGNMENT;
  }
  // the gains and code matrices in the bf16 struct's places (checked there; the
  // projections read the codes and scales through w)
  const mla_weights_t view{w->w_in_norm, w->w_q_a, w->w_q_a_norm, w->w_q_b,
                           w->w_kv_a,    w->w_kv_a_norm, w->w_kv_b, w->w_o};
  return decode_impl(&view, params, x, B, P, nullptr, k_cache, v_cache, cap, out, workspace, workspace_bytes, stream,
                     w);
}

int mla_quantize_fp8(const void* w_bf16, int rows, int cols, void* codes, float* scales, void* stream) {
  if (!w_bf16 || !codes || !scales || rows < 1 || cols < 1 || cols % 128) return MLA_ERR_INVALID_ARG;
  if (!aligned16(w_bf16) || !aligned16(codes) || (reinterpret_cast<uintptr_t>(scales) & 3)) return MLA_ERR_ALIGNMENT;
  if (launch_fp8_quantize(static_cast<const __nv_bfloat16*>(w_bf16), rows, cols, static_cast<uint8_t*>(codes), scales,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

int mla_decode_varlen(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, const int* P,
                      int P_max, void* k_cache, void* v_cache, int cap, void* out, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!P) return MLA_ERR_INVALID_ARG;
  return decode_impl(w, params, x, B, P_max, P, k_cache, v_cache, cap, out, workspace, workspace_bytes, stream);
}

int mla_decode_latent(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int P,
                      void* ckv_cache, void* kpe_cache, int cap, void* out, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return decode_latent_impl(w, params, x, B, P, nullptr, ckv_cache, kpe_cache, cap, out, workspace,
                            workspace_bytes, stream);
}

int mla_decode_latent_varlen(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, const int* P,
                             int P_max, void* ckv_cache, void* kpe_cache, int cap, void* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!P) return MLA_ERR_INVALID_ARG;
  return decode_latent_impl(w, params, x, B, P_max, P, ckv_cache, kpe_cache, cap, out, workspace, workspace_bytes,
                            stream);
}

int mla_fold_wuv_into_wo(const mla_weights_t* w, void* w_fold, void* workspace, size_t workspace_bytes,
                         void* stream) {
  int rc = check_weights(w);
  if (rc) return rc;
  if (!w_fold) return MLA_ERR_INVALID_ARG;
  if (!workspace) return MLA_ERR_WORKSPACE;
  if (!aligned16(w_fold) || !aligned16(workspace)) return MLA_ERR_ALIGNMENT;
  const Layout L = make_layout(MLA_MODE_FOLD, 1, 1, kMaxSmsForSizing);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MLA_ERR_CUDA;
  cudaStream_t stream_ = static_cast<cudaStream_t>(stream);
  const DevStatusHost st{at<uint32_t>(workspace, L.status), kDefaultWaitLimitNs};
  if (cudaMemsetAsync(st.word, 0, kStatusRegion, stream_) != cudaSuccess) return MLA_ERR_CUDA;
  // per head h: W_fold[:, h*512 .. +512] = W_o[:, h*128 .. +128] W_kv_b[h*256 + 128 .. +128, :]
  // (A = W_o's head columns, B = the head's W_UV rows as [K = 128, N = 512], N contiguous)
  GemmShape s{MLA_D, MLA_KV_LORA, MLA_V, MLA_HEADS, 0, MLA_V, MLA_QK_NOPE, 256, MLA_KV_LORA};
  GemmOperands op{static_cast<const __nv_bfloat16*>(w->w_o), MLA_HEADS * MLA_V, MLA_D,
                  static_cast<const __nv_bfloat16*>(w->w_kv_b), MLA_KV_LORA, MLA_HEADS * 256, nullptr, 0, 0, true};
  EpiArgs ea{};
  ea.out = static_cast<__nv_bfloat16*>(w_fold);
  ea.ldo = MLA_HEADS * MLA_KV_LORA;
  ea.c_col0 = 0;
  ea.c_col_step = MLA_KV_LORA;
  return launch_gemm(s, op, Epi::kStoreBf16, ea, st, sms, stream_) == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

int mla_decode_latent_folded(const mla_weights_t* w, const void* w_fold, const mla_params_t* params, const void* x,
                             int B, int P, void* ckv_cache, void* kpe_cache, int cap, void* out, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (!w_fold) return MLA_ERR_INVALID_ARG;
  return decode_latent_impl(w, params, x, B, P, nullptr, ckv_cache, kpe_cache, cap, out, workspace,
                            workspace_bytes, stream, w_fold);
}

int mla_prefill_chunk_absorbed(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T,
                               int P0, void* out, void* ckv_cache, void* kpe_cache, int cap, void* workspace,
                               size_t workspace_bytes, void* stream) {
  if (!out) return MLA_ERR_INVALID_ARG;
  return chunk_absorbed_impl(w, params, x, B, T, P0, out, ckv_cache, kpe_cache, cap, workspace, workspace_bytes,
                             stream);
}

int mla_ffn(const mla_ffn_weights_t* w, const mla_params_t* params, const void* x, int n_tok, void* out,
            void* workspace, size_t workspace_bytes, void* stream) {
  const Params p = resolve(params);
  if (!w || !x || !out || n_tok < 1 || (int64_t)n_tok > kMaxTokens) return MLA_ERR_INVALID_ARG;
  for (const void* q : {w->w_post_norm, w->w_1, w->w_3, w->w_2})
    if (!q) return MLA_ERR_INVALID_ARG;
  for (const void* q : {w->w_post_norm, w->w_1, w->w_3, w->w_2, x, (const void*)out})
    if (!aligned16(q)) return MLA_ERR_ALIGNMENT;
  if (!workspace) return MLA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MLA_ERR_ALIGNMENT;
  if (!params_ok(p)) return MLA_ERR_INVALID_ARG;
  if (bad_overlap(x, out, (size_t)n_tok * MLA_D * 2)) return MLA_ERR_INVALID_ARG;
  const Layout L = make_layout(MLA_MODE_FFN, 1, n_tok, kMaxSmsForSizing);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;
  const int sms = num_sms_of_current_device();
  if (sms <= 0) return MLA_ERR_CUDA;

  cudaStream_t stream_ = static_cast<cudaStream_t>(stream);
  const DevStatusHost st{at<uint32_t>(workspace, L.status), kDefaultWaitLimitNs};
  Stager sg{p.timing, stream_};
  int launches = 0;
  if (cudaMemsetAsync(st.word, 0, kStatusRegion, stream_) != cudaSuccess) return MLA_ERR_CUDA;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(x);

  // x_ffn = RMSNorm(x')
  sg.start(MLA_STAGE_FFN_NORM);
  MLA_TRY(launch_rmsnorm_rows(xb, static_cast<const __nv_bfloat16*>(w->w_post_norm), at<__nv_bfloat16>(workspace, L.xn),
                              n_tok, p.eps, stream_));
  launches += 1;
  sg.stop(MLA_STAGE_FFN_NORM);

  // h = SiLU(x_ffn W_1) (.) (x_ffn W_3): one product over [W_1 ; W_3], the
  // gate and up columns of each intermediate index in the same tile
  sg.start(MLA_STAGE_FFN_GATE_UP);
  {
    GemmShape s{n_tok, 2 * MLA_FFN_INTER, MLA_D, 1, 0, 0, 0, 0, MLA_FFN_INTER};
    GemmOperands op{at<__nv_bfloat16>(workspace, L.xn), MLA_D, n_tok,
                    static_cast<const __nv_bfloat16*>(w->w_1), MLA_D, MLA_FFN_INTER,
                    static_cast<const __nv_bfloat16*>(w->w_3), MLA_D, MLA_FFN_INTER, false};
    EpiArgs ea{};
    ea.out = at<__nv_bfloat16>(workspace, L.h);
    ea.ldo = MLA_FFN_INTER;
    MLA_TRY(launch_gemm(s, op, Epi::kSwiGLU, ea, st, sms, stream_));
    launches += 1;
  }
  sg.stop(MLA_STAGE_FFN_GATE_UP);

  // x_{n+1} = x' + h W_2
  sg.start(MLA_STAGE_FFN_DOWN);
  {
    GemmShape s{n_tok, MLA_D, MLA_FFN_INTER, 1, 0, 0, 0, 0, MLA_D};
    GemmOperands op{at<__nv_bfloat16>(workspace, L.h), MLA_FFN_INTER, n_tok,
                    static_cast<const __nv_bfloat16*>(w->w_2), MLA_FFN_INTER, MLA_D, nullptr, 0, 0, false};
    EpiArgs ea{};
    ea.out = static_cast<__nv_bfloat16*>(out);
    ea.ldo = MLA_D;
    ea.x = xb;
    ea.delta = p.delta;
    set_split(ea, workspace, L);
    MLA_TRY(launch_gemm(s, op, Epi::kResidual, ea, st, sms, stream_));
    launches += 1;
  }
  sg.stop(MLA_STAGE_FFN_DOWN);
  if (p.timing) p.timing->n_launches = launches;
  return MLA_OK;
}

}  // extern "C"
