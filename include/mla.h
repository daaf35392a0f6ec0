/*
 * mla.h -- C ABI of the GB300 (sm_103a) multi-head latent attention sublayer.
 *
 * The operation is the MLA sublayer of a Kimi K2 / DeepSeek-V3 style block:
 *   Kimi K2 "Dense transformer block" page, equation list (x_attn = RMSNorm(x),
 *     c^Q, c^KV, q^C/q^pe, k^C/k^pe, v, RoPE, Q = [Q^C; Q^R], K_i = [K^C_i; k^R],
 *     x' = x + Delta_attn);
 *   "Mix and project" page (decode, P = 1,000), code excerpt: scores scaled and
 *     masked, float32 softmax, P.V, heads merged head-major, o_proj;
 *   "Key-value compression" page: kv_a_proj_with_mqa gives a 512-wide latent
 *     and one 64-wide rotary key (576 features, split after the product); the
 *     latent alone is normalised; 576 cached values per position for the
 *     latent form versus 20,480 for rebuilt per-head keys and values.
 *
 * Fixed sizes (checked against the pages' 101,124,096 MLA parameters):
 *   d = 7168, H = 64 heads, q_lora = 1536, kv_lora = 512,
 *   qk = 128 (nope) + 64 (rope, 32 pairs) = 192, v = 128, no biases.
 * Other sizes are not supported.
 *
 * Conventions for every entry point
 *   - All tensors are bf16, row-major, in device memory, owned by the caller.
 *     Weights use the nn.Linear layout [out, in].
 *   - Every pointer must be 16-byte aligned (MLA_ERR_ALIGNMENT otherwise).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream).  The library never synchronises and allocates no
 *     device memory: all scratch lives in the caller's workspace, sized by
 *     mla_workspace_size().  A workspace must not be shared by calls that may
 *     run concurrently.
 *   - Decode and prefill calls of at most 4096 rows run the kv_b product on a
 *     second stream of the library's own, beside q_b (neither fills the GPU
 *     alone, or its last wave of tiles), forked from and joined back into
 *     `stream` with events: the call is still ordered on `stream` as a whole.
 *     That stream and its two events are created by the first such call of
 *     each host thread on each device (not during a stream capture: a call
 *     captured before any uncaptured call of its thread stays on `stream`)
 *     and destroyed when the thread exits.
 *   - Positions are implicit: prefill tokens sit at positions 0..T-1 with a
 *     causal mask (key j visible to query i iff j <= i); a decode token sits
 *     at position P and attends to all P + 1 keys.
 *   - RoPE is rotate-half on pairs (i, i+32), theta_i = rope_base^(-2i/64).
 *   - `out` may be the same buffer as `x` (in-place residual); any other
 *     overlap between out and x is rejected.
 *   - Arguments are checked on the host before anything is enqueued; a
 *     failed check returns a negative status and enqueues nothing.  This
 *     mirrors the shape checks (ValueError / assert) of the pages' code.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MLA_OK 0
#define MLA_ERR_INVALID_ARG (-1)  /* null pointer, B/T/P out of range, cap too small, overlap */
#define MLA_ERR_ALIGNMENT (-2)    /* a pointer is not 16-byte aligned */
#define MLA_ERR_WORKSPACE (-3)    /* workspace NULL or smaller than mla_workspace_size() */
#define MLA_ERR_UNSUPPORTED (-4)  /* a size or mode the library does not implement */
#define MLA_ERR_CUDA (-5)         /* a CUDA call or kernel launch failed */
#define MLA_ERR_TIMEOUT (-6)      /* a bounded device-side wait gave up (see mla_device_status) */

/* ---- fixed sizes -------------------------------------------------------- */
#define MLA_D 7168
#define MLA_HEADS 64
#define MLA_Q_LORA 1536
#define MLA_KV_LORA 512
#define MLA_QK_NOPE 128
#define MLA_QK_ROPE 64
#define MLA_QK 192
#define MLA_V 128
#define MLA_FFN_INTER 18432  /* SwiGLU MLP width: 396,361,728 parameters / (3 x 7168) */

/* ---- modes for mla_workspace_size ---------------------------------------- */
#define MLA_MODE_PREFILL 0
#define MLA_MODE_DECODE 1
#define MLA_MODE_DECODE_LATENT 2
#define MLA_MODE_FFN 3
#define MLA_MODE_CHUNK_LATENT 4
#define MLA_MODE_CHUNK_ABSORBED 5
#define MLA_MODE_FOLD 6

/* Weights of one MLA sublayer: device pointers to bf16, nn.Linear [out, in].
 * Key-value compression page, MLA __init__ excerpt, for the projections;
 * w_in_norm is the block's input RMSNorm gain (dense-block page). */
typedef struct {
  const void* w_in_norm;   /* [7168]          input RMSNorm gain            */
  const void* w_q_a;       /* [1536, 7168]    q_a_proj (W_DQ)               */
  const void* w_q_a_norm;  /* [1536]          q_a_layernorm gain            */
  const void* w_q_b;       /* [12288, 1536]   q_b_proj; per head [128 nope | 64 pe] */
  const void* w_kv_a;      /* [576, 7168]     kv_a_proj_with_mqa (W_DKV ; W_KR) */
  const void* w_kv_a_norm; /* [512]           kv_a_layernorm gain           */
  const void* w_kv_b;      /* [16384, 512]    kv_b_proj; per head [128 k_nope | 128 v] */
  const void* w_o;         /* [7168, 8192]    o_proj                        */
} mla_weights_t;

/* Stage ids for optional per-stage timing. */
#define MLA_STAGE_INPUT_NORM 0   /* RMSNorm(x)                               */
#define MLA_STAGE_A_PROJ 1       /* x_attn . [W_DQ ; W_DKV ; W_KR]^T          */
#define MLA_STAGE_LATENT 2       /* split, q/kv latent RMSNorm, RoPE table and RoPE(k), latent cache write */
#define MLA_STAGE_Q_B 3          /* q_b_proj + RoPE(q)                       */
#define MLA_STAGE_KV_B 4         /* kv_b_proj + per-head K/V cache write     */
#define MLA_STAGE_ATTN 5         /* attention (prefill, decode or latent decode) */
#define MLA_STAGE_COMBINE 6      /* split-KV combine                         */
#define MLA_STAGE_ABSORB_Q 7     /* latent decode: q_nope . W_UK             */
#define MLA_STAGE_ABSORB_O 8     /* latent decode: o_latent . W_UV^T         */
#define MLA_STAGE_O_PROJ 9       /* o_proj + residual                        */
#define MLA_STAGE_FFN_NORM 10    /* mla_ffn: RMSNorm(x')                     */
#define MLA_STAGE_FFN_GATE_UP 11 /* mla_ffn: [W_1 ; W_3] product + SiLU(g) * u */
#define MLA_STAGE_FFN_DOWN 12    /* mla_ffn: W_2 product + residual          */
#define MLA_MAX_STAGES 13

/* Optional per-stage timing.  start[s] / stop[s] are cudaEvent_t handles
 * created by the caller (or NULL to skip stage s); the library records them
 * on `stream` around stage s.  n_launches is written with the number of
 * kernels the call enqueued. */
typedef struct {
  void* start[MLA_MAX_STAGES];
  void* stop[MLA_MAX_STAGES];
  int n_launches;
} mla_timing_t;

/* Runtime parameters.  Passing NULL for the whole struct selects
 * eps = 1e-6, rope_base = 10000, softmax_scale = 1/sqrt(192). */
typedef struct {
  float eps;            /* RMSNorm epsilon, used by all three norms        */
  float rope_base;      /* RoPE base                                       */
  float softmax_scale;  /* multiplies Q.K before the softmax               */
  float* delta_out;     /* optional: float32 [N_tok, 7168] receives Delta_attn
                           (o_proj output before the residual); NULL = off */
  mla_timing_t* timing; /* optional per-stage events; NULL = off            */
} mla_params_t;

/* Bytes of workspace an entry point needs.
 *   mode = MLA_MODE_PREFILL:       B sequences of T = t_or_p tokens; `cap` is
 *                                  ignored (pass the cache capacity or 0).
 *   mode = MLA_MODE_DECODE / _LATENT: B sequences, P = t_or_p cached positions.
 *   mode = MLA_MODE_FFN:           B * t_or_p token rows (mla_ffn).
 *   mode = MLA_MODE_CHUNK_LATENT:  B sequences, chunks of T = t_or_p tokens,
 *                                  latent caches of `cap` positions
 *                                  (mla_prefill_chunk_latent; the size grows
 *                                  with cap: it holds the rebuilt keys and
 *                                  values of every position, 40 KB each).
 *   mode = MLA_MODE_CHUNK_ABSORBED: B sequences, chunks of T = t_or_p
 *                                  tokens, latent caches of `cap` positions
 *                                  (mla_prefill_chunk_absorbed; the size grows
 *                                  with B * T only).
 *   mode = MLA_MODE_FOLD:          mla_fold_wuv_into_wo (B, t_or_p, cap
 *                                  ignored: a status region only).
 * Returns 0 when the arguments are out of range. */
size_t mla_workspace_size(int mode, int B, int t_or_p, int cap);

/* Causal prefill of x [B, T, 7168] at positions 0..T-1.
 *   out       [B, T, 7168]        x + Delta_attn (may alias x exactly); or NULL:
 *                                 the call then only fills the caches it is
 *                                 given (a prompt-cache fill: the query path,
 *                                 attention and o_proj are skipped)
 *   k_cache   [B, 64, cap, 192]   optional (NULL): receives K rows 0..T-1, post-RoPE
 *   v_cache   [B, 64, cap, 128]   optional, given together with k_cache
 *   ckv_cache [B, cap, 512]       optional (NULL): receives the normalised latent c^KV-hat
 *   kpe_cache [B, cap, 64]        optional, given together with ckv_cache: rotated k^R
 *   cap       cache capacity in positions; must be >= T when a cache is given
 * Errors: INVALID_ARG (B < 1, T < 1, null x or weights, out NULL with no
 * cache, only one of a cache pair, cap < T, partial x/out overlap),
 * ALIGNMENT, WORKSPACE, CUDA. */
int mla_prefill(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T,
                void* out, void* k_cache, void* v_cache, void* ckv_cache, void* kpe_cache, int cap,
                void* workspace, size_t workspace_bytes, void* stream);

/* Chunked prefill: T new tokens per sequence at positions P0..P0+T-1, after
 * P0 tokens already in the rebuilt cache ("Mix and project" page: the cache
 * update appends the new keys and values after the cached ones, and the
 * additive mask of shape (B, 1, q_len, kv_seq_len), kv_seq_len = P0 + T,
 * keeps the causal order: token t sees keys 0..P0+t).
 *   x         [B, T, 7168]        the chunk's tokens
 *   out       [B, T, 7168]        x + Delta_attn (may alias x exactly)
 *   k_cache   [B, 64, cap, 192]   rows 0..P0-1 are read, rows P0..P0+T-1 written
 *   v_cache   [B, 64, cap, 128]   same (both required)
 *   ckv_cache, kpe_cache          optional latent cache, rows P0..P0+T-1 written
 * Requires P0 >= 0 and P0 + T <= cap; the workspace is that of
 * mla_workspace_size(MLA_MODE_PREFILL, B, T, cap).  P0 = 0 computes what
 * mla_prefill computes with caches.
 * Errors: INVALID_ARG (null or missing K/V cache, P0 < 0, P0 + T > cap),
 * ALIGNMENT, WORKSPACE, CUDA. */
int mla_prefill_chunk(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T,
                      int P0, void* out, void* k_cache, void* v_cache, void* ckv_cache, void* kpe_cache,
                      int cap, void* workspace, size_t workspace_bytes, void* stream);

/* Chunked prefill against the 576-value latent cache (latent-cache serving:
 * "Key-value compression" page, the per-head keys and values of every
 * position are rebuilt from its one latent).  T new tokens per sequence at
 * positions P0..P0+T-1; their latent rows are written to the cache, then the
 * keys and values of positions 0..P0+T-1 are rebuilt from the cache into the
 * workspace (kv_b product, rotary key appended) and the chunk attends to them
 * with the causal mask offset by P0, as mla_prefill_chunk.
 *   x, out          [B, T, 7168]   (out may alias x exactly; required)
 *   ckv_cache       [B, cap, 512]  rows 0..P0-1 read, rows P0..P0+T-1 written
 *   kpe_cache       [B, cap, 64]   same
 * Requires P0 >= 0, P0 + T <= cap; workspace
 * mla_workspace_size(MLA_MODE_CHUNK_LATENT, B, T, cap).
 * Errors: INVALID_ARG (null pointer, P0 < 0, P0 + T > cap), ALIGNMENT,
 * WORKSPACE, CUDA. */
int mla_prefill_chunk_latent(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T,
                             int P0, void* out, void* ckv_cache, void* kpe_cache, int cap, void* workspace,
                             size_t workspace_bytes, void* stream);

/* W_UV folded into the output projection (latent-cache serving, "Key-value
 * compression" page: the value up-projection moves past the attention, and
 * here on into W_o): for every head h,
 *   W_fold[:, h*512 .. h*512+511] = W_o[:, h*128 .. h*128+127] W_UV[h],
 * W_UV[h] = rows h*256+128 .. h*256+255 of W_kv_b ([128, 512]).
 *   w_fold     [7168, 32768] bf16, caller-allocated (470 MB), written
 *   workspace  mla_workspace_size(MLA_MODE_FOLD, 1, 1, 0) bytes
 * Errors: INVALID_ARG (null weight or w_fold), ALIGNMENT, WORKSPACE, CUDA. */
int mla_fold_wuv_into_wo(const mla_weights_t* w, void* w_fold, void* workspace, size_t workspace_bytes,
                         void* stream);

/* mla_decode_latent with the output projection through W_fold: the latent
 * attention output of all heads, o_lat [B, 64*512], times W_fold^T plus the
 * residual, one GEMM in place of W_UV and o_proj.  Arguments, workspace
 * (MLA_MODE_DECODE_LATENT) and errors as mla_decode_latent; w_fold from
 * mla_fold_wuv_into_wo (16-byte aligned).  It streams 470 MB of weights where
 * W_UV and W_o are 125 MB, so a weight-bound decode step is slower; kept for
 * comparison. */
int mla_decode_latent_folded(const mla_weights_t* w, const void* w_fold, const mla_params_t* params, const void* x,
                             int B, int P, void* ckv_cache, void* kpe_cache, int cap, void* out, void* workspace,
                             size_t workspace_bytes, void* stream);

/* The same chunk in the absorbed form (latent-cache serving, "Key-value
 * compression" page: W_UK folded into the query, W_UV applied after the
 * attention, so the cached latent is never expanded).  Every new token
 * (b, t) is one latent decode step at position P0 + t that attends to cache
 * rows 0..P0+t of sequence b: scores q_lat . [k^R ; c^KV], o_lat = P c^KV,
 * then W_UV and o_proj.  Results, arguments and errors as
 * mla_prefill_chunk_latent; the chunk's latent rows are written first.
 * Cost: the cache is read once per new token (B T (P0 + T) 1152 bytes)
 * instead of rebuilding the keys and values of every cached position (a
 * 16384 x 512 product per position), so it is the form for short chunks.
 * Requires P0 >= 0, P0 + T <= cap; workspace
 * mla_workspace_size(MLA_MODE_CHUNK_ABSORBED, B, T, cap).
 * Errors: INVALID_ARG (null pointer, P0 < 0, P0 + T > cap), ALIGNMENT,
 * WORKSPACE, CUDA. */
int mla_prefill_chunk_absorbed(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int T,
                               int P0, void* out, void* ckv_cache, void* kpe_cache, int cap, void* workspace,
                               size_t workspace_bytes, void* stream);

/* One decode step against the rebuilt per-head cache (the pinned
 * implementation's cache, "Mix and project" page at P = 1,000).
 *   x        [B, 7168]           the new token of each sequence, at position P
 *   k_cache  [B, 64, cap, 192]   positions 0..P-1 are read; row P is written
 *   v_cache  [B, 64, cap, 128]   same
 *   out      [B, 7168]           x + Delta_attn (may alias x exactly)
 * Requires 0 <= P and P + 1 <= cap.
 * Errors: INVALID_ARG, ALIGNMENT, WORKSPACE, CUDA. */
int mla_decode(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int P,
               void* k_cache, void* v_cache, int cap, void* out,
               void* workspace, size_t workspace_bytes, void* stream);

/* One decode step against the 576-value latent cache, with W_UK absorbed
 * into the query and W_UV applied after attention (the latent-caching design
 * the key-value compression page describes).
 *   ckv_cache [B, cap, 512]  normalised latent; positions 0..P-1 read, row P written
 *   kpe_cache [B, cap, 64]   rotated rotary key; same
 * Other arguments as mla_decode. */
int mla_decode_latent(const mla_weights_t* w, const mla_params_t* params, const void* x, int B,
                      int P, void* ckv_cache, void* kpe_cache, int cap, void* out,
                      void* workspace, size_t workspace_bytes, void* stream);

/* The same two decode steps for a batch of sequences of different lengths
 * (a ragged batch: "Mix and project" page, each sequence its own cache update
 * and score row).  Sequence b's new token sits at position P[b] and attends
 * to its P[b] + 1 keys; its cache row P[b] is written.
 *   P      int [B] in DEVICE memory (4-byte aligned), read by the kernels, so
 *          a captured CUDA graph can be replayed with new lengths
 *   P_max  an upper bound of every P[b]; it sizes the launch and the
 *          workspace: mla_workspace_size(MLA_MODE_DECODE or
 *          MLA_MODE_DECODE_LATENT, B, P_max, cap); requires P_max + 1 <= cap
 * A P[b] outside [0, P_max] cannot be checked on the host: the kernels clamp
 * it into that range (no access leaves the caches) and record it, and
 * mla_device_status then returns MLA_ERR_INVALID_ARG.
 * Other arguments, results and errors as mla_decode / mla_decode_latent. */
int mla_decode_varlen(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, const int* P,
                      int P_max, void* k_cache, void* v_cache, int cap, void* out, void* workspace,
                      size_t workspace_bytes, void* stream);
int mla_decode_latent_varlen(const mla_weights_t* w, const mla_params_t* params, const void* x, int B,
                             const int* P, int P_max, void* ckv_cache, void* kpe_cache, int cap, void* out,
                             void* workspace, size_t workspace_bytes, void* stream);

/* mla_decode without a workspace argument.  The pages have no counterpart
 * to this entry point: it exists for callers that cannot allocate device
 * memory (code running under a host framework that owns all device memory
 * and allows no allocation of its own, such as inference-server plugins or
 * runtimes with a fixed memory budget, and latency-critical loops that cannot
 * afford the device synchronisation an allocation may cause).
 *   Scratch: a 64 MiB static device array inside the library, held by every
 *   GPU that loads the library until the process exits.  Batches whose
 *   mla_workspace_size(MLA_MODE_DECODE, B, P, cap) exceeds 64 MiB (more than
 *   455 sequences) are rejected with MLA_ERR_WORKSPACE; nothing is allocated.
 *   The first call on each device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   Every call on a device shares the one array and it keeps the last call's
 *   contents: calls that may overlap on the GPU (different streams without
 *   ordering between them) race.  A device-side timeout is recorded only in
 *   the array, not returned.
 * Arguments, checks and results otherwise as mla_decode. */
int mla_decode_noalloc(const mla_weights_t* w, const mla_params_t* params, const void* x, int B, int P,
                       void* k_cache, void* v_cache, int cap, void* out, void* stream);

/* ---- FP8 block-scaled weights ---------------------------------------------
 * The dense-block page counts the checkpoint's tensors with its "FP8 block
 * scales" left out: the released weights are FP8 with one scale per block.
 * Block size and scale format are not printed; this library's format:
 * E4M3 codes (the OCP FP8 E4M3 encoding, largest finite 448) of the [out, in]
 * matrix, and one float scale per 128 x 128 block, always a power of two:
 * the smallest 2^k with amax(block) <= 448 * 2^k.  The weight used is
 * code * scale, exact in bfloat16, so the FP8 decode computes with exactly
 * the quantized weights (on the bf16 tensor-core path: the codes are
 * dequantized in shared memory; the bytes read from HBM halve).
 *   cols   a multiple of 128
 *   codes  uint8, block-major: block (i, j) (rows 128i.., columns 128j..) is
 *          16,384 contiguous bytes at offset (i * cols/128 + j) * 16384,
 *          row-major inside; ceil(rows/128) * cols/128 * 16384 bytes in all,
 *          the rows past the matrix zero
 *   scales [ceil(rows/128), cols/128] float */
int mla_quantize_fp8(const void* w_bf16, int rows, int cols, void* codes, float* scales, void* stream);

/* The MLA weights with the five projection matrices in that format (gains
 * stay bf16). */
typedef struct {
  const void* w_in_norm;   /* [7168] bf16                                       */
  const void* w_q_a_norm;  /* [1536] bf16                                       */
  const void* w_kv_a_norm; /* [512]  bf16                                       */
  const void* w_q_a;       /* [1536, 7168]   E4M3 codes, block-major; scales [12, 56] */
  const void* w_q_b;       /* [12288, 1536]  E4M3 codes, block-major; scales [96, 12] */
  const void* w_kv_a;      /* [576, 7168]    E4M3 codes, block-major (640 rows); scales [5, 56] */
  const void* w_kv_b;      /* [16384, 512]   E4M3 codes, block-major; scales [128, 4] */
  const void* w_o;         /* [7168, 8192]   E4M3 codes, block-major; scales [56, 64] */
  const float* s_q_a;
  const float* s_q_b;
  const float* s_kv_a;
  const float* s_kv_b;
  const float* s_o;
} mla_weights_fp8_t;

/* mla_decode with FP8 block-scaled weights: the same step, arguments,
 * workspace (MLA_MODE_DECODE) and errors; every projection reads its E4M3
 * codes and scales (codes 16-byte aligned, scales 4-byte aligned, else
 * MLA_ERR_ALIGNMENT). */
int mla_decode_fp8(const mla_weights_fp8_t* w, const mla_params_t* params, const void* x, int B, int P,
                   void* k_cache, void* v_cache, int cap, void* out, void* workspace, size_t workspace_bytes,
                   void* stream);

/* ---- the block's second half ---------------------------------------------
 * Kimi K2 "Dense transformer block" page, equation list after
 * x'_n = x_n + Delta_attn, and its DecoderLayer forward excerpt: the dense
 * block applies the MLA sublayer (mla_prefill / mla_decode /
 * mla_decode_latent: x -> x'), then
 *   x_ffn = RMSNorm(x'); g = x_ffn W_1; u = x_ffn W_3; a = g sigma(g);
 *   h = a (.) u; Delta_ffn = h W_2; x_{n+1} = x' + Delta_ffn.
 * The intermediate width is not printed; the page's parameter table gives
 * the SwiGLU MLP 396,361,728 parameters = 3 x 7168 x 18,432 (no biases). */
typedef struct {
  const void* w_post_norm; /* [7168]          post-attention RMSNorm gain   */
  const void* w_1;         /* [18432, 7168]   gate projection (g)           */
  const void* w_3;         /* [18432, 7168]   up projection (u)             */
  const void* w_2;         /* [7168, 18432]   down projection               */
} mla_ffn_weights_t;

/* x_{n+1} = x' + Delta_ffn for n_tok token rows (any mix of prefill and
 * decode rows: every row is independent).
 *   x    [n_tok, 7168]   x' (the MLA sublayer's output)
 *   out  [n_tok, 7168]   x_{n+1} (may alias x exactly)
 *   params: eps (the MLP RMSNorm's), delta_out (optional float32
 *   [n_tok, 7168] receiving Delta_ffn) and timing (stages
 *   MLA_STAGE_FFN_*); rope_base and softmax_scale are not used.  NULL
 *   selects eps = 1e-6.
 *   workspace: mla_workspace_size(MLA_MODE_FFN, 1, n_tok, 0) bytes (it holds
 *   RMSNorm(x') and h, n_tok x (7168 + 18432) bf16 values).
 * g and u accumulate in float32; SiLU(g) u is rounded once to bf16 (h), the
 * input of the down projection, whose float32 sum is added to x' in float32
 * and rounded once.
 * Errors: INVALID_ARG (null pointer, n_tok < 1, partial x/out overlap),
 * ALIGNMENT, WORKSPACE, CUDA. */
int mla_ffn(const mla_ffn_weights_t* w, const mla_params_t* params, const void* x, int n_tok, void* out,
            void* workspace, size_t workspace_bytes, void* stream);

/* Synchronises `stream` and reads the device status word the last call on
 * this workspace left: MLA_OK, MLA_ERR_TIMEOUT if a bounded device wait
 * gave up (the kernel then skipped its remaining work and returned), or
 * MLA_ERR_INVALID_ARG if a per-sequence position of a _varlen call was
 * outside [0, P_max].
 * The word describes one call only: every entry point clears it (and the
 * rest of the status region) on its stream before its first kernel, so a
 * caller that needs the status of a call must read it before enqueueing the
 * next call on the same workspace.
 * MLA_ERR_CUDA if the synchronisation itself fails. */
int mla_device_status(const void* workspace, void* stream);

/* Human-readable name of a status code (static string). */
const char* mla_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */
