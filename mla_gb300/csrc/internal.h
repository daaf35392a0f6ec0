// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace mla {

// Launch with programmatic stream serialization (see pdl_wait in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The same launch as clusters of two consecutive CTAs (grid.x even).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster2(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

struct DevStatusHost {
  uint32_t* word;
  uint64_t wait_limit_ns;
};
// Words of the status region (256 bytes before the split-K counters, zeroed
// before every call): 0 = the status word, kWorkCounterWord = the persistent
// prefill attention's work counter.
constexpr int kWorkCounterWord = 16;

// ---- tensor maps ------------------------------------------------------------
// 2D bf16 tensor map over a row-major [rows, cols] matrix with row stride
// `ld` elements, box {box_cols, box_rows}, 128-byte swizzle (box_cols * 2
// must be 128).  Returns false if the driver rejects it.
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                       uint32_t box_rows, uint32_t box_cols);

// Tensor maps for epilogue stores: 32 x 32 chunks of bf16 with 64-byte
// swizzle (64-byte chunk rows) and of float32 with 128-byte swizzle; the 3D
// bf16 map (the per-head K/V caches) stores 32 x 64 chunks with 128-byte
// swizzle, one whole 128-byte line of a cache row per chunk row.
bool make_tmap_store_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld);
bool make_tmap_store_f32_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t ld);
bool make_tmap_store_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
                             uint64_t mid_stride_bytes, uint64_t outer_stride_bytes);

// 3D bf16 tensor map over [outer][mid][inner] with byte strides for mid and
// outer, box {box_inner, box_mid, 1}, 128-byte swizzle.
bool make_tmap_bf16_3d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
                       uint64_t mid_stride_bytes, uint64_t outer_stride_bytes, uint32_t box_inner, uint32_t box_mid);

// ---- GEMM (tcgen05, TMA, persistent) --------------------------------------
// D[b][m, n] = sum_k A[m, a_col0 + b*a_col_step + k] * Bmat(b)[n, k]
// A is K-major.  B is either K-major ([N, K] rows, weight layout) taken from
// B0 for n < n_split and from B1 (rows n - n_split) otherwise, or MN-major
// ([K, N] rows, N contiguous).  Row offset b_row0 + b*b_row_step selects the
// batch's slice of B (along N for K-major, along K for MN-major).
struct GemmShape {
  int M, N, K;
  int batches;
  int a_col0, a_col_step;
  int b_row0, b_row_step;
  int n_split;
  int ksplit;   // set by launch_gemm: K slices per tile (1 = no split)
  int kb_per;   // set by launch_gemm: 64-wide K blocks per slice
  int raster_g; // set by launch_gemm: tiles walk groups of raster_g row blocks,
                // row block fastest inside a group (1 = column block fastest)
};

// Split-K (used when a GEMM has too few output tiles to fill the GPU, as
// the decode projections with M <= 128 do): each CTA of a tile's K slice
// writes its float32 partial to its own slot; the last warp to finish a
// 32-row slice of the tile (counter per tile and quarter) sums the slots in
// slice order and runs the epilogue.  Units = tiles x slices <= kMaxSplitUnits.
// A slot holds a whole BM x BN tile (BM = 64 for M <= 64, else 128).
constexpr int kMaxSplitUnits = 160;
constexpr int kMaxSplitCounters = 960;
inline size_t split_part_bytes(int M) { return (size_t)kMaxSplitUnits * (M <= 64 ? 64 : 128) * 256 * sizeof(float); }

struct GemmOperands {
  const __nv_bfloat16* A;
  int lda;
  int a_rows;  // rows of the A tensor (>= M)
  const __nv_bfloat16* B0;
  int ldb0;
  int b0_rows;
  const __nv_bfloat16* B1;  // may be null
  int ldb1;
  int b1_rows;
  bool b_mn_major;
};

enum class Epi { kStoreBf16, kStoreF32, kQRope, kKVCache, kResidual, kSwiGLU };

struct EpiArgs {
  // kStoreBf16: out[row, c_col0 + batch*c_col_step + n]; kStoreF32: out_f32[row, n]
  __nv_bfloat16* out;
  float* out_f32;
  int ldo;
  int c_col0, c_col_step;
  // kQRope: q[row, n] with RoPE on columns 128..191 of each 192 block;
  //         position index of a row = row % t_mod into cs (float2 [.., 32])
  const float2* cs;
  int t_mod;
  // kQRope, register epilogue only (decode sizes): when set, the rotated pe
  // columns of row r, head h are also written to qpe_out[(r*64 + h)*576 + 512 ..]
  __nv_bfloat16* qpe_out;
  // kKVCache: K[b, h, t, 0:128] / V[b, h, t, 0:128] / K[b, h, t, 128:192] = kpe[row]
  //           b = row / t_mod, t = t_off + row % t_mod
  __nv_bfloat16* kc;
  __nv_bfloat16* vc;
  const __nv_bfloat16* kpe;
  int t_off;
  int cap;
  // kResidual: out[row, n] = x[row, n] + acc; delta[row, n] = acc (optional)
  // kSwiGLU: out[row, j] = SiLU(g) * u for j < N / 2, g from B0 (gate) row j,
  //          u from B1 (up) row j: each BN-wide tile holds BN / 2 gate columns
  //          then the BN / 2 up columns of the same j (B0, B1 both [N / 2, K])
  const __nv_bfloat16* x;
  float* delta;
  // split-K scratch (null: no split): partial slots and zeroed counters
  float* part;
  size_t part_bytes;
  int* counters;
  // rows of the K/V caches the kv_b epilogue may write (t < t_off + t_mod)
  int B;
  // kKVCache, decode with per-sequence lengths: row b's position pos[b]
  // (clamped into [0, pos_max]) replaces t_off; null otherwise
  const int* pos;
  int pos_max;
};

cudaError_t launch_gemm(const GemmShape& s, const GemmOperands& op, Epi epi, const EpiArgs& ea,
                        const DevStatusHost& st, int num_sms, cudaStream_t stream);

// The same product with B stored as FP8 (E4M3) codes and one power-of-two
// scale per 128 x 128 block (scales [rows / 128 rounded up, K / 128]); B is
// K-major ([N, K]), K a multiple of 128, one batch; the codes are stored
// block-major: block (i, j) = rows 128i.., columns 128j.. is 16 KB at
// ((i * K/128 + j) * 128) * 128, row-major inside (rows past the matrix are
// zero).  The codes are bulk-copied and dequantized to bf16 in shared memory
// (exact: the scales are powers of two); the product runs on the bf16
// tensor-core path.  Decode-size M: the weight bytes halve.
struct GemmW8Operands {
  const __nv_bfloat16* A;
  int lda;
  int a_rows;
  const uint8_t* B0;  // rows n < n_split
  int b0_rows;
  const float* s0;
  const uint8_t* B1;  // rows n - n_split (may be null)
  int b1_rows;
  const float* s1;
};
cudaError_t launch_gemm_w8(const GemmShape& s, const GemmW8Operands& op, Epi epi, const EpiArgs& ea,
                           const DevStatusHost& st, int num_sms, cudaStream_t stream);

// bf16 [rows, cols] (cols a multiple of 128) -> E4M3 codes, block-major with
// the row count padded to 128 (zeros), and scales [ceil(rows/128), cols/128]
cudaError_t launch_fp8_quantize(const __nv_bfloat16* w, int rows, int cols, uint8_t* codes, float* scales,
                                cudaStream_t stream);

// ---- row kernels --------------------------------------------------------------
cudaError_t launch_rmsnorm_rows(const __nv_bfloat16* x, const __nv_bfloat16* g, __nv_bfloat16* y, int rows,
                                float eps, cudaStream_t stream);
// Split the A-projection output ca [rows, 2112] (float32) into RMSNorm(c^Q) [rows,1536],
// RMSNorm(c^KV) [rows,512] and RoPE(k_pe) [rows,64]; optional latent cache
// copies at ckv_cache[b, t_off + t] / kpe_cache[b, t_off + t]; also writes the
// RoPE table cs[t] = (cos, sin)((pos0 + t) theta_i) that the q_b epilogue reads.
struct LatentArgs {
  const float* ca;
  const __nv_bfloat16* g_qa;
  const __nv_bfloat16* g_kva;
  float2* cs;              // RoPE table [t_mod, 32] written here (rows of batch 0)
  double inv_freq[32];     // theta_i = base^(-2i/64), computed on the host in double
  int pos0;                // position of t = 0
  __nv_bfloat16* cq;
  __nv_bfloat16* ckv;
  __nv_bfloat16* kpe;
  __nv_bfloat16* ckv_cache;
  __nv_bfloat16* kpe_cache;
  int rows, t_mod, t_off, cap;
  float eps;
  // decode with per-sequence lengths: row r sits at position pos[r] (cache
  // row and RoPE angle; cs then holds one entry per row); positions outside
  // [0, pos_max] set kStatusBadLength in *status and are clamped
  const int* pos;
  int pos_max;
  uint32_t* status;
};
cudaError_t launch_latent_split(const LatentArgs& a, cudaStream_t stream);

// ---- attention ----------------------------------------------------------------
struct PrefillAttnArgs {
  const __nv_bfloat16* q;   // [B*T, 64*192], queries at positions past..past+T-1
  const __nv_bfloat16* k;   // [B, 64, cap, 192], keys 0..past+T-1
  const __nv_bfloat16* v;   // [B, 64, cap, 128]
  __nv_bfloat16* o;         // [B*T, 64*128]
  int B, T, cap;
  float scale;
  int past;                 // keys before the first query (chunked prefill), 0 otherwise
};
cudaError_t launch_prefill_attention(const PrefillAttnArgs& a, const DevStatusHost& st, int num_sms,
                                     cudaStream_t stream);

struct DecodeAttnArgs {
  const __nv_bfloat16* q;   // [B, 64*192]
  const __nv_bfloat16* k;   // [B, 64, cap, 192]
  const __nv_bfloat16* v;   // [B, 64, cap, 128]
  __nv_bfloat16* o;         // [B, 64*128]
  float* part_o;            // [B*64*splits, 128] split partials
  float2* part_ml;          // [B*64*splits] (max, sum)
  int B, L, cap, splits;    // L = keys attended (P + 1); with lens_pos: the largest P_b + 1
  float scale;
  const int* lens_pos;      // optional per-sequence P_b (keys 0..P_b), clamped into [0, L - 1]
};
int decode_splits(int B, int L, int num_sms);
cudaError_t launch_decode_attention(const DecodeAttnArgs& a, const DevStatusHost& st, cudaStream_t stream,
                                    int* launches);

struct LatentAttnArgs {
  const __nv_bfloat16* qlat;  // [B, 64, 576] (absorbed q_nope | rotated q_pe)
  const __nv_bfloat16* ckv;   // [B, cap, 512]
  const __nv_bfloat16* kpe;   // [B, cap, 64]
  __nv_bfloat16* olat;        // [B, 64, 512]
  float* part_o;              // [2*ctas, 64, 512]: two partial slots per CTA
  float2* part_ml;            // [2*ctas, 64]
  int B, L, cap, ctas;        // ctas = latent_ctas(B, L, SMs); with pos: L = the largest P_b + 1
  float scale;
  // decode with per-sequence lengths: P_b = pos[b] (clamped into [0, L - 1])
  // and the work plan that latent_plan_kernel writes (null: every sequence L keys)
  const int* pos;
  int* plan;                  // [latent_plan_ints(B, ctas)] workspace, written by the launch
  // sequences per cache plane: sequence b reads plane b / kv_div of the
  // caches (absorbed chunked prefill: each new token is a sequence of its own)
  int kv_div = 1;
};
int latent_ctas(int B, int L, int num_sms);
// Work plan of the latent decode for per-sequence lengths: plan[0..B] =
// first flattened 64-key tile of each sequence (plan[B] = total), then per
// CTA g: (first sequence, first tile within it, tile count).  Written by a
// one-CTA kernel that launch_latent_attention runs first when pos is set.
inline size_t latent_plan_ints(int B, int ctas) { return (size_t)B + 1 + 3 * (size_t)ctas; }
cudaError_t launch_latent_attention(const LatentAttnArgs& a, const DevStatusHost& st, cudaStream_t stream,
                                    int* launches);
// pos[i] = p0 + i % t for i < n (the positions of a chunk's tokens, row-major
// over (sequence, token)).
cudaError_t launch_chunk_positions(int* pos, int n, int t, int p0, cudaStream_t stream);

// qlat[b, h, 512:576] = q[b, h*192 + 128 : h*192 + 192]
cudaError_t launch_copy_qpe(const __nv_bfloat16* q, __nv_bfloat16* qlat, int B, cudaStream_t stream);

}  // namespace mla
