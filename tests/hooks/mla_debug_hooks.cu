// Test hooks (mla_debug.h): single kernels of the library exposed so that the
// test-suite can check them in isolation.  Linked into the test-only
// libmla_debug.so with the library's own objects; libmla.so does not carry them.
#include "../../mla_gb300/csrc/common.cuh"
#include "../../mla_gb300/csrc/internal.h"
#include "../../include/mla.h"
#include "mla_debug.h"

namespace mla {
namespace {

__global__ void wait_timeout_kernel(uint32_t* word, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  DevStatus st{word, limit_ns};
  if (threadIdx.x == 0) mbar_wait(&bar, 0, st, nullptr, 99);  // nothing ever arrives
}

// element (r, k) of a K-major tile with 64-element (128-byte) rows, 128-byte swizzle
__device__ __forceinline__ uint32_t sw128_offset(int r, int k) {
  return (uint32_t)(r * 128 + ((((k >> 3) ^ (r & 7)) & 7) << 4) + (k & 7) * 2);
}

__global__ void __launch_bounds__(128) umma_probe_kernel(float* out, int m, uint32_t* word) {
  __shared__ uint8_t raw[128 * 128 + 64 * 128 + 1024];
  __shared__ uint64_t bar;
  __shared__ uint32_t slot;
  uint8_t* sA = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sB = sA + 128 * 128;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < (128 * 128 + 64 * 128) / 4; i += 128) reinterpret_cast<uint32_t*>(sA)[i] = 0;
  __syncthreads();
  if (tid < m) {
    *reinterpret_cast<__nv_bfloat16*>(sA + sw128_offset(tid, 0)) = __float2bfloat16((float)(tid + 1));
    *reinterpret_cast<__nv_bfloat16*>(sA + sw128_offset(tid, 1)) = __float2bfloat16(128.f);
  }
  if (tid < 64) {
    *reinterpret_cast<__nv_bfloat16*>(sB + sw128_offset(tid, 0)) = __float2bfloat16(1.f);
    *reinterpret_cast<__nv_bfloat16*>(sB + sw128_offset(tid, 1)) = __float2bfloat16((float)tid);
  }
  fence_proxy_async_smem();
  if (tid == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&slot, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = slot;
  {
    // clear all 128 lanes x 64 columns so that lanes the MMA does not write read 0
    uint32_t z[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) z[i] = 0u;
    tmem_st32(tmem + ((uint32_t)(warp * 32) << 16), z);
    tmem_st32(tmem + ((uint32_t)(warp * 32) << 16) + 32, z);
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    const uint64_t da = sdesc_sw128(smem_u32(sA), 16, 1024);
    const uint64_t db = sdesc_sw128(smem_u32(sB), 16, 1024);
    umma_bf16(tmem, da, db, idesc_bf16(m, 64, false, false), 0u);
    umma_commit(&bar);
  }
  DevStatus st{word, 1000000000ull};
  const bool ok = mbar_wait(&bar, 0, st, nullptr, 98);
  __syncwarp();
  if (__all_sync(0xffffffffu, ok)) {
    tc_fence_after();
    uint32_t r0[32], r1[32];
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16), r0);
    tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + 32, r1);
    tmem_wait_ld();
    float* o = out + (size_t)(warp * 32 + lane) * 64;
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      o[c] = __uint_as_float(r0[c]);
      o[32 + c] = __uint_as_float(r1[c]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" {

int mla_debug_gemm(const void* A, int lda, const void* B, int ldb, int b_mn_major, void* C, int ldc, int M, int N,
                   int K, void* stream) {
  if (!A || !B || !C || M < 1 || N < 1 || K < 64 || K % 64) return MLA_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  GemmShape s{M, N, K, 1, 0, 0, 0, 0, N};
  GemmOperands op{static_cast<const __nv_bfloat16*>(A), lda, M, static_cast<const __nv_bfloat16*>(B), ldb,
                  b_mn_major ? K : N, nullptr, 0, 0, b_mn_major != 0};
  EpiArgs ea{};
  ea.out = static_cast<__nv_bfloat16*>(C);
  ea.ldo = ldc;
  DevStatusHost st{nullptr, 2000000000ull};
  return cuda_rc(launch_gemm(s, op, Epi::kStoreBf16, ea, st, sms, static_cast<cudaStream_t>(stream)));
}

int mla_debug_wait_timeout(void* status_word, uint64_t limit_ns, void* stream) {
  if (!status_word) return MLA_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint32_t*>(status_word),
                                                                       limit_ns);
  return cuda_rc(cudaGetLastError());
}

int mla_debug_umma_probe(float* out, int m, void* stream) {
  if (!out || (m != 64 && m != 128)) return MLA_ERR_INVALID_ARG;
  umma_probe_kernel<<<1, 128, 0, static_cast<cudaStream_t>(stream)>>>(out, m, nullptr);
  return cuda_rc(cudaGetLastError());
}

}  // extern "C"
