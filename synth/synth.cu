// Seeded synthetic input generator, GPU copy of synth/__init__.py.
//
// Holds only the generator (splitmix64 counter stream -> Irwin-Hall sum of
// four 16-bit uniforms -> bf16), step for step as the numpy version, so that
// large inputs can be drawn on the device with the same bits.  Every floating
// point step uses an explicitly rounded intrinsic so that no multiply-add is
// contracted.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kM1 = 0xBF58476D1CE4E5B9ull;
constexpr uint64_t kM2 = 0x94D049BB133111EBull;

__host__ __device__ inline uint64_t splitmix64(uint64_t x) {
  x += kGamma;
  x = (x ^ (x >> 30)) * kM1;
  x = (x ^ (x >> 27)) * kM2;
  return x ^ (x >> 31);
}

__global__ void normal_bf16_kernel(__nv_bfloat16* __restrict__ out, uint64_t count, uint64_t key,
                                   uint64_t start, double mean, double stdv) {
  const double zscale = 0x1.bb67ae8584caap-16;  // sqrt(3) / 65536
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    uint64_t r = splitmix64(key + (start + i) * kGamma);
    int64_t ks = (int64_t)(r & 0xFFFF) + (int64_t)((r >> 16) & 0xFFFF) +
                 (int64_t)((r >> 32) & 0xFFFF) + (int64_t)(r >> 48);
    double z = __dmul_rn((double)(ks - 131070), zscale);
    double v = __dadd_rn(__dmul_rn(z, stdv), mean);
    out[i] = __float2bfloat16_rn(__double2float_rn(v));
  }
}

}  // namespace

extern "C" int synth_normal_bf16(void* out, uint64_t count, uint32_t seed, uint32_t stream,
                                 uint64_t start, double mean, double stdv, void* cuda_stream) {
  if (count == 0) return 0;
  uint64_t key = splitmix64(((uint64_t)seed << 32) | (uint64_t)stream);
  int threads = 256;
  uint64_t blocks64 = (count + threads - 1) / threads;
  int blocks = (int)(blocks64 < 152ull * 64 ? blocks64 : 152ull * 64);
  normal_bf16_kernel<<<blocks, threads, 0, (cudaStream_t)cuda_stream>>>(
      (__nv_bfloat16*)out, count, key, start, mean, stdv);
  return (int)cudaGetLastError();
}
