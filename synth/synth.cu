// Seeded synthetic input generator, GPU copy of synth/__init__.py.
//
// Holds only the generator (splitmix64 counter stream -> two 53-bit uniforms
// -> Box-Muller normal variate with ln and cos by power series -> bf16), step
// for step as the numpy version, so that
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

// Series coefficients (the same hex literals as the numpy copy):
// 1 / (2k + 1), (-1)^k / (2k)!, (-1)^k / (2k + 1)!, k = 0..11.
__constant__ double kAtanh[12] = {0x1.0000000000000p+0, 0x1.5555555555555p-2, 0x1.999999999999ap-3,
                                  0x1.2492492492492p-3, 0x1.c71c71c71c71cp-4, 0x1.745d1745d1746p-4,
                                  0x1.3b13b13b13b14p-4, 0x1.1111111111111p-4, 0x1.e1e1e1e1e1e1ep-5,
                                  0x1.af286bca1af28p-5, 0x1.8618618618618p-5, 0x1.642c8590b2164p-5};
__constant__ double kCos[12] = {0x1.0000000000000p+0,  -0x1.0000000000000p-1, 0x1.5555555555555p-5,
                                -0x1.6c16c16c16c17p-10, 0x1.a01a01a01a01ap-16, -0x1.27e4fb7789f5cp-22,
                                0x1.1eed8eff8d898p-29,  -0x1.93974a8c07c9dp-37, 0x1.ae7f3e733b81fp-45,
                                -0x1.6827863b97d97p-53, 0x1.e542ba4020225p-62, -0x1.0ce396db7f853p-70};
__constant__ double kSin[12] = {0x1.0000000000000p+0,  -0x1.5555555555555p-3, 0x1.1111111111111p-7,
                                -0x1.a01a01a01a01ap-13, 0x1.71de3a556c734p-19, -0x1.ae64567f544e4p-26,
                                0x1.6124613a86d09p-33,  -0x1.ae7f3e733b81fp-41, 0x1.952c77030ad4ap-49,
                                -0x1.2f49b46814157p-57, 0x1.71b8ef6dcf572p-66, -0x1.761b41316381ap-75};
constexpr double kLn2 = 0x1.62e42fefa39efp-1;
constexpr double kHalfPi = 0x1.921fb54442d18p+0;
constexpr double kSqrtHalf = 0x1.6a09e667f3bcdp-1;

// sum_k c[k] x^k by Horner's rule from the highest term, one rounding per operation
__device__ inline double horner12(double x, const double* c) {
  double p = __dadd_rn(__dmul_rn(x, c[11]), c[10]);
  for (int k = 9; k >= 0; --k) p = __dadd_rn(__dmul_rn(p, x), c[k]);
  return p;
}

__global__ void normal_bf16_kernel(__nv_bfloat16* __restrict__ out, uint64_t count, uint64_t key,
                                   uint64_t start, double mean, double stdv) {
  uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    const uint64_t c2 = (start + i) * 2;  // value i draws counters 2i and 2i + 1
    const uint64_t r1 = splitmix64(key + c2 * kGamma) >> 11;
    const uint64_t r2 = splitmix64(key + (c2 + 1) * kGamma) >> 11;
    // u1 = (r1 + 1) 2^-53 in (0, 1]: exponent e and mantissa m in [1/2, 1), then m in [sqrt(1/2), sqrt(2))
    const double u1 = __dmul_rn((double)(r1 + 1), 0x1p-53);
    const uint64_t ub = (uint64_t)__double_as_longlong(u1);
    double e = (double)(ub >> 52) - 1022.0;
    double m = __longlong_as_double((long long)((ub & 0x000FFFFFFFFFFFFFull) | (1022ull << 52)));
    if (m < kSqrtHalf) {
      m = __dmul_rn(m, 2.0);
      e = e - 1.0;
    }
    // ln u1 = e ln 2 + 2 s sum_k s^2k / (2k + 1),  s = (m - 1) / (m + 1)
    const double s = __ddiv_rn(m - 1.0, __dadd_rn(m, 1.0));
    const double p = horner12(__dmul_rn(s, s), kAtanh);
    const double ln_u1 = __dadd_rn(__dmul_rn(e, kLn2), __dmul_rn(__dmul_rn(s, p), 2.0));
    const double R = __dsqrt_rn(-2.0 * ln_u1);
    // cos(2 pi u2) by quarter turns: q = floor(4 u2), phi = (pi/2)(4 u2 - q)
    const double t4 = __dmul_rn((double)r2, 0x1p-51);
    const int q = (int)t4;
    const double phi = __dmul_rn(t4 - (double)q, kHalfPi);
    const double x = __dmul_rn(phi, phi);
    const double cphi = horner12(x, kCos);
    const double sphi = __dmul_rn(horner12(x, kSin), phi);
    const double c = q == 0 ? cphi : q == 1 ? -sphi : q == 2 ? -cphi : sphi;
    const double z = __dmul_rn(R, c);
    const double v = __dadd_rn(__dmul_rn(z, stdv), mean);
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
