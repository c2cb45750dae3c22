// Pieces of the decode-sized expert GEMMs on tcgen05 kind::f8f6f4: the E4M3 x E4M3 MMA, the
// E4M3 conversions used by the exact two-term split of bf16 activations, and the power-of-two
// row normalizer that keeps the split inside the E4M3 range.
#pragma once
#include <cuda_fp8.h>
#include <stdint.h>

#include "moe_tc.cuh"

namespace moe {
namespace dec {

constexpr int kRows = 16;  // token rows per decode tile; hi / lo rows fill N = 32

__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);  // A, B = E4M3 (0)
}

__device__ __forceinline__ void mma_f8_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t v) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)v, __NV_E4M3);
  return __half22float2(__half2(h));
}

// Largest power of two u with amax * smax * u <= 448 (1 when the row is all zeros).
__device__ __forceinline__ float pow2_norm(float amax, float smax) {
  const float m = amax * smax;
  if (!(m > 0.f)) return 1.f;
  int e;
  frexpf(448.0f / m, &e);  // 448/m = f * 2^e, f in [0.5, 1); inf / denormal ranges clamp below
  e = e - 1 < -126 ? -126 : (e - 1 > 126 ? 126 : e - 1);
  return ldexpf(1.0f, e);
}

}  // namespace dec
}  // namespace moe
