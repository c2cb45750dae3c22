// The NVFP4 block encoder shared by the quantizers and the W4A4 gate/up epilogue (which
// quantizes h in place when the activation scales are static): one 16-element block with
// global scale gs and block maximum amax -> 8 code bytes (E2M1, element i in bits 4i..4i+3)
// and one E4M3 block scale, exactly as the format defines them (clef-omni-NVFP4, "How it was
// made"): bs = E4M3((amax / 6) * gs), q = E2M1(v / (bs / gs)).
#pragma once
#include "moe_internal.cuh"

namespace moe {

// Eight floats to eight E2M1 codes (element i in bits 4i..4i+3) with the hardware conversion:
// round to nearest, ties to the even code, saturating at 6, sign kept.
__device__ __forceinline__ uint32_t e2m1x8(const float f[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
  return r;
}

// Codes of eight elements: E2M1(fl(v / eff)), fl = fp32 division rounded to nearest.
// Bracketing: with r = fl(1/eff), a = fl(v * fl(r * (1 - 2^-20))) and b = fl(v * fl(r * (1 + 2^-20)))
// carry at most three roundings of 2^-24 each, so |a| < |v/eff| < |b| (outside the subnormal
// range, where every candidate is far below the first rounding boundary 0.25 and codes 0).
// fl is monotone, so |a| <= |fl(v/eff)| <= |b|, and because the conversion is monotone too,
// equal codes for a and b are the code of fl(v/eff).  Only a pair that straddles a rounding
// boundary pays the exact division.
__device__ __forceinline__ uint32_t e2m1x8_div(const float* v, float eff, float rd, float ru) {
  float a[8], b[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a[i] = __fmul_rn(v[i], rd);
    b[i] = __fmul_rn(v[i], ru);
  }
  const uint32_t ca = e2m1x8(a);
  if (ca == e2m1x8(b)) return ca;
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = __fdiv_rn(v[i], eff);
  return e2m1x8(a);
}

// One NVFP4 16-block of a row with global scale gs and block maximum amax = max |v|:
// 8 code bytes and 1 scale byte.
__device__ __forceinline__ void nvfp4_encode(const float v[16], float amax, float gs, uint2* codes8, uint8_t* scale) {
  const uint8_t bsc = f32_to_e4m3(__fmul_rn(__fdiv_rn(amax, 6.0f), gs));
  const float bs = e4m3_to_f32(bsc);
  uint32_t lo = 0, hi = 0;
  if (bs != 0.0f) {
    const float eff = __fdiv_rn(bs, gs);
    const float r = __frcp_rn(eff);
    const float rd = __fmul_rn(r, 1.0f - 0x1p-20f), ru = __fmul_rn(r, 1.0f + 0x1p-20f);
    lo = e2m1x8_div(v, eff, rd, ru);
    hi = e2m1x8_div(v + 8, eff, rd, ru);
  }
  *codes8 = make_uint2(lo, hi);
  *scale = bsc;
}

}  // namespace moe
