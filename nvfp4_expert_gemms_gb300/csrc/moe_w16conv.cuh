// Register-level helpers of the bf16 converters (the weight-only tensor-core GEMMs) and the
// NVFP4 converter itself, shared by the 128- and 256-token kernels.
#pragma once
#include "moe_nvfp4.cuh"

namespace moe {
namespace {

// Packed bf16 helpers on plain 32-bit registers (no address-taken temporaries).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// An empty asm that claims to read and rewrite the 32 converted words: the conversion is then
// finished before the barrier waits that follow it (register-only arithmetic may otherwise be
// scheduled after them, serialising it behind the tensor-memory slot's release).
__device__ __forceinline__ void reg_fence(uint32_t* v) {
#pragma unroll
  for (int i = 0; i < 32; i += 8)
    asm volatile("" : "+r"(v[i]), "+r"(v[i + 1]), "+r"(v[i + 2]), "+r"(v[i + 3]), "+r"(v[i + 4]), "+r"(v[i + 5]),
                 "+r"(v[i + 6]), "+r"(v[i + 7]));
}

// ---- converters: half a chunk (64 K) of one weight row -> 32 bf16x2 words -------------------
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// NVFP4: the weights come as the converter's image (nvfp4_w4a16_image_kernel): in each 32-bit
// word of eight E2M1 codes the bits sit where one shift (or rotate) and mask puts a pair of codes
// under the exponent of a bf16 pair -- code bits (e1 e0 m) at bf16 bits 8..6 and the sign at bit
// 15 give the bf16 value code * 2^-126, E2M1 subnormals on bf16 subnormals.  One packed multiply
// by bf16(block scale * 2^116) then gives w * 2^-10 exactly (at most 6 significant bits); the
// epilogue applies 2^10 / global scale.  The scale's E4M3 bits go under bf16's exponent plus 236
// (2^-120 to 2^116), or, when a block scale of the half chunk is zero or subnormal, through fp32.
__device__ __forceinline__ void conv_nvfp4(const char* sub, int r, int kh, uint32_t bs4, uint32_t* out) {
  constexpr uint32_t kPair = 0x81C081C0u;  // bf16 pair bits: sign, exponent bits 1..0, mantissa bit 6
  uint4 q[2];
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) q[cc] = *(const uint4*)(sub + r * 64 + (((kh * 2 + cc) ^ ((r >> 1) & 3)) * 16));
  uint32_t bs2[4];
  const uint32_t ex = bs4 & 0x78787878u;
  if ((((ex - 0x08080808u) & ~ex) & 0x80808080u) == 0u) {  // four normal scales
    const uint32_t m = bs4 & 0x7F7F7F7Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) bs2[b] = prmt(m, 0u, 0x4040u | (uint32_t)b | ((uint32_t)b << 8)) * 16u + 0x76007600u;
  } else {
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const float f = e4m3_to_f32((bs4 >> (8 * b)) & 0xFF) * 0x1p116f;
      bs2[b] = pack_bf16x2(f, f);
    }
  }
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {  // 16-byte piece = 32 codes = two 16-element blocks
    const uint32_t w[4] = {q[cc].x, q[cc].y, q[cc].z, q[cc].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t bs = bs2[cc * 2 + (i >> 1)], x = w[i];
      out[cc * 16 + i * 4 + 0] = bmul2((x << 6) & kPair, bs);
      out[cc * 16 + i * 4 + 1] = bmul2((x << 2) & kPair, bs);
      out[cc * 16 + i * 4 + 2] = bmul2(__funnelshift_r(x, x, 4) & kPair, bs);
      out[cc * 16 + i * 4 + 3] = bmul2((x & 0x81808180u) | ((x >> 8) & 0x00400040u), bs);
    }
  }
}

}  // namespace
}  // namespace moe
