// Device-side views of the packed canonical tensors: load 8 consecutive weights of one row
// as fp32, using each format's dequantization rule (one fp32 rounding, as the formats define):
//   FP8   (clef-omni-fp8, "Recipe"):            e4m3(code) * scale_inv[n/128][k/128]
//   INT4  (clef-omni-int4, "What was quantized"): (code - 8) * fp16 scale[k/128][n]
//   NVFP4 (clef-omni-NVFP4, "How it was made"):  (e2m1(q) * e4m3(bs[n][k/16])) / gs
//   BF16  (unquantized):                         the bf16 weight
#pragma once
#include "moe_internal.cuh"

namespace moe {

struct MatView {
  const uint8_t* a;   // codes / qweight / packed nibbles, for all experts
  const void* b;      // scale_inv / fp16 scales / E4M3 block scales
  const float* gs;    // NVFP4 global scales [E] (else null)
  int N, K;           // matrix shape [N, K] per expert
};

__host__ inline MatView mat_view(const moe_packed_desc_t& d, const char* packed, int which) {
  MatView v;
  const int N = which == 0 ? 2 * d.I : d.H, K = which == 0 ? d.H : d.I;
  v.a = (const uint8_t*)(packed + d.offset[which == 0 ? MOE_T_GU_A : MOE_T_D_A]);
  v.b = packed + d.offset[which == 0 ? MOE_T_GU_B : MOE_T_D_B];
  v.gs = (d.fmt == MOE_FMT_NVFP4_W4A16 || d.fmt == MOE_FMT_NVFP4_W4A4)
             ? (const float*)(packed + d.offset[which == 0 ? MOE_T_GU_GS : MOE_T_D_GS])
             : nullptr;
  v.N = N;
  v.K = K;
  return v;
}

// k0 is a multiple of 8.
template <int FMT>
__device__ __forceinline__ void load_w8(const MatView& m, int e, int n, int k0, float w[8]) {
  if constexpr (FMT == MOE_FMT_FP8_B128_W8A16) {
    const uint2 c = *(const uint2*)(m.a + ((size_t)e * m.N + n) * m.K + k0);
    const float s = ((const float*)m.b)[((size_t)e * (m.N / 128) + n / 128) * (m.K / 128) + k0 / 128];
#pragma unroll
    for (int i = 0; i < 4; ++i) w[i] = e4m3_to_f32((c.x >> (8 * i)) & 0xFF) * s;
#pragma unroll
    for (int i = 0; i < 4; ++i) w[4 + i] = e4m3_to_f32((c.y >> (8 * i)) & 0xFF) * s;
  } else if constexpr (FMT == MOE_FMT_BF16) {
    const uint4 c = *(const uint4*)(m.a + (((size_t)e * m.N + n) * m.K + k0) * 2);
    const uint32_t ww[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      w[2 * i] = __uint_as_float(ww[i] << 16);
      w[2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
    }
  } else if constexpr (FMT == MOE_FMT_INT4_G128_W4A16) {
    const uint32_t q = ((const uint32_t*)m.a)[((size_t)e * (m.K / 8) + k0 / 8) * m.N + n];
    const float s = __half2float(((const __half*)m.b)[((size_t)e * (m.K / 128) + k0 / 128) * m.N + n]);
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = (float)((int)((q >> (4 * i)) & 0xF) - 8) * s;
  } else {
    const uint32_t q = *(const uint32_t*)(m.a + ((size_t)e * m.N + n) * (m.K / 2) + k0 / 2);
    const float bs = e4m3_to_f32(((const uint8_t*)m.b)[((size_t)e * m.N + n) * (m.K / 16) + k0 / 16]);
    const float gs = m.gs[e];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = __fdiv_rn(e2m1_to_f32((q >> (4 * i)) & 0xF) * bs, gs);
  }
}

}  // namespace moe
