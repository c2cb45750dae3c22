// The expert half of the forward pass: picks the grouped-GEMM kernels for the format and
// shape, and (for the down kernels that do not yet combine in their epilogue) the separate
// deterministic combine.
//
// The pages dequantize the selected experts to bf16 and call a grouped matmul
// (clef-omni-NVFP4, "How it was made"; clef-omni-fp8, "How this checkpoint runs"); here the
// dequantization happens inside the GEMMs and the bf16 copy of the weights never exists.
#include "moe_formats.cuh"
#include "moe_w8a8.cuh"

namespace moe {

namespace {

// The combine (deterministic): out[t, :] = bf16( sum over slots j = 0..k-1, in order, of the
// routing-weighted down row y[inv[t*k + j], :] ) with y in bf16, one thread per 8 output columns.
__global__ void __launch_bounds__(256) finalize_kernel(const uint16_t* __restrict__ y, const int32_t* __restrict__ inv,
                                                       int k, int T, int H, uint16_t* __restrict__ out) {
  const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;  // 8 columns of one token
  const bool live = i < (size_t)T * H;
  const int t = live ? (int)(i / H) : 0, c = (int)(i % H);
  pdl_wait();
  if (!live) return;
  int src[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) src[j] = j < k ? __ldg(inv + (size_t)t * k + j) : 0;
  uint4 v[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j)
    if (j < k) v[j] = __ldcs((const uint4*)(y + (size_t)src[j] * H + c));
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        s[2 * e] += __uint_as_float(w[e] << 16);
        s[2 * e + 1] += __uint_as_float(w[e] & 0xFFFF0000u);
      }
    }
  }
  uint4 o;
  o.x = (uint32_t)bf16_bits(s[0]) | ((uint32_t)bf16_bits(s[1]) << 16);
  o.y = (uint32_t)bf16_bits(s[2]) | ((uint32_t)bf16_bits(s[3]) << 16);
  o.z = (uint32_t)bf16_bits(s[4]) | ((uint32_t)bf16_bits(s[5]) << 16);
  o.w = (uint32_t)bf16_bits(s[6]) | ((uint32_t)bf16_bits(s[7]) << 16);
  *(uint4*)(out + i) = o;
}

}  // namespace

cudaError_t launch_experts(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                           int row_block, const WsLayout& L, char* ws, __nv_bfloat16* out, const StepEvents& ev,
                           cudaStream_t s, const float* act_gs) {
  const size_t n_out = (size_t)T * d.H;
  if (T == 0) return cudaGetLastError();
  cudaError_t e;
  if (d.fmt == MOE_FMT_NVFP4_W4A4) {  // combines in the down GEMM's epilogue
    return launch_experts_fp4(d, packed, x, T, k, L, ws, ev, s, (uint16_t*)out, act_gs);
  } else if (d.fmt == MOE_FMT_FP8_B128_W8A8) {
    e = launch_experts_w8a8(d, packed, x, T, k, L, ws, ev, s);
  } else if (d.fmt == MOE_FMT_FP8_B128_W8A16 && row_block == fp8dec_row_block()) {
    e = launch_experts_fp8dec(d, packed, x, T, k, L, ws, ev, s);
  } else {
    e = launch_experts_tc(d, packed, x, T, k, row_block, L, ws, ev, s);
  }
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)((n_out / 8 + 255) / 256);
  note_launches(1);
  return launch_pdl(finalize_kernel, dim3(blocks), dim3(256), 0, s, (const uint16_t*)(ws + L.y),
                    (const int32_t*)(ws + L.inv), k, T, d.H, (uint16_t*)out);
}

}  // namespace moe
