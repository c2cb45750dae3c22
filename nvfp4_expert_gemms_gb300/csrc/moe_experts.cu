// The expert half of the forward pass: picks the grouped-GEMM kernels for the format and shape.
// Every down GEMM kernel ends with the deterministic routing-weighted combine itself.
//
// The pages dequantize the selected experts to bf16 and call a grouped matmul
// (clef-omni-NVFP4, "How it was made"; clef-omni-fp8, "How this checkpoint runs"); here the
// dequantization happens inside the GEMMs and the bf16 copy of the weights never exists.
#include "moe_formats.cuh"
#include "moe_w8a8.cuh"

namespace moe {

cudaError_t launch_experts(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                           int row_block, const WsLayout& L, char* ws, __nv_bfloat16* out, const StepEvents& ev,
                           cudaStream_t s, const float* act_gs) {
  if (T == 0) return cudaGetLastError();
  uint16_t* o = (uint16_t*)out;
  if (d.fmt == MOE_FMT_NVFP4_W4A4) return launch_experts_fp4(d, packed, x, T, k, L, ws, ev, s, o, act_gs);
  if (d.fmt == MOE_FMT_FP8_B128_W8A8) return launch_experts_w8a8(d, packed, x, T, k, L, ws, ev, s, o);
  if (d.fmt == MOE_FMT_FP8_B128_W8A16 && row_block == fp8dec_row_block()) {
    if (fp8gemv_preferred(T, k, d.E, d.I)) return launch_experts_fp8gemv(d, packed, x, T, k, row_block, L, ws, ev, s, o);
    return launch_experts_fp8dec(d, packed, x, T, k, L, ws, ev, s, o);
  }
  if (d.fmt == MOE_FMT_INT4_G128_W4A16 && int4gemv_preferred(T, k, d.E, d.H, d.I))
    return launch_experts_int4gemv(d, packed, x, T, k, row_block, L, ws, ev, s, o);
  if (d.fmt == MOE_FMT_NVFP4_W4A16 && row_block == tcw_row_block())
    return launch_experts_tcw(d, packed, x, T, k, L, ws, ev, s, o);
  return launch_experts_tc(d, packed, x, T, k, row_block, L, ws, ev, s, o);
}

}  // namespace moe
