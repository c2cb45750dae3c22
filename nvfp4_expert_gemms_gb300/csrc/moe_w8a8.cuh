// Internal declarations of the FP8 W8A8 path (FP8 block-128 weights, FP8 activations with one
// scale per 1x128 group): the activation quantizer and the two grouped GEMMs.
#pragma once
#include "moe_internal.cuh"

namespace moe {

// Rows of 128-wide groups: one fp32 scale_inv per (row, group).  The tensor-core GEMMs need
// H a multiple of 256 (down-GEMM items cover 256 output features).
bool w8a8_supported(const moe_packed_desc_t& d);
int w8a8_row_block();

// FP8 quantization of bf16 rows, one scale per 128 consecutive elements of a row:
// s = 448 / max(amax, 1e-12), code = E4M3(v * s), scale_inv = 1 / s.
// Row r's codes go to output row r, or (scatter != null) to rows scatter[r*k .. r*k+k-1].
// sf_rows = 0: scale_inv row-major [rows, K/128]; else group-major [K/128][sf_rows].
cudaError_t launch_quant_fp8_rows(const __nv_bfloat16* x, const int32_t* scatter, int k, int rows, int K, uint8_t* q,
                                  float* sinv, int sf_rows, cudaStream_t s);

// Workspace bytes of the W8A8 activation buffers (codes and group scales of x and h).
size_t w8a8_act_bytes(size_t R, int K);

// The layer's two GEMMs (after routing): x -> FP8 per permuted row, gate/up (h in bf16),
// h -> FP8, down (routing-weighted rows y), which ends with the combine into out (bf16 [T, H]).
cudaError_t launch_experts_w8a8(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                                const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, uint16_t* out);

}  // namespace moe
