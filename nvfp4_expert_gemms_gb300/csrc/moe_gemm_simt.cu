// Grouped expert GEMMs on CUDA cores (fp32 FMA), one CTA per (row block of one expert,
// column block).  Dequantization uses each format's rule on the fly; SiLU(gate)*up is fused
// into the gate/up GEMM; the down GEMM writes each permuted row times its routing weight (fp32),
// and finalize_kernel sums a token's k rows in slot order and rounds once to bf16.
//
// The pages dequantize the selected experts to bf16 and call a grouped matmul
// (clef-omni-NVFP4, "How it was made"; clef-omni-fp8, "How this checkpoint runs"); here the
// dequantization happens inside the GEMM and the bf16 copy of the weights never exists.
#include "moe_formats.cuh"
#include "moe_w8a8.cuh"

namespace moe {

namespace {

constexpr int kSimtRB = 8;   // rows (token slots) per CTA
constexpr int kSimtNB = 16;  // output columns per CTA (4 per warp)

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Activation row r of the tile into shared memory as fp32: bf16 x / h, or the NVFP4
// dequantization (e2m1 * e4m3) / gs of the W4A4 codes.
template <bool A4>
__device__ __forceinline__ void stage_rows(float* xs, int K, int rows, const uint16_t* __restrict__ src,
                                           const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf,
                                           const float* __restrict__ gs, const int* src_row) {
  for (int i = threadIdx.x; i < kSimtRB * K; i += blockDim.x) {
    const int r = i / K, c = i % K;
    float v = 0.f;
    if (r < rows) {
      const size_t sr = (size_t)src_row[r];
      if constexpr (A4) {
        const uint8_t byte = q[sr * (K / 2) + c / 2];
        const float bs = e4m3_to_f32(sf[sr * (K / 16) + c / 16]);
        v = __fdiv_rn(e2m1_to_f32((c & 1) ? (byte >> 4) : (byte & 0xF)) * bs, gs[sr]);
      } else {
        v = bf16_to_f32(src[sr * K + c]);
      }
    }
    xs[i] = v;
  }
}

template <int FMT, bool A4>
__global__ void __launch_bounds__(128) gateup_simt_kernel(MatView gu, const uint16_t* __restrict__ x,
                                                          const uint8_t* __restrict__ xq,
                                                          const uint8_t* __restrict__ xsf,
                                                          const float* __restrict__ xgs,
                                                          const int32_t* __restrict__ perm, int k, int I,
                                                          const TileEntry* __restrict__ tiles,
                                                          uint16_t* __restrict__ h) {
  extern __shared__ float xs[];
  __shared__ int src_row[kSimtRB];
  if ((int)blockIdx.x >= tiles[0].expert) return;
  const TileEntry te = tiles[1 + blockIdx.x];
  const int H = gu.K, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < kSimtRB) src_row[threadIdx.x] = threadIdx.x < te.rows ? perm[te.row0 + threadIdx.x] / k : 0;
  __syncthreads();
  stage_rows<A4>(xs, H, te.rows, x, xq, xsf, xgs, src_row);
  __syncthreads();
  for (int i = 0; i < 4; ++i) {
    const int n = blockIdx.y * kSimtNB + warp * 4 + i;
    float ag[kSimtRB], au[kSimtRB];
#pragma unroll
    for (int r = 0; r < kSimtRB; ++r) ag[r] = au[r] = 0.f;
    for (int k0 = lane * 8; k0 < H; k0 += 256) {
      float wg[8], wu[8];
      load_w8<FMT>(gu, te.expert, n, k0, wg);
      load_w8<FMT>(gu, te.expert, I + n, k0, wu);
#pragma unroll
      for (int r = 0; r < kSimtRB; ++r) {
        const float* xr = xs + r * H + k0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          ag[r] = fmaf(wg[j], xr[j], ag[r]);
          au[r] = fmaf(wu[j], xr[j], au[r]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < kSimtRB; ++r)
      for (int off = 16; off > 0; off >>= 1) {
        ag[r] += __shfl_xor_sync(0xffffffffu, ag[r], off);
        au[r] += __shfl_xor_sync(0xffffffffu, au[r], off);
      }
    if (lane == 0)
      for (int r = 0; r < te.rows; ++r) {
        const float v = silu_f(ag[r]) * au[r];
        h[(size_t)(te.row0 + r) * I + n] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
      }
  }
}

template <int FMT, bool A4>
__global__ void __launch_bounds__(128) down_simt_kernel(MatView dn, const uint16_t* __restrict__ h,
                                                        const uint8_t* __restrict__ hq,
                                                        const uint8_t* __restrict__ hsf,
                                                        const float* __restrict__ hgs,
                                                        const int32_t* __restrict__ perm,
                                                        const float* __restrict__ topk_w, int k,
                                                        const TileEntry* __restrict__ tiles,
                                                        uint16_t* __restrict__ y_out) {
  extern __shared__ float hs[];
  __shared__ int src_row[kSimtRB];
  if ((int)blockIdx.x >= tiles[0].expert) return;
  const TileEntry te = tiles[1 + blockIdx.x];
  const int I = dn.K, H = dn.N, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < kSimtRB) src_row[threadIdx.x] = te.row0 + min((int)threadIdx.x, te.rows - 1);
  __syncthreads();
  stage_rows<A4>(hs, I, te.rows, h, hq, hsf, hgs, src_row);
  __syncthreads();
  for (int i = 0; i < 4; ++i) {
    const int c = blockIdx.y * kSimtNB + warp * 4 + i;
    float acc[kSimtRB];
#pragma unroll
    for (int r = 0; r < kSimtRB; ++r) acc[r] = 0.f;
    for (int k0 = lane * 8; k0 < I; k0 += 256) {
      float w[8];
      load_w8<FMT>(dn, te.expert, c, k0, w);
#pragma unroll
      for (int r = 0; r < kSimtRB; ++r) {
        const float* hr = hs + r * I + k0;
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[r] = fmaf(w[j], hr[j], acc[r]);
      }
    }
#pragma unroll
    for (int r = 0; r < kSimtRB; ++r)
      for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
    if (lane == 0)
      for (int r = 0; r < te.rows; ++r) {
        const int p = perm[te.row0 + r];
        y_out[(size_t)(te.row0 + r) * H + c] = bf16_bits(topk_w[p] * acc[r]);
      }
  }
}

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

template <int FMT, bool A4>
cudaError_t run_simt(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                     const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, const float* h_gs = nullptr) {
  const int H = d.H, I = d.I;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  const TileEntry* tiles = (const TileEntry*)(ws + L.tiles);
  const int32_t* perm = (const int32_t*)(ws + L.perm);
  const size_t smem_gu = sizeof(float) * kSimtRB * H, smem_d = sizeof(float) * kSimtRB * I;
  cudaFuncSetAttribute(gateup_simt_kernel<FMT, A4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_gu);
  cudaFuncSetAttribute(down_simt_kernel<FMT, A4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_d);
  record_event(ev.start[0], s);
  gateup_simt_kernel<FMT, A4><<<dim3(L.max_tiles, I / kSimtNB), 128, smem_gu, s>>>(
      gu, (const uint16_t*)x, (const uint8_t*)(ws + L.xq), (const uint8_t*)(ws + L.xs),
      (const float*)(ws + L.xg), perm, k, I, tiles, (uint16_t*)(ws + L.h));
  record_event(ev.stop[0], s);
  if (A4)
    launch_quant_rows((const __nv_bfloat16*)(ws + L.h), nullptr, 1, T * k, I, (uint8_t*)(ws + L.hq), (uint8_t*)(ws + L.hs),
                      (float*)(ws + L.hg), s, false, 0, h_gs);
  record_event(ev.start[1], s);
  down_simt_kernel<FMT, A4><<<dim3(L.max_tiles, H / kSimtNB), 128, smem_d, s>>>(
      dn, (const uint16_t*)(ws + L.h), (const uint8_t*)(ws + L.hq), (const uint8_t*)(ws + L.hs),
      (const float*)(ws + L.hg), perm, (const float*)(ws + L.topk_w), k, tiles, (uint16_t*)(ws + L.y));
  record_event(ev.stop[1], s);
  note_launches(2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_experts(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                           int row_block, const WsLayout& L, char* ws, __nv_bfloat16* out, const StepEvents& ev,
                           cudaStream_t s, const float* act_gs) {
  const size_t n_out = (size_t)T * d.H;
  if (T == 0) return cudaGetLastError();
  cudaError_t e;
  if (d.fmt == MOE_FMT_NVFP4_W4A4 && fp4_supported(d)) {
    e = launch_experts_fp4(d, packed, x, T, k, L, ws, ev, s, act_gs);
  } else if (d.fmt == MOE_FMT_NVFP4_W4A4) {
    launch_quant_rows(x, nullptr, 1, T, d.H, (uint8_t*)(ws + L.xq), (uint8_t*)(ws + L.xs), (float*)(ws + L.xg), s,
                      false, 0, act_gs);
    e = run_simt<MOE_FMT_NVFP4_W4A16, true>(d, packed, x, T, k, L, ws, ev, s, act_gs ? act_gs + 1 : nullptr);
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

int simt_row_block() { return kSimtRB; }

}  // namespace moe
