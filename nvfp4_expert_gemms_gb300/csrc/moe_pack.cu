// Quantize-and-pack kernels (off the hot path) and the dequantization view.
// Every quantizer step is one IEEE fp32 operation with an explicit rounding intrinsic, so the
// packed bytes are reproducible bit for bit:
//   FP8   (clef-omni-fp8, "Recipe"): per 128x128 tile s = 448/amax, code = E4M3(w*s),
//         scale_inv = 1/s.
//   INT4  (clef-omni-int4, "What was quantized"): per (row, 128-group) s16 = fp16(amax/7),
//         q = clamp(rint(w/s16), -8, 7), code = q + 8, auto_gptq word order along K.
//   NVFP4 (clef-omni-NVFP4, "How it was made"): gs = 2688/amax(matrix); per 16-block
//         bs = E4M3((amax_b/6)*gs), q = E2M1(w/(bs/gs)).
// A zero amax is clamped to 1e-12 (FP8 tiles, NVFP4 matrices); an INT4 group with a zero
// scale stores the zero code 8.
#include "moe_formats.cuh"
#include "moe_nvfp4.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float block_max(float v, float* red) {
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = 0.f;
  for (int i = 0; i < nw; ++i) r = fmaxf(r, red[i]);
  return r;
}

// grid (K/128, N/128, E), 256 threads: thread t covers row t/2, columns (t%2)*64 .. +63.
__global__ void __launch_bounds__(256) pack_fp8_kernel(const uint16_t* __restrict__ w, int N, int K,
                                                       uint8_t* __restrict__ codes,
                                                       float* __restrict__ scale_inv) {
  __shared__ float red[8];
  const int tk = blockIdx.x, tn = blockIdx.y, e = blockIdx.z;
  const int r = threadIdx.x >> 1, c0 = (threadIdx.x & 1) * 64;
  const size_t base = ((size_t)e * N + tn * 128 + r) * K + tk * 128 + c0;
  float amax = 0.f;
  for (int c = 0; c < 64; ++c) amax = fmaxf(amax, fabsf(bf16_to_f32(w[base + c])));
  amax = block_max(amax, red);
  if (amax < 1e-12f) amax = 1e-12f;
  const float s = __fdiv_rn(448.0f, amax);
  for (int c = 0; c < 64; c += 4) {
    uint32_t word = 0;
    for (int i = 0; i < 4; ++i) word |= (uint32_t)f32_to_e4m3(__fmul_rn(bf16_to_f32(w[base + c + i]), s)) << (8 * i);
    *(uint32_t*)(codes + base + c) = word;
  }
  if (threadIdx.x == 0) scale_inv[((size_t)e * (N / 128) + tn) * (K / 128) + tk] = __fdiv_rn(1.0f, s);
}

// grid (N/128, K/128, E), 128 threads: thread = output row n of one 128-group.
__global__ void __launch_bounds__(128) pack_int4_kernel(const uint16_t* __restrict__ w, int N, int K,
                                                        uint32_t* __restrict__ qweight,
                                                        __half* __restrict__ scales) {
  const int n = blockIdx.x * 128 + threadIdx.x, g = blockIdx.y, e = blockIdx.z;
  const uint16_t* row = w + ((size_t)e * N + n) * K + g * 128;
  float amax = 0.f;
  for (int c = 0; c < 128; ++c) amax = fmaxf(amax, fabsf(bf16_to_f32(row[c])));
  const __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
  const float sf = __half2float(s16);
  scales[((size_t)e * (K / 128) + g) * N + n] = s16;
  for (int kr = 0; kr < 16; ++kr) {
    uint32_t word = 0;
    for (int j = 0; j < 8; ++j) {
      int code = 8;
      if (sf != 0.0f) {
        float q = rintf(__fdiv_rn(bf16_to_f32(row[kr * 8 + j]), sf));
        q = fminf(fmaxf(q, -8.0f), 7.0f);
        code = (int)q + 8;
      }
      word |= (uint32_t)code << (4 * j);
    }
    qweight[((size_t)e * (K / 8) + g * 16 + kr) * N + n] = word;
  }
}

// Matrix amax into the global-scale slot (as float bits; non-negative floats order like uints).
__global__ void __launch_bounds__(256) nvfp4_amax_kernel(const uint16_t* __restrict__ w, size_t per_expert,
                                                         unsigned* __restrict__ slot) {
  __shared__ float red[8];
  const int e = blockIdx.y;
  const uint16_t* m = w + (size_t)e * per_expert;
  float amax = 0.f;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < per_expert; i += (size_t)gridDim.x * blockDim.x)
    amax = fmaxf(amax, fabsf(bf16_to_f32(m[i])));
  amax = block_max(amax, red);
  if (threadIdx.x == 0) atomicMax(&slot[e], __float_as_uint(amax));
}

__device__ __forceinline__ void nvfp4_block(const float v[16], float gs, uint2* codes8, uint8_t* scale) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  nvfp4_encode(v, amax, gs, codes8, scale);
}

// thread = one (row, 16-block) of one expert matrix.
__global__ void __launch_bounds__(256) nvfp4_pack_kernel(const uint16_t* __restrict__ w, int N, int K,
                                                         const unsigned* __restrict__ amax_slot,
                                                         uint8_t* __restrict__ packed,
                                                         uint8_t* __restrict__ scales) {
  const int e = blockIdx.y;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;  // block index within the expert
  const size_t nblk = (size_t)N * K / 16;
  if (i >= nblk) return;
  float amax_m = __uint_as_float(amax_slot[e]);
  if (amax_m < 1e-12f) amax_m = 1e-12f;
  const float gs = __fdiv_rn(2688.0f, amax_m);
  const uint16_t* src = w + (size_t)e * N * K + i * 16;
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = bf16_to_f32(src[j]);
  nvfp4_block(v, gs, (uint2*)(packed + (size_t)e * N * K / 2 + i * 8), scales + (size_t)e * nblk + i);
}

// The W4A4 operand image of one expert matrix [E, N, K] (canonical codes [E, N, K/2] and block
// scales [E, N, K/16] in, ActImage layout out): thread = one row of one (tile pair, chunk) block,
// writing its 128 code bytes (16-byte pieces swizzled) and its 16 scales.  gate/up (gu): pair p
// = gate rows 128p.. over up rows I + 128p..; down: rows 256p .. 256p + 255 (rows past N zero).
// Columns past K (a last half chunk) are zero.
__global__ void __launch_bounds__(256) nvfp4_image_kernel(const uint8_t* __restrict__ codes,
                                                          const uint8_t* __restrict__ scales, int E, int N, int K,
                                                          bool gu, uint8_t* __restrict__ img) {
  const int C = nvfp4_chunks(K), P = gu ? N / 256 : (N + 255) / 256;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)E * P * C * 256) return;
  const int nl = (int)(i % 256), c = (int)((i / 256) % C), p = (int)((i / 256 / C) % P), e = (int)(i / 256 / C / P);
  const int g = nl >> 7, l = nl & 127;
  const int n = gu ? (g == 0 ? 128 * p + l : N / 2 + 128 * p + l) : 256 * p + nl;
  uint8_t* blk = img + (((size_t)e * P + p) * C + c) * kWImgBlock;
  uint8_t* tcodes = blk + g * kImgTile;
  uint8_t* tsf = blk + 2 * kImgTile + g * kImgSf;
  const int kb = min(128, K / 2 - 128 * c);  // code bytes of this row in the chunk (64 for a half chunk)
  const bool row_ok = n < N;
  const uint8_t* src = codes + ((size_t)e * N + (row_ok ? n : 0)) * (K / 2) + 128 * c;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (row_ok && 16 * j < kb) v = *(const uint4*)(src + 16 * j);
    *(uint4*)(tcodes + 128 * l + ((j ^ (l & 7)) << 4)) = v;
  }
  const uint8_t* ssrc = scales + ((size_t)e * N + (row_ok ? n : 0)) * (K / 16) + 16 * c;
  for (int b = 0; b < 16; ++b) tsf[img_wsf_byte(l, b)] = row_ok && 8 * b < kb ? ssrc[b] : (uint8_t)0;
}

// One 32-bit word of eight E2M1 codes in the bf16 converter's bit order (conv_nvfp4 in
// moe_gemm_tc.cu): element k = nibble k of the canonical word (code bits m, e0, e1, s = bits
// 0..3), its bits moved so that element pair j comes out of one shift-and-mask of the word: pair
// 0 by << 6, pair 1 by << 2, pair 2 by a rotate right by 4, pair 3 in place except the two
// mantissa bits (>> 8).
__device__ __forceinline__ uint32_t w4a16_image_word(uint32_t c) {
  constexpr uint8_t kDst[8][4] = {{0, 1, 2, 9},     {16, 17, 18, 25}, {4, 5, 6, 13},  {20, 21, 22, 29},
                                  {10, 11, 12, 19}, {26, 27, 28, 3},  {14, 7, 8, 15}, {30, 23, 24, 31}};
  uint32_t o = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k)
#pragma unroll
    for (int b = 0; b < 4; ++b) o |= ((c >> (4 * k + b)) & 1u) << kDst[k][b];
  return o;
}

// The W4A16 weight image of one expert matrix (canonical codes [E, N, K/2], scales [E, N, K/16]),
// blocks [E, K/128, N/128]: thread = one row l of one (expert, 128-column chunk c, 128-row tile b)
// block; gate/up (gu) tile b = gate rows 64b.. then up rows N/2 + 64b..; down tile b = rows 128b...
__global__ void __launch_bounds__(256) nvfp4_w4a16_image_kernel(const uint8_t* __restrict__ codes,
                                                                const uint8_t* __restrict__ scales, int E, int N,
                                                                int K, bool gu, uint8_t* __restrict__ img) {
  const int C = K / 128, NB = N / 128;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)E * NB * C * 128) return;
  const int l = (int)(i % 128), b = (int)((i / 128) % NB), c = (int)((i / 128 / NB) % C), e = (int)(i / 128 / NB / C);
  const int n = gu ? (l < 64 ? 64 * b + l : N / 2 + 64 * b + l - 64) : 128 * b + l;
  uint8_t* blk = img + (((size_t)e * C + c) * NB + b) * kW16Block;
  const uint8_t* src = codes + ((size_t)e * N + n) * (K / 2) + 64 * c;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint4 v = *(const uint4*)(src + 16 * p);
    const uint4 o = make_uint4(w4a16_image_word(v.x), w4a16_image_word(v.y), w4a16_image_word(v.z),
                               w4a16_image_word(v.w));
    *(uint4*)(blk + 64 * l + ((p ^ ((l >> 1) & 3)) << 4)) = o;
  }
  *(uint2*)(blk + kW16Codes + 8 * l) = *(const uint2*)(scales + ((size_t)e * N + n) * (K / 16) + 8 * c);
}

__global__ void nvfp4_finish_kernel(unsigned* slot, int E) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < E) {
    float a = __uint_as_float(slot[e]);
    if (a < 1e-12f) a = 1e-12f;
    ((float*)slot)[e] = __fdiv_rn(2688.0f, a);
  }
}

// Byte offset of the block scale of 16-block b of row d: row-major [rows, K/16], or with
// sf_rows > 0 chunk-major [C][sf_rows][16] (C = ceil(K/256); every 256-column chunk of a run of
// rows is one contiguous block, as the block-scaled MMA path loads it; a last half chunk fills
// 8 of its row's 16 bytes).
__device__ __forceinline__ size_t sf_index(size_t d, int b, int K, int sf_rows) {
  return sf_rows ? ((size_t)(b >> 4) * sf_rows + d) * 16 + (b & 15) : d * (K / 16) + b;
}

// Dynamic NVFP4 quantization of bf16 rows (W4A4 activations): one warp per input row r;
// gs_row = 2688 / max(amax_row, 1e-12), then blocks exactly as for weights.  The codes, scales
// and gs_row go to output row r, or, with a scatter map, to each of rows scatter[r*k .. r*k+k-1]
// (the expert-permuted copies of a token: computed once, stored k times).
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint16_t* __restrict__ x,
                                                         const int32_t* __restrict__ scatter, int k, int rows, int K,
                                                         uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                         float* __restrict__ gs_out, int sf_rows,
                                                         const float* __restrict__ static_gs, ActImage im) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (r >= rows) return;
  const uint16_t* row = x + (size_t)r * K;
  float amax = 0.f;
  for (int c = lane * 8; c < K; c += 256) {
    const uint4 u = *(const uint4*)(row + c);
    const uint32_t ww[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      amax = fmaxf(amax, fabsf(__uint_as_float(ww[i] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(ww[i] & 0xFFFF0000u)));
    }
  }
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if (amax < 1e-12f) amax = 1e-12f;
  const float gs = static_gs ? *static_gs : __fdiv_rn(2688.0f, amax);
  const int ncopy = scatter ? k : 1;
  if (gs_out && lane < ncopy) gs_out[scatter ? scatter[(size_t)r * k + lane] : r] = gs;
  for (int b = lane; b < K / 16; b += 32) {
    const uint4 u0 = *(const uint4*)(row + b * 16), u1 = *(const uint4*)(row + b * 16 + 8);
    const uint32_t ww[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float v[16];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[2 * j] = __uint_as_float(ww[j] << 16);
      v[2 * j + 1] = __uint_as_float(ww[j] & 0xFFFF0000u);
    }
    uint2 code;
    uint8_t scale;
    nvfp4_block(v, gs, &code, &scale);
    for (int c = 0; c < ncopy; ++c) {
      const size_t src = scatter ? (size_t)r * k + c : 0;
      const size_t d = scatter ? (size_t)scatter[src] : (size_t)r;
      if (im.img) {
        const int e = im.topk_idx[scatter ? src : (size_t)im.perm[d]];
        const int slot = img_slot((int)d, e, im.offsets, im.toff);
        uint8_t* blk = im.img + ((size_t)(slot >> 7) * im.chunks + (b >> 4)) * kAImgBlock;
        *(uint2*)(blk + img_code_byte(slot & 127, b & 15)) = code;
        blk[kImgTile + 16 * (slot & 127) + (b & 15)] = scale;
      } else {
        *(uint2*)(q + d * (K / 2) + b * 8) = code;
        sf[sf_index(d, b, K, sf_rows)] = scale;
      }
    }
  }
}

// The same quantization with RPW whole rows of K = 16*NBLK elements held in registers.  The
// rows are contiguous, so their 16-blocks form one flat run of RPW*NBLK blocks: lane l owns
// blocks l, l+32, ..., loads all of them before any arithmetic and reads each row once.  Block
// and row maxima are taken on the bf16 magnitude bits (for finite values the integer order of
// |v| is the float order).  EARLY: the rows were final before the preceding kernel of the stream
// passed its own pdl_wait(), so they are loaded before this kernel's wait and only the stores
// follow it.
template <int NBLK, int RPW, bool EARLY>
__global__ void __launch_bounds__(256) quant_rows_flat_kernel(const uint16_t* __restrict__ x,
                                                              const int32_t* __restrict__ scatter, int k, int rows,
                                                              uint8_t* __restrict__ q, uint8_t* __restrict__ sf,
                                                              float* __restrict__ gs_out, int sf_rows,
                                                              const float* __restrict__ static_gs, ActImage im) {
  constexpr int K = 16 * NBLK, kFlat = NBLK * RPW, NB = (kFlat + 31) / 32;
  static_assert(NB <= 8 && RPW * kMaxTopK <= 32, "flat quantizer shape");
  const int lane = threadIdx.x & 31;
  const int r0 = (blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * RPW;
  const uint4* base = (const uint4*)(x + (size_t)r0 * K);
  if (!EARLY) pdl_wait();
  uint4 u[NB][2];
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const int f = lane + 32 * j;
    if (f < kFlat && r0 + f / NBLK < rows) {
      u[j][0] = __ldcs(base + 2 * f);
      u[j][1] = __ldcs(base + 2 * f + 1);
    } else {
      u[j][0] = u[j][1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if (EARLY) pdl_wait();
  pdl_trigger();

  uint32_t bmax[NB], rmax[RPW];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) rmax[rr] = 0u;
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const uint32_t m = 0x7FFF7FFFu;
    uint32_t t = __vmaxu2(__vmaxu2(u[j][0].x & m, u[j][0].y & m), __vmaxu2(u[j][0].z & m, u[j][0].w & m));
    t = __vmaxu2(t, __vmaxu2(__vmaxu2(u[j][1].x & m, u[j][1].y & m), __vmaxu2(u[j][1].z & m, u[j][1].w & m)));
    bmax[j] = max(t & 0xFFFFu, t >> 16);
    const int row = (lane + 32 * j) / NBLK;
#pragma unroll
    for (int rr = 0; rr < RPW; ++rr)
      if (row == rr) rmax[rr] = max(rmax[rr], bmax[j]);
  }
  float gs[RPW];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) {
    float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, rmax[rr]) << 16);
    if (amax < 1e-12f) amax = 1e-12f;
    gs[rr] = static_gs ? *static_gs : __fdiv_rn(2688.0f, amax);
  }
  // destinations: lane rr*k + c holds row rr's copy c (scatter), else row r0 + rr
  const int ncopy = scatter ? k : 1;
  int my_dst = 0, my_slot = 0;  // permuted row, and with an image its slot there
  if (scatter) {
    if (lane < RPW * k && r0 + lane / k < rows) {
      const size_t src = (size_t)(r0 + lane / k) * k + lane % k;
      my_dst = scatter[src];
      if (im.img) my_slot = img_slot(my_dst, im.topk_idx[src], im.offsets, im.toff);
    }
  } else {
    my_dst = r0 + lane;
    if (im.img && lane < RPW && my_dst < rows) my_slot = img_slot(my_dst, im.topk_idx[im.perm[my_dst]], im.offsets, im.toff);
  }
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr)
    if (gs_out && lane / ncopy == rr && lane < RPW * ncopy && r0 + rr < rows) gs_out[my_dst] = gs[rr];
#pragma unroll
  for (int j = 0; j < NB; ++j) {
    const int f = lane + 32 * j, row = f / NBLK, b = f % NBLK;
    const bool live = f < kFlat && r0 + row < rows;
    float g = gs[0];
#pragma unroll
    for (int rr = 1; rr < RPW; ++rr)
      if (row == rr) g = gs[rr];
    const uint32_t ww[8] = {u[j][0].x, u[j][0].y, u[j][0].z, u[j][0].w, u[j][1].x, u[j][1].y, u[j][1].z, u[j][1].w};
    float v[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = __uint_as_float(ww[i] << 16);
      v[2 * i + 1] = __uint_as_float(ww[i] & 0xFFFF0000u);
    }
    uint2 code;
    uint8_t scale;
    nvfp4_encode(v, __uint_as_float(bmax[j] << 16), g, &code, &scale);
    for (int c = 0; c < ncopy; ++c) {  // warp-uniform trip count: the shuffle sees every lane
      const int from = (row < RPW ? row : 0) * ncopy + c;
      const int d = __shfl_sync(0xffffffffu, my_dst, from);
      const int slot = __shfl_sync(0xffffffffu, my_slot, from);
      if (live) {
        if (im.img) {
          uint8_t* blk = im.img + ((size_t)(slot >> 7) * im.chunks + (b >> 4)) * kAImgBlock;
          *(uint2*)(blk + img_code_byte(slot & 127, b & 15)) = code;
          blk[kImgTile + 16 * (slot & 127) + (b & 15)] = scale;
        } else {
          *(uint2*)(q + (size_t)d * (K / 2) + b * 8) = code;
          sf[sf_index((size_t)d, b, K, sf_rows)] = scale;
        }
      }
    }
  }
}

// out[r] = x[map[r] / k]: the expert-permuted copy of the activation rows (one warp per row).
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ map,
                                                          int k, int rows, int row_vec, uint4* __restrict__ out) {
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  pdl_wait();
  pdl_trigger();
  if (r >= rows) return;
  const uint4* src = x + (size_t)(map[r] / k) * row_vec;
  uint4* dst = out + (size_t)r * row_vec;
  for (int c = lane; c < row_vec; c += 32) dst[c] = src[c];
}

template <int FMT>
__global__ void __launch_bounds__(256) dequant_kernel(MatView m, int e, float* __restrict__ out) {
  const size_t i = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i >= (size_t)m.N * m.K) return;
  const int n = (int)(i / m.K), k0 = (int)(i % m.K);
  float w[8];
  load_w8<FMT>(m, e, n, k0, w);
#pragma unroll
  for (int j = 0; j < 8; ++j) out[i + j] = w[j];
}

}  // namespace

cudaError_t launch_pack(const moe_packed_desc_t& d, const __nv_bfloat16* wgu, const __nv_bfloat16* wd, char* packed,
                        cudaStream_t s) {
  const int E = d.E, H = d.H, I = d.I;
  for (int which = 0; which < 2; ++which) {
    const uint16_t* w = (const uint16_t*)(which == 0 ? wgu : wd);
    const int N = which == 0 ? 2 * I : H, K = which == 0 ? H : I;
    uint8_t* a = (uint8_t*)(packed + d.offset[which == 0 ? MOE_T_GU_A : MOE_T_D_A]);
    uint8_t* b = (uint8_t*)(packed + d.offset[which == 0 ? MOE_T_GU_B : MOE_T_D_B]);
    if (d.fmt == MOE_FMT_BF16) {  // unquantized: the canonical tensors are the weights themselves
      const cudaError_t e = cudaMemcpyAsync(a, w, (size_t)E * N * K * 2, cudaMemcpyDeviceToDevice, s);
      if (e != cudaSuccess) return e;
      continue;
    }
    if (d.fmt == MOE_FMT_FP8_B128_W8A16 || d.fmt == MOE_FMT_FP8_B128_W8A8) {
      pack_fp8_kernel<<<dim3(K / 128, N / 128, E), 256, 0, s>>>(w, N, K, a, (float*)b);
    } else if (d.fmt == MOE_FMT_INT4_G128_W4A16) {
      pack_int4_kernel<<<dim3(N / 128, K / 128, E), 128, 0, s>>>(w, N, K, (uint32_t*)a, (__half*)b);
    } else {
      unsigned* slot = (unsigned*)(packed + d.offset[which == 0 ? MOE_T_GU_GS : MOE_T_D_GS]);
      cudaMemsetAsync(slot, 0, sizeof(float) * E, s);
      const size_t per = (size_t)N * K;
      nvfp4_amax_kernel<<<dim3(64, E), 256, 0, s>>>(w, per, slot);
      const size_t nblk = per / 16;
      nvfp4_pack_kernel<<<dim3((unsigned)((nblk + 255) / 256), E), 256, 0, s>>>(w, N, K, slot, a, b);
      nvfp4_finish_kernel<<<(E + 127) / 128, 128, 0, s>>>(slot, E);
      note_launches(2);
      const int it = which == 0 ? MOE_T_GU_IMG : MOE_T_D_IMG;
      if (d.size[it] && d.fmt == MOE_FMT_NVFP4_W4A16) {
        const size_t n = d.size[it] / kW16Block * 128;
        nvfp4_w4a16_image_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, b, E, N, K, which == 0,
                                                                              (uint8_t*)(packed + d.offset[it]));
        note_launches(1);
      } else if (d.size[it]) {
        const size_t n = d.size[it] / kWImgBlock * 256;
        nvfp4_image_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(a, b, E, N, K, which == 0,
                                                                        (uint8_t*)(packed + d.offset[it]));
        note_launches(1);
      }
    }
    note_launches(1);
  }
  return cudaGetLastError();
}

cudaError_t launch_act_scale(const uint16_t* v, size_t n, float* gs, cudaStream_t s) {
  // the dynamic rule over a whole tensor: gs = 2688 / max(amax, 1e-12), amax over n bf16 values
  const cudaError_t e = cudaMemsetAsync(gs, 0, sizeof(float), s);
  if (e != cudaSuccess) return e;
  nvfp4_amax_kernel<<<dim3(64, 1), 256, 0, s>>>(v, n, (unsigned*)gs);
  nvfp4_finish_kernel<<<1, 128, 0, s>>>((unsigned*)gs, 1);
  note_launches(2);
  return cudaGetLastError();
}

cudaError_t launch_dequant(const moe_packed_desc_t& d, const char* packed, int e, int which, float* out,
                           cudaStream_t s) {
  const MatView m = mat_view(d, packed, which);
  const unsigned blocks = (unsigned)(((size_t)m.N * m.K / 8 + 255) / 256);
  if (d.fmt == MOE_FMT_FP8_B128_W8A16 || d.fmt == MOE_FMT_FP8_B128_W8A8)
    dequant_kernel<MOE_FMT_FP8_B128_W8A16><<<blocks, 256, 0, s>>>(m, e, out);
  else if (d.fmt == MOE_FMT_BF16) dequant_kernel<MOE_FMT_BF16><<<blocks, 256, 0, s>>>(m, e, out);
  else if (d.fmt == MOE_FMT_INT4_G128_W4A16) dequant_kernel<MOE_FMT_INT4_G128_W4A16><<<blocks, 256, 0, s>>>(m, e, out);
  else dequant_kernel<MOE_FMT_NVFP4_W4A16><<<blocks, 256, 0, s>>>(m, e, out);
  note_launches(1);
  return cudaGetLastError();
}

template <int NBLK, int RPW>
static cudaError_t launch_quant_flat(bool early, const __nv_bfloat16* x, const int32_t* scatter, int k, int rows,
                                     uint8_t* q, uint8_t* sf, float* gs, int sf_rows, const float* static_gs,
                                     const ActImage& im, cudaStream_t s) {
  const dim3 grid((rows + 8 * RPW - 1) / (8 * RPW));
  if (early)
    return launch_pdl(quant_rows_flat_kernel<NBLK, RPW, true>, grid, dim3(256), 0, s, (const uint16_t*)x, scatter, k,
                      rows, q, sf, gs, sf_rows, static_gs, im);
  return launch_pdl(quant_rows_flat_kernel<NBLK, RPW, false>, grid, dim3(256), 0, s, (const uint16_t*)x, scatter, k,
                    rows, q, sf, gs, sf_rows, static_gs, im);
}

cudaError_t launch_quant_rows(const __nv_bfloat16* x, const int32_t* scatter, int k, int rows, int K, uint8_t* q,
                              uint8_t* sf, float* gs, cudaStream_t s, bool early, int sf_rows,
                              const float* static_gs, const ActImage* img) {
  if (rows <= 0) return cudaGetLastError();
  const ActImage im = img ? *img : ActImage();
  note_launches(1);
  switch (K) {  // register-resident shapes: RPW rows fill whole 32-lane passes of 16-blocks
    case 128: return launch_quant_flat<8, 4>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    case 256: return launch_quant_flat<16, 2>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    case 512: return launch_quant_flat<32, 1>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    case 768: return launch_quant_flat<48, 2>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    case 1024: return launch_quant_flat<64, 1>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    case 1280: return launch_quant_flat<80, 2>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    case 1536: return launch_quant_flat<96, 1>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    case 2048: return launch_quant_flat<128, 1>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    case 3072: return launch_quant_flat<192, 1>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    case 4096: return launch_quant_flat<256, 1>(early, x, scatter, k, rows, q, sf, gs, sf_rows, static_gs, im, s);
    default:
      return launch_pdl(quant_rows_kernel, dim3((rows + 7) / 8), dim3(256), 0, s, (const uint16_t*)x, scatter, k, rows,
                        K, q, sf, gs, sf_rows, static_gs, im);
  }
}

cudaError_t launch_gather_rows(const __nv_bfloat16* x, const int32_t* map, int k, int rows, int K, __nv_bfloat16* out,
                               cudaStream_t s) {
  if (rows <= 0) return cudaGetLastError();
  note_launches(1);
  return launch_pdl(gather_rows_kernel, dim3((rows + 7) / 8), dim3(256), 0, s, (const uint4*)x, map, k, rows, K / 8,
                    (uint4*)out);
}

}  // namespace moe
