// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05) for the weight-only
// formats (FP8 W8A16, INT4 W4A16, NVFP4 W4A16).
//
// The pages run the experts as "dequantize, then a grouped matmul" (clef-omni-fp8, "How this
// checkpoint runs"; clef-omni-int4, same section; clef-omni-NVFP4, "How it was made").  Here the
// dequantization is fused into the GEMM and never reaches HBM:
//
//   weights (packed, HBM) --TMA--> shared memory --converter warps--> bf16 A operand in TMEM
//   activations (bf16)    --TMA gather4 / tile--> shared memory (128-byte swizzle) = B operand
//   tcgen05.mma kind::f16: D[weight row, token] += A[weight row, k] * B[token, k]   (fp32, TMEM)
//
// Weight rows are the MMA's M side (128 per sub-tile) and tokens its N side (BN = 16..128), so a
// decode step with one or two tokens per expert still issues full-rate 128-row MMAs while the
// kernel streams weights.  Each CTA covers one row block of one expert (from the routing tile
// table) and two 128-row weight sub-tiles: gate rows n0.. and up rows I+n0.. for the gate/up
// GEMM (so SiLU(gate)*up is computed in the epilogue from two TMEM accumulators), or 256
// consecutive output features for the down GEMM (whose epilogue scales by the routing weight
// and adds into the fp32 token-order accumulator).
//
// Warp roles (320 threads): warps 0-7 convert (warp w: sub-tile w/4, TMEM lanes 32*(w%4)..) and
// later run the epilogue; warp 8 issues TMA; warp 9 owns TMEM and issues the MMAs.
#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "moe_formats.cuh"
#include "moe_tc.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kKC = 128;          // K elements per pipeline chunk
constexpr int kThreads = 320;
constexpr int kStagesW = 4;       // weight chunks in flight (shared memory)
constexpr int kStagesA = 2;       // converted A chunks (TMEM)
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol = 256;   // TMEM columns [256, 512): A ring; [0, 2*BN): accumulators

template <int FMT>
struct WFmt;
template <>
struct WFmt<MOE_FMT_FP8_B128_W8A16> {
  static constexpr int kSubBytes = 128 * 128;  // 128 rows x 128 codes, 128-byte swizzle
};
template <>
struct WFmt<MOE_FMT_INT4_G128_W4A16> {
  static constexpr int kSubBytes = 16 * 128 * 4;  // 16 qweight rows (128 K) x 128 columns
};
template <>
struct WFmt<MOE_FMT_NVFP4_W4A16> {
  static constexpr int kSubBytes = 128 * 64;  // 128 rows x 64 bytes (128 codes), 64-byte swizzle
};

struct TcArgs {
  CUtensorMap wmap;  // packed weight codes of the matrix
  CUtensorMap bmap;  // activations: x (gate/up, one-row box for gather4) or h (down, BN-row box)
  const void* wscale;
  const float* wgs;
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;
  float* out_acc;
  int* err;
  int k, N, K, I, H;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// ---- converters: raw chunk of one weight row (128 K) -> 64 bf16x2 words ------------------
// FP8: e4m3 bits re-based into an fp32 exponent (value * 2^-120, exact incl. subnormals), an
// exact multiply by 2^120, then one fp32 multiply by scale_inv and one rounding to bf16.
__device__ __forceinline__ void conv_fp8(const char* sub, int r, float sc, uint32_t* out) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 q = *(const uint4*)(sub + r * 128 + ((c ^ (r & 7)) * 16));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float f[4];
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = (w[i] >> (8 * b)) & 0xFFu;
        f[b] = (__uint_as_float(((byte & 0x7Fu) << 20) | ((byte & 0x80u) << 24)) * 0x1p120f) * sc;
      }
      out[c * 8 + i * 2] = pack_bf16x2(f[0], f[1]);
      out[c * 8 + i * 2 + 1] = pack_bf16x2(f[2], f[3]);
    }
  }
}

// INT4: 16 qweight words of column r (rows kr = 0..15 of the chunk), (code - 8) * scale.
__device__ __forceinline__ void conv_int4(const char* sub, int r, float s, uint32_t* out) {
#pragma unroll
  for (int kr = 0; kr < 16; ++kr) {
    const uint32_t q = *(const uint32_t*)(sub + kr * 512 + r * 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = (float)((int)((q >> (8 * i)) & 0xF) - 8) * s;
      const float hi = (float)((int)((q >> (8 * i + 4)) & 0xF) - 8) * s;
      out[kr * 4 + i] = pack_bf16x2(lo, hi);
    }
  }
}

// NVFP4: e2m1 * e4m3 block scale is exact in bf16; the global scale is applied in the epilogue.
__device__ __forceinline__ void conv_nvfp4(const char* sub, int r, uint2 bs8, uint32_t* out) {
  const uint32_t bsw[2] = {bs8.x, bs8.y};
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // 16-byte chunk c = 32 codes = two 16-element blocks
    const uint4 q = *(const uint4*)(sub + r * 64 + ((c ^ ((r >> 1) & 3)) * 16));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int blk = c * 2 + (i >> 1);
      const float bs = e4m3_to_f32((bsw[blk >> 2] >> (8 * (blk & 3))) & 0xFF);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t byte = (w[i] >> (8 * p)) & 0xFFu;
        out[c * 16 + i * 4 + p] = pack_bf16x2(e2m1_to_f32(byte & 0xF) * bs, e2m1_to_f32(byte >> 4) * bs);
      }
    }
  }
}

// MODE 0: gate/up GEMM + SiLU(gate)*up -> h (bf16, permuted row order).
// MODE 1: down GEMM + routing weight -> fp32 red.add into the token-order accumulator.
template <int FMT, int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1) tc_expert_gemm_kernel(const __grid_constant__ TcArgs a) {
  constexpr int SB = BN >= 64 ? 2 : 4;  // activation stages
  constexpr int WSUB = WFmt<FMT>::kSubBytes;
  constexpr int WSTAGE = 2 * WSUB;
  constexpr int BSTAGE = BN * 256;  // BN rows x 128 K bf16, two 128-byte swizzle atoms
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = (char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  char* sW = smem;
  char* sB = smem + kStagesW * WSTAGE;
  __shared__ uint64_t w_full[kStagesW], w_empty[kStagesW], a_full[kStagesA], a_empty[kStagesA], b_full[SB],
      b_empty[SB], acc_full;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_tok[BN];
  __shared__ float s_w[BN];

  if ((int)blockIdx.x >= a.tiles[0].expert) return;  // header entry holds the tile count
  const TileEntry te = a.tiles[1 + blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = te.expert, row0 = te.row0, rows = te.rows;
  int nbase0, nbase1, nsub;
  if (MODE == 0) {
    nbase0 = blockIdx.y * 128;
    nbase1 = a.I + nbase0;
    nsub = 2;
  } else {
    nbase0 = blockIdx.y * 256;
    nbase1 = nbase0 + 128;
    nsub = (a.H - nbase0) >= 256 ? 2 : 1;
  }
  const int nK = a.K / kKC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesW; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], 4 * nsub);
    }
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(&a_full[i], 4 * nsub);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    mbar_init(&acc_full, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (threadIdx.x < BN) {
    const int j = threadIdx.x;
    const int p = a.perm[row0 + (j < rows ? j : rows - 1)];
    s_tok[j] = p / a.k;
    s_w[j] = j < rows ? a.topk_w[p] : 0.f;
  }
  if (warp == 9) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    prefetch_tmap(&a.wmap);
    prefetch_tmap(&a.bmap);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int armed_w[kStagesW] = {0}, armed_b[SB] = {0};
      for (int kc = 0; kc < nK && !s_abort; ++kc) {
        const int sw = kc % kStagesW;
        if (!mbar_wait(&w_empty[sw], ((kc / kStagesW) & 1) ^ 1, &s_abort)) break;
        mbar_arrive_expect_tx(&w_full[sw], nsub * WSUB);
        ++armed_w[sw];
        for (int g = 0; g < nsub; ++g) {
          char* dst = sW + sw * WSTAGE + g * WSUB;
          const int nb = g == 0 ? nbase0 : nbase1;
          if (FMT == MOE_FMT_FP8_B128_W8A16) tma_load_2d(dst, &a.wmap, &w_full[sw], kc * kKC, e * a.N + nb);
          else if (FMT == MOE_FMT_INT4_G128_W4A16) tma_load_2d(dst, &a.wmap, &w_full[sw], nb, e * (a.K / 8) + kc * 16);
          else tma_load_2d(dst, &a.wmap, &w_full[sw], kc * (kKC / 2), e * a.N + nb);
        }
        const int sb = kc % SB;
        if (!mbar_wait(&b_empty[sb], ((kc / SB) & 1) ^ 1, &s_abort)) break;
        mbar_arrive_expect_tx(&b_full[sb], BSTAGE);
        ++armed_b[sb];
        char* bd = sB + sb * BSTAGE;
#pragma unroll
        for (int at = 0; at < 2; ++at) {
          if (MODE == 0) {
            for (int j = 0; j < BN; j += 4)
              tma_gather4(bd + at * BN * 128 + j * 128, &a.bmap, &b_full[sb], kc * kKC + at * 64, s_tok[j],
                          s_tok[j + 1], s_tok[j + 2], s_tok[j + 3]);
          } else {
            tma_load_2d(bd + at * BN * 128, &a.bmap, &b_full[sb], kc * kKC + at * 64, row0);
          }
        }
      }
      if (s_abort) {  // let every issued copy land before the CTA's shared memory goes away
        volatile int no_abort = 0;
        for (int i = 0; i < kStagesW; ++i)
          if (armed_w[i]) mbar_wait(&w_full[i], (armed_w[i] - 1) & 1, &no_abort);
        for (int i = 0; i < SB; ++i)
          if (armed_b[i]) mbar_wait(&b_full[i], (armed_b[i] - 1) & 1, &no_abort);
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, BN);
      for (int kc = 0; kc < nK && !s_abort; ++kc) {
        const int sa = kc % kStagesA, sb = kc % SB;
        if (!mbar_wait(&a_full[sa], (kc / kStagesA) & 1, &s_abort)) break;
        if (!mbar_wait(&b_full[sb], (kc / SB) & 1, &s_abort)) break;
        fence_after_sync();
        const uint32_t b0 = smem_u32(sB + sb * BSTAGE);
        for (int g = 0; g < nsub; ++g)
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t bdsc = sdesc_k_sw128(b0 + (ks >> 2) * BN * 128 + (ks & 3) * 32);
            mma_f16_ts(tmem + g * BN, tmem + kACol + sa * 128 + g * 64 + ks * 8, bdsc, idesc, (kc | ks) != 0);
          }
        mma_commit(&a_empty[sa]);
        mma_commit(&b_empty[sb]);
      }
      mma_commit(&acc_full);  // always committed, so the epilogue can drain even after an abort
    }
  } else {
    // ---------------- converters: packed weights -> bf16 A in TMEM ----------------
    const int g = warp >> 2, q = warp & 3, r = q * 32 + lane;
    const int nb = g == 0 ? nbase0 : nbase1;
    if (g < nsub) {
      for (int kc = 0; kc < nK && !s_abort; ++kc) {
        const int sw = kc % kStagesW, sa = kc % kStagesA;
        float sc = 1.f;
        uint2 bs8 = make_uint2(0, 0);
        if (FMT == MOE_FMT_FP8_B128_W8A16)
          sc = ((const float*)a.wscale)[((size_t)e * (a.N / 128) + nb / 128) * (a.K / 128) + kc];
        else if (FMT == MOE_FMT_INT4_G128_W4A16)
          sc = __half2float(((const __half*)a.wscale)[((size_t)e * (a.K / 128) + kc) * a.N + nb + r]);
        else
          bs8 = *(const uint2*)((const uint8_t*)a.wscale + ((size_t)e * a.N + nb + r) * (a.K / 16) + kc * 8);
        if (!mbar_wait(&w_full[sw], (kc / kStagesW) & 1, &s_abort)) break;
        uint32_t v[64];
        const char* sub = sW + sw * WSTAGE + g * WSUB;
        if (FMT == MOE_FMT_FP8_B128_W8A16) conv_fp8(sub, r, sc, v);
        else if (FMT == MOE_FMT_INT4_G128_W4A16) conv_int4(sub, r, sc, v);
        else conv_nvfp4(sub, r, bs8, v);
        __syncwarp();
        if (lane == 0) mbar_arrive(&w_empty[sw]);
        if (!mbar_wait(&a_empty[sa], ((kc / kStagesA) & 1) ^ 1, &s_abort)) break;
        fence_after_sync();
        const uint32_t ta = taddr(tmem, q * 32, kACol + sa * 128 + g * 64);
        tmem_st_32x32(ta, v);
        tmem_st_32x32(ta + 32, v + 32);
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[sa]);
      }
    }
  }

  // ---------------- epilogue ----------------
  {
    volatile int no_abort = 0;
    mbar_wait(&acc_full, 0, &no_abort);  // bounded; drains outstanding MMAs in every case
  }
  fence_after_sync();
  if (warp < 8 && !s_abort) {
    const int q = warp & 3, half = warp >> 2, r = q * 32 + lane;
    const float gs = FMT == MOE_FMT_NVFP4_W4A16 ? a.wgs[e] : 1.f;
    if (MODE == 0) {
      const int cbeg = BN == 16 ? 0 : half * (BN / 2);
      const int cend = BN == 16 ? (half == 0 ? 16 : 0) : cbeg + BN / 2;
      const int n = nbase0 + r;
      for (int c0 = cbeg; c0 < cend; c0 += 16) {
        uint32_t G[16], U[16];
        tmem_ld_32x16(taddr(tmem, q * 32, c0), G);
        tmem_ld_32x16(taddr(tmem, q * 32, BN + c0), U);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = c0 + j;
          if (col < rows) {
            float gv = __uint_as_float(G[j]), uv = __uint_as_float(U[j]);
            if (FMT == MOE_FMT_NVFP4_W4A16) {
              gv = __fdiv_rn(gv, gs);
              uv = __fdiv_rn(uv, gs);
            }
            const float hv = gv / (1.0f + expf(-gv)) * uv;
            a.h_out[(size_t)(row0 + col) * a.I + n] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
          }
        }
      }
    } else if (half < nsub) {
      const int c = (half == 0 ? nbase0 : nbase1) + r;
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t Y[16];
        tmem_ld_32x16(taddr(tmem, q * 32, half * BN + c0), Y);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int col = c0 + j;
          if (col < rows) {
            float y = __uint_as_float(Y[j]);
            if (FMT == MOE_FMT_NVFP4_W4A16) y = __fdiv_rn(y, gs);
            atomicAdd(&a.out_acc[(size_t)s_tok[col] * a.H + c], s_w[col] * y);
          }
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 9) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && s_abort) set_dev_error(a.err, kDevTimeout);
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  });
  return fn;
}

// 2-D map: d0 = inner extent (elements), d1 = rows, row pitch in bytes, box b0 x b1.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1, uint64_t pitch,
              uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {d0, d1};
  cuuint64_t strides[1] = {pitch};
  cuuint32_t box[2] = {b0, b1};
  cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool weight_map(CUtensorMap* m, int fmt, const MatView& v, int E) {
  if (fmt == MOE_FMT_FP8_B128_W8A16)
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, v.a, v.K, (uint64_t)E * v.N, v.K, 128, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (fmt == MOE_FMT_INT4_G128_W4A16)
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, v.a, v.N, (uint64_t)E * (v.K / 8), (uint64_t)v.N * 4, 128, 16,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, v.a, v.K / 2, (uint64_t)E * v.N, v.K / 2, 64, 128,
                  CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int FMT, int MODE, int BN>
cudaError_t launch_one(const TcArgs& args, int grid_x, int grid_y, cudaStream_t s) {
  constexpr int SB = BN >= 64 ? 2 : 4;
  constexpr size_t need = 1024 + (size_t)kStagesW * 2 * WFmt<FMT>::kSubBytes + (size_t)SB * BN * 256;
  // at least 116 KB so that a single CTA (owning all 512 TMEM columns) runs per SM
  constexpr size_t smem = need > 116 * 1024 ? need : 116 * 1024;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(tc_expert_gemm_kernel<FMT, MODE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr = true;
  }
  tc_expert_gemm_kernel<FMT, MODE, BN><<<dim3(grid_x, grid_y), kThreads, smem, s>>>(args);
  return cudaGetLastError();
}

template <int FMT, int MODE>
cudaError_t launch_bn(int bn, const TcArgs& args, int gx, int gy, cudaStream_t s) {
  switch (bn) {
    case 16: return launch_one<FMT, MODE, 16>(args, gx, gy, s);
    case 32: return launch_one<FMT, MODE, 32>(args, gx, gy, s);
    case 64: return launch_one<FMT, MODE, 64>(args, gx, gy, s);
    default: return launch_one<FMT, MODE, 128>(args, gx, gy, s);
  }
}

template <int MODE>
cudaError_t launch_fmt(int fmt, int bn, const TcArgs& args, int gx, int gy, cudaStream_t s) {
  if (fmt == MOE_FMT_FP8_B128_W8A16) return launch_bn<MOE_FMT_FP8_B128_W8A16, MODE>(bn, args, gx, gy, s);
  if (fmt == MOE_FMT_INT4_G128_W4A16) return launch_bn<MOE_FMT_INT4_G128_W4A16, MODE>(bn, args, gx, gy, s);
  return launch_bn<MOE_FMT_NVFP4_W4A16, MODE>(bn, args, gx, gy, s);
}

}  // namespace

// Token rows per GEMM tile: the next power of two >= the mean rows per active expert, 16..128.
int tc_row_block(int T, int k, int E) {
  const long R = (long)T * k;
  const long active = R < E ? (R > 0 ? R : 1) : E;
  const long avg = (R + active - 1) / active;
  int bn = 16;
  while (bn < 128 && bn < avg) bn *= 2;
  return bn;
}

cudaError_t launch_experts_tc(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                              int bn, const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s) {
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  TcArgs a;
  memset(&a, 0, sizeof(a));
  a.perm = (const int32_t*)(ws + L.perm);
  a.topk_w = (const float*)(ws + L.topk_w);
  a.tiles = (const TileEntry*)(ws + L.tiles);
  a.h_out = (uint16_t*)(ws + L.h);
  a.out_acc = (float*)(ws + L.out_acc);
  a.err = (int*)(ws + L.err);
  a.k = k;
  a.I = I;
  a.H = H;
  const int gx = (int)(R / bn + (R < (size_t)E ? R : (size_t)E) + 1);

  // gate/up: A = fused [2I, H] weights, B = gathered rows of x
  if (!weight_map(&a.wmap, d.fmt, gu, E) ||
      !make_map(&a.bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, H, (uint64_t)T, (uint64_t)H * 2, 64, 1,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.wscale = gu.b;
  a.wgs = gu.gs;
  a.N = 2 * I;
  a.K = H;
  if (ev.start[0]) cudaEventRecord(ev.start[0], s);
  cudaError_t err = launch_fmt<0>(d.fmt, bn, a, gx, I / 128, s);
  if (ev.stop[0]) cudaEventRecord(ev.stop[0], s);
  if (err != cudaSuccess) return err;

  // down: A = [H, I] weights, B = rows of h (already in permuted order)
  if (!weight_map(&a.wmap, d.fmt, dn, E) ||
      !make_map(&a.bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, ws + L.h, I, (uint64_t)R, (uint64_t)I * 2, 64, bn,
                CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.wscale = dn.b;
  a.wgs = dn.gs;
  a.N = H;
  a.K = I;
  if (ev.start[1]) cudaEventRecord(ev.start[1], s);
  err = launch_fmt<1>(d.fmt, bn, a, gx, (H + 255) / 256, s);
  if (ev.stop[1]) cudaEventRecord(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
