// FP8 W8A8 grouped GEMMs: FP8 block-128 weights times FP8 activations quantized at run time,
// one scale per 1x128 group of a row (clef-omni-fp8, "What was quantized": E4M3 weights with one
// fp32 scale per 128x128 tile; activations dynamic FP8 per 1x128 group in serving engines).
//
// Both operands go to the tensor cores as stored codes (tcgen05.mma kind::f8f6f4, E4M3 x E4M3,
// fp32 accumulation).  Both scales change along K, once per 128-element block, so no single
// epilogue factor can apply them: the sum over K is
//
//   D[r, n] = sum_kb  sa[r, kb] * sw[n / 128, kb] * sum_{k in kb} qa[r, k] * qw[n, k]
//
// and each K block's partial sum has to be scaled before it joins the others ("promotion").
// The MMA warp writes the partial sum of K block kb into one of two tensor-memory buffers
// (256 columns each, all 512 columns of the SM), and sixteen promoter warps read it back, scale
// it by sa * sw and add it to accumulators they keep in registers, while the MMAs of the next K
// block fill the other buffer.  After the last block the same warps run the epilogue.
//
// One work item = 128 expert-permuted activation rows (one routing tile) x 256 weight rows:
//   P[act row, weight row] = sum_{k in kb} A[act row, k] * B[weight row, k]   M = 128, N = 256, K = 32
// gate/up: 128 gate rows over the matching 128 up rows, so a thread holds gate and up of the
// same features of its row; down: 256 consecutive output features.  Codes arrive by TMA tiles
// (128 rows x 128 bytes, the 128-byte swizzle); x is quantized straight into permuted row order,
// one copy per routed token slot, so the gate/up GEMM needs no row gather.
//
// Warps (576 threads): 0-15 promote and run the epilogue (warp w: TMEM lanes 32 (w % 4).., column
// group w / 4: 32 gate + 32 up columns, or 64 output columns), 16 issues TMA, 17 owns TMEM and
// issues the MMAs.  Persistent CTAs walk (routing tile, column block) work items handed out by a
// global counter.
#include <cudaTypedefs.h>

#include "moe_dec.cuh"
#include "moe_formats.cuh"
#include "moe_combine.cuh"
#include "moe_tc.cuh"
#include "moe_w8a8.cuh"

namespace moe {

namespace {

using namespace tc;

// ---------------------------------------------------------------------------------------------
// Activation quantizer: one warp per (row, 128-element group); lane l holds elements 4l .. 4l+3.
// ---------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quant_fp8_rows_kernel(const uint16_t* __restrict__ x,
                                                             const int32_t* __restrict__ scatter, int k, int rows,
                                                             int K, uint8_t* __restrict__ q, float* __restrict__ sinv,
                                                             int sf_rows) {
  pdl_wait();  // x may be the previous kernel's output (h)
  pdl_trigger();
  const int gpr = K / 128;
  const long wid = ((long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= (long)rows * gpr) return;
  const int r = (int)(wid / gpr), g = (int)(wid % gpr);
  const uint2 v = *(const uint2*)(x + (size_t)r * K + g * 128 + lane * 4);
  // max |v| on the bf16 bit patterns (magnitudes order like their values; NaN is left out, as
  // an ordered comparison would leave it out)
  uint32_t m = 0u;
  const uint32_t w[2] = {v.x, v.y};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t lo = w[i] & 0x7FFFu, hi = (w[i] >> 16) & 0x7FFFu;
    m = max(m, lo <= 0x7F80u ? lo : 0u);
    m = max(m, hi <= 0x7F80u ? hi : 0u);
  }
  m = __reduce_max_sync(0xffffffffu, m);
  float amax = __uint_as_float(m << 16);
  if (amax < 1e-12f) amax = 1e-12f;
  const float s = __fdiv_rn(448.0f, amax);
  const uint32_t c01 = dec::e4m3x2(__fmul_rn(bf16_to_f32(w[0] & 0xFFFFu), s), __fmul_rn(bf16_to_f32(w[0] >> 16), s));
  const uint32_t c23 = dec::e4m3x2(__fmul_rn(bf16_to_f32(w[1] & 0xFFFFu), s), __fmul_rn(bf16_to_f32(w[1] >> 16), s));
  const uint32_t codes = c01 | (c23 << 16);
  const float si = __fdiv_rn(1.0f, s);
  const int ndst = scatter ? k : 1;
  for (int j = 0; j < ndst; ++j) {
    const int dst = scatter ? scatter[(size_t)r * k + j] : r;
    *(uint32_t*)(q + (size_t)dst * K + g * 128 + lane * 4) = codes;
    if (lane == 0) sinv[sf_rows ? (size_t)g * sf_rows + dst : (size_t)dst * gpr + g] = si;
  }
}

// ---------------------------------------------------------------------------------------------
// The GEMM.
// ---------------------------------------------------------------------------------------------
constexpr int kKC = 128;                  // K per chunk = one scale block = 128 bytes of codes per row
constexpr int kRows = 128;                // activation rows per item (MMA M): the routing row block
constexpr int kStages = 4;                // chunks in flight
constexpr int kRing = 8;                  // work items handed from the producer to the other warps
constexpr int kPromWarps = 16, kProdWarp = 16, kMmaWarp = 17;
constexpr int kThreads = 18 * 32;
constexpr int kTile = 128 * 128;          // one 128-row x 128-byte E4M3 tile, 128-byte swizzle
constexpr int kWStage = 2 * kTile;        // the item's 256 weight rows
constexpr int kXStage = kTile;            // its 128 activation rows
constexpr size_t kSmem = 1024 + (size_t)kStages * (kWStage + kXStage);
constexpr uint32_t kBufCols = 256;        // TMEM: two partial-sum buffers

struct W8Args {
  CUtensorMap wcode;     // weight codes [E*N, K] E4M3
  CUtensorMap xcode;     // activation codes [R, K] E4M3, permuted row order
  const float* wsinv;    // weight scale_inv [E, N/128, K/128]
  const float* asinv;    // activation scale_inv group-major [K/128][sf_rows]
  int sf_rows;
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;
  uint8_t* hq_out;       // MODE 2 output: h's E4M3 codes [R, I] and scale_inv group-major
  float* hs_out;         //   [I/128][sf_rows] (h rounded to bf16, then quantized per 1x128 group)       // MODE 0 output [R, I] bf16
  uint16_t* y_out;       // MODE 1 output: routing-weighted rows [R, H] bf16, permuted order
  CombineTail ct;        // MODE 1: the combine that follows the GEMM items
  int* err;
  int* work_ctr;         // items handed out past each CTA's first (zeroed by routing)
  int k, N, K, I, H;
};

// 32 lanes x 8 columns of 32-bit words.
__device__ __forceinline__ void tmem_ld_32x8(uint32_t taddr, uint32_t* v) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
               : "r"(taddr)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)bf16_bits(lo) | ((uint32_t)bf16_bits(hi) << 16);
}

// MODE 0: gate/up (h in bf16), 1: down, 2: gate/up with h quantized to FP8 in the epilogue.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) w8a8_kernel(const __grid_constant__ W8Args a) {
  constexpr bool kGateUp = MODE != 1, kFuseH = MODE == 2;
  __shared__ uint32_t s_hmax[kFuseH ? 4 : 1][kFuseH ? kRows : 1];  // MODE 2: each column group's max |h| bits
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = (char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  char* sW = smem;
  char* sX = sW + kStages * kWStage;
  __shared__ uint64_t w_full[kStages], w_empty[kStages], x_full[kStages], x_empty[kStages], p_full[2], p_empty[2],
      drain;
  __shared__ uint64_t work_full[kRing], work_empty[kRing];
  __shared__ int s_work[kRing];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  // gate/up: wait for the activation quantization (and, before it, routing); down: the tile table
  // was final before the gate/up GEMM passed its own pdl_wait(), so only h's codes and scales
  // need the wait
  if (kGateUp) pdl_wait();
  const int ntiles = load_tile(a.tiles).expert;
  const int ncb = kGateUp ? a.I / 128 : a.H / 256;
  const int nwork = ntiles * ncb;
  if ((int)blockIdx.x >= nwork) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nK = a.K / kKC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], 1);
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&p_full[i], 1);
      mbar_init(&p_empty[i], kPromWarps);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&work_full[i], 1);
      mbar_init(&work_empty[i], kPromWarps + 1);  // every consuming warp
    }
    mbar_init(&drain, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, 512);
    tmem_relinquish();
  }
  if (warp == kProdWarp && lane == 0) {
    prefetch_tmap(&a.wcode);
    prefetch_tmap(&a.xcode);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;
  if (MODE == 1 && warp != kProdWarp) pdl_wait();  // the producer waits before its first h tile
  pdl_trigger();

  auto next_item = [&](int n, bool& ok) -> int {  // consumer side, whole warp
    const int slot = n % kRing;
    ok = __all_sync(0xffffffffu, mbar_wait(&work_full[slot], (n / kRing) & 1, &s_abort));
    if (!ok) return -1;
    const int wk = *(volatile int*)&s_work[slot];
    __syncwarp();
    if (lane == 0) mbar_arrive(&work_empty[slot]);
    return wk;
  };
  // item wk: routing tile wk / ncb; weight rows w0 .. w0+127 and w1 .. w1+127 of its expert
  auto item = [&](int wk, TileEntry& te, int& w0, int& w1) {
    te = load_tile(a.tiles + 1 + wk / ncb);
    const int cb = wk % ncb;
    w0 = kGateUp ? cb * 128 : cb * 256;
    w1 = kGateUp ? a.I + w0 : w0 + 128;
  };

  if (warp == kProdWarp) {
    // ---------------- TMA producer (whole warp walks the loop, lane 0 issues) ----------------
    int it = 0;
    bool ok = true;
    int armed_w[kStages] = {0}, armed_x[kStages] = {0};
    for (int n = 0; ok; ++n) {
      int wk = -1;
      if (lane == 0) {
        wk = n == 0 ? (int)blockIdx.x : (int)gridDim.x + atomicAdd(a.work_ctr, 1);
        if (wk >= nwork) wk = -1;
        const int slot = n % kRing;
        ok = mbar_wait(&work_empty[slot], ((n / kRing) & 1) ^ 1, &s_abort);
        if (ok) {
          s_work[slot] = wk;
          mbar_arrive(&work_full[slot]);
        }
      }
      wk = __shfl_sync(0xffffffffu, wk, 0);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok || wk < 0) break;
      TileEntry te;
      int w0, w1;
      item(wk, te, w0, w1);
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int st = it % kStages;
        const uint32_t par = ((it / kStages) & 1) ^ 1;
        if (lane == 0) {
          ok = mbar_wait(&w_empty[st], par, &s_abort);
          if (ok) {
            char* ws = sW + st * kWStage;
            mbar_arrive_expect_tx(&w_full[st], kWStage);
            ++armed_w[st];
            tma_load_2d(ws, &a.wcode, &w_full[st], kc * kKC, te.expert * a.N + w0);
            tma_load_2d(ws + kTile, &a.wcode, &w_full[st], kc * kKC, te.expert * a.N + w1);
          }
          if (ok) {
            ok = mbar_wait(&x_empty[st], par, &s_abort);
            if (MODE == 1 && it == 0) pdl_wait();
            if (ok) {
              mbar_arrive_expect_tx(&x_full[st], kXStage);
              ++armed_x[st];
              tma_load_2d(sX + st * kXStage, &a.xcode, &x_full[st], kc * kKC, te.row0);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0 && s_abort) {  // let every issued copy land before shared memory goes away
      volatile int no_abort = 0;
      for (int i = 0; i < kStages; ++i) {
        if (armed_w[i]) mbar_wait(&w_full[i], (armed_w[i] - 1) & 1, &no_abort);
        if (armed_x[i]) mbar_wait(&x_full[i], (armed_x[i] - 1) & 1, &no_abort);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (whole warp waits, lane 0 issues) ----------------
    const uint32_t idesc = dec::idesc_e4m3_f32(kRows, 256);
    int it = 0;
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      if (next_item(nitem, ok) < 0) break;
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int st = it % kStages, b = it & 1;
        ok = mbar_wait(&p_empty[b], ((it >> 1) & 1) ^ 1, &s_abort) &&
             mbar_wait(&w_full[st], (it / kStages) & 1, &s_abort) &&
             mbar_wait(&x_full[st], (it / kStages) & 1, &s_abort);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        fence_after_sync();
        if (lane == 0) {
          const uint32_t xa = smem_u32(sX + st * kXStage), wa = smem_u32(sW + st * kWStage);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)  // a fresh partial sum per K block
            dec::mma_f8_ss(tmem + b * kBufCols, sdesc_k_sw128(xa + ks * 32), sdesc_k_sw128(wa + ks * 32), idesc,
                           ks != 0);
          mma_commit(&w_empty[st]);
          mma_commit(&x_empty[st]);
          mma_commit(&p_full[b]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) mma_commit(&drain);
    __syncwarp();
  } else {
    // ---------------- promoters + epilogue: thread = activation row of the tile ----------------
    const int q = warp & 3, grp = warp >> 2, r = q * 32 + lane;
    int it = 0;
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      const int wk = next_item(nitem, ok);
      // the promoter warps move together: two named barriers per item, every thread reaches both
      if (!named_bar_and(1, kPromWarps * 32, ok && wk >= 0)) break;
      TileEntry te;
      int w0, w1;
      item(wk, te, w0, w1);
      const bool live = r < te.rows;
      // weight scale_inv of the thread's columns, K block kb at [kb]: gate/up: the gate tile (A)
      // and the up tile (B); down: the 128-row tile holding the thread's 64 columns
      const size_t tiles_n = (size_t)te.expert * (a.N / 128);
      const float* swA = a.wsinv + (tiles_n + (kGateUp ? w0 : w0 + 64 * grp) / 128) * nK;
      const float* swB = kGateUp ? a.wsinv + (tiles_n + w1 / 128) * nK : swA;
      // rows of the tile past its end (next expert's rows or past R) read in-bounds scales that
      // are never stored
      const float* sa = a.asinv + te.row0 + r;
      float acc[64];
#pragma unroll
      for (int i = 0; i < 64; ++i) acc[i] = 0.f;
      for (int kb = 0; kb < nK; ++kb, ++it) {
        const int b = it & 1;
        const float s_a = sa[(size_t)kb * a.sf_rows];
        const float fA = s_a * swA[kb], fB = s_a * swB[kb];
        // after a failed wait every later wait returns at once (the abort flag is set)
        ok = __all_sync(0xffffffffu, ok && mbar_wait(&p_full[b], (it >> 1) & 1, &s_abort));
        if (!ok) continue;
        fence_after_sync();
        const uint32_t base = taddr(tmem, q * 32, b * kBufCols);
#pragma unroll
        for (int h8 = 0; h8 < 8; ++h8) {
          // gate/up: h8 0-3 gate columns 32 grp + 8 h8, h8 4-7 up columns 128 + 32 grp + 8 (h8 - 4);
          // down: columns 64 grp + 8 h8
          const uint32_t col = kGateUp ? (h8 < 4 ? 32 * grp + 8 * h8 : 128 + 32 * grp + 8 * (h8 - 4))
                                       : 64 * grp + 8 * h8;
          const float f = kGateUp && h8 >= 4 ? fB : fA;
          uint32_t P[8];
          tmem_ld_32x8(base + col, P);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[8 * h8 + j] = fmaf(__uint_as_float(P[j]), f, acc[8 * h8 + j]);
        }
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_empty[b]);
      }
      if (!named_bar_and(1, kPromWarps * 32, ok)) break;
      if (kFuseH) {
        // The item's 128 features of a row are exactly one 1x128 group of h, spread over the four
        // column groups of lane quarter q (warps q, q + 4, q + 8, q + 12): h -> bf16, the group's
        // max |h| through shared memory, then E4M3 codes with s = 448 / amax, as the activation
        // quantizer does.  Every thread takes part (the rows past the tile too); only live rows
        // are stored.
        uint32_t hw[16], m = 0u;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float hv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float gv = acc[2 * j + e], uv = acc[32 + 2 * j + e];
            hv[e] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
          }
          hw[j] = pack_bf16x2(hv[0], hv[1]);
          // max |h| on the bf16 bit patterns, NaN left out (as in quant_fp8_rows_kernel)
          const uint32_t lo = hw[j] & 0x7FFFu, hi = (hw[j] >> 16) & 0x7FFFu;
          m = max(m, max(lo <= 0x7F80u ? lo : 0u, hi <= 0x7F80u ? hi : 0u));
        }
        s_hmax[grp][r] = m;
        named_bar_sync(2 + q, 4 * 32);
        m = max(max(s_hmax[0][r], s_hmax[1][r]), max(s_hmax[2][r], s_hmax[3][r]));
        named_bar_sync(2 + q, 4 * 32);  // s_hmax is rewritten for the next item
        float amax = __uint_as_float(m << 16);
        if (amax < 1e-12f) amax = 1e-12f;
        const float sc = __fdiv_rn(448.0f, amax);
        uint32_t cw[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t u0 = hw[2 * j], u1 = hw[2 * j + 1];
          const uint32_t c01 = dec::e4m3x2(__fmul_rn(__uint_as_float(u0 << 16), sc),
                                           __fmul_rn(__uint_as_float(u0 & 0xFFFF0000u), sc));
          const uint32_t c23 = dec::e4m3x2(__fmul_rn(__uint_as_float(u1 << 16), sc),
                                           __fmul_rn(__uint_as_float(u1 & 0xFFFF0000u), sc));
          cw[j] = c01 | (c23 << 16);
        }
        if (live) {
          const size_t row = (size_t)te.row0 + r;
          st_global_v8(a.hq_out + row * a.I + w0 + 32 * grp, cw);
          if (grp == 0) a.hs_out[(size_t)(w0 / 128) * a.sf_rows + row] = __fdiv_rn(1.0f, sc);
        }
        continue;
      }
      if (!live) continue;
      if (kGateUp) {
        // features w0 + 32 grp .. + 31: gate in acc[j], up in acc[32 + j]
        uint16_t* dst = a.h_out + (size_t)(te.row0 + r) * a.I + w0 + 32 * grp;
        uint32_t hw[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float hv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float gv = acc[2 * j + e], uv = acc[32 + 2 * j + e];
            hv[e] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
          }
          hw[j] = pack_bf16x2(hv[0], hv[1]);
        }
        st_global_v8(dst, hw);  // 32-byte stores: whole sectors of the thread's own row
        st_global_v8(dst + 16, hw + 8);
      } else {
        // output features w0 + 64 grp .. + 63 of the routing-weighted row
        const float rw = a.topk_w[a.perm[te.row0 + r]];
        uint16_t* dst = a.y_out + (size_t)(te.row0 + r) * a.H + w0 + 64 * grp;
        uint32_t yw[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) yw[j] = pack_bf16x2(acc[2 * j] * rw, acc[2 * j + 1] * rw);
#pragma unroll
        for (int v = 0; v < 4; ++v) st_global_v8(dst + 16 * v, yw + 8 * v);
      }
    }
  }

  {
    volatile int no_abort = 0;
    mbar_wait(&drain, 0, &no_abort);  // bounded; every MMA of this CTA has completed
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && s_abort) set_dev_error(a.err, kDevTimeout);
  if (MODE == 1) {  // the routing-weighted combine, once every working CTA is done
    __shared__ int s_flag;
    if (!combine_tail(a.ct, min((int)gridDim.x, nwork), &s_flag) && threadIdx.x == 0)
      set_dev_error(a.err, kDevTimeout);
  }
}

template <int MODE>
cudaError_t launch_w8a8(const W8Args& a, int work, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(w8a8_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    attr = true;
  }
  const int sms = tc_num_sms();
  return launch_pdl(w8a8_kernel<MODE>, dim3(work < sms ? work : sms), dim3(kThreads), kSmem, s, a);
}

}  // namespace

bool w8a8_supported(const moe_packed_desc_t& d) { return d.H % 256 == 0 && d.I % 128 == 0; }
int w8a8_row_block() { return kRows; }

size_t w8a8_act_bytes(size_t R, int K) { return R * (size_t)K + 4 * (size_t)sf_plane_rows(R) * (K / 128); }

cudaError_t launch_quant_fp8_rows(const __nv_bfloat16* x, const int32_t* scatter, int k, int rows, int K, uint8_t* q,
                                  float* sinv, int sf_rows, cudaStream_t s) {
  if (rows <= 0) return cudaGetLastError();
  const size_t threads = (size_t)rows * (K / 128) * 32;
  note_launches(1);
  return launch_pdl(quant_fp8_rows_kernel, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, s,
                    (const uint16_t*)x, scatter, k, rows, K, q, sinv, sf_rows);
}

cudaError_t launch_experts_w8a8(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                                const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, uint16_t* out) {
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  uint8_t* xq = (uint8_t*)(ws + L.xq);
  float* xs = (float*)(ws + L.xs);
  uint8_t* hq = (uint8_t*)(ws + L.hq);
  float* hs = (float*)(ws + L.hs);
  const int sf_rows = sf_plane_rows(R);
  cudaError_t err = launch_quant_fp8_rows(x, (const int32_t*)(ws + L.inv), k, T, H, xq, xs, sf_rows, s);
  if (err != cudaSuccess) return err;

  W8Args a;
  memset(&a, 0, sizeof(a));
  a.perm = (const int32_t*)(ws + L.perm);
  a.topk_w = (const float*)(ws + L.topk_w);
  a.tiles = (const TileEntry*)(ws + L.tiles);
  a.h_out = (uint16_t*)(ws + L.h);
  a.y_out = (uint16_t*)(ws + L.y);
  combine_tail_args(a.ct, L, ws, T, k, H, out);
  a.err = (int*)(ws + L.err);
  a.k = k;
  a.I = I;
  a.H = H;
  a.sf_rows = sf_rows;
  a.hq_out = hq;
  a.hs_out = hs;
  a.work_ctr = (int*)(ws + L.err) + 1;
  const int max_tiles = (int)(R / kRows + (R < (size_t)E ? R : (size_t)E) + 1);
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;

  // gate/up: A = quantized x in permuted row order, B = fused [2I, H] FP8 weights
  if (!tc_make_map(&a.wcode, u8, gu.a, H, (uint64_t)E * 2 * I, H, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc_make_map(&a.xcode, u8, xq, H, (uint64_t)R, H, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.wsinv = (const float*)gu.b;
  a.asinv = xs;
  a.N = 2 * I;
  a.K = H;
  record_event(ev.start[0], s);
  err = launch_w8a8<2>(a, max_tiles * (I / 128), s);  // h leaves the epilogue as FP8 codes and scales
  record_event(ev.stop[0], s);
  if (err != cudaSuccess) return err;

  // down: A = h rows (quantized by the gate/up epilogue), B = [H, I] weights
  if (!tc_make_map(&a.wcode, u8, dn.a, I, (uint64_t)E * H, I, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc_make_map(&a.xcode, u8, hq, I, (uint64_t)R, I, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.wsinv = (const float*)dn.b;
  a.asinv = hs;
  a.N = H;
  a.K = I;
  a.work_ctr = (int*)(ws + L.err) + 2;
  record_event(ev.start[1], s);
  err = launch_w8a8<1>(a, max_tiles * (H / 256), s);
  record_event(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
