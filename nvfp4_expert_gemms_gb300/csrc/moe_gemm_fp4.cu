// NVFP4 W4A4 grouped GEMMs on the native block-scaled FP4 tensor-core MMA
// (tcgen05.mma kind::mxf4nvf4, E2M1 operands, UE4M3 scale per 16 elements along K).
//
// Both operands stay in their packed NVFP4 form end to end (clef-flash-NVFP4-Hybrid, layer
// table: NVFP4 activations as well as weights, E4M3 scales per 16 and one fp32 global scale;
// weights: clef-omni-NVFP4, "How it was made"):
//   weights      E2M1 codes [N, K/2] + E4M3 block scales [N, K/16] + global scale gs_w (per matrix)
//   activations  E2M1 codes [rows, K/2] + E4M3 block scales [rows, K/16] + global scale gs_a (per row)
// The MMA forms sum_k (q_a * bs_a)(q_w * bs_w) exactly in fp32, and the epilogue divides by
// gs_a * gs_w.
//
// One work item = 128 expert-permuted activation rows (one routing tile) x 256 weight rows:
//   D[act row, weight row] += A[act row, k] * B[weight row, k]     M = 128, N = 256, K = 64
// gate/up: the 256 weight rows are 128 gate rows over the 128 matching up rows, so a thread
// of the epilogue holds gate and up of the same features of its token; down: 256 consecutive
// output features.  An N = 256 block-scaled MMA costs the tensor pipe the same issue time as
// N = 64 or 128, so one instruction per K step covers what two N = 128 ones did.  Codes arrive
// by TMA tiles in the 128-byte swizzle (x is quantized straight into permuted row order, one copy
// per routed token slot, so the gate/up GEMM needs no row gather).  The block scales come in
// layouts where the 128 rows of one 256-column chunk are one contiguous 2 KB block (the packed
// re-tiled weight-scale copy; the quantizer writes activation scales chunk-major), each one bulk
// copy next to its codes rather than 128 strided 16-byte pieces; the four scale warps place
// both in tensor memory in the layout the MMA reads (per K = 64 step: row r of the operand in lane
// r % 32 of column r / 32, four scales per word, repeated in every lane quarter).
//
// Warps (448 threads): 0-3 stage scale factors, 4-11 run the epilogue (thread = token row, 64
// or 128 contiguous output features), 12 issues TMA, 13 owns TMEM and issues the MMAs.
// Persistent CTAs walk (routing tile, column block) work items.
#include <cudaTypedefs.h>

#include "moe_formats.cuh"
#include "moe_nvfp4.cuh"
#include "moe_tc.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kKC = 256;                  // K per chunk: 128 bytes of codes per row
constexpr int kRows = 128;                // activation rows per item (MMA M): the routing row block
constexpr int kStagesW = 4, kStagesX = 4, kStagesS = 4;
constexpr int kRing = 8;                  // work items handed from the producer to the other warps
constexpr int kSfWarps = 4, kEpiWarp0 = 4, kEpiWarps = 8, kProdWarp = 12, kMmaWarp = 13;
constexpr int kThreads = 14 * 32;
constexpr int kWCodes = 128 * 128;        // one 128-row weight tile, 128-byte swizzle
constexpr int kWSf = 128 * 16;            // its 128 rows x 16 scales
constexpr int kWStage = 2 * kWCodes + 2 * kWSf;  // two tiles = the 256 B rows of one item
constexpr int kXCodes = kRows * 128;      // activation codes, 128-byte swizzle
constexpr int kXStage = kXCodes + kRows * 16;  // then their 128 rows x 16 scales
constexpr size_t kSmem = 1024 + (size_t)kStagesW * kWStage + (size_t)kStagesX * kXStage;
constexpr uint32_t kSfCol = 256;          // TMEM: [0, 256) accumulator, then 4 x 48 scale-factor columns
constexpr uint32_t kSfStageCols = 48;     // A (activation) scales 4 x 4 columns, B (weight) scales 4 x 8

struct Fp4Args {
  CUtensorMap wcode;        // weight codes [E*N, K/2]
  CUtensorMap xcode;        // activation codes [R, K/2], permuted row order
  const uint8_t* wsft;      // weight block scales re-tiled [E, N/128, K/256, 128, 16]
  const uint8_t* asft;      // activation block scales chunk-major [K/256][sf_rows][16]
  int sf_rows;
  const float* wgs;         // weight global scales [E]
  const float* ags;         // activation global scales [R]
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;          // MODE 0 output [R, I] bf16 (dynamic activation scales)
  const float* hgs_static;  // MODE 2 (gate/up, static activation scales): h's global scale (dev); h
  uint8_t* hq_out;          //   leaves NVFP4-quantized instead: codes [R, I/2], chunk-major block
  uint8_t* hsf_out;         //   scales [I/256][sf_rows][16] and the global scale per row [R]
  float* hg_out;
  uint16_t* y_out;          // MODE 1 output: routing-weighted rows [R, H] bf16, permuted order
  int* err;
  int* work_ctr;            // items handed out past each CTA's first (zeroed by routing)
  int k, N, K, I, H;
};

__host__ __device__ constexpr uint32_t idesc_nvf4(int M, int N) {
  // E2M1 A and B (1), K-major, N >> 3 at bit 17, UE4M3 scales (0) at bit 23, M >> 4 at bit 24
  return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_nvf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
      : "memory");
}

__device__ __forceinline__ void tmem_st_32x16(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)bf16_bits(lo) | ((uint32_t)bf16_bits(hi) << 16);
}

// MODE 0: gate/up (h in bf16), 1: down, 2: gate/up with static activation scales (h leaves as
// NVFP4 codes, block scales and global scales).
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) fp4_kernel(const __grid_constant__ Fp4Args a) {
  constexpr bool kGateUp = MODE != 1, kFuseH = MODE == 2;
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = (char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  char* sW = smem;
  char* sX = sW + kStagesW * kWStage;
  __shared__ uint64_t w_full[kStagesW], w_empty[kStagesW], x_full[kStagesX], x_empty[kStagesX], s_full[kStagesS],
      s_empty[kStagesS], acc_full, acc_empty, drain;
  __shared__ uint64_t work_full[kRing], work_empty[kRing];
  __shared__ int s_work[kRing];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  // gate/up: wait for the activation quantization (and, before it, routing); down: the tile table
  // was final before the gate/up GEMM passed its own pdl_wait(), so only the h codes need the wait
  if (kGateUp) pdl_wait();
  const int ntiles = load_tile(a.tiles).expert;
  const int ncb = kGateUp ? a.I / 128 : a.H / 256;
  const int nwork = ntiles * ncb;
  if ((int)blockIdx.x >= nwork) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nK = a.K / kKC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesW; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], 1);
    }
    for (int i = 0; i < kStagesX; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);
    }
    for (int i = 0; i < kStagesS; ++i) {
      mbar_init(&s_full[i], kSfWarps);
      mbar_init(&s_empty[i], 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&work_full[i], 1);
      mbar_init(&work_empty[i], kSfWarps + 1 + kEpiWarps);  // every consuming warp
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kEpiWarps);
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

  // Work items are handed out dynamically (SMs do not all stream at the same rate): the
  // producer takes each CTA's first item statically and the rest from a global counter, and
  // passes every item id (then -1) through a shared-memory ring to the other warps.
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
    int armed_w[kStagesW] = {0}, armed_x[kStagesX] = {0};
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
        const int sw = it % kStagesW, sx = it % kStagesX;
        if (lane == 0) {
          ok = mbar_wait(&w_empty[sw], ((it / kStagesW) & 1) ^ 1, &s_abort);
          if (ok) {
            char* ws = sW + sw * kWStage;
            mbar_arrive_expect_tx(&w_full[sw], 2 * (kWCodes + kWSf));
            ++armed_w[sw];
            for (int g = 0; g < 2; ++g) {
              const int wr = g == 0 ? w0 : w1;
              tma_load_2d(ws + g * kWCodes, &a.wcode, &w_full[sw], kc * (kKC / 2), te.expert * a.N + wr);
              // the 128 rows' scales of this chunk: one contiguous 2 KB block of the re-tiled copy
              const size_t blk = ((size_t)te.expert * (a.N / 128) + wr / 128) * nK + kc;
              bulk_load(ws + 2 * kWCodes + g * kWSf, a.wsft + blk * kWSf, kWSf, &w_full[sw]);
            }
          }
          if (ok) {
            ok = mbar_wait(&x_empty[sx], ((it / kStagesX) & 1) ^ 1, &s_abort);
            if (MODE == 1 && it == 0) pdl_wait();
            if (ok) {
              mbar_arrive_expect_tx(&x_full[sx], kXStage);
              ++armed_x[sx];
              tma_load_2d(sX + sx * kXStage, &a.xcode, &x_full[sx], kc * (kKC / 2), te.row0);
              bulk_load(sX + sx * kXStage + kXCodes, a.asft + ((size_t)kc * a.sf_rows + te.row0) * 16, kRows * 16,
                        &x_full[sx]);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0 && s_abort) {  // let every issued copy land before shared memory goes away
      volatile int no_abort = 0;
      for (int i = 0; i < kStagesW; ++i)
        if (armed_w[i]) mbar_wait(&w_full[i], (armed_w[i] - 1) & 1, &no_abort);
      for (int i = 0; i < kStagesX; ++i)
        if (armed_x[i]) mbar_wait(&x_full[i], (armed_x[i] - 1) & 1, &no_abort);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (whole warp waits, lane 0 issues) ----------------
    const uint32_t idesc = idesc_nvf4(kRows, 256);
    int it = 0;
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      if (next_item(nitem, ok) < 0) break;
      ok = mbar_wait(&acc_empty, (nitem & 1) ^ 1, &s_abort);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      fence_after_sync();
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sw = it % kStagesW, sx = it % kStagesX, ss = it % kStagesS;
        ok = mbar_wait(&w_full[sw], (it / kStagesW) & 1, &s_abort) &&
             mbar_wait(&x_full[sx], (it / kStagesX) & 1, &s_abort) &&
             mbar_wait(&s_full[ss], (it / kStagesS) & 1, &s_abort);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        fence_after_sync();
        if (lane == 0) {
          const uint32_t xa = smem_u32(sX + sx * kXStage), wa = smem_u32(sW + sw * kWStage);
          const uint32_t sfa = tmem + kSfCol + ss * kSfStageCols, sfb = sfa + 16;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_nvf4(tmem, sdesc_k_sw128(xa + ks * 32), sdesc_k_sw128(wa + ks * 32), idesc, sfa + 4 * ks,
                     sfb + 8 * ks, (kc | ks) != 0);
          mma_commit(&w_empty[sw]);
          mma_commit(&x_empty[sx]);
          mma_commit(&s_empty[ss]);
        }
        __syncwarp();
      }
      if (ok && lane == 0) mma_commit(&acc_full);
      __syncwarp();
    }
    if (lane == 0) mma_commit(&drain);
    __syncwarp();
  } else if (warp < kSfWarps) {
    // ---------------- scale factors -> tensor memory ----------------
    const int q = warp, l = lane;
    int it = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int wk = next_item(n, ok);
      if (wk < 0) break;
      TileEntry te;
      int w0, w1;
      item(wk, te, w0, w1);
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sw = it % kStagesW, sx = it % kStagesX, ss = it % kStagesS;
        ok = __all_sync(0xffffffffu, mbar_wait(&w_full[sw], (it / kStagesW) & 1, &s_abort) &&
                                         mbar_wait(&x_full[sx], (it / kStagesX) & 1, &s_abort) &&
                                         mbar_wait(&s_empty[ss], ((it / kStagesS) & 1) ^ 1, &s_abort));
        if (!ok) break;
        fence_after_sync();
        const uint32_t col = kSfCol + ss * kSfStageCols;
        // A: column 4 ks + j holds the K-step-ks word of activation row l + 32 j (rows past the
        // tile scale by 0)
        const char* xsf = sX + sx * kXStage + kXCodes;
        uint4 x4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          x4[j] = l + 32 * j < te.rows ? *(const uint4*)(xsf + (l + 32 * j) * 16) : make_uint4(0u, 0u, 0u, 0u);
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[0 + j] = x4[j].x;
          v[4 + j] = x4[j].y;
          v[8 + j] = x4[j].z;
          v[12 + j] = x4[j].w;
        }
        tmem_st_32x16(taddr(tmem, q * 32, col), v);
        // B: column 16 + 8 ks + j holds the K-step-ks word of weight row l + 32 j (j < 4: first
        // 128-row tile, j >= 4: second)
        uint4 w[8];
        const char* wsf = sW + sw * kWStage + 2 * kWCodes;
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = *(const uint4*)(wsf + (j >> 2) * kWSf + (l + 32 * (j & 3)) * 16);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[0 + j] = w[j].x;
          v[8 + j] = w[j].y;
        }
        tmem_st_32x16(taddr(tmem, q * 32, col + 16), v);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          v[0 + j] = w[j].z;
          v[8 + j] = w[j].w;
        }
        tmem_st_32x16(taddr(tmem, q * 32, col + 32), v);
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_full[ss]);
      }
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ---------------- epilogue: thread = token row of the tile ----------------
    const int q = warp & 3, half = (warp - kEpiWarp0) >> 2, r = q * 32 + lane;
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      const int wk = next_item(nitem, ok);
      // the epilogue warps leave together (they meet in a named barrier every item)
      if (!named_bar_and(1, kEpiWarps * 32, ok && wk >= 0)) break;
      TileEntry te;
      int w0, w1;
      item(wk, te, w0, w1);
      // the row's scale (1 / (gs_w gs_a), times the routing weight for the down GEMM), read
      // while the MMAs run
      const bool live = r < te.rows;
      float cs = 0.f;
      if (live) {
        const float g = a.wgs[te.expert] * a.ags[te.row0 + r];
        cs = kGateUp ? 1.0f / g : a.topk_w[a.perm[te.row0 + r]] / g;
      }
      ok = mbar_wait(&acc_full, nitem & 1, &s_abort);
      // every epilogue thread takes the same branch
      ok = named_bar_and(1, kEpiWarps * 32, ok);
      if (!ok) break;
      fence_after_sync();
      if (kGateUp) {
        // features w0 + 64 half .. + 63: gate in accumulator columns c, up in 128 + c
        uint16_t* dst = a.h_out + (size_t)(te.row0 + r) * a.I + w0 + 64 * half;
        const float ghs = kFuseH ? *a.hgs_static : 0.f;  // static scales: quantize h here
        uint32_t hall[32];  // fused: the row's 64 bf16 h values, encoded once the accumulator is free
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int c = 64 * half + 32 * b;
          uint32_t G[32], U[32];
          tmem_ld_32x16(taddr(tmem, q * 32, c), G);
          tmem_ld_32x16(taddr(tmem, q * 32, c + 16), G + 16);
          tmem_ld_32x16(taddr(tmem, q * 32, 128 + c), U);
          tmem_ld_32x16(taddr(tmem, q * 32, 128 + c + 16), U + 16);
          tmem_ld_wait();
          if (b == 1) {  // the accumulator is free once every warp has read it
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty);
          }
          uint32_t hw[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float hv[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float gv = __uint_as_float(G[2 * j + e]) * cs, uv = __uint_as_float(U[2 * j + e]) * cs;
              hv[e] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            }
            hw[j] = pack_bf16x2(hv[0], hv[1]);
          }
          if (!kFuseH) {
            if (live)  // 32-byte stores: each lane writes whole sectors of its own row
#pragma unroll
              for (int v = 0; v < 2; ++v) st_global_v8(dst + 32 * b + 16 * v, hw + 8 * v);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) hall[16 * b + j] = hw[j];
          }
        }
        uint32_t hc[8];  // fused: codes of the thread's four 16-blocks and their scales
        uint32_t hs4 = 0u;
        if (kFuseH) {
#pragma unroll
          for (int blk = 0; blk < 4; ++blk) {  // the bf16 h block -> NVFP4 with the static scale
            float v[16];
            uint32_t m = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const uint32_t w = hall[8 * blk + i];
              v[2 * i] = __uint_as_float(w << 16);
              v[2 * i + 1] = __uint_as_float(w & 0xFFFF0000u);
              m = max(m, max(w & 0x7FFFu, (w >> 16) & 0x7FFFu));
            }
            uint2 code;
            uint8_t sc;
            nvfp4_encode(v, __uint_as_float(m << 16), ghs, &code, &sc);
            hc[2 * blk] = code.x;
            hc[2 * blk + 1] = code.y;
            hs4 |= (uint32_t)sc << (8 * blk);
          }
        }
        if (kFuseH && live) {
          const size_t row = (size_t)te.row0 + r;
          const int f0 = w0 + 64 * half;  // four whole blocks of one 256-column chunk
          st_global_v8(a.hq_out + row * (a.I / 2) + f0 / 2, hc);
          *(uint32_t*)(a.hsf_out + ((size_t)(f0 >> 8) * a.sf_rows + row) * 16 + ((f0 & 255) >> 4)) = hs4;
          if (f0 == 0) a.hg_out[row] = ghs;
        }
      } else {
        // output features w0 + 128 half .. + 127 of the routing-weighted row
        uint16_t* dst = a.y_out + (size_t)(te.row0 + r) * a.H + w0 + 128 * half;
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const int c = 128 * half + 64 * b;
          uint32_t Y[64];
#pragma unroll
          for (int i = 0; i < 4; ++i) tmem_ld_32x16(taddr(tmem, q * 32, c + 16 * i), Y + 16 * i);
          tmem_ld_wait();
          if (b == 1) {
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j)  // in place: word j reads words 2j, 2j+1 >= j
            Y[j] = pack_bf16x2(__uint_as_float(Y[2 * j]) * cs, __uint_as_float(Y[2 * j + 1]) * cs);
          if (live)
#pragma unroll
            for (int v = 0; v < 4; ++v) st_global_v8(dst + 64 * b + 16 * v, Y + 8 * v);
        }
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
}

}  // namespace

// The FP4 path needs whole 256-element K chunks in both GEMMs.
bool fp4_supported(const moe_packed_desc_t& d) { return d.H % 256 == 0 && d.I % 256 == 0; }
int fp4_row_block() { return kRows; }

template <int MODE>
static cudaError_t launch_fp4(const Fp4Args& a, int work, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(fp4_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    attr = true;
  }
  const int sms = tc_num_sms();
  return launch_pdl(fp4_kernel<MODE>, dim3(work < sms ? work : sms), dim3(kThreads), kSmem, s, a);
}

cudaError_t launch_experts_fp4(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                               const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, const float* act_gs,
                               bool calibrate) {
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  uint8_t* xq = (uint8_t*)(ws + L.xq);
  uint8_t* xsf = (uint8_t*)(ws + L.xs);
  uint8_t* hq = (uint8_t*)(ws + L.hq);
  uint8_t* hsf = (uint8_t*)(ws + L.hs);
  const int sf_rows = sf_plane_rows(R);
  float* cal = calibrate ? const_cast<float*>(act_gs) : nullptr;  // calibration writes the two scales
  if (cal && launch_act_scale((const uint16_t*)x, (size_t)T * H, cal, s) != cudaSuccess) return cudaGetLastError();
  launch_quant_rows(x, (const int32_t*)(ws + L.inv), k, T, H, xq, xsf, (float*)(ws + L.xg), s, !cal, sf_rows, act_gs);

  Fp4Args a;
  memset(&a, 0, sizeof(a));
  a.perm = (const int32_t*)(ws + L.perm);
  a.topk_w = (const float*)(ws + L.topk_w);
  a.tiles = (const TileEntry*)(ws + L.tiles);
  a.h_out = (uint16_t*)(ws + L.h);
  a.hgs_static = act_gs && !calibrate ? act_gs + 1 : nullptr;
  a.hq_out = hq;
  a.hsf_out = hsf;
  a.hg_out = (float*)(ws + L.hg);
  a.y_out = (uint16_t*)(ws + L.y);
  a.err = (int*)(ws + L.err);
  a.k = k;
  a.I = I;
  a.H = H;
  a.sf_rows = sf_rows;
  a.work_ctr = (int*)(ws + L.err) + 1;
  const int max_tiles = (int)(R / kRows + (R < (size_t)E ? R : (size_t)E) + 1);
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;

  // gate/up: A = quantized x in permuted row order, B = fused [2I, H] NVFP4 weights
  if (!tc_make_map(&a.wcode, u8, gu.a, H / 2, (uint64_t)E * 2 * I, H / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc_make_map(&a.xcode, u8, xq, H / 2, (uint64_t)R, H / 2, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.wsft = (const uint8_t*)packed + d.offset[MOE_T_GU_BT];
  a.asft = xsf;
  a.wgs = gu.gs;
  a.ags = (const float*)(ws + L.xg);
  a.N = 2 * I;
  a.K = H;
  record_event(ev.start[0], s);
  cudaError_t err = a.hgs_static ? launch_fp4<2>(a, max_tiles * (I / 128), s) : launch_fp4<0>(a, max_tiles * (I / 128), s);
  record_event(ev.stop[0], s);
  if (err != cudaSuccess) return err;

  if (cal) return launch_act_scale((const uint16_t*)(ws + L.h), R * I, cal + 1, s);  // h's scale; no down GEMM
  // h -> NVFP4 per permuted row (its own global scale; with static scales the gate/up epilogue
  // has already quantized it), then down: A = h rows, B = [H, I] weights
  if (!act_gs)
    launch_quant_rows((const __nv_bfloat16*)(ws + L.h), nullptr, 1, (int)R, I, hq, hsf, (float*)(ws + L.hg), s, false,
                      sf_rows);
  if (!tc_make_map(&a.wcode, u8, dn.a, I / 2, (uint64_t)E * H, I / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc_make_map(&a.xcode, u8, hq, I / 2, (uint64_t)R, I / 2, 128, kRows, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.wsft = (const uint8_t*)packed + d.offset[MOE_T_D_BT];
  a.asft = hsf;
  a.wgs = dn.gs;
  a.ags = (const float*)(ws + L.hg);
  a.N = H;
  a.K = I;
  a.work_ctr = (int*)(ws + L.err) + 2;
  record_event(ev.start[1], s);
  err = launch_fp4<1>(a, max_tiles * (H / 256), s);
  record_event(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
