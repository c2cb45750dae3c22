// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05) for the weight-only
// formats (FP8 W8A16, INT4 W4A16, NVFP4 W4A16).
//
// The pages run the experts by dequantizing them, then calling a grouped matmul (clef-omni-fp8,
// "How this checkpoint runs"; clef-omni-int4, same section; clef-omni-NVFP4, "How it was made").
// Here the dequantization is fused into the GEMM and never reaches HBM:
//
//   weights (packed, HBM) --TMA--> shared memory --converter warps--> bf16 A operand in TMEM
//   activations (bf16)    --TMA tile / cp.async gather--> shared memory (128-byte swizzle) = B operand
//   tcgen05.mma kind::f16: D[weight row, token] += A[weight row, k] * B[token, k]   (fp32, TMEM)
//
// Weight rows are the MMA's M side (128 per sub-tile) and tokens its N side (BN = 16..128), so a
// decode step with one or two tokens per expert still issues full-rate 128-row MMAs while the
// kernel streams weights.  Each CTA covers one row block of one expert (from the routing tile
// table) and two 128-row weight sub-tiles: gate rows n0.. and up rows I+n0.. for the gate/up
// GEMM (so SiLU(gate)*up is computed in the epilogue from two TMEM accumulators), or 256
// consecutive output features for the down GEMM (whose epilogue writes the row times its
// routing weight, fp32, for the slot-ordered combine).
//
// Warp roles (640 threads): warps 0-15 convert (warp w: sub-tile (w/4)%2, K half w/8, TMEM lanes
// 32*(w%4)..) and later run the epilogue; warp 16 issues TMA; warp 17 owns TMEM and issues the
// MMAs.  The gate/up GEMM reads x rows in expert-permuted order: for row blocks of 64 or more a
// separate pass writes that permuted copy and the kernel loads it in TMA tiles; for smaller row
// blocks warps 18-19 gather the token rows with 16-byte cp.async copies.  (A TMA gather4 per four
// 128-byte rows moved about one row per 35 SM cycles, and a few cp.async warps reach only about
// 20-40 GB/s per SM, both far below what the MMAs consume at 64-128 tokens per tile.)
#include <cudaTypedefs.h>

#include <mutex>
#include <unordered_map>

#include "moe_formats.cuh"
#include "moe_combine.cuh"
#include "moe_tc.cuh"
#include "moe_w16conv.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kKC = 128;          // K elements per pipeline chunk
constexpr int kConvWarps = 16;    // warps 0-15: converters + epilogue
constexpr int kProdWarp = 16;     // TMA producer
constexpr int kMmaWarp = 17;      // TMEM owner and MMA issuer
constexpr int kGathWarp0 = 18, kGathWarps = 2;  // activations: row gather (small BN) or warp 18 issues TMA tiles
constexpr int kRing = 8;           // work items handed from the producer to the other warps
constexpr int kThreads = 20 * 32;
constexpr uint32_t kTmemCols = 512;
// TMEM columns: [0, 2*BN) accumulators (two sub-tiles), then a ring of converted A chunks of 128
// columns (both sub-tiles, 64 columns each): three stages from column 128 when BN <= 64, two from
// column 256 when BN = 128.

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
  static constexpr int kSubBytes = kW16Block;  // one image block (128 rows' codes, then their scales)
};
template <>
struct WFmt<MOE_FMT_BF16> {
  static constexpr int kSubBytes = 2 * 128 * 128;  // two 128-byte swizzle atoms (64 K each) x 128 rows
};

// Shared-memory rings: weight chunks (kStagesW) and activation chunks (SB, each BN rows x 128 K
// bf16 as two 128-byte swizzle atoms); the gather threads keep LAG chunks in flight.
// Weight stages fill what the activation ring leaves of ~220 KB, up to 12: a weight stream from
// HBM needs ~150 KB in flight per SM (about 3.4 us of latency under load at its bandwidth share).
template <int FMT, int BN>
struct TcCfg {
  static constexpr int kWSub = WFmt<FMT>::kSubBytes;
  static constexpr int kBStage = BN * 256;
  static constexpr int SB = BN <= 32 ? 4 : (BN == 64 ? 4 : (FMT == MOE_FMT_BF16 ? 2 : 3));  // BF16: 32 KB weight sub-tiles
  static constexpr int kWFree = 220 * 1024 - 1024 - SB * kBStage;
  // per weight stage, the chunk's scales (copied by the producer warp next to the TMA tile):
  // FP8 one fp32 per sub-tile, INT4 128 fp16 per sub-tile; NVFP4's are in its image blocks, BF16 has none
  static constexpr int kScaleSlot = FMT == MOE_FMT_BF16 || FMT == MOE_FMT_NVFP4_W4A16 ? 0 : 2048;
  static constexpr int kStagesWFit = kWFree / (2 * kWSub + kScaleSlot);
  static constexpr int kStagesW = kStagesWFit > 12 ? 12 : (kStagesWFit < 2 ? 2 : kStagesWFit);
  static constexpr int LAG = SB - 2;
  static constexpr size_t kSmem = 1024 + (size_t)kStagesW * 2 * kWSub + (size_t)SB * kBStage +
                                  (size_t)kStagesW * kScaleSlot;
};

struct TcArgs {
  CUtensorMap wmap;  // packed weight codes of the matrix
  CUtensorMap bmap;  // activation rows in permuted order as [K/64 atoms][rows][64], boxes of BN rows x 2 atoms
  const uint8_t* wimg;  // NVFP4: the weight image [E, K/128, N/128, kW16Block]
  const __nv_bfloat16* x;  // activations of the gate/up GEMM [T, K], gathered by token (small row blocks)
  const void* wscale;
  const float* wgs;
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;
  uint16_t* y_out;  // down: routing-weighted rows [R, H] bf16, permuted order
  CombineTail ct;        // MODE 1: the combine that follows the GEMM items
  int* err;
  int* work_ctr;  // items handed out past each CTA's first (zeroed by routing)
  int k, N, K, I, H;
};

__device__ __forceinline__ uint32_t bsub2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// FP8: each e4m3 byte becomes bf16 bits of (value * 2^-120) by moving its magnitude bits under
// the bf16 exponent (exact, with e4m3 subnormals landing on bf16 subnormals), then one packed
// bf16 multiply by bf16(scale_inv * 2^120) gives the dequantized weight rounded once to bf16.
// When scale_inv * 2^120 does not fit bf16 (|w| > ~1e5) the exact fp32 route is taken instead.
// (The shared-memory loads are issued first and the path choice sits outside the loops: both
// matter several-fold for the converter's issue rate.)
__device__ __forceinline__ void conv_fp8_exact(const char* sub, int r, int kh, float scale, uint32_t* out) {
  for (int cc = 0; cc < 4; ++cc) {
    const int c = kh * 4 + cc;
    const uint4 q = *(const uint4*)(sub + r * 128 + ((c ^ (r & 7)) * 16));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    for (int i = 0; i < 4; ++i) {
      float f[4];
      for (int b = 0; b < 4; ++b) {
        const uint32_t byte = (w[i] >> (8 * b)) & 0xFFu;
        f[b] = (__uint_as_float(((byte & 0x7Fu) << 20) | ((byte & 0x80u) << 24)) * 0x1p120f) * scale;
      }
      out[cc * 8 + i * 2] = pack_bf16x2(f[0], f[1]);
      out[cc * 8 + i * 2 + 1] = pack_bf16x2(f[2], f[3]);
    }
  }
}

__device__ __forceinline__ void conv_fp8(const char* sub, int r, int kh, float scale, uint32_t* out) {
  const float big = scale * 0x1p120f;
  if (!(big < 3.0e38f)) {
    conv_fp8_exact(sub, r, kh, scale, out);
    return;
  }
  const uint32_t sc = pack_bf16x2(big, big);
  uint4 q[4];
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) q[cc] = *(const uint4*)(sub + r * 128 + (((kh * 4 + cc) ^ (r & 7)) * 16));
#pragma unroll
  for (int cc = 0; cc < 4; ++cc) {
    const uint32_t w[4] = {q[cc].x, q[cc].y, q[cc].z, q[cc].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t m = w[i] & 0x7F7F7F7Fu, sg = w[i] & 0x80808080u;
      out[cc * 8 + i * 2] = bmul2((prmt(m, 0u, 0x4140u) << 4) | prmt(sg, 0u, 0x1404u), sc);
      out[cc * 8 + i * 2 + 1] = bmul2((prmt(m, 0u, 0x4342u) << 4) | prmt(sg, 0u, 0x3424u), sc);
    }
  }
}

// INT4: nibble pair (k, k+1) of byte i -> bf16x2 (128 + n) by placing the nibbles under the
// exponent of 128, minus 136 (exact), times the bf16-rounded group scale.
__device__ __forceinline__ void conv_int4(const char* sub, int r, int kh, float scale, uint32_t* out) {
  const uint32_t sc = pack_bf16x2(scale, scale);
  const uint32_t off = 0x43084308u;  // bf16x2 (136, 136)
  uint32_t qs[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) qs[j] = *(const uint32_t*)(sub + (kh * 8 + j) * 512 + r * 4);
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t q = qs[j], q4 = q >> 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      // out byte 0 = byte i of q (low nibble = k 2i), out byte 2 = byte i of q >> 4 (low nibble = k 2i+1)
      const uint32_t t = prmt(q, q4, 0x4040u | (uint32_t)i | ((uint32_t)(4 + i) << 8));
      const uint32_t v = (t & 0x000F000Fu) | 0x43004300u;
      out[j * 4 + i] = bmul2(bsub2(v, off), sc);
    }
  }
}

// BF16: the weights are the operand already; half a chunk of row r is unswizzled out of its
// 128-byte atom (chunk c of row r sits at chunk position c ^ (r % 8)).
__device__ __forceinline__ void conv_bf16(const char* sub, int r, int kh, uint32_t* out) {
  uint4 q[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) q[c] = *(const uint4*)(sub + kh * 128 * 128 + r * 128 + ((c ^ (r & 7)) * 16));
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    out[c * 4 + 0] = q[c].x;
    out[c * 4 + 1] = q[c].y;
    out[c * 4 + 2] = q[c].z;
    out[c * 4 + 3] = q[c].w;
  }
}

// Persistent kernel: one CTA per SM walks the work items (row tile of one expert x column block)
// with a stride of gridDim.x; the pipeline rings keep their phases across items, so the TMA for
// the next item runs while the current item's epilogue executes.
// MODE 0: gate/up GEMM + SiLU(gate)*up -> h (bf16, permuted row order).
// MODE 1: down GEMM x routing weight -> fp32 rows [R, H] in permuted order (combined later).
template <int FMT, int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1) tc_expert_gemm_kernel(const __grid_constant__ TcArgs a) {
  using Cfg = TcCfg<FMT, BN>;
  constexpr bool kGather = MODE == 0 && BN < kTcPermuteFromRows;
  constexpr int kStagesW = Cfg::kStagesW;
  constexpr int SB = Cfg::SB;  // activation stages
  constexpr int kStagesA = BN <= 64 ? 3 : 2;
  constexpr uint32_t kACol = BN <= 64 ? 128 : 256;
  // Row blocks of 32 or fewer: two accumulators (one per item in flight) fit below the A ring, so
  // the next item's first chunks are converted and multiplied while the previous item's epilogue
  // runs; larger row blocks keep one accumulator, drained before the next item's conversion.
  constexpr bool kDB = BN <= 32;
  static_assert(!kDB || 4 * BN <= (int)kACol, "two accumulators fit below the A ring");
  constexpr int WSUB = WFmt<FMT>::kSubBytes;
  constexpr int WSTAGE = 2 * WSUB;
  constexpr int BSTAGE = Cfg::kBStage;  // BN rows x 128 K bf16, two 128-byte swizzle atoms
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = (char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  char* sW = smem;
  char* sB = smem + kStagesW * WSTAGE;
  char* sS = sB + SB * BSTAGE;  // scale slots, one per weight stage
  constexpr int kScaleSlot = Cfg::kScaleSlot;
  __shared__ uint64_t w_full[kStagesW], w_empty[kStagesW], a_full[kStagesA], a_empty[kStagesA], b_full[SB],
      b_empty[SB], acc_full[2], acc_empty[2], drain;
  __shared__ uint64_t work_full[kRing], work_empty[kRing];
  __shared__ int s_work[kRing];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_tok[2][BN];     // gather: token of each row of the item (double-buffered)
  __shared__ float s_cw[2][BN];    // down epilogue: routing weight / global scale of each column

  // gate/up: the tile table may come from the launch right before this one; down: it was final
  // before the gate/up GEMM passed its own pdl_wait(), so only the activations need the wait
  if (MODE == 0) pdl_wait();
  const int ntiles = load_tile(a.tiles).expert;  // header entry holds the tile count
  const int ncb = MODE == 0 ? a.I / 128 : (a.H + 255) / 256;
  const int nwork = ntiles * ncb;
  if ((int)blockIdx.x >= nwork) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nK = a.K / kKC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesW; ++i) {
      // the TMA issue, plus (scales by cp.async) one arrival per producer lane
      mbar_init(&w_full[i], FMT == MOE_FMT_NVFP4_W4A16 ? 1 : 1 + 32);
      mbar_init(&w_empty[i], kConvWarps);
    }
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(&a_full[i], kConvWarps);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(&b_full[i], kGather ? kGathWarps : 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&work_full[i], 1);
      mbar_init(&work_empty[i], (kGather ? kGathWarps : 1) + 1 + kConvWarps);  // every consuming warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kConvWarps);
    }
    mbar_init(&drain, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProdWarp && lane == 0) {
    if (FMT != MOE_FMT_NVFP4_W4A16) prefetch_tmap(&a.wmap);
    if (!kGather) prefetch_tmap(&a.bmap);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;
  if (MODE == 1 && warp != kProdWarp) pdl_wait();  // the weight producer needs nothing from the gate/up GEMM
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
  // per-item geometry
  auto item = [&](int wk, TileEntry& te, int& nb0, int& nb1, int& nsub) {
    const int tile = wk / ncb, cb = wk % ncb;
    te = load_tile(a.tiles + 1 + tile);
    if (MODE == 0) {
      nb0 = cb * 128;
      nb1 = a.I + nb0;
      nsub = 2;
    } else {
      nb0 = cb * 256;
      nb1 = nb0 + 128;
      nsub = (a.H - nb0) >= 256 ? 2 : 1;
    }
  };

  if (warp == kProdWarp) {
    // ---------------- TMA producer (the whole warp walks the loop, lane 0 issues) ----------------
    int it = 0;
    int armed_w[kStagesW] = {0};
    for (int n = 0;; ++n) {
      int wk = -1;
      bool ok = true;
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
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sw = it % kStagesW;
        if (lane == 0) {
          ok = mbar_wait(&w_empty[sw], ((it / kStagesW) & 1) ^ 1, &s_abort);
          if (ok) {
            mbar_arrive_expect_tx(&w_full[sw], nsub * WSUB);
            ++armed_w[sw];
            if (FMT == MOE_FMT_NVFP4_W4A16)  // the item's (one or) two adjacent image blocks
              bulk_load(sW + sw * WSTAGE,
                        a.wimg + (((size_t)te.expert * nK + kc) * (a.N / 128) + 2 * (wk % ncb)) * kW16Block,
                        nsub * kW16Block, &w_full[sw]);
            else
            for (int g = 0; g < nsub; ++g) {
              char* dst = sW + sw * WSTAGE + g * WSUB;
              const int nb = g == 0 ? nb0 : nb1;
              if (FMT == MOE_FMT_BF16) {  // two 64-K boxes of the bf16 rows
                tma_load_2d(dst, &a.wmap, &w_full[sw], kc * kKC, te.expert * a.N + nb);
                tma_load_2d(dst + 128 * 128, &a.wmap, &w_full[sw], kc * kKC + 64, te.expert * a.N + nb);
              } else if (FMT == MOE_FMT_FP8_B128_W8A16)
                tma_load_2d(dst, &a.wmap, &w_full[sw], kc * kKC, te.expert * a.N + nb);
              else
                tma_load_2d(dst, &a.wmap, &w_full[sw], nb, te.expert * (a.K / 8) + kc * 16);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        {  // this chunk's weight scales into the stage's slot, completing on the same barrier
          char* ss = sS + sw * kScaleSlot;
          const int e = te.expert;
          if (FMT == MOE_FMT_NVFP4_W4A16) {
            // in the image blocks
          } else if (FMT == MOE_FMT_BF16) {
            // no scales: the arrival below still completes this lane's share of the barrier
          } else if (FMT == MOE_FMT_FP8_B128_W8A16) {
            if (lane < nsub)
              cp_async_4(smem_u32(ss + lane * 4),
                         (const float*)a.wscale + ((size_t)e * (a.N / 128) + (lane == 0 ? nb0 : nb1) / 128) * (a.K / 128) + kc);
          } else if (FMT == MOE_FMT_INT4_G128_W4A16) {
            const int g = lane >> 4, piece = lane & 15;
            if (g < nsub)
              cp_async_16(smem_u32(ss + g * 256 + piece * 16),
                          (const char*)a.wscale + (((size_t)e * (a.K / 128) + kc) * a.N + (g == 0 ? nb0 : nb1)) * 2 +
                              piece * 16);
          }
          if (FMT != MOE_FMT_NVFP4_W4A16) cp_async_mbar_arrive_noinc(&w_full[sw]);
        }
      }
      if (!ok) break;
    }
    if (lane == 0 && s_abort) {  // let every issued copy land before shared memory goes away
      volatile int no_abort = 0;
      for (int i = 0; i < kStagesW; ++i)
        if (armed_w[i]) mbar_wait(&w_full[i], (armed_w[i] - 1) & 1, &no_abort);
    }
    __syncwarp();
  } else if (!kGather && warp == kGathWarp0) {
    // ---------------- activation tiles by TMA (a warp of their own, so that the weight stream
    // runs as far ahead as its stages allow instead of at the pace of the activation ring) -------
    int it = 0;
    int armed_b[SB] = {0};
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      const int wk = next_item(nitem, ok);
      if (wk < 0) break;
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sb = it % SB;
        if (lane == 0) {
          ok = mbar_wait(&b_empty[sb], ((it / SB) & 1) ^ 1, &s_abort);
          if (ok) {
            char* bd = sB + sb * BSTAGE;
            mbar_arrive_expect_tx(&b_full[sb], BSTAGE);
            ++armed_b[sb];
            tma_load_3d(bd, &a.bmap, &b_full[sb], 0, te.row0, kc * 2);  // both 64-K atoms
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0 && s_abort) {  // let every issued copy land before shared memory goes away
      volatile int no_abort = 0;
      for (int i = 0; i < SB; ++i)
        if (armed_b[i]) mbar_wait(&b_full[i], (armed_b[i] - 1) & 1, &no_abort);
    }
    __syncwarp();
  } else if (kGather && warp >= kGathWarp0) {
    // ---------------- gate/up activation rows: token rows of x -> shared memory ----------------
    // 16 threads per row (16-byte pieces of the 256-byte chunk row), 4 rows per pass.  Piece p of
    // row j lands in swizzle atom p / 8 (K 0-63 or 64-127) at piece (p % 8) ^ (j % 8).
    constexpr int LAG = Cfg::LAG;
    constexpr int RP = BN / 4;
    const int gt = (warp - kGathWarp0) * 32 + lane;
    const int piece = gt & 15, rsub = gt >> 4;
    const uint32_t dpiece = (uint32_t)(piece >> 3) * BN * 128;
    int it = 0, pend = 0;
    bool ok = true;
    for (int nitem = 0;; ++nitem) {
      const int wk = next_item(nitem, ok);
      // the gather warps leave together (they meet in a named barrier every item)
      if (!named_bar_and(2, kGathWarps * 32, ok && wk >= 0)) break;
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      int* tb = s_tok[nitem & 1];
      if (ok)
        for (int j = gt; j < BN; j += kGathWarps * 32) tb[j] = a.perm[te.row0 + (j < te.rows ? j : te.rows - 1)] / a.k;
      ok = named_bar_and(2, kGathWarps * 32, ok);
      if (!ok) break;
      const char* xrow = (const char*)a.x + piece * 16;
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sb = it % SB;
        ok = __all_sync(0xffffffffu, mbar_wait(&b_empty[sb], ((it / SB) & 1) ^ 1, &s_abort));
        if (!ok) break;
        const uint32_t bs = smem_u32(sB + sb * BSTAGE) + dpiece;
        const char* xk = xrow + kc * (kKC * 2);
#pragma unroll 8
        for (int i = 0; i < RP; ++i) {
          const int j = rsub + 4 * i;
          cp_async_16(bs + j * 128 + ((((uint32_t)piece & 7u) ^ (uint32_t)(j & 7)) << 4),
                      xk + (size_t)tb[j] * (a.K * 2));
        }
        cp_async_commit();
        if (pend == LAG) {  // the chunk LAG behind this one has landed: publish it
          cp_async_wait<LAG>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&b_full[(it - LAG) % SB]);
        } else {
          ++pend;
        }
      }
    }
    cp_async_wait<0>();
    if (ok) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0)
        for (int p = pend; p > 0; --p) mbar_arrive(&b_full[(it - p) % SB]);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer ----------------
    // The whole warp walks the loop and waits together (lane 0 issues): a lane left idling in a
    // barrier wait would hold the diverged warp, and with it the issuing lane, asleep.
    int it = 0;
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      const int wk = next_item(nitem, ok);
      if (wk < 0) break;
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      // the MMA's N: the item's rows rounded up to 16 (a routing tile of a small expert is mostly
      // padding, and the tensor pipe's time per MMA scales with N)
      const int nmma = ((te.rows + 15) & ~15) < BN ? ((te.rows + 15) & ~15) : BN;
      const uint32_t idesc = idesc_bf16_f32(128, nmma);
      const int ab = kDB ? nitem & 1 : 0;
      const uint32_t acc = tmem + ab * 2 * BN;
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sa = it % kStagesA, sb = it % SB;
        ok = mbar_wait(&a_full[sa], (it / kStagesA) & 1, &s_abort) &&
             mbar_wait(&b_full[sb], (it / SB) & 1, &s_abort) &&
             (!kDB || kc != 0 || mbar_wait(&acc_empty[ab], ((nitem >> 1) & 1) ^ 1, &s_abort));
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        fence_after_sync();
        if (lane == 0) {
          const uint32_t b0 = smem_u32(sB + sb * BSTAGE);
          for (int g = 0; g < nsub; ++g)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t bdsc = sdesc_k_sw128(b0 + (ks >> 2) * BN * 128 + (ks & 3) * 32);
              mma_f16_ts(acc + g * BN, tmem + kACol + sa * 128 + g * 64 + ks * 8, bdsc, idesc, (kc | ks) != 0);
            }
          mma_commit(&a_empty[sa]);
          mma_commit(&b_empty[sb]);
        }
        __syncwarp();
      }
      if (ok && lane == 0) mma_commit(&acc_full[ab]);
      __syncwarp();
    }
    if (lane == 0) mma_commit(&drain);  // completes once every MMA issued by this thread has finished
    __syncwarp();
  } else if (warp < kConvWarps) {
    // ---------------- converters (16 warps) and epilogue ----------------
    const int g = (warp >> 2) & 1, kh = warp >> 3, q = warp & 3, r = q * 32 + lane;
    int it = 0;
    bool ok = true;
    // one K chunk of the item into the A ring: this thread's row of sub-tile g, K half kh
    auto convert = [&](int nsub) -> bool {
      const bool active = g < nsub;
      const int sw = it % kStagesW, sa = it % kStagesA;
      if (!__all_sync(0xffffffffu, mbar_wait(&w_full[sw], (it / kStagesW) & 1, &s_abort))) return false;
      // the chunk's scale for this thread's row (or sub-tile), from the stage's scale slot
      const char* ss = sS + sw * kScaleSlot;
      uint32_t sc_raw = 0u;
      if (active && FMT != MOE_FMT_BF16) {
        if (FMT == MOE_FMT_FP8_B128_W8A16) sc_raw = *(const uint32_t*)(ss + g * 4);
        else if (FMT == MOE_FMT_INT4_G128_W4A16) sc_raw = __float_as_uint(__half2float(*(const __half*)(ss + g * 256 + r * 2)));
      }
      const float sc = __uint_as_float(sc_raw);
      uint32_t v[32];
      if (active) {
        const char* sub = sW + sw * WSTAGE + g * WSUB;
        if (FMT == MOE_FMT_BF16) conv_bf16(sub, r, kh, v);
        else if (FMT == MOE_FMT_FP8_B128_W8A16) conv_fp8(sub, r, kh, sc, v);
        else if (FMT == MOE_FMT_INT4_G128_W4A16) conv_int4(sub, r, kh, sc, v);
        else {  // image block of this row: gate/up blocks hold 64 gate rows, then the up rows
          const int blk = MODE == 0 ? r >> 6 : g, row = MODE == 0 ? 64 * g + (r & 63) : r;
          const char* b = sW + sw * WSTAGE + blk * WSUB;
          conv_nvfp4(b, row, kh, *(const uint32_t*)(b + kW16Codes + row * 8 + kh * 4), v);
        }
        reg_fence(v);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&w_empty[sw]);
      if (!__all_sync(0xffffffffu, mbar_wait(&a_empty[sa], ((it / kStagesA) & 1) ^ 1, &s_abort))) return false;
      fence_after_sync();
      if (active) {
        tmem_st_32x32(taddr(tmem, q * 32, kACol + sa * 128 + g * 64 + kh * 32), v);
        tmem_st_wait();
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[sa]);
      return true;
    };
    // epilogue of item n from accumulator buffer ab (the caller has waited for acc_full); with
    // two accumulators the buffer is released as soon as this warp has read its columns
    auto epilogue = [&](int n, int ab, const TileEntry& te, int nb0, int nb1, int nsub, float inv_gs) {
      const uint32_t acc = tmem + ab * 2 * BN;
      const int cend = te.rows < BN ? te.rows : BN;  // warp-uniform: no column group past the rows
      auto release = [&]() {
        if (kDB) {
          fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[ab]);
        }
      };
      if (MODE == 0) {
        const int part = warp >> 2;  // 0..3: 16-column chunks part, part+4, ...
        const int n_out = nb0 + r;
        bool released = false;
        for (int c0 = part * 16; c0 < cend; c0 += 64) {
          uint32_t G[16], U[16];
          tmem_ld_32x16(taddr(acc, q * 32, c0), G);
          tmem_ld_32x16(taddr(acc, q * 32, BN + c0), U);
          tmem_ld_wait();
          if (c0 + 64 >= cend) {  // this warp's last read of the accumulator
            release();
            released = true;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (col < te.rows) {
              const float gv = __uint_as_float(G[j]) * inv_gs, uv = __uint_as_float(U[j]) * inv_gs;
              const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
              a.h_out[(size_t)(te.row0 + col) * a.I + n_out] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
            }
          }
        }
        if (!released) release();
      } else {
        const bool active = g < nsub;
        const int c = (g == 0 ? nb0 : nb1) + r;
        const float* cw = s_cw[n & 1];
        bool released = false;
        for (int c0 = kh * 16; active && c0 < cend; c0 += 32) {
          uint32_t Y[16];
          tmem_ld_32x16(taddr(acc, q * 32, g * BN + c0), Y);
          tmem_ld_wait();
          if (c0 + 32 >= cend) {
            release();
            released = true;
          }
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (col < te.rows) a.y_out[(size_t)(te.row0 + col) * a.H + c] = bf16_bits(cw[col] * __uint_as_float(Y[j]));
          }
        }
        if (!released) release();
      }
    };
    bool have_prev = false;
    TileEntry te_p;
    int nb0_p = 0, nb1_p = 0, nsub_p = 0;
    float igs_p = 1.f;
    for (int nitem = 0;; ++nitem) {
      const int wk = next_item(nitem, ok);
      // the converter warps leave together (they meet in a named barrier every item)
      const bool live = named_bar_and(1, kConvWarps * 32, ok && wk >= 0);
      if (!kDB && !live) break;
      TileEntry te;
      int nb0 = 0, nb1 = 0, nsub = 0, d = 0;
      float inv_gs = 1.f;
      if (live) {
        item(wk, te, nb0, nb1, nsub);
        inv_gs = FMT == MOE_FMT_NVFP4_W4A16 ? 0x1p10f / a.wgs[te.expert] : 1.f;  // see conv_nvfp4
        if (MODE == 1 && threadIdx.x < BN) {  // column table of the down epilogue: routing weights
          const int col = threadIdx.x;
          s_cw[nitem & 1][col] = col < te.rows ? a.topk_w[a.perm[te.row0 + col]] * inv_gs : 0.f;
        }
        if (kDB) {  // the item's first chunks go into the A ring before the previous item's epilogue
          d = nK < kStagesA ? nK : kStagesA;
          for (int kc = 0; kc < d && ok; ++kc, ++it) ok = convert(nsub);
        }
      }
      if (kDB) {
        if (have_prev && ok) {
          const int n = nitem - 1, ab = n & 1;
          ok = __all_sync(0xffffffffu, mbar_wait(&acc_full[ab], (n >> 1) & 1, &s_abort));
          if (ok) {
            fence_after_sync();
            epilogue(n, ab, te_p, nb0_p, nb1_p, nsub_p, igs_p);
          }
        }
        if (!live) break;  // (a warp whose wait failed skips its work but still meets the barrier)
        for (int kc = d; kc < nK && ok; ++kc, ++it) ok = convert(nsub);
        te_p = te;
        nb0_p = nb0;
        nb1_p = nb1;
        nsub_p = nsub;
        igs_p = inv_gs;
        have_prev = true;
      } else {
        for (int kc = 0; kc < nK && ok; ++kc, ++it) ok = convert(nsub);
        // epilogue of this item; every converter thread takes the same branch here
        if (ok) ok = mbar_wait(&acc_full[0], nitem & 1, &s_abort);
        ok = named_bar_and(1, kConvWarps * 32, ok);
        if (!ok) break;
        fence_after_sync();
        epilogue(nitem, 0, te, nb0, nb1, nsub, inv_gs);
        fence_before_sync();  // accumulator reads are ordered before the next item's MMAs
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
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && s_abort) set_dev_error(a.err, kDevTimeout);
  if (MODE == 1) {  // the routing-weighted combine, once every working CTA is done
    __shared__ int s_flag;
    if (!combine_tail(a.ct, min((int)gridDim.x, nwork), &s_flag) && threadIdx.x == 0)
      set_dev_error(a.err, kDevTimeout);
  }
}

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
int num_sms() {
  static int n[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!n[dev]) cudaDeviceGetAttribute(&n[dev], cudaDevAttrMultiProcessorCount, dev);
  return n[dev] > 0 ? n[dev] : 148;
}

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
  if (fmt == MOE_FMT_BF16)
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, v.a, v.K, (uint64_t)E * v.N, (uint64_t)v.K * 2, 64, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (fmt == MOE_FMT_FP8_B128_W8A16)
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, v.a, v.K, (uint64_t)E * v.N, v.K, 128, 128,
                    CU_TENSOR_MAP_SWIZZLE_128B);
  if (fmt == MOE_FMT_INT4_G128_W4A16)
    return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, v.a, v.N, (uint64_t)E * (v.K / 8), (uint64_t)v.N * 4, 128, 16,
                    CU_TENSOR_MAP_SWIZZLE_NONE);
  return true;  // NVFP4: image blocks by bulk copy
}

// Activation rows [R, K] bf16 viewed as [K/64 atoms][R rows][64]: one copy brings BN rows x
// 128 K as two 128-byte swizzle atoms.
bool act_map(CUtensorMap* m, const void* base, uint64_t R, int K, int bn) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, R, (cuuint64_t)K / 64};
  cuuint64_t strides[2] = {(cuuint64_t)K * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)bn, 2};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int FMT, int MODE, int BN>
cudaError_t launch_one(const TcArgs& args, int grid_x, int grid_y, cudaStream_t s) {
  constexpr size_t need = TcCfg<FMT, BN>::kSmem;
  // at least 116 KB so that a single CTA (owning all 512 TMEM columns) runs per SM
  constexpr size_t smem = need > 116 * 1024 ? need : 116 * 1024;
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(tc_expert_gemm_kernel<FMT, MODE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    attr = true;
  }
  return launch_pdl(tc_expert_gemm_kernel<FMT, MODE, BN>,
                    dim3(grid_x * grid_y < num_sms() ? grid_x * grid_y : num_sms()), dim3(kThreads), smem, s, args);
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
  if (fmt == MOE_FMT_BF16) return launch_bn<MOE_FMT_BF16, MODE>(bn, args, gx, gy, s);
  return launch_bn<MOE_FMT_NVFP4_W4A16, MODE>(bn, args, gx, gy, s);
}

}  // namespace

bool tc_make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1, uint64_t pitch,
                 uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw) {
  return make_map(m, dt, base, d0, d1, pitch, b0, b1, sw);
}
int tc_num_sms() { return num_sms(); }
bool tc_act_map(CUtensorMap* m, const void* base, uint64_t R, int K, int bn) { return act_map(m, base, R, K, bn); }

// Token rows per GEMM tile: the next power of two >= the mean rows per active expert, 16..128.
// The weight-converting formats (INT4, NVFP4 W4A16) take twice that: their MMA and conversion
// cost per tile does not depend on the rows it holds (an M = 128 MMA costs the same up to
// N = 128), so fewer, fuller tiles convert and stream each expert's weights fewer times; NVFP4
// W4A16 goes on to 256-row tiles (moe_gemm_tcw.cu) past 128.
int tc_row_block(int fmt, int T, int k, int E) {
  const long R = (long)T * k;
  const long active = R < E ? (R > 0 ? R : 1) : E;
  long avg = (R + active - 1) / active;
  if (fmt == MOE_FMT_INT4_G128_W4A16 || fmt == MOE_FMT_NVFP4_W4A16) avg *= 2;
  int bn = 16;
  while (bn < 128 && bn < avg) bn *= 2;
  if (fmt == MOE_FMT_NVFP4_W4A16 && bn == 128 && avg > 128) bn = tcw_row_block();  // 256-row tiles
  return bn;
}

cudaError_t launch_experts_tc(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                              int bn, const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, uint16_t* out) {
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  // NVFP4: weight image blocks (codes in the converter's bit order, then scales)
  if (d.fmt == MOE_FMT_NVFP4_W4A16 && (!d.size[MOE_T_GU_IMG] || !d.size[MOE_T_D_IMG])) return cudaErrorInvalidValue;
  TcArgs a;
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
  const int gx = (int)(R / bn + (R < (size_t)E ? R : (size_t)E) + 1);

  // gate/up: A = fused [2I, H] weights, B = gathered rows of x
  if (!weight_map(&a.wmap, d.fmt, gu, E)) return cudaErrorInvalidValue;
  a.wimg = (const uint8_t*)(packed + d.offset[MOE_T_GU_IMG]);
  a.x = x;
  if (bn >= kTcPermuteFromRows) {
    __nv_bfloat16* xp = (__nv_bfloat16*)(ws + L.xp);
    if (launch_gather_rows(x, a.perm, k, (int)R, H, xp, s) != cudaSuccess || !act_map(&a.bmap, xp, R, H, bn))
      return cudaErrorInvalidValue;
  }
  a.wscale = gu.b;
  a.wgs = gu.gs;
  a.N = 2 * I;
  a.work_ctr = (int*)(ws + L.err) + 1;
  a.K = H;
  record_event(ev.start[0], s);
  cudaError_t err = launch_fmt<0>(d.fmt, bn, a, gx, I / 128, s);
  record_event(ev.stop[0], s);
  if (err != cudaSuccess) return err;

  // down: A = [H, I] weights, B = rows of h (already in permuted order)
  if (!weight_map(&a.wmap, d.fmt, dn, E) || !act_map(&a.bmap, ws + L.h, R, I, bn)) return cudaErrorInvalidValue;
  a.wimg = (const uint8_t*)(packed + d.offset[MOE_T_D_IMG]);
  a.wscale = dn.b;
  a.wgs = dn.gs;
  a.N = H;
  a.work_ctr = (int*)(ws + L.err) + 2;
  a.K = I;
  record_event(ev.start[1], s);
  err = launch_fmt<1>(d.fmt, bn, a, gx, (H + 255) / 256, s);
  record_event(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
