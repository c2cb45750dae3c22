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
// N = 64 or 128, so one instruction per K step covers what two N = 128 ones did.
// Both operands are read from operand images (moe_internal.cuh, ActImage): the packed weights
// and the quantized activations are laid out in global memory exactly as one K chunk of an item
// sits in shared memory -- codes in the 128-byte swizzle, block scales in the order the scale
// warps move them -- so a chunk of each operand arrives by ONE bulk copy.  (A TMA unit's cost
// is per copy and nearly independent of its size up to tens of KB: three 16 KB tensor tiles and
// three 2 KB scale copies per chunk took ~1.07 us, the two image copies ~0.94 us.)  x is
// quantized straight into its image (one copy per routed token slot, at its routing tile's row),
// so the gate/up GEMM needs no row gather; h likewise.  The weight scale image keeps, per K = 64
// step, a 512-byte atom whose row l holds the four scales of tile rows l, l + 32, l + 64, l + 96;
// the activation scales are 16 bytes per row; four scale warps move both into tensor memory
// with tcgen05.st (measured faster than tcgen05.cp issued by the MMA thread, which shares the
// tensor pipe with the MMAs).  K need not be a multiple of 256: a last half chunk (128 columns)
// issues two K steps, its upper half (zero in the images) unread.
//
// The down GEMM also combines, deterministically: its epilogue stores the routing-weighted bf16
// row of (token t, slot j) at row t * k + j of a slot-ordered buffer, a signal warp publishes
// each finished item and counts it, and after the GEMM items the work queue hands out combine
// items (kCombTokens tokens each): once every GEMM item is counted, the producer bulk-copies
// each token's k contiguous rows into the (now idle) stage memory and the epilogue warps sum
// them in slot order in fp32 and write out[t] in bf16.
//
// Warps: 0-7 epilogue (thread = token row, 64 or 128 contiguous output features), 8-11 scale
// warps, (down) 12 signal warp, then the TMA producer and the MMA issuer (which owns TMEM).
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
constexpr int kCPS = 2;                   // K chunks per stage: one bulk copy per operand covers them
constexpr int kStages = 4 / kCPS;         // stages in flight
constexpr int kRing = 16;                 // work items handed from the producer to the other warps
constexpr int kCombRing = 4;              // down: items whose stored rows await the signal warp
constexpr int kWCodes = 128 * 128;        // one 128-row weight tile, 128-byte swizzle
constexpr int kSfBlock = 2048;            // scales of one (128-row tile, chunk): four 512-byte atoms
constexpr int kWChunk = 2 * kWCodes + 2 * kSfBlock;  // two tiles = the 256 B rows of one item
constexpr int kXCodes = kRows * 128;      // activation codes, 128-byte swizzle
constexpr int kXChunk = kXCodes + kSfBlock;
constexpr int kWStage = kCPS * kWChunk, kXStage = kCPS * kXChunk;
constexpr size_t kSmem = 1024 + (size_t)kStages * (kWStage + kXStage);
constexpr uint32_t kSfCol = 256;          // TMEM: [0, 256) accumulator, then the stages' scale columns
constexpr uint32_t kSfChunkCols = 48;     // per K step: A (activation) scales 4 columns, B (weight) 8
constexpr uint32_t kSfStageCols = kCPS * kSfChunkCols;
static_assert(kWChunk == kWImgBlock && kXChunk == kAImgBlock, "a stage holds whole image blocks");
static_assert(kSfCol + kStages * kSfStageCols <= 512, "tensor memory columns");
constexpr int kCombTokens = 24;           // tokens per combine item of the down GEMM
constexpr int kCombBuf = 96 * 1024;       // combine: two buffers of partial rows in the stage memory

// Warp roles: 0-7 epilogue (warp w reads TMEM lane quarter w % 4), 8-11 scale warps (quarter
// w % 4), then (down only) a signal warp, the TMA producer and the MMA issuer.
constexpr int kEpiWarps = 8, kSfWarp0 = 8, kSfWarps = 4, kSigWarp = 12;
template <int MODE>
struct Roles {
  static constexpr int kSigWarps = MODE == 1 ? 1 : 0;
  static constexpr int kProdWarp = kSigWarp + kSigWarps, kMmaWarp = kProdWarp + 1;
  static constexpr int kThreads = (kMmaWarp + 1) * 32;
};
static_assert(2 * kCombBuf <= kStages * (kWStage + kXStage), "combine buffers live in the stage memory");

struct Fp4Args {
  const uint8_t* wimg;      // weight operand image [E, P, C, kWImgBlock] (P = tile pairs per expert)
  const uint8_t* aimg;      // activation operand image [tiles, C, kAImgBlock]
  int C, P;                 // K chunks, weight tile pairs
  const float* wgs;         // weight global scales [E]
  const float* ags;         // activation global scales [R]
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;          // MODE 0 output [R, I] bf16 (dynamic activation scales)
  const float* hgs_static;  // MODE 2 (gate/up, static activation scales): h's global scale (dev); h
  uint8_t* hq_out;          //   leaves NVFP4-quantized instead, into its operand image [tiles, C(I), ..]
  int hC;                   //   (C(I) chunks), with the global scale per routed row [R]
  float* hg_out;
  uint16_t* comb;           // MODE 1: routing-weighted rows [T*k, H] bf16, row t*k + j = (token t, slot j)
  int* done;                // MODE 1: GEMM items finished (their rows published), zero on entry
  uint16_t* out;            // MODE 1 output [T, H] bf16
  int T;
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

__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

// Orders global data acquired by generic loads before later bulk (async-proxy) copies of it.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// The routing-weighted partial rows stream through L2 once each (written by the epilogue, read
// back by the combine much later), so they are written evict-first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void st_global_v8_hint(void* p, const uint32_t* v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8}, %9;" ::"l"(p), "r"(v[0]),
               "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "l"(pol)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return (uint32_t)bf16_bits(lo) | ((uint32_t)bf16_bits(hi) << 16);
}

// MODE 0: gate/up (h in bf16), 1: down + combine, 2: gate/up with static activation scales (h
// leaves as NVFP4 codes, block scales and global scales).
template <int MODE>
__global__ void __launch_bounds__(Roles<MODE>::kThreads, 1) fp4_kernel(const __grid_constant__ Fp4Args a) {
  constexpr bool kGateUp = MODE != 1, kFuseH = MODE == 2;
  constexpr int kSigWarps = Roles<MODE>::kSigWarps, kProdWarp = Roles<MODE>::kProdWarp,
                kMmaWarp = Roles<MODE>::kMmaWarp;
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = (char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  char* sW = smem;
  char* sX = sW + kStages * kWStage;
  __shared__ uint64_t w_full[kStages], w_empty[kStages], x_full[kStages], x_empty[kStages], s_full[kStages],
      s_empty[kStages], acc_full, acc_empty, drain;
  __shared__ uint64_t work_full[kRing], work_empty[kRing];
  __shared__ uint64_t rows_stored[kCombRing], rows_taken[kCombRing], c_full[2], c_empty[2];
  __shared__ int s_work[kRing];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  // gate/up: wait for the activation quantization (and, before it, routing); down: the tile table
  // was final before the gate/up GEMM passed its own pdl_wait(), so only the h codes need the wait
  if (kGateUp) pdl_wait();
  const int ntiles = load_tile(a.tiles).expert;
  const int ncb = kGateUp ? a.I / 128 : (a.H + 255) / 256;
  // down: after the ngemm GEMM items, one combine item per kCombTokens tokens
  const int ngemm = ntiles * ncb;
  const int nslices = kGateUp || a.k == 1 ? 0 : (a.T + kCombTokens - 1) / kCombTokens;
  const int nwork = ngemm + nslices;
  // combine items move partial rows in segments of (token, cseg columns) -- each one contiguous
  // run of k rows when cseg = H -- packed nseg to a buffer
  const int cseg = !kGateUp && a.k * a.H * 2 > kCombBuf ? kCombBuf / (a.k * 2) / 256 * 256 : a.H;
  const int nsegc = (a.H + cseg - 1) / cseg, nseg = max(1, kCombBuf / (a.k * cseg * 2));
  if ((int)blockIdx.x >= nwork) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nK = (a.K + kKC - 1) / kKC;           // chunks; the last is a half chunk when K % 256 = 128
  const int last_ks = (a.K % kKC) ? 2 : 4;        // K = 64 steps of the last chunk
  const int nKP = (nK + kCPS - 1) / kCPS;         // stages per item

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], 1);
      mbar_init(&x_full[i], 1);
      mbar_init(&x_empty[i], 1);
      mbar_init(&s_full[i], kSfWarps);
      mbar_init(&s_empty[i], 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&work_full[i], 1);
      mbar_init(&work_empty[i], 1 + kEpiWarps + kSfWarps + kSigWarps);  // every consuming warp
    }
    for (int i = 0; i < kCombRing; ++i) {
      mbar_init(&rows_stored[i], kEpiWarps);
      mbar_init(&rows_taken[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&c_full[i], 1);
      mbar_init(&c_empty[i], kEpiWarps);
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
  // Item wk: a combine item (down, wk >= ngemm; returns false), or routing tile `tile`, weight
  // rows w0 .. w0+127 and w1 .. w1+127 of its expert.  GEMM items run tile by tile, so a tile's
  // activations are reused by its column blocks while in L2.
  auto item = [&](int wk, TileEntry& te, int& tile, int& w0, int& w1) -> bool {
    if (!kGateUp && wk >= ngemm) return false;
    tile = wk / ncb;
    const int cb = wk % ncb;
    te = load_tile(a.tiles + 1 + tile);
    w0 = kGateUp ? cb * 128 : cb * 256;
    w1 = kGateUp ? a.I + w0 : w0 + 128;
    return true;
  };

  if (warp == kProdWarp) {
    // ---------------- TMA producer (whole warp walks the loop, lane 0 issues) ----------------
    int it = 0, cg = 0;  // chunks, combine buffer groups
    bool ok = true, comb_ready = false;
    int armed_w[kStages] = {0}, armed_x[kStages] = {0}, armed_c[2] = {0};
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
      int tile, w0, w1;
      if (!item(wk, te, tile, w0, w1)) {
        // combine item: stream its tokens' partial rows into the two buffers.  The first one waits
        // until every GEMM item of the grid is done -- then also this CTA's stage memory is free.
        if (lane == 0) {
          if (!comb_ready) {
            const long long t0 = clock64();
            while (ok && ld_acquire_gpu(a.done) < ngemm) {
              if (*(volatile int*)&s_abort || clock64() - t0 > kWaitLimitCycles) {
                *(volatile int*)&s_abort = 1;
                ok = false;
              }
            }
            fence_proxy_async_global();  // the rows acquired above, read next by bulk copies
            comb_ready = true;
          }
          const int tb = (wk - ngemm) * kCombTokens, te_ = min(a.T, tb + kCombTokens);
          for (int g0 = 0; ok && g0 < (te_ - tb) * nsegc; g0 += nseg, ++cg) {
            const int b = cg & 1, ng_ = min(nseg, (te_ - tb) * nsegc - g0);
            ok = mbar_wait(&c_empty[b], ((cg >> 1) & 1) ^ 1, &s_abort);
            if (!ok) break;
            mbar_arrive_expect_tx(&c_full[b], (uint32_t)(ng_ * a.k * min(cseg, a.H) * 2));
            ++armed_c[b];
            for (int u = 0; u < ng_; ++u) {
              const int sg = g0 + u, t = tb + sg / nsegc, c0 = (sg % nsegc) * cseg, cw = min(cseg, a.H - c0);
              char* dst = smem + (size_t)b * kCombBuf + (size_t)u * a.k * cseg * 2;
              const uint16_t* src = a.comb + (size_t)t * a.k * a.H + c0;
              if (cw == a.H)
                bulk_load(dst, src, (uint32_t)(a.k * a.H * 2), &c_full[b]);
              else
                for (int j = 0; j < a.k; ++j)
                  bulk_load(dst + (size_t)j * cw * 2, src + (size_t)j * a.H, (uint32_t)(cw * 2), &c_full[b]);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        continue;
      }
      for (int kp = 0; kp < nKP; ++kp, ++it) {
        const int st = it % kStages, kc0 = kp * kCPS, nch = min(kCPS, nK - kc0);
        if (lane == 0) {
          ok = mbar_wait(&w_empty[st], ((it / kStages) & 1) ^ 1, &s_abort);
          if (ok) {  // one bulk copy: both weight tiles' codes and scales of the stage's chunks
            mbar_arrive_expect_tx(&w_full[st], (uint32_t)(nch * kWChunk));
            ++armed_w[st];
            const int pair = kGateUp ? w0 / 128 : w0 / 256;
            bulk_load(sW + st * kWStage, a.wimg + (((size_t)te.expert * a.P + pair) * a.C + kc0) * kWChunk,
                      (uint32_t)(nch * kWChunk), &w_full[st]);
          }
          if (ok) {
            ok = mbar_wait(&x_empty[st], ((it / kStages) & 1) ^ 1, &s_abort);
            if (MODE == 1 && it == 0) pdl_wait();
            if (ok) {  // one bulk copy: the routing tile's codes and scales of the stage's chunks
              mbar_arrive_expect_tx(&x_full[st], (uint32_t)(nch * kXChunk));
              ++armed_x[st];
              bulk_load(sX + st * kXStage, a.aimg + ((size_t)tile * a.C + kc0) * kXChunk, (uint32_t)(nch * kXChunk),
                        &x_full[st]);
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
      for (int i = 0; i < 2; ++i)
        if (armed_c[i]) mbar_wait(&c_full[i], (armed_c[i] - 1) & 1, &no_abort);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (whole warp waits, lane 0 issues) ----------------
    const uint32_t idesc = idesc_nvf4(kRows, 256);
    int it = 0, ng = 0;  // chunks and GEMM items so far
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int wk = next_item(n, ok);
      if (wk < 0) break;
      if (!kGateUp && wk >= ngemm) continue;  // a combine item
      const int nitem = ng++;
      ok = mbar_wait(&acc_empty, (nitem & 1) ^ 1, &s_abort);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      fence_after_sync();
      for (int kp = 0; kp < nKP; ++kp, ++it) {
        const int st = it % kStages, kc0 = kp * kCPS, nch = min(kCPS, nK - kc0);
        ok = mbar_wait(&w_full[st], (it / kStages) & 1, &s_abort) &&
             mbar_wait(&x_full[st], (it / kStages) & 1, &s_abort) &&
             mbar_wait(&s_full[st], (it / kStages) & 1, &s_abort);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        fence_after_sync();
        if (lane == 0) {
          for (int j = 0; j < nch; ++j) {
            const int kc = kc0 + j;
            const uint32_t xa = smem_u32(sX + st * kXStage + j * kXChunk), wa = smem_u32(sW + st * kWStage + j * kWChunk);
            const uint32_t sfa = tmem + kSfCol + st * kSfStageCols + j * kSfChunkCols, sfb = sfa + 16;
            const int nks = kc == nK - 1 ? last_ks : 4;
            for (int ks = 0; ks < nks; ++ks)
              mma_nvf4(tmem, sdesc_k_sw128(xa + ks * 32), sdesc_k_sw128(wa + ks * 32), idesc, sfa + 4 * ks,
                       sfb + 8 * ks, (kc | ks) != 0);
          }
          mma_commit(&w_empty[st]);
          mma_commit(&x_empty[st]);
          mma_commit(&s_empty[st]);
        }
        __syncwarp();
      }
      if (ok && lane == 0) mma_commit(&acc_full);
      __syncwarp();
    }
    if (lane == 0) mma_commit(&drain);
    __syncwarp();
  } else if (warp >= kSfWarp0 && warp < kSfWarp0 + kSfWarps) {
    // ---------------- scale warps: block scales -> tensor memory (warp = lane quarter) -------
    // TMEM lane l, column 4 ks + j: K step ks's four scales of activation row l + 32 j (from the
    // row's 16 chunk bytes); column 16 + 8 ks + 4 g + j: those of weight row l + 32 j of tile g
    // (atom row l of the packed copy).  Every lane quarter gets a copy.
    const int q = warp & 3;
    int it = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int wk = next_item(n, ok);
      if (wk < 0) break;
      TileEntry te;
      int tile, w0, w1;
      if (!item(wk, te, tile, w0, w1)) continue;  // a combine item
      for (int kp = 0; kp < nKP; ++kp, ++it) {
        const int st = it % kStages, nch = min(kCPS, nK - kp * kCPS);
        ok = __all_sync(0xffffffffu, mbar_wait(&w_full[st], (it / kStages) & 1, &s_abort) &&
                                         mbar_wait(&x_full[st], (it / kStages) & 1, &s_abort) &&
                                         mbar_wait(&s_empty[st], ((it / kStages) & 1) ^ 1, &s_abort));
        if (!ok) break;
        fence_after_sync();
        for (int jc = 0; jc < nch; ++jc) {
        const uint32_t col = kSfCol + st * kSfStageCols + jc * kSfChunkCols;
        const char* xsf = sX + st * kXStage + jc * kXChunk + kXCodes + 16 * lane;
        const char* wsf = sW + st * kWStage + jc * kWChunk + 2 * kWCodes + 16 * lane;
        uint32_t v[16];
        uint4 x4[4];  // activations: row l + 32 j's 16 scales (word = K step)
#pragma unroll
        for (int j = 0; j < 4; ++j) x4[j] = *(const uint4*)(xsf + 512 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[j] = x4[j].x;
          v[4 + j] = x4[j].y;
          v[8 + j] = x4[j].z;
          v[12 + j] = x4[j].w;
        }
        tmem_st_32x16(taddr(tmem, q * 32, col), v);
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // weight columns of K steps 2h, 2h + 1
#pragma unroll
          for (int kk = 0; kk < 2; ++kk)
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              const uint4 u = *(const uint4*)(wsf + g * kSfBlock + (2 * h + kk) * 512);
              v[8 * kk + 4 * g] = u.x;
              v[8 * kk + 4 * g + 1] = u.y;
              v[8 * kk + 4 * g + 2] = u.z;
              v[8 * kk + 4 * g + 3] = u.w;
            }
          tmem_st_32x16(taddr(tmem, q * 32, col + 16 + 16 * h), v);
        }
        }
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_full[st]);
      }
    }
  } else if (warp == kSigWarp) {
    // ---------------- signal warp (down): per GEMM item, take the epilogue's stored rows
    // (freeing the ring slot), publish them at GPU scope and count the item done ----------------
    int ng = 0;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int wk = next_item(n, ok);
      if (!ok || wk < 0) break;
      if (wk >= ngemm) continue;
      const int nitem = ng++, rs = nitem % kCombRing;
      ok = __all_sync(0xffffffffu, mbar_wait(&rows_stored[rs], (nitem / kCombRing) & 1, &s_abort));
      if (!ok) break;
      if (a.k > 1 && lane == 0) {
        fence_acq_rel_gpu();  // the epilogue's stores (observed through the barrier) before the count
        atomicAdd(a.done, 1);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&rows_taken[rs]);
    }
  } else {
    // ---------------- epilogue: thread = token row of the tile ----------------
    const int q = warp & 3, half = warp >> 2, r = q * 32 + lane;
    bool ok = true;
    int ng = 0, cg = 0;  // GEMM items, combine buffer groups so far
    for (int n = 0; ok; ++n) {
      const int wk = next_item(n, ok);
      // the epilogue warps leave together (they meet in a named barrier every item)
      if (!named_bar_and(1, kEpiWarps * 32, ok && wk >= 0)) break;
      TileEntry te;
      int tile, w0, w1;
      if (!item(wk, te, tile, w0, w1)) {
        // combine item: per buffer group, each (token, column segment): out = bf16 of the sum of
        // the token's k routing-weighted rows in slot order (thread: 8 columns at a time)
        bool cok = true;
        const int tb = (wk - ngemm) * kCombTokens, te_ = min(a.T, tb + kCombTokens);
        for (int g0 = 0; g0 < (te_ - tb) * nsegc; g0 += nseg, ++cg) {
          const int b = cg & 1, ng_ = min(nseg, (te_ - tb) * nsegc - g0);
          cok = cok && mbar_wait(&c_full[b], (cg >> 1) & 1, &s_abort);
          if (cok) {
            for (int u = 0; u < ng_; ++u) {
              const int sg = g0 + u, t = tb + sg / nsegc, c0 = (sg % nsegc) * cseg, cw = min(cseg, a.H - c0);
              const char* seg = smem + (size_t)b * kCombBuf + (size_t)u * a.k * cseg * 2;
              for (int c = 8 * (int)threadIdx.x; c < cw; c += 8 * kEpiWarps * 32) {
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // slot order
                for (int j = 0; j < a.k; ++j) {
                  const uint4 v = *(const uint4*)(seg + ((size_t)j * cw + c) * 2);
                  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    acc[2 * e] += __uint_as_float(w[e] << 16);
                    acc[2 * e + 1] += __uint_as_float(w[e] & 0xFFFF0000u);
                  }
                }
                *(uint4*)(a.out + (size_t)t * a.H + c0 + c) =
                    make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                               pack_bf16x2(acc[6], acc[7]));
              }
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&c_empty[b]);
        }
        if (!named_bar_and(1, kEpiWarps * 32, cok)) break;  // the epilogue warps leave together
        continue;
      }
      const int nitem = ng++;
      // the row's scale (1 / (gs_w gs_a), times the routing weight for the down GEMM) and, for
      // the down GEMM, its (token, slot) entry, read while the MMAs run
      const bool live = r < te.rows;
      float cs = 0.f;
      int p = 0;
      if (live) {
        const float g = a.wgs[te.expert] * a.ags[te.row0 + r];
        if (kGateUp) {
          cs = 1.0f / g;
        } else {
          p = a.perm[te.row0 + r];
          cs = a.topk_w[p] / g;
        }
      }
      ok = mbar_wait(&acc_full, nitem & 1, &s_abort);
      if (MODE == 1 && ok && nitem >= kCombRing)  // the signal warp has taken this ring slot's rows
        ok = mbar_wait(&rows_taken[nitem % kCombRing], ((nitem / kCombRing) & 1) ^ 1, &s_abort);
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
        if (kFuseH && live) {  // into h's operand image: row r of routing tile `tile`
          const int f0 = w0 + 64 * half;  // four whole blocks = one K step of one 256-column chunk
          const int b0 = (f0 & 255) >> 4;
          uint8_t* blk = a.hq_out + ((size_t)tile * a.hC + (f0 >> 8)) * kAImgBlock;
          *(uint4*)(blk + img_code_byte(r, b0)) = make_uint4(hc[0], hc[1], hc[2], hc[3]);
          *(uint4*)(blk + img_code_byte(r, b0 + 2)) = make_uint4(hc[4], hc[5], hc[6], hc[7]);
          *(uint32_t*)(blk + kImgTile + 16 * r + b0) = hs4;
          if (f0 == 0) a.hg_out[te.row0 + r] = ghs;
        }
      } else {
        // output features fb .. fb + 127 of the routing-weighted row of (token t, slot p % k): to
        // the slot-ordered buffer (the combine items sum the k rows), or with one slot straight
        // to the output
        const int fb = w0 + 128 * half;
        const bool mine = live && fb < a.H;
        const uint64_t stream = policy_evict_first();
        uint16_t* dst = a.k == 1 ? a.out + (size_t)(p / a.k) * a.H + fb : a.comb + (size_t)p * a.H + fb;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          uint32_t Y[32];
          tmem_ld_32x16(taddr(tmem, q * 32, 128 * half + 32 * b), Y);
          tmem_ld_32x16(taddr(tmem, q * 32, 128 * half + 32 * b + 16), Y + 16);
          tmem_ld_wait();
          if (b == 3) {
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty);
          }
#pragma unroll
          for (int j = 0; j < 16; ++j)  // in place: word j reads words 2j, 2j+1 >= j
            Y[j] = pack_bf16x2(__uint_as_float(Y[2 * j]) * cs, __uint_as_float(Y[2 * j + 1]) * cs);
          if (mine) {
            if (a.k > 1)  // 32-byte stores of whole sectors
#pragma unroll
              for (int v = 0; v < 2; ++v) st_global_v8_hint(dst + 32 * b + 16 * v, Y + 8 * v, stream);
            else  // one slot: the row is the output (16-byte aligned)
#pragma unroll
              for (int v = 0; v < 4; ++v)
                *(uint4*)(dst + 32 * b + 8 * v) = make_uint4(Y[4 * v], Y[4 * v + 1], Y[4 * v + 2], Y[4 * v + 3]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&rows_stored[nitem % kCombRing]);  // release: the stores above
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

int fp4_row_block() { return kRows; }

template <int MODE>
static cudaError_t launch_fp4(const Fp4Args& a, int work, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(fp4_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    attr = true;
  }
  const int sms = tc_num_sms();
  return launch_pdl(fp4_kernel<MODE>, dim3(work < sms ? work : sms), dim3(Roles<MODE>::kThreads), kSmem, s, a);
}

cudaError_t launch_experts_fp4(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                               const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, uint16_t* out,
                               const float* act_gs, bool calibrate) {
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  // x and h go straight into their operand images (slot of routed row p: 128 toff[e] + p - off[e])
  ActImage xim, him;
  xim.img = (uint8_t*)(ws + L.xi);
  xim.chunks = nvfp4_chunks(H);
  xim.topk_idx = (const int32_t*)(ws + L.topk_idx);
  xim.perm = (const int32_t*)(ws + L.perm);
  xim.offsets = (const int32_t*)(ws + L.offsets);
  xim.toff = (const int32_t*)(ws + L.toff);
  him = xim;
  him.img = (uint8_t*)(ws + L.hi);
  him.chunks = nvfp4_chunks(I);
  float* cal = calibrate ? const_cast<float*>(act_gs) : nullptr;  // calibration writes the two scales
  if (cal && launch_act_scale((const uint16_t*)x, (size_t)T * H, cal, s) != cudaSuccess) return cudaGetLastError();
  launch_quant_rows(x, (const int32_t*)(ws + L.inv), k, T, H, nullptr, nullptr, (float*)(ws + L.xg), s, !cal, 0, act_gs,
                    &xim);

  Fp4Args a;
  memset(&a, 0, sizeof(a));
  a.perm = (const int32_t*)(ws + L.perm);
  a.topk_w = (const float*)(ws + L.topk_w);
  a.tiles = (const TileEntry*)(ws + L.tiles);
  a.h_out = (uint16_t*)(ws + L.h);
  a.hgs_static = act_gs && !calibrate ? act_gs + 1 : nullptr;
  a.hq_out = him.img;
  a.hC = him.chunks;
  a.hg_out = (float*)(ws + L.hg);
  a.comb = (uint16_t*)(ws + L.y);
  a.done = (int*)(ws + L.cnt);
  a.T = T;
  a.out = out;
  a.err = (int*)(ws + L.err);
  a.k = k;
  a.I = I;
  a.H = H;
  a.work_ctr = (int*)(ws + L.err) + 1;
  const int max_tiles = (int)(R / kRows + (R < (size_t)E ? R : (size_t)E) + 1);

  // gate/up: A = x's image (routing tiles), B = the fused [2I, H] weights' image (gate/up tile pairs)
  a.wimg = (const uint8_t*)packed + d.offset[MOE_T_GU_IMG];
  a.aimg = xim.img;
  a.C = xim.chunks;
  a.P = I / 128;
  a.wgs = gu.gs;
  a.ags = (const float*)(ws + L.xg);
  a.N = 2 * I;
  a.K = H;
  record_event(ev.start[0], s);
  cudaError_t err = a.hgs_static ? launch_fp4<2>(a, max_tiles * (I / 128), s) : launch_fp4<0>(a, max_tiles * (I / 128), s);
  record_event(ev.stop[0], s);
  if (err != cudaSuccess) return err;

  if (cal) return launch_act_scale((const uint16_t*)(ws + L.h), R * I, cal + 1, s);  // h's scale; no down GEMM
  // h -> NVFP4 per routed row (its own global scale; with static scales the gate/up epilogue has
  // already quantized it), then down: A = h's image, B = the [H, I] weights' image; the epilogue combines
  if (!act_gs)
    launch_quant_rows((const __nv_bfloat16*)(ws + L.h), nullptr, 1, (int)R, I, nullptr, nullptr, (float*)(ws + L.hg),
                      s, false, 0, nullptr, &him);
  a.wimg = (const uint8_t*)packed + d.offset[MOE_T_D_IMG];
  a.aimg = him.img;
  a.C = him.chunks;
  a.P = (H + 255) / 256;
  a.wgs = dn.gs;
  a.ags = (const float*)(ws + L.hg);
  a.N = H;
  a.K = I;
  a.work_ctr = (int*)(ws + L.err) + 2;
  record_event(ev.start[1], s);
  const int slices = k > 1 ? (T + kCombTokens - 1) / kCombTokens : 0;
  err = launch_fp4<1>(a, max_tiles * ((H + 255) / 256) + slices, s);
  record_event(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
