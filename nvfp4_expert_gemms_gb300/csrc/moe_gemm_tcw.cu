// NVFP4 W4A16 grouped expert GEMMs for routing tiles of up to 256 token rows (the prefill sizes).
//
// Same dataflow as the 128-token kernel (moe_gemm_tc.cu): weight image blocks --bulk copy-->
// shared memory --converter warps--> bf16 A operand in tensor memory; activation tiles --TMA-->
// shared memory; tcgen05.mma kind::f16 with A from tensor memory.  What differs is the shape of
// an item: one 128-row weight tile against up to 256 token rows, the MMA's N.  For the gate/up
// GEMM the tile holds 64 gate rows and the same features' up rows, interleaved by 16 in tensor
// memory (lanes 32q..32q+15 gate, 32q+16.. up), so the epilogue pairs them with one lane
// exchange; for the down GEMM it holds 128 output features.
//
// Why: an MMA's completion reaches the warps that reuse its A operand slot some 2000 SM cycles
// after it was issued, so the A ring must hold more MMA time than that or the tensor pipe waits
// at every chunk.  With N = 256 each 64-column A stage (one 128 x 128 chunk) is 8 MMAs of twice
// the work of the 128-token kernel's, and four stages fit next to the 256-column accumulator.
// The accumulator is single; the next item's first four chunks are converted before the previous
// item's epilogue, which releases the accumulator as soon as it has read it.
//
// Warp roles (640 threads): warps 0-15 convert (two groups of eight take alternate K chunks;
// warp w: TMEM lanes 32*(w%4).., K half (w/4)%2) and all sixteen run the epilogues; warp 16
// issues the weight image copies; warp 17 owns TMEM and issues the MMAs; warp 18 issues the
// activation tile copies.
#include "moe_formats.cuh"
#include "moe_combine.cuh"
#include "moe_tc.cuh"
#include "moe_w16conv.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kBN = 256;         // token rows per routing tile (the MMA's largest N)
constexpr int kKC = 128;         // K per chunk
constexpr int kConvWarps = 16;   // warps 0-15: converters + epilogue
constexpr int kProdWarp = 16;    // weight image copies
constexpr int kMmaWarp = 17;     // TMEM owner and MMA issuer
constexpr int kActWarp = 18;     // activation tile copies
constexpr int kRing = 8;         // work items handed from the weight producer to the other warps
constexpr int kThreads = 20 * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kACol = kBN;  // [0, 256) accumulator, then the A ring
constexpr int kStagesA = 4;      // 64 columns each: one 128-row x 128-K chunk in bf16
constexpr int kSB = 2;           // activation stages: 256 rows x 128 K bf16 = 64 KB each
constexpr int kBStage = kBN * 256;
constexpr int kStagesW = (220 * 1024 - 1024 - kSB * kBStage) / kW16Block;
constexpr size_t kSmem = 1024 + (size_t)kStagesW * kW16Block + (size_t)kSB * kBStage;
static_assert(kACol + kStagesA * 64 <= kTmemCols, "accumulator and A ring fit tensor memory");
static_assert(kStagesW >= 4, "enough weight stages in flight");

struct TcwArgs {
  CUtensorMap bmap;      // activation rows [R, K] as [K/64 atoms][R][64], boxes of 256 rows x 2 atoms
  const uint8_t* wimg;   // weight image [E, K/128, N/128, kW16Block]
  const float* wgs;      // global scales [E]
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;       // gate/up: h bf16 [R, I], permuted row order
  uint16_t* y_out;       // down: routing-weighted rows bf16 [R, H], permuted order
  CombineTail ct;        // MODE 1: the combine that follows the GEMM items
  int* err;
  int* work_ctr;         // items handed out past each CTA's first (zeroed by routing)
  int k, N, K, I, H;
};

// MODE 0: gate/up GEMM + SiLU(gate)*up -> h.  MODE 1: down GEMM x routing weight, then the combine.
template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) tcw_expert_gemm_kernel(const __grid_constant__ TcwArgs a) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = (char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  char* sB = smem;                      // activation stages (1024-aligned for the 128-byte swizzle)
  char* sW = smem + kSB * kBStage;      // weight image blocks
  __shared__ uint64_t w_full[kStagesW], w_empty[kStagesW], a_full[kStagesA], a_empty[kStagesA], b_full[kSB],
      b_empty[kSB], acc_full, acc_empty, drain;
  __shared__ uint64_t work_full[kRing], work_empty[kRing];
  __shared__ int s_work[kRing];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ float s_cw[2][kBN];  // down epilogue: routing weight x 2^10 / global scale of each column

  // gate/up: the tile table may come from the launch right before this one; down: it was final
  // before the gate/up GEMM passed its own pdl_wait(), so only the activations need the wait
  if (MODE == 0) pdl_wait();
  const int ntiles = load_tile(a.tiles).expert;  // header entry holds the tile count
  const int ncb = a.N / 128;                     // 128-row weight tiles per matrix
  const int nwork = ntiles * ncb;
  if ((int)blockIdx.x >= nwork) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nK = a.K / kKC;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStagesW; ++i) {
      mbar_init(&w_full[i], 1);
      mbar_init(&w_empty[i], kConvWarps / 2);
    }
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(&a_full[i], kConvWarps / 2);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < kSB; ++i) {
      mbar_init(&b_full[i], 1);
      mbar_init(&b_empty[i], 1);
    }
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&work_full[i], 1);
      mbar_init(&work_empty[i], 1 + 1 + kConvWarps);  // activation warp, MMA warp, converters
    }
    mbar_init(&acc_full, 1);
    mbar_init(&acc_empty, kConvWarps);
    mbar_init(&drain, 1);
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&s_tmem, kTmemCols);
    tmem_relinquish();
  }
  if (warp == kActWarp && lane == 0) prefetch_tmap(&a.bmap);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;
  if (MODE == 1 && warp != kProdWarp) pdl_wait();  // the weight producer needs nothing from the gate/up GEMM
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

  if (warp == kProdWarp) {
    // ---------------- weight image blocks (lane 0 issues; each CTA's first item static) ----------
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
        if (ok && wk >= 0) {
          const int e = load_tile(a.tiles + 1 + wk / ncb).expert, b = wk % ncb;
          for (int kc = 0; kc < nK && ok; ++kc, ++it) {
            const int sw = it % kStagesW;
            ok = mbar_wait(&w_empty[sw], ((it / kStagesW) & 1) ^ 1, &s_abort);
            if (ok) {
              mbar_arrive_expect_tx(&w_full[sw], kW16Block);
              ++armed_w[sw];
              bulk_load(sW + sw * kW16Block, a.wimg + (((size_t)e * nK + kc) * ncb + b) * kW16Block, kW16Block,
                        &w_full[sw]);
            }
          }
        }
      }
      wk = __shfl_sync(0xffffffffu, wk, 0);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok || wk < 0) break;
    }
    if (lane == 0 && s_abort) {  // let every issued copy land before shared memory goes away
      volatile int no_abort = 0;
      for (int i = 0; i < kStagesW; ++i)
        if (armed_w[i]) mbar_wait(&w_full[i], (armed_w[i] - 1) & 1, &no_abort);
    }
    __syncwarp();
  } else if (warp == kActWarp) {
    // ---------------- activation tiles: 256 rows x 128 K per copy ----------------
    int it = 0;
    int armed_b[kSB] = {0};
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      const int wk = next_item(nitem, ok);
      if (wk < 0) break;
      const TileEntry te = load_tile(a.tiles + 1 + wk / ncb);
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sb = it % kSB;
        if (lane == 0) {
          ok = mbar_wait(&b_empty[sb], ((it / kSB) & 1) ^ 1, &s_abort);
          if (ok) {
            mbar_arrive_expect_tx(&b_full[sb], kBStage);
            ++armed_b[sb];
            tma_load_3d(sB + sb * kBStage, &a.bmap, &b_full[sb], 0, te.row0, kc * 2);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0 && s_abort) {
      volatile int no_abort = 0;
      for (int i = 0; i < kSB; ++i)
        if (armed_b[i]) mbar_wait(&b_full[i], (armed_b[i] - 1) & 1, &no_abort);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (the whole warp waits, lane 0 issues) ----------------
    int it = 0;
    bool ok = true;
    for (int nitem = 0; ok; ++nitem) {
      const int wk = next_item(nitem, ok);
      if (wk < 0) break;
      const TileEntry te = load_tile(a.tiles + 1 + wk / ncb);
      const int nmma = ((te.rows + 15) & ~15) < kBN ? ((te.rows + 15) & ~15) : kBN;
      const uint32_t idesc = idesc_bf16_f32(128, nmma);
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sa = it % kStagesA, sb = it % kSB;
        ok = mbar_wait(&a_full[sa], (it / kStagesA) & 1, &s_abort) &&
             mbar_wait(&b_full[sb], (it / kSB) & 1, &s_abort) &&
             (kc != 0 || mbar_wait(&acc_empty, (nitem & 1) ^ 1, &s_abort));
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        fence_after_sync();
        if (lane == 0) {
          const uint32_t b0 = smem_u32(sB + sb * kBStage);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t bdsc = sdesc_k_sw128(b0 + (ks >> 2) * kBN * 128 + (ks & 3) * 32);
            mma_f16_ts(tmem, tmem + kACol + sa * 64 + ks * 8, bdsc, idesc, (kc | ks) != 0);
          }
          mma_commit(&a_empty[sa]);
          mma_commit(&b_empty[sb]);
        }
        __syncwarp();
      }
      if (ok && lane == 0) mma_commit(&acc_full);
      __syncwarp();
    }
    if (lane == 0) mma_commit(&drain);  // completes once every MMA issued by this thread has finished
    __syncwarp();
  } else if (warp < kConvWarps) {
    // ---------------- converters (two groups of 8 warps, alternate chunks) and epilogues ----------
    const int grp = warp >> 3, kh = (warp >> 2) & 1, q = warp & 3, part = warp >> 2;
    // the tile row this thread converts into TMEM lane 32 q + lane (gate/up: lanes 32q..32q+15
    // take gate rows 16q.., lanes 32q+16.. the up rows of the same features)
    const int r = MODE == 0 ? (lane < 16 ? 16 * q + lane : 48 + 16 * q + lane) : 32 * q + lane;
    int it = 0;
    bool ok = true;
    auto convert = [&]() -> bool {  // chunk `it` into the A ring
      const int sw = it % kStagesW, sa = it % kStagesA;
      if (!__all_sync(0xffffffffu, mbar_wait(&w_full[sw], (it / kStagesW) & 1, &s_abort))) return false;
      const char* blk = sW + sw * kW16Block;
      uint32_t v[32];
      conv_nvfp4(blk, r, kh, *(const uint32_t*)(blk + kW16Codes + r * 8 + kh * 4), v);
      reg_fence(v);
      __syncwarp();
      if (lane == 0) mbar_arrive(&w_empty[sw]);
      if (!__all_sync(0xffffffffu, mbar_wait(&a_empty[sa], ((it / kStagesA) & 1) ^ 1, &s_abort))) return false;
      fence_after_sync();
      tmem_st_32x32(taddr(tmem, q * 32, kACol + sa * 64 + kh * 32), v);
      tmem_st_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[sa]);
      return true;
    };
    // epilogue of item n: this warp's accumulator columns part*16 + 64 i, i = 0..3, read in two
    // halves (registers) and turned into packed bf16 results; the accumulator is released once
    // the second half is read, and the stores follow
    auto epilogue = [&](int n, const TileEntry& te, int nb, float inv_gs) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full, n & 1, &s_abort))) return false;
      fence_after_sync();
      const int cend = te.rows < kBN ? te.rows : kBN;  // warp-uniform
      const bool gl = lane < 16;
      uint32_t P[4][8];  // bf16 pairs: gate/up 8 results per group (4 words), down 16 (8 words)
      const int ngr = cend > part * 16 ? (cend - part * 16 + 63) / 64 : 0;  // this warp's groups
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {  // one group at a time: load, (last one: release), compute
        const int c0 = part * 16 + 64 * gi;
        uint32_t X[16];
        if (gi < ngr) {
          tmem_ld_32x16(taddr(tmem, q * 32, c0), X);
          tmem_ld_wait();
        }
        if (gi == (ngr > 0 ? ngr - 1 : 0)) {
          fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty);
        }
        if (gi >= ngr) continue;
        if (MODE == 0) {
          // lanes 0-15 hold gate values of feature nb + 16q + lane, lanes 16-31 the same
          // features' up values; the low half computes columns c0..c0+7, the high half c0+8..
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            float hv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t recv = __shfl_xor_sync(0xffffffffu, gl ? X[8 + j + u] : X[j + u], 16);
              const float gv = __uint_as_float(gl ? X[j + u] : recv) * inv_gs;
              const float uv = __uint_as_float(gl ? recv : X[8 + j + u]) * inv_gs;
              hv[u] = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            }
            P[gi][j >> 1] = pack_bf16x2(hv[0], hv[1]);
          }
        } else {
          const float* cw = s_cw[n & 1];
#pragma unroll
          for (int j = 0; j < 16; j += 2)
            P[gi][j >> 1] = pack_bf16x2(cw[c0 + j] * __uint_as_float(X[j]), cw[c0 + j + 1] * __uint_as_float(X[j + 1]));
        }
      }
#pragma unroll
      for (int gi = 0; gi < 4; ++gi) {
        const int c0 = part * 16 + 64 * gi;
        if (c0 >= cend) continue;
        if (MODE == 0) {
          const int n_out = nb + 16 * q + (lane & 15);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int col = c0 + (gl ? 0 : 8) + j;
            if (col < te.rows) a.h_out[(size_t)(te.row0 + col) * a.I + n_out] = (uint16_t)(P[gi][j >> 1] >> (16 * (j & 1)));
          }
        } else {
          const int c = nb + 32 * q + lane;
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int col = c0 + j;
            if (col < te.rows) a.y_out[(size_t)(te.row0 + col) * a.H + c] = (uint16_t)(P[gi][j >> 1] >> (16 * (j & 1)));
          }
        }
      }
      return true;
    };
    bool have_prev = false;
    TileEntry te_p;
    int nb_p = 0;
    float igs_p = 1.f;
    for (int nitem = 0;; ++nitem) {
      const int wk = next_item(nitem, ok);
      // the converter warps leave together (they meet in a named barrier every item)
      const bool live = named_bar_and(1, kConvWarps * 32, ok && wk >= 0);
      TileEntry te;
      int nb = 0, d = 0;
      float igs = 1.f;
      if (live) {
        te = load_tile(a.tiles + 1 + wk / ncb);
        nb = (wk % ncb) * (MODE == 0 ? 64 : 128);
        igs = 0x1p10f / a.wgs[te.expert];  // conv_nvfp4 leaves the weights times 2^-10
        if (MODE == 1 && threadIdx.x < kBN) {  // column table of this item's down epilogue
          const int col = threadIdx.x;
          s_cw[nitem & 1][col] = col < te.rows ? a.topk_w[a.perm[te.row0 + col]] * igs : 0.f;
        }
        // the item's first chunks go into the A ring before the previous item's epilogue
        d = nK < kStagesA ? nK : kStagesA;
        for (int kc = 0; kc < d && ok; ++kc, ++it)
          if ((it & 1) == grp) ok = convert();
      }
      if (have_prev && ok) ok = epilogue(nitem - 1, te_p, nb_p, igs_p);
      if (!live) break;  // (a warp whose wait failed skips its work but still meets the barrier)
      for (int kc = d; kc < nK && ok; ++kc, ++it)
        if ((it & 1) == grp) ok = convert();
      te_p = te;
      nb_p = nb;
      igs_p = igs;
      have_prev = true;
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

template <int MODE>
cudaError_t launch_tcw(const TcwArgs& args, int items, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(tcw_expert_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    attr = true;
  }
  const int sms = tc_num_sms();
  return launch_pdl(tcw_expert_gemm_kernel<MODE>, dim3(items < sms ? items : sms), dim3(kThreads), kSmem, s, args);
}

}  // namespace

int tcw_row_block() { return kBN; }

cudaError_t launch_experts_tcw(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                               const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, uint16_t* out) {
  if (d.fmt != MOE_FMT_NVFP4_W4A16 || !d.size[MOE_T_GU_IMG] || !d.size[MOE_T_D_IMG]) return cudaErrorInvalidValue;
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  TcwArgs a;
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
  const int gx = (int)(R / kBN + (R < (size_t)E ? R : (size_t)E) + 1);  // routing tiles, at most

  // gate/up: activations = x rows in expert-permuted order (a copy), weights = the [2I, H] image
  __nv_bfloat16* xp = (__nv_bfloat16*)(ws + L.xp);
  if (launch_gather_rows(x, a.perm, k, (int)R, H, xp, s) != cudaSuccess || !tc_act_map(&a.bmap, xp, R, H, kBN))
    return cudaErrorInvalidValue;
  a.wimg = (const uint8_t*)(packed + d.offset[MOE_T_GU_IMG]);
  a.wgs = gu.gs;
  a.N = 2 * I;
  a.K = H;
  a.work_ctr = (int*)(ws + L.err) + 1;
  record_event(ev.start[0], s);
  cudaError_t err = launch_tcw<0>(a, gx * (I / 64), s);
  record_event(ev.stop[0], s);
  if (err != cudaSuccess) return err;

  // down: activations = h rows (already in permuted order), weights = the [H, I] image
  if (!tc_act_map(&a.bmap, ws + L.h, R, I, kBN)) return cudaErrorInvalidValue;
  a.wimg = (const uint8_t*)(packed + d.offset[MOE_T_D_IMG]);
  a.wgs = dn.gs;
  a.N = H;
  a.K = I;
  a.work_ctr = (int*)(ws + L.err) + 2;
  record_event(ev.start[1], s);
  err = launch_tcw<1>(a, gx * (H / 128), s);
  record_event(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
