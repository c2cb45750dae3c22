// NVFP4 W4A4 grouped GEMMs on the native block-scaled FP4 tensor-core MMA
// (tcgen05.mma kind::mxf4nvf4, E2M1 operands, UE4M3 scale per 16 elements along K).
//
// Both operands stay in their packed NVFP4 form end to end (clef-flash-NVFP4-Hybrid, layer
// table: "16-element groups, FP8 group scales, one FP32 global scale"; weights: clef-omni-NVFP4,
// "How it was made"):
//   weights      E2M1 codes [N, K/2] + E4M3 block scales [N, K/16] + global scale gs_w (per matrix)
//   activations  E2M1 codes [rows, K/2] + E4M3 block scales [rows, K/16] + global scale gs_a (per row)
// The MMA forms sum_k (q_w * bs_w)(q_a * bs_a) exactly in fp32, and the epilogue divides by
// gs_w * gs_a.  Codes arrive by TMA tiles in the 128-byte swizzle: weights in 128-row tiles,
// activations in BN-row tiles of their expert-permuted rows (x is quantized straight into that
// order, one copy per routed token slot, so the gate/up GEMM needs no row gather).  The weight block
// scales arrive by TMA next to their codes; the activation block scales are read from global
// memory by the four scale warps (16 bytes per row and chunk, fetched one chunk ahead), which
// place both in tensor memory in the layout the MMA reads (per K = 64 step and 128 rows:
// 4 columns; lane l, column j = the four scales of row l + 32 j, repeated in every lane quarter).
//
//   D[weight row, act row] += A[weight row, k] * B[act row, k]     M = 128, N = BN <= 128, K = 64
//
// Warps (448 threads): 0-3 stage scale factors, 4-11 run the epilogue (thread = weight row),
// 12 issues TMA, 13 owns TMEM and issues the MMAs.  Persistent CTAs walk (row tile, column
// block) work items.
#include <cudaTypedefs.h>

#include "moe_formats.cuh"
#include "moe_tc.cuh"

namespace moe {

namespace {

using namespace tc;

constexpr int kKC = 256;                  // K per chunk: 128 bytes of codes per row
constexpr int kStagesX = 4, kStagesS = 4;
constexpr int kSfWarps = 4, kEpiWarp0 = 4, kEpiWarps = 8, kProdWarp = 12, kMmaWarp = 13;
constexpr int kThreads = 14 * 32;
constexpr int kWCodes = 128 * 128;        // 128 rows x 128 B (256 codes), 128-byte swizzle
constexpr int kWSf = 128 * 16;            // 128 rows x 16 scales
constexpr int kWStage = 2 * kWCodes + 2 * kWSf;
constexpr uint32_t kSfCol = 256;          // TMEM: [0, 2*BN) accumulators, then 4 x 48 scale-factor columns
constexpr uint32_t kSfStageCols = 48;     // sub-tile 0 A scales (16), sub-tile 1 (16), B scales (16)

// Shared memory: weight stages, activation stages, and (gate/up) the h tile staged for
// coalesced stores: BN token rows x 128 intermediate columns of bf16.
template <int MODE, int BN>
struct Fp4Cfg {
  static constexpr int kStagesW = MODE == 0 ? 3 : 4;
  static constexpr int kXBytes = BN * 128;                        // codes, 128-byte swizzle
  static constexpr int kXStage = (kXBytes + 1023) / 1024 * 1024;  // stages start 1024-aligned
  static constexpr int kHBytes = MODE == 0 ? BN * 256 : 0;
  static constexpr size_t kSmem = 1024 + (size_t)kStagesW * kWStage + (size_t)kStagesX * kXStage + kHBytes;
};

struct Fp4Args {
  CUtensorMap wcode, wsf;   // weight codes [E*N, K/2], scales [E*N, K/16]
  CUtensorMap xcode;        // activation codes [R, K/2] in permuted row order
  const uint8_t* asf;       // activation block scales [R, K/16]
  const float* wgs;         // weight global scales [E]
  const float* ags;         // activation global scales [R]
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;          // MODE 0 output [R, I] bf16
  uint16_t* y_out;          // MODE 1 output: routing-weighted rows [R, H] bf16, permuted order
  int* err;
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

// Scale tile [rows][16 bytes] -> 16 TMEM words for lane l: word (4*ks + j) = bytes 4ks..4ks+3 of
// row l + 32j (zero for rows >= nrows).
__device__ __forceinline__ void sf_words(const char* tile, int l, int nrows, uint32_t* v) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int row = l + 32 * j;
    const uint4 s = row < nrows ? *(const uint4*)(tile + row * 16) : make_uint4(0, 0, 0, 0);
    v[0 + j] = s.x;
    v[4 + j] = s.y;
    v[8 + j] = s.z;
    v[12 + j] = s.w;
  }
}

template <int MODE, int BN>
__global__ void __launch_bounds__(kThreads, 1) fp4_kernel(const __grid_constant__ Fp4Args a) {
  constexpr int kStagesW = Fp4Cfg<MODE, BN>::kStagesW;
  constexpr int kXStage = Fp4Cfg<MODE, BN>::kXStage;
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = (char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  char* sW = smem;
  char* sX = sW + kStagesW * kWStage;
  char* sH = sX + kStagesX * kXStage;
  __shared__ uint64_t w_full[kStagesW], w_empty[kStagesW], x_full[kStagesX], x_empty[kStagesX], s_full[kStagesS],
      s_empty[kStagesS], acc_full, acc_empty, drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  // per output column of the current item (double-buffered by item parity): the scale that
  // undoes both global scales (times the routing weight for the down GEMM) and the token row
  __shared__ __align__(16) float s_cs[2][BN];
  __shared__ __align__(16) int s_ct[2][BN];

  // gate/up: wait for the activation quantization (and, before it, routing); down: the tile table
  // was final before the gate/up GEMM passed its own pdl_wait(), so only the h codes need the wait
  if (MODE == 0) pdl_wait();
  const int ntiles = load_tile(a.tiles).expert;
  const int ncb = MODE == 0 ? a.I / 128 : (a.H + 255) / 256;
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
    prefetch_tmap(&a.wsf);
    prefetch_tmap(&a.xcode);
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;
  if (MODE == 1 && warp != kProdWarp) pdl_wait();  // the producer waits before its first h tile
  pdl_trigger();

  auto item = [&](int wk, TileEntry& te, int& nb0, int& nb1, int& nsub) {
    te = load_tile(a.tiles + 1 + wk / ncb);
    const int cb = wk % ncb;
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
    // ---------------- TMA producer (whole warp walks the loop, lane 0 issues) ----------------
    int it = 0;
    bool ok = true;
    int armed_w[kStagesW] = {0}, armed_x[kStagesX] = {0};
    for (int wk = blockIdx.x; wk < nwork && ok; wk += gridDim.x) {
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sw = it % kStagesW, sx = it % kStagesX;
        if (lane == 0) {
          ok = mbar_wait(&w_empty[sw], ((it / kStagesW) & 1) ^ 1, &s_abort);
          if (ok) {
            char* ws = sW + sw * kWStage;
            mbar_arrive_expect_tx(&w_full[sw], nsub * (kWCodes + kWSf));
            ++armed_w[sw];
            for (int g = 0; g < nsub; ++g) {
              const int row = te.expert * a.N + (g == 0 ? nb0 : nb1);
              tma_load_2d(ws + g * kWCodes, &a.wcode, &w_full[sw], kc * (kKC / 2), row);
              tma_load_2d(ws + 2 * kWCodes + g * kWSf, &a.wsf, &w_full[sw], kc * (kKC / 16), row);
            }
          }
          if (ok) {
            ok = mbar_wait(&x_empty[sx], ((it / kStagesX) & 1) ^ 1, &s_abort);
            if (MODE == 1 && it == 0) pdl_wait();
            if (ok) {
              mbar_arrive_expect_tx(&x_full[sx], Fp4Cfg<MODE, BN>::kXBytes);
              ++armed_x[sx];
              tma_load_2d(sX + sx * kXStage, &a.xcode, &x_full[sx], kc * (kKC / 2), te.row0);
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
    const uint32_t idesc = idesc_nvf4(128, BN);
    int it = 0, nitem = 0;
    bool ok = true;
    for (int wk = blockIdx.x; wk < nwork && ok; wk += gridDim.x, ++nitem) {
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
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
          const uint32_t xa = smem_u32(sX + sx * kXStage);
          for (int g = 0; g < nsub; ++g) {
            const uint32_t wa = smem_u32(sW + sw * kWStage + g * kWCodes);
            const uint32_t sfa = tmem + kSfCol + ss * kSfStageCols + g * 16, sfb = tmem + kSfCol + ss * kSfStageCols + 32;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_nvf4(tmem + g * BN, sdesc_k_sw128(wa + ks * 32), sdesc_k_sw128(xa + ks * 32), idesc, sfa + 4 * ks,
                       sfb + 4 * ks, (kc | ks) != 0);
          }
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
    for (int wk = blockIdx.x; wk < nwork && ok; wk += gridDim.x) {
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      // source rows of the activation scales this lane places: tile rows l + 32 j
      const uint8_t* src[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int row = l + 32 * j;
        src[j] = nullptr;
        if (row < te.rows && row < BN) src[j] = a.asf + (size_t)(te.row0 + row) * (a.K / 16);
      }
      uint4 nxt[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) nxt[j] = src[j] ? *(const uint4*)(src[j]) : make_uint4(0, 0, 0, 0);
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sw = it % kStagesW, ss = it % kStagesS;
        uint4 cur[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          cur[j] = nxt[j];
          if (kc + 1 < nK) nxt[j] = src[j] ? *(const uint4*)(src[j] + (kc + 1) * 16) : make_uint4(0, 0, 0, 0);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&w_full[sw], (it / kStagesW) & 1, &s_abort) &&
                                         mbar_wait(&s_empty[ss], ((it / kStagesS) & 1) ^ 1, &s_abort));
        if (!ok) break;
        fence_after_sync();
        const uint32_t col = kSfCol + ss * kSfStageCols;
        uint32_t v[16];
        for (int g = 0; g < nsub; ++g) {
          sf_words(sW + sw * kWStage + 2 * kWCodes + g * kWSf, l, 128, v);
          tmem_st_32x16(taddr(tmem, q * 32, col + g * 16), v);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[0 + j] = cur[j].x;
          v[4 + j] = cur[j].y;
          v[8 + j] = cur[j].z;
          v[12 + j] = cur[j].w;
        }
        tmem_st_32x16(taddr(tmem, q * 32, col + 32), v);
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_full[ss]);
      }
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ---------------- epilogue: thread = weight row, columns = activation rows ----------------
    const int ge = (warp - kEpiWarp0) >> 2, q = warp & 3, r = q * 32 + lane;
    const int et = threadIdx.x - kEpiWarp0 * 32;
    int nitem = 0;
    bool ok = true;
    for (int wk = blockIdx.x; wk < nwork; wk += gridDim.x, ++nitem) {
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      const int buf = nitem & 1;
      // column table of this item, filled while its MMAs run
      if (et < BN) {
        float cs = 0.f;
        int ct = 0;
        if (et < te.rows) {
          const float gw = a.wgs[te.expert];
          if (MODE == 0) {
            cs = 1.0f / (gw * a.ags[te.row0 + et]);
          } else {
            const int p = a.perm[te.row0 + et];
            cs = a.topk_w[p] / (gw * a.ags[te.row0 + et]);
            ct = p / a.k;
          }
        }
        s_cs[buf][et] = cs;
        s_ct[buf][et] = ct;
      }
      ok = mbar_wait(&acc_full, nitem & 1, &s_abort);
      // every epilogue thread takes the same branch: the table is complete and no one has aborted
      ok = named_bar_and(1, kEpiWarps * 32, ok);
      if (!ok) break;
      fence_after_sync();
      const float* cs = s_cs[buf];
      if (MODE == 0) {
        // both warp groups own the same weight rows (gate in sub-tile 0, up in sub-tile 1) and
        // split the token columns; h goes to the staged tile [token][weight row] first
        const int c_beg = BN <= 16 ? (ge == 0 ? 0 : BN) : ge * (BN / 2);
        const int c_end = BN <= 16 ? (ge == 0 ? BN : BN) : c_beg + BN / 2;
        uint16_t* sh = (uint16_t*)sH;
        for (int c0 = c_beg; c0 < c_end; c0 += 16) {
          uint32_t G[16], U[16];
          tmem_ld_32x16(taddr(tmem, q * 32, c0), G);
          tmem_ld_32x16(taddr(tmem, q * 32, BN + c0), U);
          float sc[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) *(float4*)(sc + 4 * i) = *(const float4*)(cs + c0 + 4 * i);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float gv = __uint_as_float(G[j]) * sc[j], uv = __uint_as_float(U[j]) * sc[j];
            const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
            sh[(c0 + j) * 128 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(hv));
          }
        }
        // the tile's valid token rows leave as 256-byte row segments in 16-byte stores
        named_bar_sync(2, kEpiWarps * 32);
        const int nrows = te.rows < BN ? te.rows : BN;
        for (int idx = et; idx < nrows * 16; idx += kEpiWarps * 32) {
          const int row = idx >> 4, piece = idx & 15;
          *(uint4*)(a.h_out + (size_t)(te.row0 + row) * a.I + nb0 + piece * 8) =
              *(const uint4*)(sH + row * 256 + piece * 16);
        }
      } else if (ge < nsub) {
        const int c = (ge == 0 ? nb0 : nb1) + r;
        const int* ct = s_ct[buf];
        for (int c0 = 0; c0 < BN; c0 += 16) {
          uint32_t Y[16];
          tmem_ld_32x16(taddr(tmem, q * 32, ge * BN + c0), Y);
          float sc[16];
          int tok[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            *(float4*)(sc + 4 * i) = *(const float4*)(cs + c0 + 4 * i);
            *(int4*)(tok + 4 * i) = *(const int4*)(ct + c0 + 4 * i);
          }
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j)
            if (c0 + j < te.rows)
              a.y_out[(size_t)(te.row0 + c0 + j) * a.H + c] = bf16_bits(sc[j] * __uint_as_float(Y[j]));
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty);
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

template <int MODE, int BN>
static cudaError_t launch_fp4_one(const Fp4Args& a, int work, cudaStream_t s) {
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(fp4_kernel<MODE, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)Fp4Cfg<MODE, BN>::kSmem);
    attr = true;
  }
  const int sms = tc_num_sms();
  return launch_pdl(fp4_kernel<MODE, BN>, dim3(work < sms ? work : sms), dim3(kThreads), Fp4Cfg<MODE, BN>::kSmem, s,
                    a);
}

template <int MODE>
static cudaError_t launch_fp4_bn(int bn, const Fp4Args& a, int work, cudaStream_t s) {
  switch (bn) {
    case 16: return launch_fp4_one<MODE, 16>(a, work, s);
    case 32: return launch_fp4_one<MODE, 32>(a, work, s);
    case 64: return launch_fp4_one<MODE, 64>(a, work, s);
    default: return launch_fp4_one<MODE, 128>(a, work, s);
  }
}

cudaError_t launch_experts_fp4(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                               int bn, const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s) {
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  uint8_t* xq = (uint8_t*)(ws + L.xq);
  uint8_t* xsf = (uint8_t*)(ws + L.xs);
  uint8_t* hq = (uint8_t*)(ws + L.hq);
  uint8_t* hsf = (uint8_t*)(ws + L.hs);
  launch_quant_rows(x, (const int32_t*)(ws + L.inv), k, T, H, xq, xsf, (float*)(ws + L.xg), s, true);

  Fp4Args a;
  memset(&a, 0, sizeof(a));
  a.perm = (const int32_t*)(ws + L.perm);
  a.topk_w = (const float*)(ws + L.topk_w);
  a.tiles = (const TileEntry*)(ws + L.tiles);
  a.h_out = (uint16_t*)(ws + L.h);
  a.y_out = (uint16_t*)(ws + L.y);
  a.err = (int*)(ws + L.err);
  a.k = k;
  a.I = I;
  a.H = H;
  const int max_tiles = (int)(R / bn + (R < (size_t)E ? R : (size_t)E) + 1);
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;

  // gate/up: A = fused [2I, H] NVFP4 weights, B = quantized x in permuted row order
  if (!tc_make_map(&a.wcode, u8, gu.a, H / 2, (uint64_t)E * 2 * I, H / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc_make_map(&a.wsf, u8, gu.b, H / 16, (uint64_t)E * 2 * I, H / 16, 16, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !tc_make_map(&a.xcode, u8, xq, H / 2, (uint64_t)R, H / 2, 128, bn, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.asf = xsf;
  a.wgs = gu.gs;
  a.ags = (const float*)(ws + L.xg);
  a.N = 2 * I;
  a.K = H;
  record_event(ev.start[0], s);
  cudaError_t err = launch_fp4_bn<0>(bn, a, max_tiles * (I / 128), s);
  record_event(ev.stop[0], s);
  if (err != cudaSuccess) return err;

  // h -> NVFP4 per permuted row (its own global scale), then down: A = [H, I] weights, B = h rows
  launch_quant_rows((const __nv_bfloat16*)(ws + L.h), nullptr, 1, (int)R, I, hq, hsf, (float*)(ws + L.hg), s);
  if (!tc_make_map(&a.wcode, u8, dn.a, I / 2, (uint64_t)E * H, I / 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tc_make_map(&a.wsf, u8, dn.b, I / 16, (uint64_t)E * H, I / 16, 16, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !tc_make_map(&a.xcode, u8, hq, I / 2, (uint64_t)R, I / 2, 128, bn, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.asf = hsf;
  a.wgs = dn.gs;
  a.ags = (const float*)(ws + L.hg);
  a.N = H;
  a.K = I;
  record_event(ev.start[1], s);
  err = launch_fp4_bn<1>(bn, a, max_tiles * ((H + 255) / 256), s);
  record_event(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
