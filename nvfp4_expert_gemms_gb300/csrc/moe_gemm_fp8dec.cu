// FP8 W8A16 grouped GEMMs for decode-sized tiles (16 token rows per tile) on tcgen05 kind::f8f6f4.
//
// At decode the layer streams weights: each routed expert sees one or two tokens, so the kernel's
// job is to move 4.7 MB of E4M3 codes per expert through the tensor cores at HBM speed.  Here the
// packed weights (clef-omni-fp8, "What was quantized": E4M3 codes, one fp32 scale per 128x128
// tile) go from HBM to shared memory by TMA and straight into the MMA as the B operand -- there is
// no dequantization pass at all.  The activations become the A operand instead:
//
//   v = x * scale_inv(tile) * u_row          (u_row: a power of two putting max|v| <= 448)
//   v = hi + lo,  hi = E4M3(v),  lo = E4M3(v - hi)
//
// A bf16 value has 8 significant bits; hi keeps the top 4 and the rounding residual v - hi has at
// most 4 more, so hi + lo equals v exactly unless lo falls below the E4M3 subnormal step (elements
// under ~1/1800 of the row maximum, whose products are then off by at most 2^-4 of themselves).
// The hi and lo rows of each token are two N columns of one MMA (columns j and 16 + j), and the
// epilogue adds them and divides by u_row.  The tile scale is folded in per 128-K chunk because
// it changes along K; the fp32 product x * scale is rounded once, to about bf16 precision, by the
// split (the same rounding a bf16 copy of the dequantized weights would carry).
//
//   D[weight row, act row] += A[weight row, k] * B[act row, k]   (M = 128 weight rows per
//                            sub-tile, N = 32 activation rows, K = 32 per instruction, fp32)
//
// Warps (448 threads): 0-3 build the B chunk (split activations), 4-11 run the epilogue (warp w:
// sub-tile (w-4)/4, TMEM lanes 32*(w%4).., one thread per weight row), 12 issues the weight TMA,
// 13 owns TMEM and issues the MMAs.  The builders read their 32 bytes of activations per chunk
// straight from global memory (two chunks ahead): staging the 16 rows through TMA gather4 took
// the producer thread longer per chunk than the weight tiles take to stream.  Persistent CTAs walk (row tile, column block) work items; two TMEM
// accumulator buffers let the epilogue of one item overlap the MMAs of the next.
#include <cudaTypedefs.h>

#include "moe_dec.cuh"
#include "moe_formats.cuh"
#include "moe_combine.cuh"
#include "moe_tc.cuh"

namespace moe {

namespace {

using namespace tc;
using namespace dec;

constexpr int kKC = 128;         // K per chunk = one FP8 scale block
constexpr int kStagesW = 5;      // weight chunks in flight
constexpr int kStagesA = 4;      // split-activation chunks
constexpr int kPrepWarps = 4, kEpiWarp0 = 4, kEpiWarps = 8, kProdWarp = 12, kMmaWarp = 13;
constexpr int kThreads = 14 * 32;
constexpr int kWSub = 128 * 128;       // one 128x128 E4M3 tile (128-byte swizzle)
constexpr int kASub = 32 * 128;        // split-activation tile: 32 rows (hi, lo) x 128 K of E4M3
constexpr uint32_t kTmemCols = 128;    // two accumulator buffers x two sub-tiles x 32 columns
constexpr size_t kSmem = 1024 + (size_t)kStagesW * 2 * kWSub + (size_t)kStagesA * 2 * kASub;

struct Fp8Args {
  CUtensorMap wmap;    // E4M3 codes [E*N, K]
  const uint16_t* act;     // activations (bf16): x [T, K] (rows by token) or h [R, K] (permuted rows)
  const float* scale_inv;  // [E, N/128, K/128]
  const float* rowmax;     // max |activation| per source row (x: per token, h: per permuted row)
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;         // MODE 0 output [R, I] bf16
  unsigned* h_rowmax;      // MODE 0: running max |h| per permuted row (fp32 bits)
  uint16_t* y_out;         // MODE 1 output: routing-weighted rows [R, H] bf16, permuted order
  CombineTail ct;        // MODE 1: the combine that follows the GEMM items
  int* err;
  int k, N, K, I, H;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) fp8dec_kernel(const __grid_constant__ Fp8Args a) {
  extern __shared__ __align__(1024) char smem_raw[];
  char* smem = (char*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  char* sW = smem;
  char* sA = sW + kStagesW * 2 * kWSub;
  __shared__ uint64_t w_full[kStagesW], w_empty[kStagesW], a_full[kStagesA], a_empty[kStagesA], acc_full[2],
      acc_empty[2], drain;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  // The gate/up GEMM follows the routing launch that writes the tile table; the down GEMM
  // follows the gate/up GEMM, whose own pdl_wait() came after routing had finished.
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
    for (int i = 0; i < kStagesA; ++i) {
      mbar_init(&a_full[i], kPrepWarps);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], kEpiWarps);
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
    prefetch_tmap(&a.wmap);
  }
  fence_proxy_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = s_tmem;
  // Down GEMM: the weight producer starts streaming at once (packed weights and the tile table
  // only); every other role waits for the gate/up GEMM's h and row maxima.
  if (MODE == 1 && warp != kProdWarp) pdl_wait();
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
  auto scale_at = [&](const TileEntry& te, int nb, int kc) {
    return a.scale_inv[((size_t)te.expert * (a.N / 128) + nb / 128) * (a.K / 128) + kc];
  };
  // The item's largest tile scale over both sub-tiles and all K chunks (one warp, no block sync),
  // and the power-of-two normalizer of tile row j; builders and epilogue compute them alike.
  auto item_smax = [&](const TileEntry& te, int nb0, int nb1, int nsub) {
    float m = 0.f;
    for (int i = lane; i < nsub * nK; i += 32) m = fmaxf(m, scale_at(te, i < nK ? nb0 : nb1, i % nK));
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    return m;
  };
  auto row_norm = [&](const TileEntry& te, int j, float smax) {
    if (j >= te.rows) return 1.f;
    const int src = MODE == 0 ? a.perm[te.row0 + j] / a.k : te.row0 + j;
    return pow2_norm(__ldcg(a.rowmax + src), smax);
  };

  if (warp == kProdWarp) {
    // ---------------- TMA producer (weights only; whole warp walks the loop) ----------------
    int it = 0;
    bool ok = true;
    int armed[kStagesW] = {0};
    for (int wk = blockIdx.x; wk < nwork && ok; wk += gridDim.x) {
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sw = it % kStagesW;
        if (lane == 0) {
          ok = mbar_wait(&w_empty[sw], ((it / kStagesW) & 1) ^ 1, &s_abort);
          if (ok) {
            mbar_arrive_expect_tx(&w_full[sw], nsub * kWSub);
            ++armed[sw];
            tma_load_2d(sW + sw * 2 * kWSub, &a.wmap, &w_full[sw], kc * kKC, te.expert * a.N + nb0);
            if (nsub == 2) tma_load_2d(sW + sw * 2 * kWSub + kWSub, &a.wmap, &w_full[sw], kc * kKC, te.expert * a.N + nb1);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    if (lane == 0 && s_abort) {  // let every issued copy land before shared memory goes away
      volatile int no_abort = 0;
      for (int i = 0; i < kStagesW; ++i)
        if (armed[i]) mbar_wait(&w_full[i], (armed[i] - 1) & 1, &no_abort);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer (whole warp waits, lane 0 issues) ----------------
    const uint32_t idesc = idesc_e4m3_f32(128, 32);
    int it = 0, nitem = 0;
    bool ok = true;
    for (int wk = blockIdx.x; wk < nwork && ok; wk += gridDim.x, ++nitem) {
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      const int ab = nitem & 1;
      ok = mbar_wait(&acc_empty[ab], ((nitem >> 1) & 1) ^ 1, &s_abort);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      fence_after_sync();
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sw = it % kStagesW, sa = it % kStagesA;
        ok = mbar_wait(&w_full[sw], (it / kStagesW) & 1, &s_abort) &&
             mbar_wait(&a_full[sa], (it / kStagesA) & 1, &s_abort);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        fence_after_sync();
        if (lane == 0) {
          for (int g = 0; g < nsub; ++g) {
            const uint32_t wa = smem_u32(sW + sw * 2 * kWSub + g * kWSub), aa = smem_u32(sA + (sa * 2 + g) * kASub);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_f8_ss(tmem + ab * 64 + g * 32, sdesc_k_sw128(wa + ks * 32), sdesc_k_sw128(aa + ks * 32), idesc,
                        (kc | ks) != 0);
          }
          mma_commit(&w_empty[sw]);
          mma_commit(&a_empty[sa]);
        }
        __syncwarp();
      }
      if (ok && lane == 0) mma_commit(&acc_full[ab]);
      __syncwarp();
    }
    if (lane == 0) mma_commit(&drain);
    __syncwarp();
  } else if (warp < kPrepWarps) {
    // ---------------- A builders: split activations into E4M3 hi/lo rows ----------------
    const int t = threadIdx.x, j = t >> 3, q = t & 7;  // row j, 16-element group q of the chunk
    int it = 0, nitem = 0;
    bool ok = true;
    // Per-item setup (tile entry, then the row map / row maxima and tile scales that depend on it,
    // then the reductions) for the next item is spread over the current item's chunks -- the
    // tile entry after chunk 0, its dependent loads after chunk 1, the reductions after the last
    // chunk -- so item boundaries cost the builders no load latency.
    struct Setup {
      TileEntry te;
      int nb0, nb1, nsub;
      float u, sc0, sc1;
      const uint16_t* xrow;
    };
    auto setup = [&](int wk, Setup& st) {
      item(wk, st.te, st.nb0, st.nb1, st.nsub);
      st.u = row_norm(st.te, j, item_smax(st.te, st.nb0, st.nb1, st.nsub));
      st.sc0 = scale_at(st.te, st.nb0, 0);
      st.sc1 = st.nsub == 2 ? scale_at(st.te, st.nb1, 0) : 0.f;
      st.xrow = nullptr;
      if (j < st.te.rows)
        st.xrow = a.act + (size_t)(MODE == 0 ? a.perm[st.te.row0 + j] / a.k : st.te.row0 + j) * a.K + q * 16;
    };
    Setup cur;
    if ((int)blockIdx.x < nwork) setup(blockIdx.x, cur);
    bool pref = false;  // n0*, n1* already hold chunks 0 and 1 of the item (loaded during the previous one)
    uint4 n0a, n0b, n1a, n1b;
    for (int wk = blockIdx.x; wk < nwork && ok; wk += gridDim.x, ++nitem) {
      const TileEntry te = cur.te;
      const int nb0 = cur.nb0, nb1 = cur.nb1, nsub = cur.nsub;
      const bool real = j < te.rows;
      const float u = cur.u;
      const uint16_t* xrow = cur.xrow;
      const int wk_next = wk + gridDim.x;
      Setup nxt;
      float nx_smax = 0.f, nx_rmax = 0.f;
      int nx_src = 0;
      // 16 bf16 of row j at K = 128 kc + 16q .. +15, loaded two chunks ahead of their use; the
      // last two chunks of an item load the next item's first two once its row is known
      auto load_from = [&](const uint16_t* row, int kc, uint4& v0, uint4& v1) {
        if (row != nullptr && kc < nK) {
          v0 = __ldcg((const uint4*)(row + kc * kKC));
          v1 = __ldcg((const uint4*)(row + kc * kKC + 8));
        } else {
          v0 = v1 = make_uint4(0u, 0u, 0u, 0u);
        }
      };
      if (!pref) {
        load_from(xrow, 0, n0a, n0b);
        load_from(xrow, 1, n1a, n1b);
      }
      bool next_x = false, next0 = false;
      float sc_next0 = cur.sc0, sc_next1 = cur.sc1;
      for (int kc = 0; kc < nK; ++kc, ++it) {
        const int sa = it % kStagesA;
        const float f0 = sc_next0 * u, f1 = sc_next1 * u;
        if (kc + 1 < nK) {
          sc_next0 = scale_at(te, nb0, kc + 1);
          if (nsub == 2) sc_next1 = scale_at(te, nb1, kc + 1);
        }
        const uint4 x0 = n0a, x1 = n0b;
        n0a = n1a;
        n0b = n1b;
        if (kc + 2 < nK) {
          load_from(xrow, kc + 2, n1a, n1b);
        } else if (next_x) {
          load_from(nxt.xrow, kc + 2 - nK, n1a, n1b);
          next0 |= kc + 2 == nK;
        } else {
          n1a = n1b = make_uint4(0u, 0u, 0u, 0u);
        }
        ok = __all_sync(0xffffffffu, mbar_wait(&a_empty[sa], ((it / kStagesA) & 1) ^ 1, &s_abort));
        if (!ok) break;
        const uint32_t xw[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        for (int g = 0; g < nsub; ++g) {
          const float f = g == 0 ? f0 : f1;
          uint32_t hiw[4], low[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            float v[4];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const uint32_t w = xw[p * 2 + h2];
              v[h2 * 2] = real ? __uint_as_float(w << 16) * f : 0.f;
              v[h2 * 2 + 1] = real ? __uint_as_float(w & 0xFFFF0000u) * f : 0.f;
            }
            const uint16_t h01 = e4m3x2(v[0], v[1]), h23 = e4m3x2(v[2], v[3]);
            const float2 d01 = e4m3x2_to_f2(h01), d23 = e4m3x2_to_f2(h23);
            const uint16_t l01 = e4m3x2(v[0] - d01.x, v[1] - d01.y), l23 = e4m3x2(v[2] - d23.x, v[3] - d23.y);
            hiw[p] = (uint32_t)h01 | ((uint32_t)h23 << 16);
            low[p] = (uint32_t)l01 | ((uint32_t)l23 << 16);
          }
          char* at = sA + (sa * 2 + g) * kASub;
          *(uint4*)(at + j * 128 + ((q ^ (j & 7)) * 16)) = make_uint4(hiw[0], hiw[1], hiw[2], hiw[3]);
          const int jl = kRows + j;
          *(uint4*)(at + jl * 128 + ((q ^ (jl & 7)) * 16)) = make_uint4(low[0], low[1], low[2], low[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_full[sa]);
        if (wk_next < nwork) {
          const int kB = nK > 2 ? 1 : 0, kB2 = kB + 1 < nK ? kB + 1 : nK - 1;
          if (kc == 0) item(wk_next, nxt.te, nxt.nb0, nxt.nb1, nxt.nsub);
          if (kc == kB) {
            for (int i = lane; i < nxt.nsub * nK; i += 32)
              nx_smax = fmaxf(nx_smax, scale_at(nxt.te, i < nK ? nxt.nb0 : nxt.nb1, i % nK));
            nxt.sc0 = scale_at(nxt.te, nxt.nb0, 0);
            nxt.sc1 = nxt.nsub == 2 ? scale_at(nxt.te, nxt.nb1, 0) : 0.f;
            if (j < nxt.te.rows) nx_src = MODE == 0 ? a.perm[nxt.te.row0 + j] / a.k : nxt.te.row0 + j;
          }
          if (kc == kB2) {
            if (j < nxt.te.rows) nx_rmax = __ldcg(a.rowmax + nx_src);
            nxt.xrow = j < nxt.te.rows ? a.act + (size_t)nx_src * a.K + q * 16 : nullptr;
            next_x = true;
          }
          if (kc == nK - 1) {
            for (int off = 16; off > 0; off >>= 1) nx_smax = fmaxf(nx_smax, __shfl_xor_sync(0xffffffffu, nx_smax, off));
            nxt.u = j < nxt.te.rows ? pow2_norm(nx_rmax, nx_smax) : 1.f;
          }
        }
      }
      cur = nxt;
      pref = next0;
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + kEpiWarps) {
    // ---------------- epilogue: thread = weight row, columns = activation rows ----------------
    const int g = (warp - kEpiWarp0) >> 2, q = warp & 3, r = q * 32 + lane;
    int nitem = 0;
    bool ok = true;
    for (int wk = blockIdx.x; wk < nwork && ok; wk += gridDim.x, ++nitem) {
      TileEntry te;
      int nb0, nb1, nsub;
      item(wk, te, nb0, nb1, nsub);
      const int ab = nitem & 1;
      // normalizers of the tile's rows (lane j < 16 computes row j's, then broadcast), loaded
      // before the accumulator is ready
      const float smax = item_smax(te, nb0, nb1, nsub);
      const float u_l = row_norm(te, lane & 15, smax);
      int p_l = 0;
      float w_l = 0.f;
      if (MODE == 1 && lane < te.rows && lane < kRows) {
        p_l = a.perm[te.row0 + lane];
        w_l = a.topk_w[p_l];
      }
      ok = mbar_wait(&acc_full[ab], (nitem >> 1) & 1, &s_abort);
      if (!ok) break;
      fence_after_sync();
      if (MODE == 0) {
        if (g == 0) {  // sub-tile 0 threads own gate row r and up row r of the column block
          uint32_t G[32], U[32];
          tmem_ld_32x16(taddr(tmem, q * 32, ab * 64), G);
          tmem_ld_32x16(taddr(tmem, q * 32, ab * 64 + 16), G + 16);
          tmem_ld_32x16(taddr(tmem, q * 32, ab * 64 + 32), U);
          tmem_ld_32x16(taddr(tmem, q * 32, ab * 64 + 48), U + 16);
          tmem_ld_wait();
          const int n = nb0 + r;
#pragma unroll
          for (int j = 0; j < kRows; ++j) {
            const float inv_u = 1.0f / __shfl_sync(0xffffffffu, u_l, j);  // exact: a power of two
            if (j < te.rows) {
              const float gv = (__uint_as_float(G[j]) + __uint_as_float(G[16 + j])) * inv_u;
              const float uv = (__uint_as_float(U[j]) + __uint_as_float(U[16 + j])) * inv_u;
              const __nv_bfloat16 hb = __float2bfloat16_rn(gv * __frcp_rn(1.0f + __expf(-gv)) * uv);
              a.h_out[(size_t)(te.row0 + j) * a.I + n] = __bfloat16_as_ushort(hb);
              float m = fabsf(__bfloat162float(hb));
              for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
              if (lane == 0) atomicMax(&a.h_rowmax[te.row0 + j], __float_as_uint(m));
            }
          }
        }
      } else if (g < nsub) {
        uint32_t Y[32];
        tmem_ld_32x16(taddr(tmem, q * 32, ab * 64 + g * 32), Y);
        tmem_ld_32x16(taddr(tmem, q * 32, ab * 64 + g * 32 + 16), Y + 16);
        tmem_ld_wait();
        const int c = (g == 0 ? nb0 : nb1) + r;
#pragma unroll
        for (int j = 0; j < kRows; ++j) {
          const float inv_u = 1.0f / __shfl_sync(0xffffffffu, u_l, j);
          const int p = __shfl_sync(0xffffffffu, p_l, j);
          const float w = __shfl_sync(0xffffffffu, w_l, j);
          if (j < te.rows) {
            const float y = (__uint_as_float(Y[j]) + __uint_as_float(Y[16 + j])) * inv_u * w;
            a.y_out[(size_t)(te.row0 + j) * a.H + c] = bf16_bits(y);
          }
        }
      }
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[ab]);
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

}  // namespace


int fp8dec_row_block() { return kRows; }

cudaError_t launch_experts_fp8dec(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T,
                                  int k, const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s,
                                  uint16_t* out) {
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  static bool attr = false;
  if (!attr) {
    cudaFuncSetAttribute(fp8dec_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    cudaFuncSetAttribute(fp8dec_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    attr = true;
  }
  Fp8Args a;
  memset(&a, 0, sizeof(a));
  a.perm = (const int32_t*)(ws + L.perm);
  a.topk_w = (const float*)(ws + L.topk_w);
  a.tiles = (const TileEntry*)(ws + L.tiles);
  a.h_out = (uint16_t*)(ws + L.h);
  a.h_rowmax = (unsigned*)(ws + L.hmax);
  a.y_out = (uint16_t*)(ws + L.y);
  combine_tail_args(a.ct, L, ws, T, k, H, out);
  a.err = (int*)(ws + L.err);
  a.k = k;
  a.I = I;
  a.H = H;
  const int sms = tc_num_sms();
  const int max_tiles = (int)(R / kRows + (R < (size_t)E ? R : (size_t)E) + 1);

  // x row maxima and the zeroed h row maxima come from the routing launch (RoutePrelude)

  if (!tc_make_map(&a.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, gu.a, H, (uint64_t)E * 2 * I, H, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.act = (const uint16_t*)x;
  a.scale_inv = (const float*)gu.b;
  a.rowmax = (const float*)(ws + L.xmax);
  a.N = 2 * I;
  a.K = H;
  int grid = max_tiles * (I / 128);
  record_event(ev.start[0], s);
  cudaError_t err = launch_pdl(fp8dec_kernel<0>, dim3(grid < sms ? grid : sms), dim3(kThreads), kSmem, s, a);
  if (err != cudaSuccess) return err;
  record_event(ev.stop[0], s);

  if (!tc_make_map(&a.wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, dn.a, I, (uint64_t)E * H, I, 128, 128,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  a.act = (const uint16_t*)(ws + L.h);
  a.scale_inv = (const float*)dn.b;
  a.rowmax = (const float*)(ws + L.hmax);
  a.N = H;
  a.K = I;
  grid = max_tiles * ((H + 255) / 256);
  record_event(ev.start[1], s);
  err = launch_pdl(fp8dec_kernel<1>, dim3(grid < sms ? grid : sms), dim3(kThreads), kSmem, s, a);
  record_event(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
