// Routing: warp-level top-k with a renormalised softmax, per-expert histogram, exclusive
// scan, and a deterministic permutation of (token, slot) rows by (expert, token, slot).
//
// The pages leave the router unquantized (clef-omni-fp8, page header and "What was
// quantized") and run the experts as one grouped matmul per layer (clef-omni-fp8, "How this
// checkpoint runs"; clef-omni-int4, same section); grouping rows by expert is what a grouped
// matmul consumes.  Three launches, no atomics whose order reaches the output:
//   1. route_topk_kernel   one warp per token; per-block expert histogram in shared memory
//   2. route_scan_kernel   one block: expert totals, offsets, per-block bases, GEMM tile table
//   3. route_scatter_kernel rank of each row inside its block from per-warp ballot masks
// Up to kRouteTB tokens (decode) all three steps run in one block of one launch
// (route_small_kernel), which produces the same outputs.
#include "moe_internal.cuh"

namespace moe {

namespace {


struct Cand {
  float v;
  int i;
};

// Zero this forward pass's running maxima (grid-stride over all launched threads).
__device__ __forceinline__ void zero_prelude(const RoutePrelude& pre) {
  const size_t g = (size_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (size_t)gridDim.x * blockDim.x;
  for (size_t i = g; i < pre.n_u32; i += stride) pre.zero_u32[i] = 0u;
  for (size_t i = g; i < pre.n2_u32; i += stride) pre.zero2_u32[i] = 0u;
}

// max |x| of token t's activation row (one warp); all loads are issued before use.
__device__ __forceinline__ void row_absmax(const RoutePrelude& pre, int t, int lane) {
  float m = 0.f;
  const uint16_t* row = pre.x + (size_t)t * pre.H;
  for (int c0 = lane * 8; c0 < pre.H; c0 += 256 * 8) {
    uint4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = c0 + u * 256 < pre.H ? *(const uint4*)(row + c0 + u * 256) : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[i] << 16)), fabsf(__uint_as_float(w4[i] & 0xFFFF0000u))));
    }
  }
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  if (lane == 0) pre.xmax[t] = m;
}

// Top-k of token t (one warp): writes its k expert indices and renormalised softmax weights and
// returns, in lane j < k, the j-th selected expert.
__device__ __forceinline__ int route_token(const float* __restrict__ logits, int t, int E, int k, int lane,
                                           int32_t* __restrict__ topk_idx, float* __restrict__ topk_w) {
  float v[kMaxE / 32];
#pragma unroll
  for (int m = 0; m < kMaxE / 32; ++m) {
    const int e = lane + 32 * m;
    float x = e < E ? logits[(size_t)t * E + e] : -INFINITY;
    v[m] = isnan(x) ? -INFINITY : x;
  }
  // Order-preserving 32-bit keys (larger key = larger logit; -0 counts as +0, as a float compare
  // does).  Each round takes the largest key over the warp, then the lowest expert index among
  // the candidates holding it: two warp reductions instead of a five-step shuffle tournament.
  uint32_t key[kMaxE / 32];
#pragma unroll
  for (int m = 0; m < kMaxE / 32; ++m) {
    const uint32_t u = __float_as_uint(v[m] == 0.f ? 0.f : v[m]);
    key[m] = lane + 32 * m < E ? ((u & 0x80000000u) ? ~u : (u | 0x80000000u)) : 0u;  // 0: no candidate
  }
  float selv[kMaxTopK];
  int seli[kMaxTopK];
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int be = INT_MAX;
#pragma unroll
    for (int m = 0; m < kMaxE / 32; ++m)  // ascending m: the lane's lowest index wins its ties
      if (key[m] > bk) {
        bk = key[m];
        be = lane + 32 * m;
      }
    const uint32_t wk = __reduce_max_sync(0xffffffffu, bk);
    const int bi = (int)__reduce_min_sync(0xffffffffu, bk == wk ? (uint32_t)be : 0xFFFFFFFFu);
    if ((bi & 31) == lane) key[bi >> 5] = 0u;  // taken
    selv[j] = __uint_as_float((wk & 0x80000000u) ? (wk & 0x7FFFFFFFu) : ~wk);
    seli[j] = bi;
  }
  // renormalised softmax over the selected logits (descending: selv[0] is the max)
  float den = 0.f;
  for (int j = 0; j < k; ++j) den += expf(selv[j] - selv[0]);
  float mine = selv[0];
  int mi = seli[0];
  for (int j = 1; j < k; ++j)
    if (j == lane) {
      mine = selv[j];
      mi = seli[j];
    }
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = mi;
    topk_w[(size_t)t * k + lane] = expf(mine - selv[0]) / den;
  }
  return mi;
}

// Exclusive scans of rows and tiles per expert by one warp (lane l owns experts 8l .. 8l+7):
// off_s[e] = first permuted row of expert e, toff_s[e] = its first tile (both for e = 0..E), and
// the tile table's header entry.
__device__ __forceinline__ void expert_scan(const int* cnt, int E, int row_block, int max_tiles, int* off_s,
                                            int* toff_s, TileEntry* tiles, int lane) {
  constexpr int kPer = kMaxE / 32;
  int rows[kPer], ntl[kPer], ra = 0, ta = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane * kPer + i;
    rows[i] = e < E ? cnt[e] : 0;
    ntl[i] = (rows[i] + row_block - 1) / row_block;
    ra += rows[i];
    ta += ntl[i];
  }
  int ri = ra, ti = ta;  // inclusive warp scans of the per-lane sums
  for (int off = 1; off < 32; off <<= 1) {
    const int rv = __shfl_up_sync(0xffffffffu, ri, off), tv = __shfl_up_sync(0xffffffffu, ti, off);
    if (lane >= off) {
      ri += rv;
      ti += tv;
    }
  }
  int a = ri - ra, b = ti - ta;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    const int e = lane * kPer + i;
    if (e <= E) {
      off_s[e] = a;
      toff_s[e] = b;
    }
    a += rows[i];
    b += ntl[i];
  }
  if (lane == 31) {
    TileEntry h;
    h.expert = min(ti, max_tiles);
    h.row0 = ri;
    h.rows = row_block;
    h.pad = 0;
    tiles[0] = h;
    if (E == kMaxE) {  // off_s[E] and toff_s[E] lie past the last lane's experts
      off_s[E] = ri;
      toff_s[E] = ti;
    }
  }
}

__global__ void __launch_bounds__(1024) route_topk_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                         int32_t* __restrict__ topk_idx,
                                                         float* __restrict__ topk_w,
                                                         int32_t* __restrict__ blkcnt, int* err, RoutePrelude pre) {
  __shared__ int cnt[kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  pdl_wait();
  pdl_trigger();
  zero_prelude(pre);
  if (blockIdx.x == 0 && tid == 0) reset_status(err);  // each forward pass reports its own errors
  __syncthreads();
  const int t_end = min(T, (int)(blockIdx.x + 1) * kRouteTB);
  for (int t = blockIdx.x * kRouteTB + warp; t < t_end; t += 32) {  // 4 tokens per warp
    if (pre.x) row_absmax(pre, t, lane);
    const int mi = route_token(logits, t, E, k, lane, topk_idx, topk_w);
    if (lane < k) atomicAdd(&cnt[mi], 1);
  }
  __syncthreads();
  for (int e = tid; e < E; e += blockDim.x) blkcnt[(size_t)blockIdx.x * E + e] = cnt[e];
}

// One block of 1024 threads.  Thread e < E owns expert e.
__global__ void __launch_bounds__(1024) route_scan_kernel(const int32_t* __restrict__ blkcnt, int nb, int E,
                                                          int row_block, int max_tiles,
                                                          int32_t* __restrict__ offsets,
                                                          int32_t* __restrict__ toffsets,
                                                          int32_t* __restrict__ blkbase,
                                                          TileEntry* __restrict__ tiles, int* err) {
  __shared__ int tot[kMaxE], ntl[kMaxE], off_s[kMaxE + 1], toff_s[kMaxE + 1];
  __shared__ int psum[1024];  // [part][expert]: the blocks of each expert split into 1024 / E parts
  const int tid = threadIdx.x, e = tid;
  const int parts = 1024 / E, pe = tid % E, pp = tid / E;  // thread (part pp, expert pe)
  const int chunk = (nb + parts - 1) / parts, b0 = pp * chunk, b1 = min(nb, b0 + chunk);
  pdl_wait();
  pdl_trigger();
  if (pp < parts) {
    int s = 0;
#pragma unroll 8
    for (int b = b0; b < b1; ++b) s += blkcnt[(size_t)b * E + pe];
    psum[pp * E + pe] = s;
  }
  __syncthreads();
  if (e < E) {
    int s = 0;
    for (int p = 0; p < parts; ++p) s += psum[p * E + e];
    tot[e] = s;
    ntl[e] = (s + row_block - 1) / row_block;
  }
  __syncthreads();
  if (e < 32) expert_scan(tot, E, row_block, max_tiles, off_s, toff_s, tiles, e);
  __syncthreads();
  if (e <= E) {
    offsets[e] = off_s[e];
    toffsets[e] = toff_s[e];
  }
  if (pp < parts) {  // each part's blocks start after the earlier parts' rows of the expert
    int run = off_s[pe];
    for (int p = 0; p < pp; ++p) run += psum[p * E + pe];
#pragma unroll 8
    for (int b = b0; b < b1; ++b) {
      blkbase[(size_t)b * E + pe] = run;
      run += blkcnt[(size_t)b * E + pe];
    }
  }
  if (e < E) {
    const int t0 = toff_s[e];
    for (int i = 0; i < ntl[e]; ++i) {
      if (t0 + i >= max_tiles) {
        set_dev_error(err, kDevFault);
        break;
      }
      TileEntry te;
      te.expert = e;
      te.row0 = off_s[e] + i * row_block;
      te.rows = min(row_block, tot[e] - i * row_block);
      te.pad = 0;
      tiles[1 + t0 + i] = te;
    }
  }
}

__global__ void __launch_bounds__(kRouteTB) route_scatter_kernel(const int32_t* __restrict__ topk_idx, int T,
                                                                 int E, int k,
                                                                 const int32_t* __restrict__ blkbase,
                                                                 int32_t* __restrict__ perm,
                                                                 int32_t* __restrict__ inv) {
  __shared__ uint32_t mask[kRouteTB / 32][kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int i = tid; i < (kRouteTB / 32) * kMaxE; i += blockDim.x) (&mask[0][0])[i] = 0u;
  pdl_wait();
  pdl_trigger();
  __syncthreads();
  const int t = blockIdx.x * kRouteTB + tid;
  int ex[kMaxTopK];
  if (t < T)
    for (int j = 0; j < k; ++j) {
      ex[j] = topk_idx[(size_t)t * k + j];
      atomicOr(&mask[warp][ex[j]], 1u << lane);
    }
  __syncthreads();
  if (t < T) {
    const uint32_t lt = (1u << lane) - 1u;
    for (int j = 0; j < k; ++j) {
      const int e = ex[j];
      int rank = __popc(mask[warp][e] & lt);
      for (int w = 0; w < warp; ++w) rank += __popc(mask[w][e]);
      const int pos = blkbase[(size_t)blockIdx.x * E + e] + rank;
      perm[pos] = t * k + j;
      inv[(size_t)t * k + j] = pos;
    }
  }
}

// All of routing in one block of 1024 threads (T <= kRouteTB): top-k by warps with the expert
// histogram and per-32-token membership masks in shared memory, then the scan and tile table,
// then each row's rank among the rows of its expert (tokens in order), as the three kernels
// above compute them.
__global__ void __launch_bounds__(1024) route_small_kernel(const float* __restrict__ logits, int T, int E, int k,
                                                           int row_block, int max_tiles,
                                                           int32_t* __restrict__ topk_idx,
                                                           float* __restrict__ topk_w, int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ toffsets,
                                                           int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                                           TileEntry* __restrict__ tiles, int* err, RoutePrelude pre) {
  __shared__ int cnt[kMaxE], off_s[kMaxE + 1], toff_s[kMaxE + 1];
  __shared__ uint32_t mask[kRouteTB / 32][kMaxE];
  __shared__ uint8_t sel_e[kRouteTB][kMaxTopK];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
  for (int i = tid; i < (kRouteTB / 32) * kMaxE; i += blockDim.x) (&mask[0][0])[i] = 0u;
  pdl_wait();  // the previous kernel of the stream may still read the accumulators zeroed here
  pdl_trigger();
  zero_prelude(pre);
  if (tid == 0) reset_status(err);
  __syncthreads();
  for (int t = warp; t < T; t += 32) {
    if (pre.x) row_absmax(pre, t, lane);
    const int mi = route_token(logits, t, E, k, lane, topk_idx, topk_w);
    if (lane < k) {
      atomicAdd(&cnt[mi], 1);
      atomicOr(&mask[t >> 5][mi], 1u << (t & 31));
      sel_e[t][lane] = (uint8_t)mi;
    }
  }
  __syncthreads();
  if (warp == 0) expert_scan(cnt, E, row_block, max_tiles, off_s, toff_s, tiles, lane);
  __syncthreads();
  if (tid <= E) {
    offsets[tid] = off_s[tid];
    toffsets[tid] = toff_s[tid];
  }
  if (tid < E) {
    const int ntl = (cnt[tid] + row_block - 1) / row_block, t0 = toff_s[tid];
    for (int i = 0; i < ntl; ++i) {
      if (t0 + i >= max_tiles) {
        set_dev_error(err, kDevFault);
        break;
      }
      TileEntry te;
      te.expert = tid;
      te.row0 = off_s[tid] + i * row_block;
      te.rows = min(row_block, cnt[tid] - i * row_block);
      te.pad = 0;
      tiles[1 + t0 + i] = te;
    }
  }
  if (tid < T) {
    const int t = tid, g = t >> 5;
    const uint32_t lt = (1u << (t & 31)) - 1u;
    for (int j = 0; j < k; ++j) {
      const int e = sel_e[t][j];
      int rank = __popc(mask[g][e] & lt);
      for (int w = 0; w < g; ++w) rank += __popc(mask[w][e]);
      const int pos = off_s[e] + rank;
      perm[pos] = t * k + j;
      inv[(size_t)t * k + j] = pos;
    }
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int row_block, const WsLayout& L, char* ws,
                         const RoutePrelude& pre, cudaStream_t s) {
  int* err = (int*)(ws + L.err);
  int32_t* idx = (int32_t*)(ws + L.topk_idx);
  float* w = (float*)(ws + L.topk_w);
  int32_t* blkcnt = (int32_t*)(ws + L.blkcnt);
  int32_t* blkbase = (int32_t*)(ws + L.blkbase);
  int32_t* off = (int32_t*)(ws + L.offsets);
  int32_t* toff = (int32_t*)(ws + L.toff);
  int32_t* perm = (int32_t*)(ws + L.perm);
  int32_t* inv = (int32_t*)(ws + L.inv);
  TileEntry* tiles = (TileEntry*)(ws + L.tiles);
  const int nb = L.nb;
  if (T > 0 && T <= kRouteTB) {
    note_launches(1);
    return launch_pdl(route_small_kernel, dim3(1), dim3(1024), 0, s, logits, T, E, k, row_block, L.max_tiles, idx,
                      w, off, toff, perm, inv, tiles, err, pre);
  }
  cudaError_t e = cudaSuccess;
  if (T > 0) e = launch_pdl(route_topk_kernel, dim3(nb), dim3(1024), 0, s, logits, T, E, k, idx, w, blkcnt, err, pre);
  else e = cudaMemsetAsync(err, 0, sizeof(int), s);
  if (e == cudaSuccess)
    e = launch_pdl(route_scan_kernel, dim3(1), dim3(1024), 0, s, (const int32_t*)blkcnt, T > 0 ? nb : 0, E, row_block,
                   L.max_tiles, off, toff, blkbase, tiles, err);
  if (e == cudaSuccess && T > 0)
    e = launch_pdl(route_scatter_kernel, dim3(nb), dim3(kRouteTB), 0, s, (const int32_t*)idx, T, E, k,
                   (const int32_t*)blkbase, perm, inv);
  note_launches(T > 0 ? 3 : 1);
  return e;
}

}  // namespace moe
