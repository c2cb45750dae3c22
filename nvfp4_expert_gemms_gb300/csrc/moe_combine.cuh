// The routing-weighted combine at the end of a down GEMM kernel (deterministic):
//   out[t, :] = bf16( sum over slots j = 0..k-1, in order, of y[inv[t*k + j], :] )
// where y holds the kernel's routing-weighted bf16 rows in permuted order (as its epilogue
// stores them: a tile's rows are consecutive).  Every CTA of the grid that ran GEMM items calls
// it after its last one: the CTA publishes its rows and counts itself done, waits (bounded)
// until every such CTA has, and then sums its own slice of tokens.
// The wait needs all those CTAs resident together, which holds for these persistent kernels
// (one CTA per SM, at most one CTA per SM launched; a dependent kernel starts only after every
// CTA of this one has started).
#pragma once
#include "moe_internal.cuh"
#include "moe_tc.cuh"

namespace moe {

struct CombineTail {
  const uint16_t* y;     // routing-weighted rows [R, H] bf16, permuted order
  const int32_t* inv;    // [T*k]: permuted row of (token t, slot j) at t*k + j
  uint16_t* out;         // [T, H] bf16 (16-byte aligned)
  int* done;             // CTAs finished, zero on entry (reset by routing)
  int k, T, H;
};

inline void combine_tail_args(CombineTail& c, const WsLayout& L, char* ws, int T, int k, int H, uint16_t* out) {
  c.y = (const uint16_t*)(ws + L.y);
  c.inv = (const int32_t*)(ws + L.inv);
  c.out = out;
  c.done = (int*)(ws + L.cnt);
  c.k = k;
  c.T = T;
  c.H = H;
}

// 8 columns of k rows (v[0 .. k-1]) summed in slot order in fp32, stored as bf16 (the loop is
// unrolled over the largest k so v stays in registers).
__device__ __forceinline__ void sum_slots_store(const uint4* v, int k, uint16_t* dst) {
  float s[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j >= k) break;
    const uint32_t w[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      s[2 * e] += __uint_as_float(w[e] << 16);
      s[2 * e + 1] += __uint_as_float(w[e] & 0xFFFF0000u);
    }
  }
  uint4 o;
  o.x = (uint32_t)bf16_bits(s[0]) | ((uint32_t)bf16_bits(s[1]) << 16);
  o.y = (uint32_t)bf16_bits(s[2]) | ((uint32_t)bf16_bits(s[3]) << 16);
  o.z = (uint32_t)bf16_bits(s[4]) | ((uint32_t)bf16_bits(s[5]) << 16);
  o.w = (uint32_t)bf16_bits(s[6]) | ((uint32_t)bf16_bits(s[7]) << 16);
  *(uint4*)dst = o;
}

// All threads of the CTA, after its last y store.  Returns false if the wait gave up (the
// caller records the timeout).  (Measured against this plain loop and found slower: streaming
// the rows through shared memory with bulk copies, two column groups per thread in flight,
// staging the slice's row indices in shared memory, and slot-ordered rows, which slow the
// epilogue's stores.)
__device__ __forceinline__ bool combine_tail(const CombineTail& c, int active_ctas, int* s_flag) {
  __syncthreads();  // every thread's y stores are issued
  if (threadIdx.x == 0) {
    asm volatile("fence.acq_rel.gpu;" ::: "memory");  // ... and visible at GPU scope before the count
    atomicAdd(c.done, 1);
    const long long t0 = clock64();
    int ok = 1;
    for (;;) {
      int v;
      asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(c.done) : "memory");
      if (v >= active_ctas) break;
      if (clock64() - t0 > tc::kWaitLimitCycles) {
        ok = 0;
        break;
      }
    }
    *s_flag = ok;
  }
  __syncthreads();  // thread 0 acquired every CTA's rows; the barrier passes it on
  if (!*s_flag) return false;
  const int cta = blockIdx.x;
  const int t0 = (int)((long long)c.T * cta / active_ctas), t1 = (int)((long long)c.T * (cta + 1) / active_ctas);
  const int per_tok = c.H / 8;  // 8 columns per thread and step
  for (int i = threadIdx.x; i < (t1 - t0) * per_tok; i += blockDim.x) {
    const int t = t0 + i / per_tok, col = 8 * (i % per_tok);
    uint4 v[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < c.k) v[j] = __ldcg((const uint4*)(c.y + (size_t)__ldg(c.inv + (size_t)t * c.k + j) * c.H + col));
    sum_slots_store(v, c.k, c.out + (size_t)t * c.H + col);
  }
  return true;
}

}  // namespace moe
