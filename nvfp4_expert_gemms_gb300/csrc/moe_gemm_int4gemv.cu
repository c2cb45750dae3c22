// INT4 W4A16 grouped GEMMs as CUDA-core GEMVs for decode steps with few routed experts, each
// seeing one or two tokens (int4gemv_preferred).
//
// The packed weights keep auto_gptq's order (clef-omni-int4, "What was quantized"): qweight
// [E, K/8, N] int32, word (kr, n) holding k = 8 kr + j in nibble j as q + 8, and one fp16 scale
// per (128-column group, row n).  Output rows are contiguous along N, so a lane takes one output
// row and a warp reads 32 consecutive words of each qweight row (128 bytes, coalesced).  To keep
// enough loads in flight, K is split over the warps: warp w of a CTA takes the 128-column group w
// (16 qweight rows), issues its 16 (gate/up: 32) word loads at once, and the CTA adds the groups'
// partial sums in shared memory.  Each group's sum is scaled once by the group's fp16 scale.
//
//   gate/up (MODE 0): item = (routing tile, features f0..f0+31); lane l: gate row f0 + l and
//     up row I + f0 + l; then h = SiLU(gate) * up -> bf16 [R, I]
//   down (MODE 1): item = (routing tile, rows n0..n0+31) times each row's routing weight -> bf16
//     y [R, H], then the deterministic combine
//
// One CTA of 16 warps per SM walks the items with a stride of the grid.  K / 128 <= 16.
#include "moe_formats.cuh"
#include "moe_combine.cuh"
#include "moe_tc.cuh"

namespace moe {

namespace {

constexpr int kWarps = 16, kThreads = kWarps * 32;
constexpr int kRowGroup = 4;  // token rows per pass over the weights

struct I4Args {
  const uint32_t* qweight;  // [E, K/8, N]
  const __half* scales;     // [E, K/128, N]
  const uint16_t* act;      // bf16: x [T, K] (rows by token) or h [R, K] (permuted rows)
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;
  uint16_t* y_out;
  CombineTail ct;
  int* err;
  int k, N, K, I, H;
};

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) int4gemv_kernel(const I4Args a) {
  __shared__ float red[kWarps][kRowGroup][2][32];  // per K group: partial sums (row, gate/up, lane)
  pdl_wait();  // the routing tables (and, for the down GEMM, h) come from the launches before
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = load_tile(a.tiles).expert;  // header entry holds the tile count
  const int nfb = (MODE == 0 ? a.I : a.H) / 32;
  const int nwork = ntiles * nfb;
  const int K = a.K, ngroups = K / 128;
  for (int wk = blockIdx.x; wk < nwork; wk += gridDim.x) {
    const TileEntry te = load_tile(a.tiles + 1 + wk / nfb);
    const int e = te.expert, f = (wk % nfb) * 32 + lane;
    const int n0 = f, n1 = MODE == 0 ? a.I + f : f;  // (down: one row per lane)
    const bool kw = warp < ngroups;                  // this warp's K group exists
    uint32_t q0[16], q1[16];
    float sc0 = 0.f, sc1 = 0.f;
    if (kw) {
      const uint32_t* col = a.qweight + ((size_t)e * (K / 8) + warp * 16) * a.N;
#pragma unroll
      for (int i = 0; i < 16; ++i) {  // the group's words first: 16 (32) loads in flight per lane
        q0[i] = __ldg(col + (size_t)i * a.N + n0);
        if (MODE == 0) q1[i] = __ldg(col + (size_t)i * a.N + n1);
      }
      const __half* sg = a.scales + ((size_t)e * ngroups + warp) * a.N;
      sc0 = __half2float(sg[n0]);
      if (MODE == 0) sc1 = __half2float(sg[n1]);
    }
    for (int rg = 0; rg < te.rows; rg += kRowGroup) {
      const int nr = te.rows - rg < kRowGroup ? te.rows - rg : kRowGroup;
      if (kw) {
#pragma unroll 1
        for (int r = 0; r < nr; ++r) {
          const int row = te.row0 + rg + r;
          const int src = MODE == 0 ? __ldcg(a.perm + row) / a.k : row;
          const uint4* xp = (const uint4*)(a.act + (size_t)src * K + warp * 128);  // (written before this grid's wait)
          float p0 = 0.f, p1 = 0.f;
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {  // qweight row i: k = 8 i .. 8 i + 7 of the group
            const uint4 u = __ldg(xp + i);  // the same 16 bytes for every lane: one broadcast
            const uint32_t xv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float x = __uint_as_float(j & 1 ? xv[j >> 1] & 0xFFFF0000u : xv[j >> 1] << 16);
              p0 = fmaf((float)((int)((q0[i] >> (4 * j)) & 0xFu) - 8), x, p0);
              if (MODE == 0) p1 = fmaf((float)((int)((q1[i] >> (4 * j)) & 0xFu) - 8), x, p1);
            }
          }
          red[warp][r][0][lane] = p0 * sc0;
          red[warp][r][1][lane] = p1 * sc1;
        }
      }
      __syncthreads();
      // thread (row r, lane) of warps 0..nr-1 adds the K groups in order and stores
      if (warp < nr) {
        float g = 0.f, u = 0.f;
        for (int w = 0; w < ngroups; ++w) {
          g += red[w][warp][0][lane];
          u += red[w][warp][1][lane];
        }
        const int row = te.row0 + rg + warp;
        if (MODE == 0) {
          const float hv = __fdividef(g, 1.0f + __expf(-g)) * u;
          a.h_out[(size_t)row * a.I + f] = bf16_bits(hv);
        } else {
          a.y_out[(size_t)row * a.H + f] = bf16_bits(__ldcg(a.topk_w + __ldcg(a.perm + row)) * g);
        }
      }
      __syncthreads();  // red is free for the next pass
    }
  }
  if (MODE == 1) {  // the routing-weighted combine, once every CTA is done
    __shared__ int s_flag;
    if (!combine_tail(a.ct, (int)gridDim.x, &s_flag) && threadIdx.x == 0) set_dev_error(a.err, kDevTimeout);
  }
}

}  // namespace

// Measured on one GB300 at H = 2048, I = 768, top-8 (tokens/s of one layer): T = 1 29.4k here
// against 25.4k on the tensor-core kernel (48 gate/up items for 152 SMs); T = 2 39.4k against
// 47.6k (96 items).  So, as for FP8: active experts averaging at most two rows, fewer gate/up
// items (128 rows each) than half the SMs, and K <= 2048 on both GEMMs.
bool int4gemv_preferred(int T, int k, int E, int H, int I) {
  const long R = (long)T * k, active = R < E ? (R > 0 ? R : 1) : E;
  return H <= 2048 && I <= 2048 && (R + active - 1) / active <= 2 && 2 * active * (I / 128) < tc_num_sms();
}

cudaError_t launch_experts_int4gemv(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T,
                                    int k, int row_block, const WsLayout& L, char* ws, const StepEvents& ev,
                                    cudaStream_t s, uint16_t* out) {
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  I4Args a;
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
  const int sms = tc_num_sms();
  const size_t tiles = R / row_block + (R < (size_t)E ? R : (size_t)E) + 1;  // routing tiles, at most

  a.qweight = (const uint32_t*)gu.a;
  a.scales = (const __half*)gu.b;
  a.act = (const uint16_t*)x;
  a.N = 2 * I;
  a.K = H;
  size_t items = tiles * (size_t)(I / 32);
  record_event(ev.start[0], s);
  cudaError_t err =
      launch_pdl(int4gemv_kernel<0>, dim3((unsigned)(items < (size_t)sms ? items : sms)), dim3(kThreads), 0, s, a);
  record_event(ev.stop[0], s);
  if (err != cudaSuccess) return err;

  a.qweight = (const uint32_t*)dn.a;
  a.scales = (const __half*)dn.b;
  a.act = (const uint16_t*)(ws + L.h);
  a.N = H;
  a.K = I;
  items = tiles * (size_t)(H / 32);
  record_event(ev.start[1], s);
  err = launch_pdl(int4gemv_kernel<1>, dim3((unsigned)(items < (size_t)sms ? items : sms)), dim3(kThreads), 0, s, a);
  record_event(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
