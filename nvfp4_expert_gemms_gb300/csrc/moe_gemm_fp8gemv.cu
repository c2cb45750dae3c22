// FP8 W8A16 grouped GEMMs as CUDA-core GEMVs for decode steps with few routed experts, each
// seeing one or two tokens (fp8gemv_preferred).
//
// There an M = 128 tensor-core MMA costs the same at N = 16 as at N = 128 (about 64-94 SM cycles
// per 128 x 16 weight block, measured), so the tensor-core kernels are bound by the MMA
// instruction rate, not by HBM; and at one token a layer has only 8 routed experts, 48 gate/up
// tiles of 128 rows for 152 SMs.  Here every warp streams two weight rows with 512-byte
// coalesced loads (one 16-byte piece per lane), turns the E4M3 codes into fp32 (through the
// hardware's E4M3 -> f16 pair conversion, exact), and multiplies them against the routing tile's
// token rows (read through L1, where every warp of the tile finds them), four rows at a time.  Each 128-column block of a
// row carries one fp32 scale (clef-omni-fp8, "What was quantized"): a lane's 16 products share
// it, so the lane sums them first and scales the sum.  The warp then reduces over its lanes.
//
//   gate/up (MODE 0): task = (routing tile, feature f): gate row f and up row I + f against each
//     token row, then h = SiLU(gate) * up -> bf16 [R, I]
//   down (MODE 1): task = (routing tile, rows 2p, 2p + 1) times the row's routing weight -> bf16
//     y [R, H], then the deterministic combine
//
// One CTA of 16 warps per SM; each warp walks tasks with a stride of all the grid's warps, with
// no block-wide synchronisation, so an SM keeps 16 tasks' weight loads in flight.
#include <cuda_fp8.h>

#include "moe_formats.cuh"
#include "moe_combine.cuh"
#include "moe_tc.cuh"

namespace moe {

namespace {

constexpr int kWarps = 16, kThreads = kWarps * 32;
constexpr int kRowGroup = 4;  // token rows multiplied per pass over the weights
constexpr int kSegBytes = 512;  // one warp load: 32 lanes x 16 bytes of one weight row
constexpr int kSegBatch = 4;    // segments loaded before the multiplies (8 loads in flight per lane)

struct GemvArgs {
  const uint8_t* codes;    // E4M3 [E, N, K]
  const float* scale_inv;  // [E, N/128, K/128]
  const uint16_t* act;     // bf16: x [T, K] (rows by token) or h [R, K] (permuted rows)
  const int32_t* perm;
  const float* topk_w;
  const TileEntry* tiles;
  uint16_t* h_out;  // gate/up: h [R, I]
  uint16_t* y_out;  // down: routing-weighted rows [R, H]
  CombineTail ct;
  int* err;
  int k, N, K, I, H;
};

// 16 E4M3 codes -> fp32 (exact: every E4M3 value is an f16 value)
__device__ __forceinline__ void e4m3x16_to_f32(const uint4& c, float* w) {
  const uint32_t v[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v[i] >> (16 * h)), __NV_E4M3);
      const float2 f = __half22float2(*(const __half2*)&r);
      w[4 * i + 2 * h] = f.x;
      w[4 * i + 2 * h + 1] = f.y;
    }
  }
}

// 16 bf16 activations -> fp32
__device__ __forceinline__ void bf16x16_to_f32(const uint4& u0, const uint4& u1, float* x) {
  const uint32_t v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(v[i] << 16);
    x[2 * i + 1] = __uint_as_float(v[i] & 0xFFFF0000u);
  }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) fp8gemv_kernel(const GemvArgs a) {
  pdl_wait();  // the routing tables (and, for the down GEMM, h) come from the launches before
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = load_tile(a.tiles).expert;  // header entry holds the tile count
  const int nrp = MODE == 0 ? a.I : a.H / 2;     // weight-row pairs per matrix: one task each
  const long ntask = (long)ntiles * nrp;
  const int K = a.K, nseg = (K + kSegBytes - 1) / kSegBytes;
  // warps walk (routing tile, row pair) tasks on their own, so that each SM keeps its 16 warps'
  // weight loads in flight without block-wide synchronisation
  for (long t = (long)blockIdx.x * kWarps + warp; t < ntask; t += (long)gridDim.x * kWarps) {
    const TileEntry te = load_tile(a.tiles + 1 + t / nrp);
    const int p = (int)(t % nrp), e = te.expert;
    const int n0 = MODE == 0 ? p : 2 * p;
    const int n1 = MODE == 0 ? a.I + p : 2 * p + 1;
    const uint8_t* w0 = a.codes + ((size_t)e * a.N + n0) * K;
    const uint8_t* w1 = a.codes + ((size_t)e * a.N + n1) * K;
    const float* s0 = a.scale_inv + ((size_t)e * (a.N / 128) + n0 / 128) * (K / 128);
    const float* s1 = a.scale_inv + ((size_t)e * (a.N / 128) + n1 / 128) * (K / 128);
    for (int rg = 0; rg < te.rows; rg += kRowGroup) {
      const int nr = te.rows - rg < kRowGroup ? te.rows - rg : kRowGroup;
      const uint16_t* xrow[kRowGroup];  // the group's activation rows
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) {
        const int row = te.row0 + rg + (r < nr ? r : 0);
        const int src = MODE == 0 ? __ldcg(a.perm + row) / a.k : row;
        xrow[r] = a.act + (size_t)src * K;
      }
      float acc[kRowGroup][2];
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r) acc[r][0] = acc[r][1] = 0.f;
      for (int j0 = 0; j0 < nseg; j0 += kSegBatch) {
        uint4 c0[kSegBatch], c1[kSegBatch];
#pragma unroll
        for (int j = 0; j < kSegBatch; ++j) {  // the batch's weight loads first
          const int kk = (j0 + j) * kSegBytes + lane * 16;
          if (j0 + j < nseg && kk < K) {
            c0[j] = __ldg((const uint4*)(w0 + kk));
            c1[j] = __ldg((const uint4*)(w1 + kk));
          }
        }
#pragma unroll
        for (int j = 0; j < kSegBatch; ++j) {
          const int kk = (j0 + j) * kSegBytes + lane * 16;
          if (j0 + j >= nseg || kk >= K) continue;
          const float sc0 = __ldg(s0 + kk / 128), sc1 = __ldg(s1 + kk / 128);
          float wa[16], wb[16];
          e4m3x16_to_f32(c0[j], wa);
          e4m3x16_to_f32(c1[j], wb);
#pragma unroll
          for (int r = 0; r < kRowGroup; ++r) {
            if (r >= nr) break;
            const uint4* xp = (const uint4*)(xrow[r] + kk);
            float xv[16];
            bf16x16_to_f32(__ldg(xp), __ldg(xp + 1), xv);  // (written before this grid's wait)
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              p0 = fmaf(wa[i], xv[i], p0);
              p1 = fmaf(wb[i], xv[i], p1);
            }
            acc[r][0] = fmaf(p0, sc0, acc[r][0]);
            acc[r][1] = fmaf(p1, sc1, acc[r][1]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kRowGroup; ++r)
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          acc[r][0] += __shfl_xor_sync(0xffffffffu, acc[r][0], o);
          acc[r][1] += __shfl_xor_sync(0xffffffffu, acc[r][1], o);
        }
      if (lane < nr) {  // lane r stores token row r of the group
        float g = acc[0][0], u = acc[0][1];
#pragma unroll
        for (int r = 1; r < kRowGroup; ++r)
          if (lane == r) {
            g = acc[r][0];
            u = acc[r][1];
          }
        const int row = te.row0 + rg + lane;
        if (MODE == 0) {
          const float hv = __fdividef(g, 1.0f + __expf(-g)) * u;
          a.h_out[(size_t)row * a.I + n0] = bf16_bits(hv);
        } else {
          const float tw = __ldcg(a.topk_w + __ldcg(a.perm + row));
          a.y_out[(size_t)row * a.H + n0] = bf16_bits(tw * g);
          a.y_out[(size_t)row * a.H + n1] = bf16_bits(tw * u);
        }
      }
    }
  }
  if (MODE == 1) {  // the routing-weighted combine, once every CTA is done
    __shared__ int s_flag;
    if (!combine_tail(a.ct, (int)gridDim.x, &s_flag) && threadIdx.x == 0) set_dev_error(a.err, kDevTimeout);
  }
}

}  // namespace

// Measured on one GB300 at H = 2048, I = 768, top-8 (FP8 decode, tokens/s of one layer): T = 1
// 34.1k here against 29.4k on the tensor-core decode kernel, whose 48 gate/up items then leave
// most SMs idle; T = 4 57.4k against 73.9k and T = 16 80.7k against 157k once that kernel has
// an item for every SM (and the INT4 GEMVs lose already at T = 2, 96 items).  So the GEMVs take
// the steps whose active experts average at most two rows and give the tensor-core kernel fewer
// gate/up items (128 rows each) than half the SMs.
bool fp8gemv_preferred(int T, int k, int E, int I) {
  const long R = (long)T * k, active = R < E ? (R > 0 ? R : 1) : E;
  return (R + active - 1) / active <= 2 && 2 * active * (I / 128) < tc_num_sms();
}

cudaError_t launch_experts_fp8gemv(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T,
                                   int k, int row_block, const WsLayout& L, char* ws, const StepEvents& ev,
                                   cudaStream_t s, uint16_t* out) {
  const int E = d.E, H = d.H, I = d.I;
  const size_t R = (size_t)T * k;
  const MatView gu = mat_view(d, packed, 0), dn = mat_view(d, packed, 1);
  GemvArgs a;
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

  a.codes = gu.a;
  a.scale_inv = (const float*)gu.b;
  a.act = (const uint16_t*)x;
  a.N = 2 * I;
  a.K = H;
  size_t ctas = (tiles * (size_t)I + kWarps - 1) / kWarps;  // one task per warp at least
  record_event(ev.start[0], s);
  cudaError_t err =
      launch_pdl(fp8gemv_kernel<0>, dim3((unsigned)(ctas < (size_t)sms ? ctas : sms)), dim3(kThreads), 0, s, a);
  record_event(ev.stop[0], s);
  if (err != cudaSuccess) return err;

  a.codes = dn.a;
  a.scale_inv = (const float*)dn.b;
  a.act = (const uint16_t*)(ws + L.h);
  a.N = H;
  a.K = I;
  ctas = (tiles * (size_t)(H / 2) + kWarps - 1) / kWarps;
  record_event(ev.start[1], s);
  err = launch_pdl(fp8gemv_kernel<1>, dim3((unsigned)(ctas < (size_t)sms ? ctas : sms)), dim3(kThreads), 0, s, a);
  record_event(ev.stop[1], s);
  note_launches(2);
  return err;
}

}  // namespace moe
