// Internal declarations shared by the library's translation units (not installed).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe_gb300.h"

namespace moe {

constexpr int kMaxE = 256;      // router width supported by the warp top-k (8 logits per lane)
constexpr int kMaxTopK = 8;     // slots per token
constexpr int kRouteTB = 128;   // tokens per routing block (histogram granularity)
constexpr int kMinRowBlock = 8; // smallest GEMM row block; bounds the tile table

// Device error word values (written with atomicCAS so the first failure is kept).
enum : int { kDevOk = 0, kDevTimeout = MOE_ERR_DEVICE_TIMEOUT, kDevFault = MOE_ERR_DEVICE_FAULT };

__device__ __forceinline__ void set_dev_error(int* err, int code) { atomicCAS(err, 0, code); }

// The workspace status block (256 bytes): int 0 is the device error word; ints 1 .. kSchedCounters
// are the work counters of the persistent GEMM kernels that hand out items dynamically.  The
// routing kernel of every forward pass resets them all.
constexpr int kSchedCounters = 2;
__device__ __forceinline__ void reset_status(int* status) {
  status[0] = kDevOk;
  for (int i = 1; i <= kSchedCounters; ++i) status[i] = 0;
}

// ---- scalar codecs (device) --------------------------------------------------------------
__device__ __forceinline__ float bf16_to_f32(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint16_t bf16_bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }

// E4M3 ("e4m3fn") code -> float; exact.
__device__ __forceinline__ float e4m3_to_f32(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}
// float -> E4M3, round to nearest even, saturating at +-448 (hardware conversion).
__device__ __forceinline__ uint8_t f32_to_e4m3(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}
// E2M1 magnitude table {0, .5, 1, 1.5, 2, 3, 4, 6}; bit 3 is the sign.
__device__ __forceinline__ float e2m1_to_f32(uint32_t c) {
  const float m[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  float v = m[c & 7];
  return (c & 8) ? -v : v;
}

// ---- routing tile table ------------------------------------------------------------------
// One entry per GEMM row block: rows [row0, row0 + rows) of the permuted order, all routed
// to `expert`.  Entry 0 of the table is a header whose .expert field holds the tile count.
struct TileEntry {
  int32_t expert, row0, rows, pad;
};
// Tile-table entries are read through L2 only (ld.global.cg): a GEMM that starts before its
// predecessor has finished reads them before griddepcontrol.wait, and the table of an earlier
// forward pass may still sit in this SM's L1.
__device__ __forceinline__ TileEntry load_tile(const TileEntry* p) {
  const int4 v = __ldcg((const int4*)p);
  TileEntry t;
  t.expert = v.x;
  t.row0 = v.y;
  t.rows = v.z;
  t.pad = v.w;
  return t;
}

// ---- workspace layout ----------------------------------------------------------------------
struct WsLayout {
  size_t err, topk_idx, topk_w, blkcnt, blkbase, offsets, perm, inv, tiles;
  size_t toff;  // first routing tile of each expert [E + 1]
  size_t h, y, xq, xs, xg, hq, hs, hg;  // y: routing-weighted down rows [R, H] bf16
  size_t xi, hi;  // W4A4: x and h as tensor-core operand images (ActImage)
  size_t cnt;         // the down GEMM's completion counter (zeroed by routing)
  size_t xp;          // expert-permuted bf16 copy of x (tensor-core path, row blocks >= 64)
  size_t xmax, hmax;  // per-row max |activation| (FP8 decode path)
  size_t x_stage, lg_stage, out_stage;
  size_t total;
  int nb;         // routing blocks
  int max_tiles;  // capacity of the tile table (excluding the header)
};

WsLayout ws_layout(int fmt, int E, int H, int I, int T, int k, bool host_io);
// The routing part alone (error word, top-k, histograms, offsets, permutation, tile table): the
// prefix every ws_layout starts with, and all that routing by itself needs.
WsLayout route_layout(int E, int T, int k);
// MOE_OK on an sm_103 device (the only target the kernels are built for), else
// MOE_ERR_UNSUPPORTED (or MOE_ERR_CUDA if the device cannot be queried).
moe_status_t device_ok();

// ---- launches (each returns cudaGetLastError() after enqueueing) -------------------------
// Work folded into the first routing launch: zero the h row maxima and (optionally) record the
// max |x| of every activation row (FP8 decode path).
struct RoutePrelude {
  unsigned* zero_u32 = nullptr;
  size_t n_u32 = 0;
  unsigned* zero2_u32 = nullptr;  // a second range (the combine counters)
  size_t n2_u32 = 0;
  const uint16_t* x = nullptr;  // bf16 [T, H] or null
  int H = 0;
  float* xmax = nullptr;
};
cudaError_t launch_route(const float* logits, int T, int E, int k, int row_block, const WsLayout& L,
                         char* ws, const RoutePrelude& pre, cudaStream_t s);
cudaError_t launch_pack(const moe_packed_desc_t& d, const __nv_bfloat16* wgu, const __nv_bfloat16* wd,
                        char* packed, cudaStream_t s);
cudaError_t launch_dequant(const moe_packed_desc_t& d, const char* packed, int e, int which, float* out,
                           cudaStream_t s);
// ---- NVFP4 W4A4 tensor-core operand images --------------------------------------------------
// One block-scaled MMA step reads, per 128-row tile and 256-column chunk, 16 KB of E2M1 codes in
// the 128-byte swizzle layout and 2 KB of E4M3 block scales.  The W4A4 path keeps both operands
// in exactly that shape in global memory, so each stage of the GEMMs is one bulk copy per
// operand (a TMA unit's cost is per copy, nearly independent of its size):
//   weights     (packed buffer)  [E, pairs, C, kWImgBlock]: two 128-row tiles (gate/up: a gate
//               tile and the matching up tile; down: 256 consecutive output rows) -> codes of
//               tile 0, codes of tile 1, scales of tile 0, scales of tile 1, the scales in the
//               order tensor memory takes them (per K = 64 step a 512-byte atom whose 16-byte
//               row l holds the four scales of tile rows l, l + 32, l + 64, l + 96);
//   activations (workspace)      [tiles, C, kAImgBlock]: one routing tile -> codes, then the
//               scales row by row (16 bytes per row).
// C = ceil(K / 256); a last half chunk leaves its upper 64 bytes per row unused.
constexpr int kImgTile = 16384, kImgSf = 2048;
// NVFP4 W4A16 weight image block ([E, K/128, N/128] of them): one 128-row tile (gate/up: 64 gate
// rows, then the same features' up rows) of one 128-column chunk -- 64 code bytes per row in the bf16 converter's bit
// order, 16-byte piece p of row l at piece p ^ ((l / 2) % 4), then 8 E4M3 scales per row.
constexpr int kW16Codes = 128 * 64, kW16Block = kW16Codes + 128 * 8;
constexpr int kWImgBlock = 2 * kImgTile + 2 * kImgSf, kAImgBlock = kImgTile + kImgSf;
__host__ __device__ inline int nvfp4_chunks(int K) { return (K + 255) / 256; }
// Byte of the 8 codes of 16-block b (0..15 of the chunk) of tile row l within a tile's codes.
__host__ __device__ inline int img_code_byte(int l, int b) { return 128 * l + (((b >> 1) ^ (l & 7)) << 4) + 8 * (b & 1); }
// Weight scale of tile row l, 16-block b (0..15 of the chunk), within a tile's scale atoms.
__host__ __device__ inline int img_wsf_byte(int l, int b) { return 512 * (b >> 2) + 16 * (l & 31) + 4 * (l >> 5) + (b & 3); }
// Routed row p of expert e is row slot % 128 of routing tile slot / 128 (128-row tiles).
__device__ __forceinline__ int img_slot(int p, int e, const int32_t* offsets, const int32_t* toff) {
  return 128 * toff[e] + p - offsets[e];
}
// Where a quantizer puts NVFP4 activation rows instead of row-major codes: the operand image.
// Rows are routed (permuted) rows; a row's expert comes from topk_idx at its (token, slot) index
// (the scatter index for x, perm[row] for h).
struct ActImage {
  uint8_t* img = nullptr;
  int chunks = 0;
  const int32_t* topk_idx = nullptr;
  const int32_t* perm = nullptr;
  const int32_t* offsets = nullptr;
  const int32_t* toff = nullptr;
};
// NVFP4 quantization of bf16 rows; row r's codes go to output row r, or (scatter != null) to
// rows scatter[r*k .. r*k+k-1].  early: x was final before the preceding kernel of the stream
// passed its pdl_wait() (true only right after routing), so x is read before this launch's wait.
// sf_rows = 0: scales row-major [rows, K/16]; else chunk-major [C][sf_rows][16], C = ceil(K/256).
// static_gs (dev, one float) != null: that global scale for every row instead of each row's own.
// gs may be null (the per-row scales are then not stored).
// img != null: codes and scales go to the operand image instead (q, sf unused).
cudaError_t launch_quant_rows(const __nv_bfloat16* x, const int32_t* scatter, int k, int rows, int K, uint8_t* q,
                              uint8_t* sf, float* gs, cudaStream_t s, bool early = false, int sf_rows = 0,
                              const float* static_gs = nullptr, const ActImage* img = nullptr);
// Rows of one chunk plane of chunk-major activation scales for R routed rows: a 128-row tile
// starting at any row below R stays inside its plane.
inline int sf_plane_rows(size_t R) { return (int)R + 128; }
// out[r] = x[map[r] / k] for r < rows (rows of K bf16).
cudaError_t launch_gather_rows(const __nv_bfloat16* x, const int32_t* map, int k, int rows, int K, __nv_bfloat16* out,
                               cudaStream_t s);
// Row block from which the tensor-core path reads a permuted copy of x instead of gathering rows.
constexpr int kTcPermuteFromRows = 64;
// Optional events around the two GEMM steps (0 = gate/up, 1 = down); null entries are skipped.
struct StepEvents {
  cudaEvent_t start[2] = {nullptr, nullptr}, stop[2] = {nullptr, nullptr};
};
// act_gs (dev, [2]; W4A4 only): null = dynamic per-row activation scales, else the static global
// scales of x and h.
cudaError_t launch_experts(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T,
                           int k, int row_block, const WsLayout& L, char* ws, __nv_bfloat16* out,
                           const StepEvents& ev, cudaStream_t s, const float* act_gs = nullptr);
// gs = 2688 / max(amax over n bf16 values, 1e-12) into *gs (dev): a static activation scale.
cudaError_t launch_act_scale(const uint16_t* v, size_t n, float* gs, cudaStream_t s);
// Programmatic dependent launch.  A kernel started with launch_pdl may begin while the previous
// kernel of the stream is still running (in a CUDA graph the edge becomes programmatic): it sets
// up shared and tensor memory, then calls pdl_wait() before it touches memory that earlier
// kernels write or read, and pdl_trigger() to let its own dependent start setting up.  Only
// read-only data (packed weights), the routing tile table (final before the previous GEMM
// passed its own pdl_wait()) and, in the activation quantizer that follows routing, the layer
// input x (final before the routing kernels, which wait before they trigger, started) may be
// read before pdl_wait().
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
// Record a timing event on s; under stream capture it becomes an event-record node of the graph.
inline void record_event(cudaEvent_t ev, cudaStream_t s) {
  if (!ev) return;
  cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &st);
  if (st == cudaStreamCaptureStatusActive) cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else cudaEventRecord(ev, s);
}
// Running count of kernels enqueued by the library (moe_kernel_launch_count).
void note_launches(int n);
// Tensor-core path (FP8 W8A16, INT4 W4A16, NVFP4 W4A16, BF16): row block per tile, and the two GEMMs.
int tc_row_block(int fmt, int T, int k, int E);
bool tc_make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t d0, uint64_t d1, uint64_t pitch,
                 uint32_t b0, uint32_t b1, CUtensorMapSwizzle sw);
int tc_num_sms();
// Activation rows [R, K] bf16 as a 3-D map ([K/64 atoms][R rows][64]) whose box brings bn rows x
// 128 K, both 128-byte swizzle atoms, in one copy.
bool tc_act_map(CUtensorMap* m, const void* base, uint64_t R, int K, int bn);
// FP8 decode path (16-row tiles, weights straight into kind::f8f6f4 MMAs).
int fp8dec_row_block();
// Each down GEMM ends with the deterministic routing-weighted combine into out (bf16 [T, H]).
cudaError_t launch_experts_fp8dec(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T,
                                  int k, const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s,
                                  uint16_t* out);
// NVFP4 W4A4 path on block-scaled FP4 MMAs (128-row routing tiles; any H, I multiples of 128).
int fp4_row_block();
// The down GEMM combines each token's k routing-weighted rows in its epilogue and writes out
// (bf16 [T, H]).  act_gs: static activation scales (dev, [2]) or null; calibrate: instead of the
// layer, write the static scales of this batch into act_gs (x's from x, then h's from the gate/up
// output; out unused).
cudaError_t launch_experts_fp4(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                               const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, uint16_t* out,
                               const float* act_gs = nullptr, bool calibrate = false);
cudaError_t launch_experts_tc(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                              int bn, const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, uint16_t* out);
// FP8 W8A16 decode steps whose active experts average at most two rows: CUDA-core GEMVs.
cudaError_t launch_experts_fp8gemv(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T,
                                   int k, int row_block, const WsLayout& L, char* ws, const StepEvents& ev,
                                   cudaStream_t s, uint16_t* out);
bool fp8gemv_preferred(int T, int k, int E, int I);
// INT4 W4A16 decode steps, the same way (moe_gemm_int4gemv.cu).
cudaError_t launch_experts_int4gemv(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T,
                                    int k, int row_block, const WsLayout& L, char* ws, const StepEvents& ev,
                                    cudaStream_t s, uint16_t* out);
bool int4gemv_preferred(int T, int k, int E, int H, int I);
// NVFP4 W4A16 with 256-row routing tiles (tc_row_block's choice at prefill sizes).
int tcw_row_block();
cudaError_t launch_experts_tcw(const moe_packed_desc_t& d, const char* packed, const __nv_bfloat16* x, int T, int k,
                               const WsLayout& L, char* ws, const StepEvents& ev, cudaStream_t s, uint16_t* out);


}  // namespace moe
