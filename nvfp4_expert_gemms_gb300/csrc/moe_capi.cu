// Host side of the C ABI declared in include/moe_gb300.h: argument checks, the packed and
// workspace layouts, and the launch sequence of the forward pass.
#include <string.h>

#include <atomic>

#include "moe_internal.cuh"
#include "moe_w8a8.cuh"

namespace moe {

static std::atomic<uint64_t> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
static thread_local StepEvents g_pending_events;

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

WsLayout route_layout(int E, int T, int k) {
  WsLayout L;
  memset(&L, 0, sizeof(L));
  size_t cur = 0;
  auto take = [&](size_t bytes) {
    const size_t o = cur;
    cur += align256(bytes);
    return o;
  };
  const size_t R = (size_t)T * k;
  L.nb = T > 0 ? (T + kRouteTB - 1) / kRouteTB : 1;
  L.max_tiles = (int)(R / kMinRowBlock + (R < (size_t)E ? R : (size_t)E) + 1);
  L.err = take(256);
  L.topk_idx = take(4 * R);
  L.topk_w = take(4 * R);
  L.blkcnt = take(4 * (size_t)L.nb * E);
  L.blkbase = take(4 * (size_t)L.nb * E);
  L.offsets = take(4 * (size_t)(E + 1));
  L.toff = take(4 * (size_t)(E + 1));
  L.perm = take(4 * R);
  L.inv = take(4 * R);
  L.tiles = take(sizeof(TileEntry) * (size_t)(L.max_tiles + 1));
  L.total = cur;
  return L;
}

WsLayout ws_layout(int fmt, int E, int H, int I, int T, int k, bool host_io) {
  WsLayout L = route_layout(E, T, k);
  size_t cur = L.total;
  auto take = [&](size_t bytes) {
    const size_t o = cur;
    cur += align256(bytes);
    return o;
  };
  const size_t R = (size_t)T * k;
  L.h = take(2 * R * I);
  L.y = take(2 * R * (size_t)H);
  L.cnt = take(256);
  L.xmax = take(4 * (size_t)T);
  L.hmax = take(4 * R);
  if (fmt == MOE_FMT_NVFP4_W4A4) {  // x and h as operand images per 128-row routing tile + row scales
    const size_t tiles = R / 128 + (R < (size_t)E ? R : (size_t)E) + 1;
    L.xi = take(tiles * nvfp4_chunks(H) * kAImgBlock);
    L.xg = take(4 * R);
    L.hi = take(tiles * nvfp4_chunks(I) * kAImgBlock);
    L.hg = take(4 * R);
  }
  if (fmt == MOE_FMT_FP8_B128_W8A8) {  // E4M3 codes per permuted row + group-major 1x128 scales
    L.xq = take(R * H);
    L.xs = take(4 * (size_t)sf_plane_rows(R) * (H / 128));
    L.hq = take(R * I);
    L.hs = take(4 * (size_t)sf_plane_rows(R) * (I / 128));
  }
  if (fmt != MOE_FMT_NVFP4_W4A4 && fmt != MOE_FMT_FP8_B128_W8A8 && tc_row_block(fmt, T, k, E) >= kTcPermuteFromRows)
    L.xp = take(2 * R * H);
  if (host_io) {
    L.x_stage = take(2 * (size_t)T * H);
    L.lg_stage = take(4 * (size_t)T * E);
    L.out_stage = take(2 * (size_t)T * H);
  }
  L.total = cur;
  return L;
}

static bool fmt_ok(int f) { return f >= MOE_FMT_FP8_B128_W8A16 && f <= MOE_FMT_FP8_B128_W8A8; }

static bool desc_ok(const moe_packed_desc_t* d) {
  return d && fmt_ok(d->fmt) && d->E >= 1 && d->E <= kMaxE && d->H >= 128 && d->I >= 128 && d->H % 128 == 0 &&
         d->I % 128 == 0;
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// The kernels are built for sm_103a only; refuse other devices before launching anything.
moe_status_t device_ok() {
  static int checked[64];  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev >= 0 && dev < 64 && checked[dev]) return checked[dev] == 1 ? MOE_OK : MOE_ERR_UNSUPPORTED;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < 64) checked[dev] = ok ? 1 : 2;
  return ok ? MOE_OK : MOE_ERR_UNSUPPORTED;
}

static moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }



// act_gs: null, or the static activation scales (dev, [2], W4A4 only).  calibrate: act_gs is
// the output of the calibration instead (out unused, fp4 shapes only).
static moe_status_t forward_checked(const void* x, const float* logits, int T, const moe_packed_desc_t* d,
                                    const void* packed, int k, void* out, void* ws, size_t ws_bytes,
                                    cudaStream_t s, bool host_io_layout, const float* act_gs = nullptr,
                                    bool calibrate = false) {
  if (!desc_ok(d) || T < 0 || k < 1 || k > kMaxTopK || k > d->E) return MOE_ERR_INVALID_ARG;
  if (act_gs && (d->fmt != MOE_FMT_NVFP4_W4A4 || !aligned(act_gs, 4))) return MOE_ERR_INVALID_ARG;
  if (calibrate) {
    if (!act_gs || T < 1) return MOE_ERR_INVALID_ARG;
    out = (void*)act_gs;  // checked below like an output; never written as one
  }
  if (T > 0 && (!x || !logits || !packed || !out || !ws)) return MOE_ERR_INVALID_ARG;
  if (!aligned(ws, 256) || !aligned(x, 16) || !aligned(out, calibrate ? 4 : 16) || !aligned(packed, 256))
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && x == out) return MOE_ERR_INVALID_ARG;
  if (d->fmt == MOE_FMT_FP8_B128_W8A8 && !w8a8_supported(*d)) return MOE_ERR_UNSUPPORTED;
  const WsLayout L = ws_layout(d->fmt, d->E, d->H, d->I, T, k, host_io_layout);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  const moe_status_t dv = device_ok();
  if (dv != MOE_OK) return dv;
  char* w = (char*)ws;
  const int rb = d->fmt == MOE_FMT_FP8_B128_W8A8 ? w8a8_row_block()
                 : d->fmt == MOE_FMT_NVFP4_W4A4  ? fp4_row_block()
                                                 : tc_row_block(d->fmt, T, k, d->E);
  RoutePrelude pre;
  if (d->fmt == MOE_FMT_FP8_B128_W8A16 && rb == fp8dec_row_block()) {  // FP8 decode path needs row maxima
    pre.zero_u32 = (unsigned*)(w + L.hmax);
    pre.n_u32 = (size_t)T * k;
    pre.x = (const uint16_t*)x;
    pre.H = d->H;
    pre.xmax = (float*)(w + L.xmax);
  }
  if (!calibrate) {  // the down GEMM's completion counter (its combine waits on it) starts at zero
    pre.zero2_u32 = (unsigned*)(w + L.cnt);
    pre.n2_u32 = 1;
  }
  if (launch_route(logits, T, d->E, k, rb, L, w, pre, s) != cudaSuccess) return MOE_ERR_CUDA;
  const StepEvents ev = g_pending_events;
  g_pending_events = StepEvents();
  if (calibrate)
    return cuda_status(launch_experts_fp4(*d, (const char*)packed, (const __nv_bfloat16*)x, T, k, L, w, ev, s,
                                          nullptr, act_gs, true));
  return cuda_status(launch_experts(*d, (const char*)packed, (const __nv_bfloat16*)x, T, k, rb, L, w,
                                    (__nv_bfloat16*)out, ev, s, act_gs));
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status_t moe_packed_size(int fmt, int E, int H, int I, moe_packed_desc_t* d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  memset(d, 0, sizeof(*d));
  d->fmt = fmt;
  d->E = E;
  d->H = H;
  d->I = I;
  if (!desc_ok(d)) return MOE_ERR_INVALID_ARG;
  const size_t e = (size_t)E, gu = (size_t)2 * I * H, dn = (size_t)H * I;
  size_t sz[MOE_T_COUNT] = {0};
  switch (fmt) {
    case MOE_FMT_FP8_B128_W8A16:
    case MOE_FMT_FP8_B128_W8A8:  // the same stored weights
      sz[MOE_T_GU_A] = e * gu;
      sz[MOE_T_GU_B] = e * gu / (128 * 128) * 4;
      sz[MOE_T_D_A] = e * dn;
      sz[MOE_T_D_B] = e * dn / (128 * 128) * 4;
      break;
    case MOE_FMT_INT4_G128_W4A16:
      sz[MOE_T_GU_A] = e * gu / 2;
      sz[MOE_T_GU_B] = e * gu / 128 * 2;
      sz[MOE_T_D_A] = e * dn / 2;
      sz[MOE_T_D_B] = e * dn / 128 * 2;
      break;
    case MOE_FMT_BF16:
      sz[MOE_T_GU_A] = e * gu * 2;
      sz[MOE_T_D_A] = e * dn * 2;
      break;
    default:
      sz[MOE_T_GU_A] = e * gu / 2;
      sz[MOE_T_GU_B] = e * gu / 16;
      sz[MOE_T_D_A] = e * dn / 2;
      sz[MOE_T_D_B] = e * dn / 16;
      sz[MOE_T_GU_GS] = e * 4;
      sz[MOE_T_D_GS] = e * 4;
      if (fmt == MOE_FMT_NVFP4_W4A4) {  // codes and scales again, as the tensor-core operand image
        sz[MOE_T_GU_IMG] = e * ((size_t)I / 128) * nvfp4_chunks(H) * kWImgBlock;
        sz[MOE_T_D_IMG] = e * (((size_t)H + 255) / 256) * nvfp4_chunks(I) * kWImgBlock;
      } else {  // W4A16: codes (in the bf16 converter's bit order) and scales again, per tile and chunk
        sz[MOE_T_GU_IMG] = e * ((size_t)H / 128) * ((size_t)2 * I / 128) * kW16Block;
        sz[MOE_T_D_IMG] = e * ((size_t)I / 128) * ((size_t)H / 128) * kW16Block;
      }
      break;
  }
  size_t cur = 0;
  for (int i = 0; i < MOE_T_COUNT; ++i) {
    if (!sz[i]) continue;
    d->offset[i] = cur;
    d->size[i] = sz[i];
    cur += align256(sz[i]);
  }
  d->bytes = cur;
  return MOE_OK;
}

moe_status_t moe_pack_experts(const moe_packed_desc_t* d, const void* w_gate_up, const void* w_down, void* packed,
                              moe_stream_t stream) {
  if (!desc_ok(d) || !w_gate_up || !w_down || !packed || !aligned(packed, 256)) return MOE_ERR_INVALID_ARG;
  moe_packed_desc_t ref;
  if (moe_packed_size(d->fmt, d->E, d->H, d->I, &ref) != MOE_OK || ref.bytes != d->bytes) return MOE_ERR_INVALID_ARG;
  const moe_status_t dv = device_ok();
  if (dv != MOE_OK) return dv;
  return cuda_status(launch_pack(*d, (const __nv_bfloat16*)w_gate_up, (const __nv_bfloat16*)w_down, (char*)packed,
                                 (cudaStream_t)stream));
}

moe_status_t moe_workspace_size(const moe_packed_desc_t* d, int T, int top_k, size_t* bytes) {
  if (!desc_ok(d) || !bytes || T < 0 || top_k < 1 || top_k > kMaxTopK || top_k > d->E) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(d->fmt, d->E, d->H, d->I, T, top_k, false).total;
  return MOE_OK;
}

moe_status_t moe_workspace_size_host_io(const moe_packed_desc_t* d, int T, int top_k, size_t* bytes) {
  if (!desc_ok(d) || !bytes || T < 0 || top_k < 1 || top_k > kMaxTopK || top_k > d->E) return MOE_ERR_INVALID_ARG;
  *bytes = ws_layout(d->fmt, d->E, d->H, d->I, T, top_k, true).total;
  return MOE_OK;
}

moe_status_t moe_layer_forward(const void* x, const float* router_logits, int T, const moe_packed_desc_t* d,
                               const void* packed, int top_k, void* out, void* workspace, size_t ws_bytes,
                               moe_stream_t stream) {
  return forward_checked(x, router_logits, T, d, packed, top_k, out, workspace, ws_bytes, (cudaStream_t)stream,
                         false);
}

moe_status_t moe_layer_forward_static_act(const void* x, const float* router_logits, int T,
                                          const moe_packed_desc_t* d, const void* packed, int top_k,
                                          const float* act_gs, void* out, void* workspace, size_t ws_bytes,
                                          moe_stream_t stream) {
  if (!act_gs) return MOE_ERR_INVALID_ARG;
  return forward_checked(x, router_logits, T, d, packed, top_k, out, workspace, ws_bytes, (cudaStream_t)stream,
                         false, act_gs);
}

moe_status_t moe_calibrate_act_scales(const void* x, const float* router_logits, int T, const moe_packed_desc_t* d,
                                      const void* packed, int top_k, float* act_gs, void* workspace,
                                      size_t ws_bytes, moe_stream_t stream) {
  return forward_checked(x, router_logits, T, d, packed, top_k, nullptr, workspace, ws_bytes, (cudaStream_t)stream,
                         false, act_gs, true);
}

moe_status_t moe_layer_forward_host(const void* x_host, const float* logits_host, int T, const moe_packed_desc_t* d,
                                    const void* packed, int top_k, void* out_host, void* workspace, size_t ws_bytes,
                                    moe_stream_t stream) {
  if (!desc_ok(d) || T < 0 || top_k < 1 || top_k > kMaxTopK || top_k > d->E) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x_host || !logits_host || !out_host || !workspace)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(d->fmt, d->E, d->H, d->I, T, top_k, true);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)workspace;
  if (T > 0) {
    if (cudaMemcpyAsync(w + L.x_stage, x_host, 2 * (size_t)T * d->H, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(w + L.lg_stage, logits_host, 4 * (size_t)T * d->E, cudaMemcpyHostToDevice, s) !=
            cudaSuccess)
      return MOE_ERR_CUDA;
  }
  const moe_status_t st = forward_checked(w + L.x_stage, (const float*)(w + L.lg_stage), T, d, packed, top_k,
                                          w + L.out_stage, workspace, ws_bytes, s, true);
  if (st != MOE_OK) return st;
  if (T > 0 && cudaMemcpyAsync(out_host, w + L.out_stage, 2 * (size_t)T * d->H, cudaMemcpyDeviceToHost, s) !=
                   cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status_t moe_get_device_error(void* workspace, moe_stream_t stream, int32_t* code) {
  if (!workspace || !code) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  *code = v;
  return MOE_OK;
}

uint64_t moe_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status_t moe_time_next_step(int step, void* start, void* stop) {
  if (step != 0 && step != 1) return MOE_ERR_INVALID_ARG;
  if ((start == nullptr) != (stop == nullptr)) return MOE_ERR_INVALID_ARG;
  g_pending_events.start[step] = (cudaEvent_t)start;
  g_pending_events.stop[step] = (cudaEvent_t)stop;
  return MOE_OK;
}

const char* moe_status_string(int st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported device or request";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_FAULT: return "device-side bounds check failed";
    default: return "unknown status";
  }
}

moe_status_t moe_debug_route(const float* logits, int T, int E, int top_k, int32_t* topk_idx, float* topk_w,
                             int32_t* offsets, int32_t* perm, int32_t* inv, void* workspace, size_t ws_bytes,
                             moe_stream_t stream) {
  if (T < 0 || E < 1 || E > kMaxE || top_k < 1 || top_k > kMaxTopK || top_k > E || !workspace || !offsets)
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_idx || !topk_w || !perm || !inv)) return MOE_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(MOE_FMT_FP8_B128_W8A16, E, 128, 128, T, top_k, false);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  const moe_status_t dv = device_ok();
  if (dv != MOE_OK) return dv;
  cudaStream_t s = (cudaStream_t)stream;
  char* w = (char*)workspace;
  if (launch_route(logits, T, E, top_k, kMinRowBlock, L, w, RoutePrelude(), s) != cudaSuccess) return MOE_ERR_CUDA;
  const size_t R = (size_t)T * top_k;
  cudaError_t e = cudaMemcpyAsync(offsets, w + L.offsets, 4 * (size_t)(E + 1), cudaMemcpyDeviceToDevice, s);
  if (R) {
    if (e == cudaSuccess) e = cudaMemcpyAsync(topk_idx, w + L.topk_idx, 4 * R, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(topk_w, w + L.topk_w, 4 * R, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(perm, w + L.perm, 4 * R, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(inv, w + L.inv, 4 * R, cudaMemcpyDeviceToDevice, s);
  }
  return cuda_status(e);
}

moe_status_t moe_debug_dequant(const moe_packed_desc_t* d, const void* packed, int expert, int which, float* out,
                               moe_stream_t stream) {
  if (!desc_ok(d) || !packed || !out || expert < 0 || expert >= d->E || (which != 0 && which != 1))
    return MOE_ERR_INVALID_ARG;
  const moe_status_t dv = device_ok();
  if (dv != MOE_OK) return dv;
  return cuda_status(launch_dequant(*d, (const char*)packed, expert, which, out, (cudaStream_t)stream));
}

moe_status_t moe_debug_quant_act_static(const void* x, int T, int H, const float* gs_static, uint8_t* codes,
                                        uint8_t* scales, moe_stream_t stream) {
  if (T < 0 || H < 16 || H % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !codes || !scales || !gs_static || !aligned(x, 16) || !aligned(gs_static, 4)))
    return MOE_ERR_INVALID_ARG;
  const moe_status_t dv = device_ok();
  if (dv != MOE_OK) return dv;
  return cuda_status(launch_quant_rows((const __nv_bfloat16*)x, nullptr, 1, T, H, codes, scales, nullptr,
                                       (cudaStream_t)stream, false, 0, gs_static));
}

moe_status_t moe_debug_quant_act_fp8(const void* x, int T, int H, uint8_t* codes, float* scale_inv,
                                     moe_stream_t stream) {
  if (T < 0 || H < 128 || H % 128 != 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !codes || !scale_inv || !aligned(x, 16) || !aligned(codes, 4) || !aligned(scale_inv, 4)))
    return MOE_ERR_INVALID_ARG;
  const moe_status_t dv = device_ok();
  if (dv != MOE_OK) return dv;
  return cuda_status(
      launch_quant_fp8_rows((const __nv_bfloat16*)x, nullptr, 1, T, H, codes, scale_inv, 0, (cudaStream_t)stream));
}

moe_status_t moe_debug_quant_act(const void* x, int T, int H, uint8_t* codes, uint8_t* scales, float* gs,
                                 moe_stream_t stream) {
  if (T < 0 || H < 16 || H % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !codes || !scales || !gs || !aligned(x, 16))) return MOE_ERR_INVALID_ARG;
  const moe_status_t dv = device_ok();
  if (dv != MOE_OK) return dv;
  return cuda_status(launch_quant_rows((const __nv_bfloat16*)x, nullptr, 1, T, H, codes, scales, gs, (cudaStream_t)stream));
}

}  // extern "C"
