// Routing for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device memory for this step: a plugin or callback run by a
// host engine that owns every device allocation and hands out no scratch for it, or a serving
// loop whose memory pool was sized at start-up and in which a cudaMalloc (with the device-wide
// synchronisation it implies) would stall the other streams.  moe_route_noalloc gives them the
// routing step (top-k, renormalised softmax, per-expert offsets and the permutation) with its
// scratch -- per-block expert histograms, per-block bases, the GEMM tile table and the error
// word -- kept in a fixed array compiled into the library.  The caller still passes the logits
// and the output buffers.
//
// The array is a file-scope __device__ variable, so every GPU that loads the library holds it
// until the process exits.  On the host its name is only a stand-in for the symbol, not a device
// address: the first call on each device asks the runtime for the address (cudaGetSymbolAddress,
// with that device current) and caches it; the kernels receive that pointer.  Every call shares
// the one array and it keeps the previous call's contents; everything a call reads is written
// earlier in the same call, and the error word is cleared by the call's first launch.  Calls
// whose work overlaps on the GPU (on different streams) race on the array.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

static __device__ __align__(256) unsigned char g_route_scratch[MOE_ROUTE_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
char* g_scratch[64];  // device address of g_route_scratch, per device ordinal

// Set-up, once per device: resolve the array's device address with that device current.
moe_status_t scratch_address(char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
    g_scratch[dev] = (char*)p;
  }
  *out = g_scratch[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_noalloc(const float* logits, int T, int E, int top_k, int32_t* topk_idx,
                                          float* topk_w, int32_t* offsets, int32_t* perm, int32_t* inv,
                                          moe_stream_t stream) {
  using namespace moe;
  if (T < 0 || E < 1 || E > kMaxE || top_k < 1 || top_k > kMaxTopK || top_k > E || !offsets)
    return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!logits || !topk_idx || !topk_w || !perm || !inv)) return MOE_ERR_INVALID_ARG;
  if (T > MOE_ROUTE_NOALLOC_MAX_TOKENS) return MOE_ERR_WORKSPACE;
  // the same routing layout the workspace-based entry points use, packed into the static array
  const WsLayout L = route_layout(E, T, top_k);
  if (L.total > (size_t)MOE_ROUTE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
  const moe_status_t dv = device_ok();
  if (dv != MOE_OK) return dv;
  char* w = nullptr;
  const moe_status_t st = scratch_address(&w);
  if (st != MOE_OK) return st;
  cudaStream_t s = (cudaStream_t)stream;
  if (launch_route(logits, T, E, top_k, kMinRowBlock, L, w, RoutePrelude(), s) != cudaSuccess) return MOE_ERR_CUDA;
  const size_t R = (size_t)T * top_k;
  cudaError_t e = cudaMemcpyAsync(offsets, w + L.offsets, 4 * (size_t)(E + 1), cudaMemcpyDeviceToDevice, s);
  if (R) {
    if (e == cudaSuccess) e = cudaMemcpyAsync(topk_idx, w + L.topk_idx, 4 * R, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(topk_w, w + L.topk_w, 4 * R, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(perm, w + L.perm, 4 * R, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(inv, w + L.inv, 4 * R, cudaMemcpyDeviceToDevice, s);
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
