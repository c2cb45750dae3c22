// Test-only check of the failure-detection path: a wait that is never satisfied must give up,
// record MOE_ERR_DEVICE_TIMEOUT in the workspace error word and leave the context usable.
//
// One thread waits on an mbarrier that nothing ever arrives on, through the same bounded wait
// (tc::mbar_wait, about 2*10^9 SM cycles) that every producer / MMA / epilogue wait of the GEMM
// kernels uses; when it gives up, the kernel records the timeout exactly as a stalled GEMM CTA
// does and returns.  Nothing faults or traps.
#include "moe_internal.cuh"
#include "moe_tc.cuh"

namespace moe {

namespace {

__global__ void __launch_bounds__(32) wait_timeout_kernel(int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !tc::mbar_wait(&bar, 0, &abort_flag)) set_dev_error(err, kDevTimeout);
}

}  // namespace

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_debug_wait_timeout(void* workspace, moe_stream_t stream) {
  if (!workspace || ((uintptr_t)workspace % 256) != 0) return MOE_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((int*)workspace);
  note_launches(1);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
