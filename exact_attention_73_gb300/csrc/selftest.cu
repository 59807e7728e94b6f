// Check of the kernels' failure path: a bounded wait that runs out.
//
// Every wait inside the library's kernels polls an mbarrier for a limited
// time (mbar_wait in ptx.cuh); when the limit passes the kernel records
// ATTN_ERR_TIMEOUT in the device status word and returns. This entry point
// launches one warp whose first lane waits on a barrier that nothing ever
// completes, with a caller-chosen limit, so the whole path — the wait ending,
// the status word, attn_get_device_status — can be exercised without making
// any real kernel stall and without faulting the GPU.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/libattn.h"
#include "ops.h"
#include "ptx.cuh"

namespace attn {
namespace {

__global__ void __launch_bounds__(32) wait_runs_out(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // expects one arrival; none is ever made
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, status, limit_ns);
  __syncwarp();
}

}  // namespace
}  // namespace attn

extern "C" attn_status attn_selftest_wait_timeout(unsigned int limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 10000) return ATTN_ERR_SHAPE;
  int* status;
  attn_status s = attn::device_context(&status);
  if (s != ATTN_OK) return s;
  attn::wait_runs_out<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      status, static_cast<unsigned long long>(limit_ms) * 1000000ull);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
