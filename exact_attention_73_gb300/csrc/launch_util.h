// Host-side launch helpers shared by the library's translation units.
#pragma once
#include <atomic>

#include <cuda_runtime.h>

namespace attn {

// Raises kernel Kern's dynamic shared-memory limit to `bytes` once per device:
// the attribute lasts for the process, so later calls skip the driver call.
template <auto Kern>
cudaError_t smem_attr_once(int bytes) {
  static std::atomic<unsigned long long> done{0};   // one bit per device 0..63
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Checks once that kernel Kern is built with at least `regs` registers per
// thread for blocks of `threads`: a register split by role (setmaxnreg)
// hands out the registers the block was launched with, and a split larger
// than that would never be granted.
template <auto Kern>
cudaError_t reg_pool_once(int threads, int regs) {
  static std::atomic<int> state{0};   // 0 unknown, 1 enough, 2 too few
  int s = state.load(std::memory_order_acquire);
  if (s == 0) {
    cudaFuncAttributes fa{};
    const cudaError_t e = cudaFuncGetAttributes(&fa, Kern);
    if (e != cudaSuccess) return e;
    s = fa.numRegs >= regs && fa.maxThreadsPerBlock >= threads ? 1 : 2;
    state.store(s, std::memory_order_release);
  }
  return s == 1 ? cudaSuccess : cudaErrorLaunchOutOfResources;
}

}  // namespace attn
