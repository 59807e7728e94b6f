// Backward entry point for callers that cannot allocate device memory.
//
// attn_bwd needs a caller-provided workspace (the FP32 dQ accumulator and
// D = rowsum(dO o O)). Some callers cannot make that allocation: a process
// whose device memory is already owned by another allocator (a framework's
// caching pool that has reserved almost all of HBM, so cudaMalloc fails or
// fragments the pool), or a serving path that must not allocate once it is
// running (cudaMalloc/cudaFree can synchronise the whole device and stall
// every other stream). attn_bwd_noalloc gives them the same backward with its
// workspace in a fixed array of device memory that belongs to this library.
//
// The array is a file-scope __device__ object of ATTN_BWD_NOALLOC_MAX_BYTES.
// Every GPU on which this code is loaded holds it until the process exits.
// Host code cannot pass the array's name to a kernel (on the host it is only
// a stand-in symbol, not a device address), so the first call on each device
// looks up its device address with cudaGetSymbolAddress while that device is
// current, and caches it. Make that first call before any stream capture.
// With lazy module loading (CUDA's default) that lookup is also when the
// driver loads this file's module and reserves the array on the device, so
// the first call can fail with ATTN_ERR_CUDA if the device is already full:
// callers whose memory pool takes nearly all of HBM should make one call at
// start-up, before the pool reserves its memory.
// All calls share the one array: calls whose kernels overlap on the GPU (two
// streams, or two host threads) race on it and give wrong results. The
// backward's first kernel clears the dQ accumulator and writes D, so nothing
// left by an earlier call leaks into the next one.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/libattn.h"
#include "ops.h"

namespace {

constexpr size_t kScratchBytes = ATTN_BWD_NOALLOC_MAX_BYTES;

static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_bwd_scratch on the current device (looked up once).
attn_status scratch_on_current_device(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_NODEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_scratch) != cudaSuccess || p == nullptr) return ATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                        const float* lse, const void* dout, void* dq, void* dk, void* dv,
                                        int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                                        attn_dtype dtype, void* stream) {
  // Every argument error, a problem too large for the array included, is
  // reported before the array's address is looked up. q stands in for the
  // workspace pointer here (the array itself is non-null and aligned).
  attn_status s = attn::bwd_check_dense(q, k, v, o, lse, dout, dq, dk, dv, q, kScratchBytes, B, Hq, Hkv, N, d,
                                        dtype);
  if (s != ATTN_OK) return s;
  // a device that is not sm_103 is reported as every other entry point does
  int* status = nullptr;
  if ((s = attn::device_context(&status)) != ATTN_OK) return s;
  void* ws = nullptr;
  if ((s = scratch_on_current_device(&ws)) != ATTN_OK) return s;
  return attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, ws, kScratchBytes, B, Hq, Hkv, N, d, scale, causal, dtype,
                  stream);
}
