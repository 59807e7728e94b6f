// C ABI of libattn: argument checks, TMA descriptors, launches.
#include <cstdint>
#include <cstdio>
#include <cmath>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/libattn.h"
#include "internal.h"
#include "ops.h"

namespace attn {

__device__ int g_status;   // written by a kernel whose bounded wait ran out

namespace {

constexpr int kMaxDev = 64;

struct DevInfo {
  bool probed = false;
  bool ok = false;
  int* status = nullptr;
};
DevInfo g_dev[kMaxDev];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

attn_status current_device(int* dev_out, int** status_out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return ATTN_ERR_NODEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  DevInfo& di = g_dev[dev];
  if (!di.probed) {
    di.probed = true;
    cudaDeviceProp p;
    if (cudaGetDeviceProperties(&p, dev) != cudaSuccess) return ATTN_ERR_NODEVICE;
    di.ok = (p.major == 10 && p.minor == 3);
    if (di.ok) {
      void* ptr = nullptr;
      if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) { di.ok = false; return ATTN_ERR_CUDA; }
      di.status = static_cast<int*>(ptr);
    }
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn) {
        di.ok = false;
        return ATTN_ERR_CUDA;
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  if (!di.ok) return ATTN_ERR_NODEVICE;
  *dev_out = dev;
  *status_out = di.status;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Encoded maps, keyed by everything the encode reads: a caller that repeats a
// call on the same buffers (a training or serving loop) skips the encode. A
// map holds only the address, shape and box, so a hit is the same map the
// encode would produce.
struct MapKey {
  int dev, dt, sw;
  const void* base;
  uint64_t dims[4], strides[3];
  uint32_t box[4];
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapEntry {
  bool used = false;
  MapKey key;
  CUtensorMap map;
};
constexpr int kMapCache = 64;
MapEntry g_maps[kMapCache];
int g_map_next = 0;
std::mutex g_map_mu;

// 4-D tiled map over a tensor whose rows hold d contiguous elements.
// dims (innermost first) and byte strides of dims 1..3; box = (box_e, b1, b2, 1).
bool encode_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, const uint64_t dims[4],
                const uint64_t strides[3], const uint32_t box[4], CUtensorMapSwizzle sw) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));   // padding takes part in the comparison
  if (cudaGetDevice(&key.dev) != cudaSuccess) return false;
  key.dt = static_cast<int>(dt);
  key.sw = static_cast<int>(sw);
  key.base = base;
  std::memcpy(key.dims, dims, sizeof(key.dims));
  std::memcpy(key.strides, strides, sizeof(key.strides));
  std::memcpy(key.box, box, sizeof(key.box));
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (const MapEntry& e : g_maps)
      if (e.used && e.key == key) {
        *m = e.map;
        return true;
      }
  }
  cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gs[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = g_encode(m, dt, 4, const_cast<void*>(base), gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  MapEntry& e = g_maps[g_map_next];
  g_map_next = (g_map_next + 1) % kMapCache;
  e.used = true;
  e.key = key;
  e.map = *m;
  return true;
}

CUtensorMapDataType tma_type(int dt) {
  switch (dt) {
    case kBF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    case kFP16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    default: return CU_TENSOR_MAP_DATA_TYPE_UINT8;
  }
}

attn_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  if (e == cudaErrorInvalidValue || e == cudaErrorLaunchOutOfResources) return ATTN_ERR_LAUNCH;
  return ATTN_ERR_CUDA;
}

attn_status check_heads(int Hq, int Hkv, int d) {
  if (Hq < 1 || Hkv < 1 || Hq > 65535) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_HEADDIM;
  if (Hq % Hkv) return ATTN_ERR_GQA;
  return ATTN_OK;
}

cudaError_t launch_fwd(int dt, int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const FwdArgs& a, int rows, int gy, int gz, cudaStream_t st) {
  switch (dt) {
    case kBF16: return launch_fwd_bf16(d, q, k, v, a, rows, gy, gz, st);
    case kFP16: return launch_fwd_fp16(d, q, k, v, a, rows, gy, gz, st);
    default: return launch_fwd_e4m3(d, q, k, v, a, rows, gy, gz, st);
  }
}

constexpr float kLog2e = 1.4426950408889634f;

}  // namespace

// Shared by the other translation units of the library.
attn_status device_context(int** status) {
  int dev;
  return current_device(&dev, status);
}

bool accum_map(CUtensorMap* m, const float* base, int d, bool packed, int B, int H, long long rows, int box_rows,
               int box_e) {
  const uint64_t esz = 4;
  const uint32_t br = static_cast<uint32_t>(box_rows);
  const uint32_t be = static_cast<uint32_t>(box_e);
  if (packed) {   // dims (d, H, T, 1)
    const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(H), static_cast<uint64_t>(rows), 1};
    const uint64_t str[3] = {d * esz, static_cast<uint64_t>(H) * d * esz, static_cast<uint64_t>(rows) * H * d * esz};
    const uint32_t box[4] = {be, 1, br, 1};
    return encode_map(m, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(rows), static_cast<uint64_t>(H),
                            static_cast<uint64_t>(B)};
  const uint64_t str[3] = {d * esz, static_cast<uint64_t>(rows) * d * esz, static_cast<uint64_t>(H) * rows * d * esz};
  const uint32_t box[4] = {be, br, 1, 1};
  return encode_map(m, base, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dims, str, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

// Map over dense [B, H, N, d] or packed [T, H, d] operands with boxes of
// `box_rows` rows and the widest swizzled inner extent (64 or 128 bytes).
bool operand_map(CUtensorMap* m, const void* base, int dt, int d, bool packed, int B, int H, long long rows,
                 int box_rows) {
  const uint64_t esz = dt == kE4M3 ? 1 : 2;
  const uint32_t box_e = static_cast<uint32_t>(fwd_box_elems(dt, d));
  const uint32_t br = static_cast<uint32_t>(box_rows);
  const CUtensorMapSwizzle sw = box_e * esz == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (packed) {   // dims (d, H, T, 1)
    const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(H), static_cast<uint64_t>(rows), 1};
    const uint64_t str[3] = {d * esz, static_cast<uint64_t>(H) * d * esz, static_cast<uint64_t>(rows) * H * d * esz};
    const uint32_t box[4] = {box_e, 1, br, 1};
    return encode_map(m, base, tma_type(dt), dims, str, box, sw);
  }
  // dims (d, N, H, B)
  const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(rows), static_cast<uint64_t>(H),
                            static_cast<uint64_t>(B)};
  const uint64_t str[3] = {d * esz, static_cast<uint64_t>(rows) * d * esz, static_cast<uint64_t>(H) * rows * d * esz};
  const uint32_t box[4] = {box_e, br, 1, 1};
  return encode_map(m, base, tma_type(dt), dims, str, box, sw);
}

}  // namespace attn

using namespace attn;

namespace {
// Dense forward with a key window (left, right); -1 means no bound.
attn_status fwd_dense(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq, int Hkv,
                      int N, int d, float scale, int win_left, int win_right, attn_dtype dtype, void* stream) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_ALIGN;
  if (B < 1 || B > 65535 || N < 1 || win_left < -1 || win_right < -1) return ATTN_ERR_SHAPE;
  attn_status s = check_heads(Hq, Hkv, d);
  if (s != ATTN_OK) return s;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_DTYPE;
  int* status;
  if ((s = device_context(&status)) != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  if (!operand_map(&tq, q, dtype, d, false, B, Hq, N, 128) || !operand_map(&tk, k, dtype, d, false, B, Hkv, N, 128) ||
      !operand_map(&tv, v, dtype, d, false, B, Hkv, N, 128))
    return ATTN_ERR_CUDA;
  FwdArgs a{};
  a.o = o;
  a.lse = lse;
  a.o_sn = d;
  a.o_sh = static_cast<long long>(N) * d;
  a.o_sb = static_cast<long long>(Hq) * N * d;
  a.l_sh = N;
  a.l_sb = static_cast<long long>(Hq) * N;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = Hq / Hkv;
  a.N = N;
  a.cu_seqlens = nullptr;
  a.scale_log2 = scale * kLog2e;
  a.win_left = win_left;
  a.win_right = win_right;
  a.causal = (win_left < 0 && win_right == 0) ? 1 : 0;
  a.status = status;
  return from_cuda(launch_fwd(dtype, d, tq, tk, tv, a, N, Hq, B, static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_NULL: return "ATTN_ERR_NULL: a required pointer is NULL";
    case ATTN_ERR_ALIGN: return "ATTN_ERR_ALIGN: a pointer is not 16-byte aligned";
    case ATTN_ERR_SHAPE: return "ATTN_ERR_SHAPE: a size is out of range";
    case ATTN_ERR_HEADDIM: return "ATTN_ERR_HEADDIM: d must be 64, 128 or 256";
    case ATTN_ERR_GQA: return "ATTN_ERR_GQA: Hq must be a positive multiple of Hkv";
    case ATTN_ERR_DTYPE: return "ATTN_ERR_DTYPE: dtype not accepted here";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE: workspace missing or too small";
    case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH: kernel resources not granted";
    case ATTN_ERR_TIMEOUT: return "ATTN_ERR_TIMEOUT: a device-side wait ran out";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA: CUDA error";
    case ATTN_ERR_NODEVICE: return "ATTN_ERR_NODEVICE: no sm_103 device is current";
  }
  return "unknown attn_status";
}

const char* attn_version(void) { return "libattn 0.1 sm_103a"; }


attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                     attn_dtype dtype, void* stream) {
  return fwd_dense(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, -1, causal ? 0 : -1, dtype, stream);
}

attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int N, int d, float scale, int window_left,
                            int window_right, attn_dtype dtype, void* stream) {
  return fwd_dense(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, window_left, window_right, dtype, stream);
}

attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens, int nseq, int T, int max_seqlen,
                            int Hq, int Hkv, int d, float scale, int causal,
                            attn_dtype dtype, void* stream) {
  if (!q || !k || !v || !o || !lse || !cu_seqlens) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(cu_seqlens))
    return ATTN_ERR_ALIGN;
  if (nseq < 1 || nseq > 65535 || T < 1 || max_seqlen < 1 || max_seqlen > T) return ATTN_ERR_SHAPE;
  attn_status s = check_heads(Hq, Hkv, d);
  if (s != ATTN_OK) return s;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_DTYPE;
  int* status;
  if ((s = device_context(&status)) != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  if (!operand_map(&tq, q, dtype, d, true, 1, Hq, T, 128) || !operand_map(&tk, k, dtype, d, true, 1, Hkv, T, 128) ||
      !operand_map(&tv, v, dtype, d, true, 1, Hkv, T, 128))
    return ATTN_ERR_CUDA;
  FwdArgs a{};
  a.o = o;
  a.lse = lse;
  a.o_sn = static_cast<long long>(Hq) * d;
  a.o_sh = d;
  a.o_sb = 0;
  a.l_sh = T;
  a.l_sb = 0;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = Hq / Hkv;
  a.N = 0;
  a.cu_seqlens = cu_seqlens;
  a.scale_log2 = scale * kLog2e;
  a.causal = causal ? 1 : 0;
  a.win_left = -1;
  a.win_right = causal ? 0 : -1;
  a.status = status;
  return from_cuda(launch_fwd(dtype, d, tq, tk, tv, a, max_seqlen, Hq, nseq, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
// Dense FP8 forward with a key window (left, right); -1 means no bound.
attn_status fwd_fp8_dense(const void* q8, const void* k8, const void* v8, const float* sq, const float* sk,
                          const float* sv, void* o, float* lse, int B, int Hq, int Hkv, int N, int d, float scale,
                          int win_left, int win_right, void* stream) {
  if (!q8 || !k8 || !v8 || !sq || !sk || !sv || !o || !lse) return ATTN_ERR_NULL;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(sq) || !aligned16(sk) ||
      !aligned16(sv) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_ALIGN;
  if (B < 1 || B > 65535 || N < 1 || win_left < -1 || win_right < -1) return ATTN_ERR_SHAPE;
  attn_status s = check_heads(Hq, Hkv, d);
  if (s != ATTN_OK) return s;
  int* status;
  if ((s = device_context(&status)) != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  const int kv_rows = fwd_e4m3_kv_rows(d);
  if (!operand_map(&tq, q8, kE4M3, d, false, B, Hq, N, 128) ||
      !operand_map(&tk, k8, kE4M3, d, false, B, Hkv, N, kv_rows) ||
      !operand_map(&tv, v8, kE4M3, d, false, B, Hkv, N, kv_rows))
    return ATTN_ERR_CUDA;
  FwdArgs a{};
  a.o = o;
  a.lse = lse;
  a.o_sn = d;
  a.o_sh = static_cast<long long>(N) * d;
  a.o_sb = static_cast<long long>(Hq) * N * d;
  a.l_sh = N;
  a.l_sb = static_cast<long long>(Hq) * N;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = Hq / Hkv;
  a.N = N;
  a.cu_seqlens = nullptr;
  a.scale_log2 = scale * kLog2e;
  a.win_left = win_left;
  a.win_right = win_right;
  a.causal = (win_left < 0 && win_right == 0) ? 1 : 0;
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.nblk = (N + 127) / 128;
  a.status = status;
  return from_cuda(launch_fwd(kE4M3, d, tq, tk, tv, a, N, Hq, B, static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" {

attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8,
                         const float* sq, const float* sk, const float* sv,
                         void* o, float* lse,
                         int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                         void* stream) {
  return fwd_fp8_dense(q8, k8, v8, sq, sk, sv, o, lse, B, Hq, Hkv, N, d, scale, -1, causal ? 0 : -1, stream);
}

attn_status attn_fwd_fp8_window(const void* q8, const void* k8, const void* v8,
                                const float* sq, const float* sk, const float* sv,
                                void* o, float* lse,
                                int B, int Hq, int Hkv, int N, int d, float scale, int window_left,
                                int window_right, void* stream) {
  return fwd_fp8_dense(q8, k8, v8, sq, sk, sv, o, lse, B, Hq, Hkv, N, d, scale, window_left, window_right,
                       stream);
}

attn_status attn_fwd_fp8_varlen(const void* q8, const void* k8, const void* v8,
                                const float* sq, const float* sk, const float* sv,
                                void* o, float* lse, const int* cu_seqlens, int nseq, int T, int max_seqlen,
                                int Hq, int Hkv, int d, float scale, int causal, void* stream) {
  if (!q8 || !k8 || !v8 || !sq || !sk || !sv || !o || !lse || !cu_seqlens) return ATTN_ERR_NULL;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(sq) || !aligned16(sk) ||
      !aligned16(sv) || !aligned16(o) || !aligned16(lse) || !aligned16(cu_seqlens))
    return ATTN_ERR_ALIGN;
  if (nseq < 1 || nseq > 65535 || T < 1 || max_seqlen < 1 || max_seqlen > T) return ATTN_ERR_SHAPE;
  attn_status s = check_heads(Hq, Hkv, d);
  if (s != ATTN_OK) return s;
  int* status;
  if ((s = device_context(&status)) != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  const int kv_rows = fwd_e4m3_kv_rows(d);
  if (!operand_map(&tq, q8, kE4M3, d, true, 1, Hq, T, 128) ||
      !operand_map(&tk, k8, kE4M3, d, true, 1, Hkv, T, kv_rows) ||
      !operand_map(&tv, v8, kE4M3, d, true, 1, Hkv, T, kv_rows))
    return ATTN_ERR_CUDA;
  FwdArgs a{};
  a.o = o;
  a.lse = lse;
  a.o_sn = static_cast<long long>(Hq) * d;
  a.o_sh = d;
  a.o_sb = 0;
  a.l_sh = T;
  a.l_sb = 0;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = Hq / Hkv;
  a.N = 0;
  a.cu_seqlens = cu_seqlens;
  a.scale_log2 = scale * kLog2e;
  a.causal = causal ? 1 : 0;
  a.win_left = -1;
  a.win_right = causal ? 0 : -1;
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.nblk = (max_seqlen + 127) / 128;
  a.status = status;
  return from_cuda(launch_fwd(kE4M3, d, tq, tk, tv, a, max_seqlen, Hq, nseq, static_cast<cudaStream_t>(stream)));
}

int attn_fwd_fp8_kv_tile(int d) { return fwd_e4m3_kv_rows(d); }

attn_status attn_get_device_status(void* stream) {
  int* status;
  attn_status s = device_context(&status);
  if (s != ATTN_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int host = 0;
  if (cudaMemcpyAsync(&host, status, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess) return ATTN_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
  if (host != 0) {
    const int zero = 0;
    if (cudaMemcpyAsync(status, &zero, sizeof(int), cudaMemcpyHostToDevice, st) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return ATTN_ERR_CUDA;
    return host == kDevTimeout ? ATTN_ERR_TIMEOUT : ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

}  // extern "C"

namespace {
attn_status quantize(const void* x, attn_dtype in_dtype, void* x8, float* scales, int B, int H, int N, int d,
                     const float* rope_cos, const float* rope_sin, const int8_t* hadamard_signs, void* stream) {
  if (!x || !x8 || !scales) return ATTN_ERR_NULL;
  if (!aligned16(x) || !aligned16(x8) || !aligned16(scales) || (hadamard_signs && !aligned16(hadamard_signs)) ||
      (rope_cos && !aligned16(rope_cos)) || (rope_sin && !aligned16(rope_sin)))
    return ATTN_ERR_ALIGN;
  if (B < 1 || B > 65535 || H < 1 || H > 65535 || N < 1) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_HEADDIM;
  if (in_dtype != ATTN_BF16 && in_dtype != ATTN_FP16) return ATTN_ERR_DTYPE;
  int* status;
  attn_status s = device_context(&status);
  if (s != ATTN_OK) return s;
  const float inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  return from_cuda(launch_quant_fp8(x, in_dtype, static_cast<uint8_t*>(x8), scales, B, H, N, d, hadamard_signs,
                                    inv_sqrt_d, rope_cos, rope_sin, static_cast<cudaStream_t>(stream)));
}
}  // namespace

extern "C" attn_status attn_quantize_fp8(const void* x, attn_dtype in_dtype, void* x8, float* scales,
                                         int B, int H, int N, int d, const int8_t* hadamard_signs,
                                         void* stream) {
  return quantize(x, in_dtype, x8, scales, B, H, N, d, nullptr, nullptr, hadamard_signs, stream);
}

extern "C" attn_status attn_quantize_fp8_varlen(const void* x, attn_dtype in_dtype, void* x8, float* scales,
                                                const int* cu_seqlens, int nseq, int T, int max_seqlen, int H,
                                                int d, const int8_t* hadamard_signs, void* stream) {
  if (!x || !x8 || !scales || !cu_seqlens) return ATTN_ERR_NULL;
  if (!aligned16(x) || !aligned16(x8) || !aligned16(scales) || !aligned16(cu_seqlens) ||
      (hadamard_signs && !aligned16(hadamard_signs)))
    return ATTN_ERR_ALIGN;
  if (nseq < 1 || nseq > 65535 || T < 1 || max_seqlen < 1 || max_seqlen > T || H < 1 || H > 65535)
    return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_HEADDIM;
  if (in_dtype != ATTN_BF16 && in_dtype != ATTN_FP16) return ATTN_ERR_DTYPE;
  int* status;
  attn_status s = device_context(&status);
  if (s != ATTN_OK) return s;
  const float inv_sqrt_d = static_cast<float>(1.0 / std::sqrt(static_cast<double>(d)));
  return from_cuda(launch_quant_fp8_varlen(x, in_dtype, static_cast<uint8_t*>(x8), scales, cu_seqlens, nseq,
                                           max_seqlen, H, d, hadamard_signs, inv_sqrt_d,
                                           static_cast<cudaStream_t>(stream)));
}

extern "C" attn_status attn_quantize_fp8_rope(const void* x, attn_dtype in_dtype, void* x8, float* scales,
                                              int B, int H, int N, int d, const float* rope_cos,
                                              const float* rope_sin, const int8_t* hadamard_signs, void* stream) {
  if (!rope_cos || !rope_sin) return ATTN_ERR_NULL;
  return quantize(x, in_dtype, x8, scales, B, H, N, d, rope_cos, rope_sin, hadamard_signs, stream);
}
