// FP8 decode over a block-quantised KV cache (split-KV): the forward kernel in
// its decode form writes one partial result per split, then a combine kernel
// merges the splits of every (batch, query head) by their log-sum-exp
// weights: LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
// The decode step reads the whole cache once: it is HBM-bound.
#include <climits>
#include <cmath>
#include <cstdint>

#include <cuda_bf16.h>

#include "../../include/libattn.h"
#include "decode_kernel.cuh"
#include "internal.h"
#include "ops.h"

namespace attn {

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// one CTA per (batch, query head), one thread per head-dim element
__global__ void __launch_bounds__(256) decode_combine_kernel(const float* __restrict__ o_part,
                                                             const float* __restrict__ lse_part,
                                                             __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
                                                             int splits, int rows, int d) {
  const int r = blockIdx.x, t = threadIdx.x;
  float mx = -INFINITY;
  for (int s = 0; s < splits; ++s) mx = fmaxf(mx, lse_part[static_cast<long long>(s) * rows + r]);
  if (mx == -INFINITY) {   // no key at all (empty cache): O = 0, LSE = -inf
    o[static_cast<long long>(r) * d + t] = __float2bfloat16(0.f);
    if (t == 0) lse[r] = -INFINITY;
    return;
  }
  float tot = 0.f, acc = 0.f;
  for (int s = 0; s < splits; ++s) {
    const float w = expf(lse_part[static_cast<long long>(s) * rows + r] - mx);
    tot += w;
    acc += w * o_part[(static_cast<long long>(s) * rows + r) * d + t];
  }
  o[static_cast<long long>(r) * d + t] = __float2bfloat16(acc / tot);
  if (t == 0) lse[r] = mx + logf(tot);
}

// persistent: at most one CTA per SM, each walking the (split, KV head,
// batch) items with a stride of the grid size
template <int D>
cudaError_t launch_decode_inst(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdArgs& a,
                               int splits, int items, cudaStream_t st) {
  using C = DecCfg<D>;
  auto kern = decode_kernel<D>;
  cudaError_t e = smem_attr_once<decode_kernel<D>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  const int grid = items < sms ? items : sms;
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, st>>>(q, k, v, a, splits, items);
  return cudaGetLastError();
}

}  // namespace

}  // namespace attn

using namespace attn;

extern "C" size_t attn_decode_fp8_workspace_size(int B, int Hq, int d, int num_splits) {
  if (B < 1 || Hq < 1 || d < 1 || num_splits < 1) return 0;
  const size_t rows = static_cast<size_t>(num_splits) * B * Hq;
  return (rows * d * 4 + 255) / 256 * 256 + (rows * 4 + 255) / 256 * 256;
}

extern "C" attn_status attn_decode_fp8(const void* q8, const float* sq, const void* k8, const void* v8,
                                       const float* sk, const float* sv, const int* seqlens, void* o, float* lse,
                                       void* workspace, size_t ws_bytes, int B, int Hq, int Hkv, int Nmax, int d,
                                       float scale, int num_splits, void* stream) {
  if (!q8 || !sq || !k8 || !v8 || !sk || !sv || !o || !lse || !workspace) return ATTN_ERR_NULL;
  const void* ptrs[] = {q8, sq, k8, v8, sk, sv, o, lse, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return ATTN_ERR_ALIGN;
  if (seqlens && !aligned16(seqlens)) return ATTN_ERR_ALIGN;
  if (B < 1 || B > 65535 || Nmax < 1 || Hq < 1 || Hkv < 1 || Hkv > 65535) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_HEADDIM;
  if (Hq % Hkv) return ATTN_ERR_GQA;
  const int g = Hq / Hkv;
  const int ntiles = (Nmax + 127) / 128;
  if (g > 128 || num_splits < 1 || num_splits > ntiles) return ATTN_ERR_SHAPE;
  // one combine CTA per (sequence, query head): the row count is an int
  if (static_cast<long long>(B) * Hq > INT_MAX) return ATTN_ERR_SHAPE;
  if (ws_bytes < attn_decode_fp8_workspace_size(B, Hq, d, num_splits)) return ATTN_ERR_WORKSPACE;
  int* status;
  attn_status s = device_context(&status);
  if (s != ATTN_OK) return s;
  CUtensorMap tq, tk, tv;
  // q [B, Hq, d] is the same memory as [B, Hkv, g, d]: one 128-row Q tile per group
  if (!operand_map(&tq, q8, kE4M3, d, false, B, Hkv, g, 128) ||
      !operand_map(&tk, k8, kE4M3, d, false, B, Hkv, Nmax, 128) ||
      !operand_map(&tv, v8, kE4M3, d, false, B, Hkv, Nmax, 128))
    return ATTN_ERR_CUDA;
  const int tps = (ntiles + num_splits - 1) / num_splits;
  const size_t rows = static_cast<size_t>(num_splits) * B * Hq;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + (rows * d * 4 + 255) / 256 * 256);
  FwdArgs a{};
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = g;
  a.N = Nmax;
  a.cu_seqlens = nullptr;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.causal = 0;
  a.win_left = -1;
  a.win_right = -1;
  a.sq = sq;
  a.sk = sk;
  a.sv = sv;
  a.nblk = ntiles;
  a.seqlens = seqlens;
  a.tiles_per_split = tps;
  a.batch = B;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.status = status;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int splits = (ntiles + tps - 1) / tps;   // splits that hold a tile of a full-length cache
  const long long items = static_cast<long long>(splits) * Hkv * B;
  if (items > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  cudaError_t e;
  switch (d) {
    case 64: e = launch_decode_inst<64>(tq, tk, tv, a, splits, static_cast<int>(items), st); break;
    case 128: e = launch_decode_inst<128>(tq, tk, tv, a, splits, static_cast<int>(items), st); break;
    default: e = launch_decode_inst<256>(tq, tk, tv, a, splits, static_cast<int>(items), st); break;
  }
  if (e == cudaSuccess) {
    decode_combine_kernel<<<static_cast<unsigned>(B * Hq), d, 0, st>>>(o_part, lse_part,
                                                                       static_cast<__nv_bfloat16*>(o), lse, splits,
                                                                       B * Hq, d);
    e = cudaGetLastError();
  }
  if (e == cudaSuccess) return ATTN_OK;
  return e == cudaErrorInvalidValue || e == cudaErrorLaunchOutOfResources ? ATTN_ERR_LAUNCH : ATTN_ERR_CUDA;
}
