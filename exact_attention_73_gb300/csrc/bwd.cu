// Backward launchers: D = rowsum(dO o O) with the dQ accumulator cleared,
// the tcgen05 main kernel (head dim 64, 128 or 256), and the FP32 -> BF16/FP16
// dQ conversion.
//
// The two helper kernels are HBM-bound streams: one warp per row of d
// elements (pre) and four elements per thread (convert), coalesced.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "bwd_kernel.cuh"
#include "ops.h"

namespace attn {

namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x);
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }
template <>
__device__ __forceinline__ float to_f<__half>(__half x) { return __half2float(x); }

// rows = B*Hq*N (dense, row r = (b*Hq + h)*N + n) or T*Hq (packed, r = t*Hq + h).
template <typename T, int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const T* __restrict__ o, const T* __restrict__ dout,
                                                      float* __restrict__ dvec, float* __restrict__ dq_acc,
                                                      long long rows, int Hq, int T_tokens, int packed) {
  constexpr int c = D / 32;
  const long long r = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const T* po = o + r * D + lane * c;
  const T* pd = dout + r * D + lane * c;
  float acc = 0.f;
#pragma unroll
  for (int e = 0; e < c; ++e) acc = fmaf(to_f(po[e]), to_f(pd[e]), acc);
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (dq_acc) {   // absent for the deterministic backward (dQ written directly)
    float* z = dq_acc + r * D + lane * c;
    if constexpr (c % 4 == 0) {
#pragma unroll
      for (int e = 0; e < c / 4; ++e) reinterpret_cast<float4*>(z)[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      static_assert(c % 2 == 0, "row chunk per lane");
#pragma unroll
      for (int e = 0; e < c / 2; ++e) reinterpret_cast<float2*>(z)[e] = make_float2(0.f, 0.f);
    }
  }
  if (lane == 0) {
    long long idx = r;
    if (packed) idx = static_cast<long long>(r % Hq) * T_tokens + r / Hq;
    dvec[idx] = acc;
  }
}

template <typename T>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc, T* __restrict__ dq,
                                                         long long n4, float scale) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n4) return;
  const float4 x = reinterpret_cast<const float4*>(acc)[i];
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x.x * scale, x.y * scale);
    __nv_bfloat162 b = __floats2bfloat162_rn(x.z * scale, x.w * scale);
    reinterpret_cast<uint2*>(dq)[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  } else {
    __half2 a = __floats2half2_rn(x.x * scale, x.y * scale);
    __half2 b = __floats2half2_rn(x.z * scale, x.w * scale);
    reinterpret_cast<uint2*>(dq)[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
}

// Tail split. Without masks every unit (key tile x DSPLIT, KV head, batch)
// walks the same query tiles, so the grid runs in waves of one unit per SM
// and the last wave holds units % SMs of them. When that remainder R is at
// most half the SMs, the common instance runs the first units - R as whole
// waves (a 1-D grid) and the split instance the last R as 2R CTAs in
// clusters of two, each CTA walking half of its unit's query tiles: the last
// wave takes about half as long. The two halves' dK and dV are summed in a
// fixed order (deterministic).
int tail_split_units(const BwdArgs& a, long long units, int per_head, int sms) {
  if (a.cu_seqlens != nullptr || a.win_left >= 0 || a.win_right >= 0) return 0;
  if (sms < 2 || static_cast<long long>(a.group) * per_head < 2) return 0;
  const long long r = units % sms;
  return 2 * r <= sms ? static_cast<int>(r) : 0;
}

// Short unmasked rows run persistent: one CTA per SM walks the units, so a
// unit's dV/dK write-out overlaps the next unit's first products and the
// CTA set-up is paid once (at d = 64 also the next unit's K/V load, from a
// second buffer). That pays while a unit holds few query tiles (N = 512:
// 6 % at d = 128, 13 % at d = 64); from about N = 1024 on the unit's own
// walk hides it and the walk's extra state costs as much as it saves.
constexpr int kBwdPersistMaxRows = 768;

template <int DT, int D, bool kDQ>
cudaError_t launch_main(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q, const CUtensorMap& d,
                        const CUtensorMap& dq, const BwdArgs& a, int max_len, int nz, cudaStream_t st) {
  using C = BwdCfg<DT, D>;
  // At d = 256 the kSplit instance runs every grid: its build of the common
  // path measured 3 % faster there (at d = 64 9 % slower, so d = 64 and 128
  // use the instance without the split code for their whole-unit grids).
  constexpr bool kSplitAll = D == 256;
  const int tiles_x = (max_len + C::BC - 1) / C::BC * C::DSPLIT;
  const long long units = static_cast<long long>(tiles_x) * a.Hkv * nz;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if constexpr (kDQ && D <= 128) {
    if (a.cu_seqlens == nullptr && a.win_left < 0 && a.win_right < 0 && max_len <= kBwdPersistMaxRows &&
        units > sms && units <= INT32_MAX) {
      BwdArgs g = a;
      g.tiles_x = tiles_x;
      g.unit0 = 0;
      g.nsplit = 1;
      g.units = static_cast<int>(units);
      return launch_bwd_persist<DT, D>(k, v, q, d, dq, g, sms, st);
    }
  }
  const int tail = units <= INT32_MAX ? tail_split_units(a, units, (a.N + C::BR - 1) / C::BR, sms) : 0;
  auto whole = [&](dim3 grid, const BwdArgs& g) -> cudaError_t {
    if constexpr (kSplitAll) {
      return launch_bwd_split<DT, D, kDQ>(k, v, q, d, dq, g, 0, grid, st);
    } else {
      cudaError_t r = smem_attr_once<bwd_kernel<DT, D, kDQ, false>>(C::SMEM_BYTES);
      if (r != cudaSuccess) return r;
      if ((r = reg_pool_once<bwd_kernel<DT, D, kDQ, false>>(C::NTHREADS, C::kRegsSplit)) != cudaSuccess) return r;
      bwd_kernel<DT, D, kDQ, false><<<grid, C::NTHREADS, C::SMEM_BYTES, st>>>(k, v, q, d, dq, g);
      return cudaGetLastError();
    }
  };
  BwdArgs g = a;
  g.tiles_x = 0;
  g.unit0 = 0;
  g.nsplit = 1;
  if (tail == 0) return whole(dim3(tiles_x, a.Hkv, nz), g);
  g.tiles_x = tiles_x;
  if (units > tail && (e = whole(dim3(static_cast<unsigned>(units - tail)), g)) != cudaSuccess) return e;
  g.unit0 = static_cast<int>(units - tail);
  g.nsplit = 2;
  return launch_bwd_split<DT, D, kDQ>(k, v, q, d, dq, g, tail, dim3(), st);
}

template <bool kDQ>
cudaError_t launch_main_dt(int dt, int hd, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                           const CUtensorMap& d, const CUtensorMap& dq, const BwdArgs& a, int max_len, int nz,
                           cudaStream_t st) {
  if (hd == 128)
    return dt == kBF16 ? launch_main<kBF16, 128, kDQ>(k, v, q, d, dq, a, max_len, nz, st)
                       : launch_main<kFP16, 128, kDQ>(k, v, q, d, dq, a, max_len, nz, st);
  if (hd == 64)
    return dt == kBF16 ? launch_main<kBF16, 64, kDQ>(k, v, q, d, dq, a, max_len, nz, st)
                       : launch_main<kFP16, 64, kDQ>(k, v, q, d, dq, a, max_len, nz, st);
  if (hd == 256 && kDQ)
    return dt == kBF16 ? launch_main<kBF16, 256, true>(k, v, q, d, dq, a, max_len, nz, st)
                       : launch_main<kFP16, 256, true>(k, v, q, d, dq, a, max_len, nz, st);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_bwd_pre(int dt, int d, const void* o, const void* dout, float* dvec, float* dq_acc, long long rows,
                           int Hq, int T_tokens, int packed, cudaStream_t st) {
  const dim3 grid(static_cast<unsigned>((rows + 7) / 8));
  const auto* ob = static_cast<const __nv_bfloat16*>(o);
  const auto* db = static_cast<const __nv_bfloat16*>(dout);
  const auto* oh = static_cast<const __half*>(o);
  const auto* dh = static_cast<const __half*>(dout);
  if (d == 128) {
    if (dt == kBF16) bwd_pre_kernel<__nv_bfloat16, 128><<<grid, 256, 0, st>>>(ob, db, dvec, dq_acc, rows, Hq, T_tokens, packed);
    else bwd_pre_kernel<__half, 128><<<grid, 256, 0, st>>>(oh, dh, dvec, dq_acc, rows, Hq, T_tokens, packed);
  } else if (d == 64) {
    if (dt == kBF16) bwd_pre_kernel<__nv_bfloat16, 64><<<grid, 256, 0, st>>>(ob, db, dvec, dq_acc, rows, Hq, T_tokens, packed);
    else bwd_pre_kernel<__half, 64><<<grid, 256, 0, st>>>(oh, dh, dvec, dq_acc, rows, Hq, T_tokens, packed);
  } else if (d == 256) {
    if (dt == kBF16) bwd_pre_kernel<__nv_bfloat16, 256><<<grid, 256, 0, st>>>(ob, db, dvec, dq_acc, rows, Hq, T_tokens, packed);
    else bwd_pre_kernel<__half, 256><<<grid, 256, 0, st>>>(oh, dh, dvec, dq_acc, rows, Hq, T_tokens, packed);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_bwd_main(int dt, int d, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                            const CUtensorMap& dout, const CUtensorMap& dq_acc, const BwdArgs& a, int max_len, int nz,
                            cudaStream_t st) {
  return launch_main_dt<true>(dt, d, k, v, q, dout, dq_acc, a, max_len, nz, st);
}

int bwd_dq_rows(int d) {
  return d == 64 ? BwdCfg<kBF16, 64>::DQ_ROWS : d == 256 ? BwdCfg<kBF16, 256>::DQ_ROWS : BwdCfg<kBF16, 128>::DQ_ROWS;
}
int bwd_dq_dims(int d) {
  return d == 64 ? BwdCfg<kBF16, 64>::DH : d == 256 ? BwdCfg<kBF16, 256>::DH : BwdCfg<kBF16, 128>::DH;
}

cudaError_t launch_bwd_dkdv(int dt, int d, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                            const CUtensorMap& dout, const BwdArgs& a, int max_len, int nz, cudaStream_t st) {
  // the dQ map is never read without the dQ product; K's map stands in for it
  return launch_main_dt<false>(dt, d, k, v, q, dout, k, a, max_len, nz, st);
}

cudaError_t launch_dq_convert(int dt, const float* acc, void* dq, long long n, float scale, cudaStream_t st) {
  const long long n4 = n / 4;
  const dim3 grid(static_cast<unsigned>((n4 + 255) / 256));
  if (dt == kBF16)
    dq_convert_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(acc, static_cast<__nv_bfloat16*>(dq), n4, scale);
  else
    dq_convert_kernel<__half><<<grid, 256, 0, st>>>(acc, static_cast<__half*>(dq), n4, scale);
  return cudaGetLastError();
}

}  // namespace attn
