// Block quantisation to E4M3 with optional incoherent processing.
//
// FlashAttention-3 (zenmind.me summary) §3.5: one scale per 128-row block
// of each (batch, head); before quantising Q and K, each row may be rotated
// by diag(random signs) * Hadamard / sqrt(d) to spread outliers.
// m.xxqk.cn FA3 walkthrough §4.2: power-of-two scale factors.
//
// One CTA per (128-row block, head, batch). Without rotation and RoPE a
// lighter instance keeps the inputs packed (quant_plain_kernel). Otherwise a
// lane holds EPL consecutive
// elements of a row (d / EPL lanes per row): EPL = 32 for the rotation
// instance (8 warps of 16 rows, 16-byte loads), EPL = d / 32 for
// the RoPE instance (a warp per row, 16 warps of 8 rows). The fast
// Walsh-Hadamard transform runs in FP32 in radix-2 stages of stride 1, 2, 4,
// ...: strides below EPL inside a lane, larger ones across the lanes of a row
// with shuffles; each butterfly computes a + b and a - b exactly once, so the
// result does not depend on which lane holds which operand. This kernel is
// HBM-bound: it reads 2 bytes and writes 1 byte per element.
// Optional rotary position embedding first (kRope; the paper fuses
// quantisation into the RoPE step that produces Q and K): rotate-half pairs
// (i, i + d/2) with the caller's cos/sin tables [N, d/2]; the first half of a
// row sits in the first half of the row's lanes, so a lane's partner is half
// the row's lanes away. Each product and sum is rounded on its own (no fused multiply-add).
#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ops.h"
#include "ptx.cuh"

namespace attn {

namespace {

// Radix-2 FWHT of one row held as EPL consecutive elements per lane over
// D / EPL lanes; li is the lane's position within its row.
template <int D, int EPL>
__device__ __forceinline__ void fwht_row(float (&x)[EPL], int li) {
#pragma unroll
  for (int h = 1; h < D; h <<= 1) {
    if (h < EPL && (h == 1 || D < 128)) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        if ((e & h) == 0) {
          const float a = x[e], b = x[e + h];
          x[e] = a + b;
          x[e + h] = a - b;
        }
      }
    } else if (h < EPL) {
      // d >= 128: two butterflies (e, e + h), (e + 1, e + h + 1) per packed
      // FP32 pair (d = 128: 37.5 -> 35.5 us per call; d = 64 measured a step
      // slower); a - b as a fused multiply-add with b * (-1) exact: rounded
      // once, as the plain subtract is
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        if ((e & h) == 0) {
          const float2 a = make_float2(x[e], x[e + 1]), b = make_float2(x[e + h], x[e + h + 1]);
          const float2 sum = fadd2(a, b);
          const float2 dif = ffma2(b, make_float2(-1.f, -1.f), a);
          x[e] = sum.x;
          x[e + 1] = sum.y;
          x[e + h] = dif.x;
          x[e + h + 1] = dif.y;
        }
      }
    } else {
      const int lm = h / EPL;
      // the upper lane of a pair computes other - x, the lower x + other:
      // one fused multiply-add with x * (-1 or 1) exact, so the sum is
      // rounded once, as the plain add or subtract would be
      const float sgn = (li & lm) != 0 ? -1.f : 1.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, x[e], lm);
        x[e] = fmaf(x[e], sgn, other);
      }
    }
  }
}

// Largest e with amax * 2^e <= 448 (448 = 0.875 * 2^9), 0 for amax == 0.
__device__ __forceinline__ int e4m3_scale_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  int k;
  const float m = frexpf(amax, &k);   // amax = m * 2^k, m in [0.5, 1)
  return (m <= 0.875f) ? 9 - k : 8 - k;
}

template <typename T>
__device__ __forceinline__ float to_f32(uint32_t bits16) {
  if constexpr (std::is_same<T, __nv_bfloat16>::value) return __uint_as_float(bits16 << 16);
  else return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// Where a CTA's 128-row block lives. Dense [B, H, N, d]: grid (blocks, H,
// B). Packed [T, H, d] (cu_seqlens non-null): grid (blocks of the longest
// sequence, H, sequences), each sequence blocked from its own first row.
// Either way block blk of (batch or sequence z, head h) has factor index
// (z * H + h) * gridDim.x + blk.
struct QuantGeom {
  int H, N;
  const int* cu_seqlens;
};
struct QuantBlock {
  long long row0;   // element offset of row 0 of this (sequence or batch, head)
  long long rs;     // elements from one row to the next
  long long si;     // factor index of this block
  int L;            // rows of this (sequence or batch, head)
};
// kLayout: 0 dense, 1 packed, 2 decided by g.cu_seqlens at run time
template <int D, int kLayout = 2>
__device__ __forceinline__ QuantBlock quant_block(const QuantGeom& g, int blk, int h, int z) {
  QuantBlock q;
  if (kLayout == 1 || (kLayout == 2 && g.cu_seqlens != nullptr)) {
    const int seq0 = g.cu_seqlens[z];
    q.L = g.cu_seqlens[z + 1] - seq0;
    q.row0 = (static_cast<long long>(seq0) * g.H + h) * D;
    q.rs = static_cast<long long>(g.H) * D;
  } else {
    q.L = g.N;
    q.row0 = (static_cast<long long>(z) * g.H + h) * g.N * D;
    q.rs = D;
  }
  q.si = (static_cast<long long>(z) * g.H + h) * gridDim.x + blk;
  return q;
}

// Layout per instance. The rotation instance: a lane holds 32 consecutive
// elements of a row (d/32 lanes per row), so five Hadamard stages run in
// registers, with 16-byte loads; 8 warps of 16 rows. The RoPE
// instance: a warp holds one row at a time (d/32 elements per lane); 16 warps
// of 8 rows, which keeps more cos/sin table loads in flight (measured faster
// for it than the 32-per-lane layout).
template <int D, bool kRope>
__host__ __device__ constexpr int quant_epl() { return kRope ? D / 32 : 32; }
template <int D, bool kRope>
__host__ __device__ constexpr int quant_threads() { return kRope ? 512 : 256; }

// n consecutive 16-bit elements (n = 2, 4 or a multiple of 8) as floats
template <typename T, int n>
__device__ __forceinline__ void load_row_part(const T* src, float* v) {
  if constexpr (n % 8 == 0) {
#pragma unroll
    for (int q = 0; q < n / 8; ++q) {
      const uint4 w = reinterpret_cast<const uint4*>(src)[q];
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        v[8 * q + 2 * u] = to_f32<T>(wv[u] & 0xFFFFu);
        v[8 * q + 2 * u + 1] = to_f32<T>(wv[u] >> 16);
      }
    }
  } else {
    uint32_t wv[n / 2];
    if constexpr (n == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(src);
      wv[0] = w.x;
      wv[1] = w.y;
    } else {
      wv[0] = *reinterpret_cast<const uint32_t*>(src);
    }
#pragma unroll
    for (int u = 0; u < n / 2; ++u) {
      v[2 * u] = to_f32<T>(wv[u] & 0xFFFFu);
      v[2 * u + 1] = to_f32<T>(wv[u] >> 16);
    }
  }
}

template <typename T, int D, bool kRope>
__global__ void __launch_bounds__(quant_threads<D, kRope>()) quant_kernel(const T* __restrict__ x, uint8_t* __restrict__ x8,
                                                             float* __restrict__ scales, const QuantGeom geo,
                                                             const int8_t* __restrict__ signs, float inv_sqrt_d,
                                                             const float* __restrict__ rope_cos,
                                                             const float* __restrict__ rope_sin) {
  constexpr int EPL = quant_epl<D, kRope>();   // elements per lane
  constexpr int R = D / EPL;           // lanes per row
  constexpr int RP = 32 / R;           // rows per warp at a time
  constexpr int NW = quant_threads<D, kRope>() / 32;
  constexpr int RPW = 128 / NW;        // rows per warp
  static_assert(RPW >= RP && RPW % RP == 0, "a warp's rows must cover whole rows of lanes");
  constexpr int NPASS = RPW / RP;
  __shared__ float red[NW];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int lr = lane / R, li = lane % R;
  const int blk = blockIdx.x;
  const QuantBlock qb = quant_block<D>(geo, blk, blockIdx.y, blockIdx.z);
  if (blk * 128 >= qb.L) return;   // a packed sequence shorter than the longest
  const int N = qb.L;
  const int row0 = blk * 128 + warp * RPW;
  float v[NPASS][EPL];
  float amax = 0.f;
  // Without RoPE and with at most two passes (d <= 128) every pass's 16-byte
  // loads are issued before the first pass is transformed, so their
  // latencies overlap (at d = 256 the four passes' raw values would not fit
  // in registers next to the transformed ones).
  constexpr bool kPre = !kRope && NPASS <= 2;
  constexpr int NRAW = kPre ? EPL / 8 : 1;
  uint4 raw[kPre ? NPASS : 1][NRAW];
  if constexpr (kPre) {
#pragma unroll
    for (int p = 0; p < NPASS; ++p) {
      const int row = row0 + p * RP + lr;
#pragma unroll
      for (int q = 0; q < NRAW; ++q)
        raw[p][q] = row < N ? reinterpret_cast<const uint4*>(x + qb.row0 + row * qb.rs + li * EPL)[q]
                            : make_uint4(0, 0, 0, 0);
    }
  }
#pragma unroll
  for (int p = 0; p < NPASS; ++p) {
    const int row = row0 + p * RP + lr;
    const bool valid = row < N;
    if constexpr (kPre) {
#pragma unroll
      for (int q = 0; q < NRAW; ++q) {
        const uint32_t wv[4] = {raw[p][q].x, raw[p][q].y, raw[p][q].z, raw[p][q].w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          v[p][8 * q + 2 * u] = to_f32<T>(wv[u] & 0xFFFFu);
          v[p][8 * q + 2 * u + 1] = to_f32<T>(wv[u] >> 16);
        }
      }
    } else if (valid) {
      load_row_part<T, EPL>(x + qb.row0 + row * qb.rs + li * EPL, v[p]);
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[p][e] = 0.f;
    }
    if constexpr (kRope) {   // partner d/2 elements away: R/2 lanes away; every lane shuffles
      float cs[EPL], sn[EPL];
      if (valid) {
        const long long t = static_cast<long long>(row) * (D / 2) + (li % (R / 2)) * EPL;
        if constexpr (EPL % 4 == 0) {
#pragma unroll
          for (int q = 0; q < EPL / 4; ++q) {
            const float4 a = reinterpret_cast<const float4*>(rope_cos + t)[q];
            const float4 bq = reinterpret_cast<const float4*>(rope_sin + t)[q];
            cs[4 * q] = a.x; cs[4 * q + 1] = a.y; cs[4 * q + 2] = a.z; cs[4 * q + 3] = a.w;
            sn[4 * q] = bq.x; sn[4 * q + 1] = bq.y; sn[4 * q + 2] = bq.z; sn[4 * q + 3] = bq.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            cs[e] = rope_cos[t + e];
            sn[e] = rope_sin[t + e];
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) cs[e] = sn[e] = 0.f;
      }
      const bool second = li >= R / 2;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, v[p][e], R / 2);
        v[p][e] = second ? __fadd_rn(__fmul_rn(v[p][e], cs[e]), __fmul_rn(other, sn[e]))
                         : __fsub_rn(__fmul_rn(v[p][e], cs[e]), __fmul_rn(other, sn[e]));
      }
    }
    if (signs) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[p][e] *= static_cast<float>(signs[li * EPL + e]);
      fwht_row<D, EPL>(v[p], li);
#pragma unroll
      for (int e = 0; e < EPL; ++e) v[p][e] *= inv_sqrt_d;
    }
#pragma unroll
    for (int e = 0; e + 1 < EPL; e += 2) amax = fmax3(amax, fabsf(v[p][e]), fabsf(v[p][e + 1]));
    if constexpr (EPL % 2 != 0) amax = fmaxf(amax, fabsf(v[p][EPL - 1]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) amax = fmaxf(amax, red[w]);
  const int e = e4m3_scale_exponent(amax);
  if (threadIdx.x == 0) scales[qb.si] = ldexpf(1.f, -e);
  // x * 2^e in one multiply when 2^e is a normal float (exact either way:
  // a power-of-two scaling), else in two steps
  const int e1 = e / 2, e2 = e - e1;
  const bool one = e >= -126 && e <= 127;
  if (!one) {
    const float fa = ldexpf(1.f, e1);
#pragma unroll
    for (int p = 0; p < NPASS; ++p)
#pragma unroll
      for (int q = 0; q < EPL; ++q) v[p][q] *= fa;
  }
  const float f1 = ldexpf(1.f, one ? e : e2);   // the (last) factor applied at the store
#pragma unroll
  for (int p = 0; p < NPASS; ++p) {
    const int row = row0 + p * RP + lr;
    if (row >= N) continue;
    uint8_t* dst = x8 + qb.row0 + row * qb.rs + li * EPL;
    if constexpr (EPL == 2) {
      uint16_t pq;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pq) : "f"(v[p][1] * f1), "f"(v[p][0] * f1));
      *reinterpret_cast<uint16_t*>(dst) = pq;
    } else {
      uint32_t pk[EPL / 4];
#pragma unroll
      for (int u = 0; u < EPL / 4; ++u)
        pk[u] = pack_e4m3x4(v[p][4 * u] * f1, v[p][4 * u + 1] * f1, v[p][4 * u + 2] * f1, v[p][4 * u + 3] * f1);
      if constexpr (EPL % 16 == 0) {
#pragma unroll
        for (int q = 0; q < EPL / 16; ++q)
          reinterpret_cast<uint4*>(dst)[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      } else {
#pragma unroll
        for (int u = 0; u < EPL / 4; ++u) reinterpret_cast<uint32_t*>(dst)[u] = pk[u];
      }
    }
  }
}

// Plain instance (no rotation, no RoPE): the 16-bit inputs stay packed in
// registers between the load and the store (a quarter of the registers of
// the float layout above), so more CTAs fit on an SM and each issues all of
// its block's loads before its first use; a lane holds 8 consecutive
// elements per row part (one 16-byte load), 256 threads per 128-row block.
// The codes and factors equal those of the float layout: the same amax (of
// the same values), the same power-of-two factor, each element scaled once.
// CTAs per SM the plain instance is built for (its whole block's loads in
// flight per CTA; more CTAs per SM keep more bytes in flight)
template <int D>
__host__ __device__ constexpr int quant_plain_ctas() { return D == 64 ? 4 : (D == 128 ? 3 : 1); }

template <typename T, int D, bool kPacked>
__global__ void __launch_bounds__(256, quant_plain_ctas<D>()) quant_plain_kernel(const T* __restrict__ x, uint8_t* __restrict__ x8,
                                                          float* __restrict__ scales, const QuantGeom geo) {
  constexpr int VPR = D / 8;                 // 16-byte vectors per row
  constexpr int NV = 128 * VPR / 256;        // vectors per thread
  __shared__ float red[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x;
  const QuantBlock qb = quant_block<D, kPacked ? 1 : 0>(geo, blk, blockIdx.y, blockIdx.z);
  if (blk * 128 >= qb.L) return;   // a packed sequence shorter than the longest
  const int rows = min(128, qb.L - blk * 128);
  // vector i of this thread: row i * RSTEP + r0 of the block, 8 elements from
  // column 8 * (threadIdx.x % VPR) (consecutive threads on consecutive
  // vectors of a row). Dense rows are D elements apart, so the block is one
  // contiguous run of vectors; packed rows are H * D apart.
  constexpr int RSTEP = 256 / VPR;
  const int r0 = static_cast<int>(threadIdx.x) / VPR;
  auto voff = [&](int i) -> long long {
    if constexpr (kPacked)
      return qb.row0 + (static_cast<long long>(blk) * 128 + i * RSTEP + r0) * qb.rs + (threadIdx.x % VPR) * 8;
    else
      return qb.row0 + static_cast<long long>(blk) * 128 * D + (static_cast<long long>(i) * 256 + threadIdx.x) * 8;
  };
  uint4 w[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i)
    w[i] = i * RSTEP + r0 < rows ? *reinterpret_cast<const uint4*>(x + voff(i)) : make_uint4(0, 0, 0, 0);
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const uint32_t wv[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
      amax = fmax3(amax, fabsf(to_f32<T>(wv[u] & 0xFFFFu)), fabsf(to_f32<T>(wv[u] >> 16)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, red[i]);
  const int e = e4m3_scale_exponent(amax);
  if (threadIdx.x == 0) scales[qb.si] = ldexpf(1.f, -e);
  // x * 2^e in one multiply when 2^e is a normal float (exact either way:
  // a power-of-two scaling), else in two steps
  const int e1 = e / 2, e2 = e - e1;
  const bool one = e >= -126 && e <= 127;
  const float f = one ? ldexpf(1.f, e) : ldexpf(1.f, e1), f2 = one ? 1.f : ldexpf(1.f, e2);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    if (i * RSTEP + r0 >= rows) continue;
    const uint32_t wv[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
    float y[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      y[2 * u] = to_f32<T>(wv[u] & 0xFFFFu) * f;
      y[2 * u + 1] = to_f32<T>(wv[u] >> 16) * f;
    }
    if (!one) {
#pragma unroll
      for (int u = 0; u < 8; ++u) y[u] *= f2;
    }
    *reinterpret_cast<uint2*>(x8 + voff(i)) =
        make_uint2(pack_e4m3x4(y[0], y[1], y[2], y[3]), pack_e4m3x4(y[4], y[5], y[6], y[7]));
  }
}

template <typename T, bool kRope>
cudaError_t launch_typed(const void* x, uint8_t* x8, float* scales, dim3 grid, const QuantGeom& geo, int d,
                         const int8_t* signs, float inv_sqrt_d, const float* rc, const float* rs, cudaStream_t st) {
  const T* xt = static_cast<const T*>(x);
  if (!kRope && signs == nullptr) {
    const bool pk = geo.cu_seqlens != nullptr;
    switch (d) {
      case 64:
        if (pk) quant_plain_kernel<T, 64, true><<<grid, 256, 0, st>>>(xt, x8, scales, geo);
        else quant_plain_kernel<T, 64, false><<<grid, 256, 0, st>>>(xt, x8, scales, geo);
        break;
      case 128:
        if (pk) quant_plain_kernel<T, 128, true><<<grid, 256, 0, st>>>(xt, x8, scales, geo);
        else quant_plain_kernel<T, 128, false><<<grid, 256, 0, st>>>(xt, x8, scales, geo);
        break;
      case 256:
        if (pk) quant_plain_kernel<T, 256, true><<<grid, 256, 0, st>>>(xt, x8, scales, geo);
        else quant_plain_kernel<T, 256, false><<<grid, 256, 0, st>>>(xt, x8, scales, geo);
        break;
      default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  switch (d) {
    case 64: quant_kernel<T, 64, kRope><<<grid, quant_threads<64, kRope>(), 0, st>>>(xt, x8, scales, geo, signs, inv_sqrt_d, rc, rs); break;
    case 128: quant_kernel<T, 128, kRope><<<grid, quant_threads<128, kRope>(), 0, st>>>(xt, x8, scales, geo, signs, inv_sqrt_d, rc, rs); break;
    case 256: quant_kernel<T, 256, kRope><<<grid, quant_threads<256, kRope>(), 0, st>>>(xt, x8, scales, geo, signs, inv_sqrt_d, rc, rs); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_geo(const void* x, int in_dt, uint8_t* x8, float* scales, dim3 grid, const QuantGeom& geo, int d,
                       const int8_t* signs, float inv_sqrt_d, const float* rope_cos, const float* rope_sin,
                       cudaStream_t st) {
  const bool rope = rope_cos != nullptr;
  if (in_dt == 0)
    return rope ? launch_typed<__nv_bfloat16, true>(x, x8, scales, grid, geo, d, signs, inv_sqrt_d, rope_cos, rope_sin, st)
                : launch_typed<__nv_bfloat16, false>(x, x8, scales, grid, geo, d, signs, inv_sqrt_d, nullptr, nullptr, st);
  return rope ? launch_typed<__half, true>(x, x8, scales, grid, geo, d, signs, inv_sqrt_d, rope_cos, rope_sin, st)
              : launch_typed<__half, false>(x, x8, scales, grid, geo, d, signs, inv_sqrt_d, nullptr, nullptr, st);
}

}  // namespace

cudaError_t launch_quant_fp8(const void* x, int in_dt, uint8_t* x8, float* scales, int B, int H, int N, int d,
                             const int8_t* signs, float inv_sqrt_d, const float* rope_cos, const float* rope_sin,
                             cudaStream_t st) {
  const QuantGeom geo{H, N, nullptr};
  return launch_geo(x, in_dt, x8, scales, dim3((N + 127) / 128, H, B), geo, d, signs, inv_sqrt_d, rope_cos, rope_sin,
                    st);
}

cudaError_t launch_quant_fp8_varlen(const void* x, int in_dt, uint8_t* x8, float* scales, const int* cu_seqlens,
                                    int nseq, int max_len, int H, int d, const int8_t* signs, float inv_sqrt_d,
                                    cudaStream_t st) {
  const QuantGeom geo{H, 0, cu_seqlens};
  return launch_geo(x, in_dt, x8, scales, dim3((max_len + 127) / 128, H, nseq), geo, d, signs, inv_sqrt_d, nullptr,
                    nullptr, st);
}

}  // namespace attn
