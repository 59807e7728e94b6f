// Block quantisation to E4M3 with optional incoherent processing.
//
// FlashAttention-3 (zenmind.me summary) §3.5: one scale per 128-row block
// of each (batch, head); before quantising Q and K, each row may be rotated
// by diag(random signs) * Hadamard / sqrt(d) to spread outliers.
// m.xxqk.cn FA3 walkthrough §4.2: power-of-two scale factors.
//
// One CTA per (128-row block, head, batch), 8 warps, each warp owns 16 rows;
// lane l holds elements [l*c, l*c + c) of a row (c = d / 32), so loads and
// stores are coalesced. The fast Walsh-Hadamard transform runs in FP32 in
// radix-2 stages of stride 1, 2, 4, ...: strides below c inside a lane,
// larger strides across lanes with shuffles; each butterfly computes a + b
// and a - b exactly once, so the result does not depend on which lane holds
// which operand. This kernel is HBM-bound: it reads 2 bytes and writes 1
// byte per element.
// Optional rotary position embedding first (kRope; the paper fuses
// quantisation into the RoPE step that produces Q and K): rotate-half pairs
// (i, i + d/2) with the caller's cos/sin tables [N, d/2]; lanes 0-15 hold the
// first half of a row and lanes 16-31 the second, so a lane's partner is 16
// lanes away. Each product and sum is rounded on its own (no fused
// multiply-add). It is a separate instance so that the plain quantiser's code
// is unchanged by it.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ops.h"
#include "ptx.cuh"

namespace attn {

namespace {

template <int D>
__device__ __forceinline__ void fwht_row(float (&x)[D / 32], int lane) {
  constexpr int c = D / 32;
#pragma unroll
  for (int h = 1; h < D; h <<= 1) {
    if (h < c) {
#pragma unroll
      for (int e = 0; e < c; ++e) {
        if ((e & h) == 0) {
          const float a = x[e], b = x[e + h];
          x[e] = a + b;
          x[e + h] = a - b;
        }
      }
    } else {
      const int lm = h / c;
      const bool upper = (lane & lm) != 0;
#pragma unroll
      for (int e = 0; e < c; ++e) {
        const float other = __shfl_xor_sync(0xffffffffu, x[e], lm);
        x[e] = upper ? (other - x[e]) : (x[e] + other);
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

// warps per CTA: 8 rows of 16 for the plain quantiser; the RoPE instance uses
// 16 warps of 8 rows, so more rows' table loads are in flight at once
template <bool kRope>
__host__ __device__ constexpr int quant_warps() { return kRope ? 16 : 8; }

template <typename T, int D, bool kRope>
__global__ void __launch_bounds__(32 * quant_warps<kRope>()) quant_kernel(const T* __restrict__ x, uint8_t* __restrict__ x8,
                                                    float* __restrict__ scales, int H, int N,
                                                    const int8_t* __restrict__ signs, float inv_sqrt_d,
                                                    const float* __restrict__ rope_cos,
                                                    const float* __restrict__ rope_sin) {
  constexpr int c = D / 32;
  constexpr int NW = quant_warps<kRope>();
  constexpr int RPW = 128 / NW;   // rows per warp
  __shared__ float red[NW];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const long long head_off = (static_cast<long long>(b) * H + h) * N;
  const int row0 = blk * 128 + warp * RPW;
  float v[RPW][c];
  float sg[c];
#pragma unroll
  for (int e = 0; e < c; ++e) sg[e] = signs ? static_cast<float>(signs[lane * c + e]) : 1.f;
  float amax = 0.f;
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int row = row0 + r;
    if (row < N) {
      const T* src = x + (head_off + row) * D + lane * c;
#pragma unroll
      for (int e = 0; e < c; ++e) {
        if constexpr (sizeof(T) == 2 && std::is_same<T, __nv_bfloat16>::value) v[r][e] = __bfloat162float(src[e]);
        else v[r][e] = __half2float(src[e]);
      }
      if constexpr (kRope) {   // row < N is the same for the whole warp
        const long long t = static_cast<long long>(row) * (D / 2) + (lane & 15) * c;
        float cs4[c], sn4[c];
        if constexpr (c % 4 == 0) {
#pragma unroll
          for (int e = 0; e < c; e += 4) {
            const float4 a = *reinterpret_cast<const float4*>(rope_cos + t + e);
            const float4 b = *reinterpret_cast<const float4*>(rope_sin + t + e);
            cs4[e] = a.x; cs4[e + 1] = a.y; cs4[e + 2] = a.z; cs4[e + 3] = a.w;
            sn4[e] = b.x; sn4[e + 1] = b.y; sn4[e + 2] = b.z; sn4[e + 3] = b.w;
          }
        } else {
#pragma unroll
          for (int e = 0; e < c; ++e) {
            cs4[e] = rope_cos[t + e];
            sn4[e] = rope_sin[t + e];
          }
        }
#pragma unroll
        for (int e = 0; e < c; ++e) {
          const float other = __shfl_xor_sync(0xffffffffu, v[r][e], 16);
          const float cs = cs4[e], sn = sn4[e];
          v[r][e] = lane < 16 ? __fsub_rn(__fmul_rn(v[r][e], cs), __fmul_rn(other, sn))
                              : __fadd_rn(__fmul_rn(v[r][e], cs), __fmul_rn(other, sn));
        }
      }
    } else {
#pragma unroll
      for (int e = 0; e < c; ++e) v[r][e] = 0.f;
    }
    if (signs) {
#pragma unroll
      for (int e = 0; e < c; ++e) v[r][e] *= sg[e];
      fwht_row<D>(v[r], lane);
#pragma unroll
      for (int e = 0; e < c; ++e) v[r][e] *= inv_sqrt_d;
    }
#pragma unroll
    for (int e = 0; e < c; ++e) amax = fmaxf(amax, fabsf(v[r][e]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) amax = fmaxf(amax, red[w]);
  const int e = e4m3_scale_exponent(amax);
  const int e1 = e / 2, e2 = e - e1;
  const float f1 = ldexpf(1.f, e1), f2 = ldexpf(1.f, e2);
  if (threadIdx.x == 0) scales[(static_cast<long long>(b) * H + h) * gridDim.x + blk] = ldexpf(1.f, -e);
#pragma unroll
  for (int r = 0; r < RPW; ++r) {
    const int row = row0 + r;
    if (row >= N) break;
    uint8_t* dst = x8 + (head_off + row) * D + lane * c;
    if constexpr (c == 2) {
      uint16_t p;
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(p) : "f"(v[r][1] * f1 * f2), "f"(v[r][0] * f1 * f2));
      *reinterpret_cast<uint16_t*>(dst) = p;
    } else {
#pragma unroll
      for (int q = 0; q < c / 4; ++q) {
        const uint32_t p = pack_e4m3x4(v[r][4 * q] * f1 * f2, v[r][4 * q + 1] * f1 * f2,
                                       v[r][4 * q + 2] * f1 * f2, v[r][4 * q + 3] * f1 * f2);
        reinterpret_cast<uint32_t*>(dst)[q] = p;
      }
    }
  }
}

template <typename T, bool kRope>
cudaError_t launch_typed(const void* x, uint8_t* x8, float* scales, int B, int H, int N, int d, const int8_t* signs,
                         float inv_sqrt_d, const float* rc, const float* rs, cudaStream_t st) {
  const dim3 grid((N + 127) / 128, H, B);
  const T* xt = static_cast<const T*>(x);
  switch (d) {
    case 64: quant_kernel<T, 64, kRope><<<grid, 32 * quant_warps<kRope>(), 0, st>>>(xt, x8, scales, H, N, signs, inv_sqrt_d, rc, rs); break;
    case 128: quant_kernel<T, 128, kRope><<<grid, 32 * quant_warps<kRope>(), 0, st>>>(xt, x8, scales, H, N, signs, inv_sqrt_d, rc, rs); break;
    case 256: quant_kernel<T, 256, kRope><<<grid, 32 * quant_warps<kRope>(), 0, st>>>(xt, x8, scales, H, N, signs, inv_sqrt_d, rc, rs); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_fp8(const void* x, int in_dt, uint8_t* x8, float* scales, int B, int H, int N, int d,
                             const int8_t* signs, float inv_sqrt_d, const float* rope_cos, const float* rope_sin,
                             cudaStream_t st) {
  const bool rope = rope_cos != nullptr;
  if (in_dt == 0)
    return rope ? launch_typed<__nv_bfloat16, true>(x, x8, scales, B, H, N, d, signs, inv_sqrt_d, rope_cos, rope_sin, st)
                : launch_typed<__nv_bfloat16, false>(x, x8, scales, B, H, N, d, signs, inv_sqrt_d, nullptr, nullptr, st);
  return rope ? launch_typed<__half, true>(x, x8, scales, B, H, N, d, signs, inv_sqrt_d, rope_cos, rope_sin, st)
              : launch_typed<__half, false>(x, x8, scales, B, H, N, d, signs, inv_sqrt_d, nullptr, nullptr, st);
}

}  // namespace attn
