// dQ kernel of the deterministic backward for sm_103a (BF16 / FP16, head dim 64
// or 128).
//
// Method: FlashAttention-3 (zenmind.me summary) §3.1 backward chain with P
// recomputed from the forward's log-sum-exp and §4 step 5 (paper App. B.1)
// D = rowsum(dO o O), so dS = P o (dP - D) and dQ = scale * dS K. The fused
// backward adds the dQ partials of every KV tile into global memory, in an
// order that varies from run to run; here one CTA owns 128 query rows of one
// (batch, head), walks the KV tiles that hold a visible key in increasing
// order and keeps dQ in tensor memory, so every dQ element is summed by one
// CTA in one order and repeated runs give identical bits. (dK and dV come from
// the key-stationary kernel with its dQ product left out.)
//
// Tensor memory (512 columns): S [128 q x 128 keys] FP32 at 0..127, dP at
// 128..255, dQ [128 q x d dims] FP32 from 256, dS (16-bit pairs, two
// buffers) at 384..447 and 448..511.
// Shared memory: Q and dO tiles (loaded once), a ring of three K tiles and a
// ring of two V tiles; 128-byte-swizzled boxes of 64 elements x 128 rows.
// Warps: 0 TMA, 1 MMA (one lane), 4..11 two warpgroups; warpgroup g turns the
// scores of keys 64g .. 64g + 63 into dS (thread = query row of its lane
// quarter) and, at the end, writes dims 64g .. 64g + 63 of dQ (at d = 64 the
// first warpgroup writes them all).
// MMA order for KV step j: S(j) = Q K_j^T and dP(j) = dO V_j^T once the
// compute warps hold S(j-1)/dP(j-1) in registers, then dQ += dS(j-1) K_{j-1}
// once dS(j-1) is in tensor memory; so S(j)/dP(j) run while dS(j-1) is formed.
#pragma once
#include <cmath>
#include <cstdint>
#include <cuda.h>

#include "bwd_kernel.cuh"
#include "ptx.cuh"

namespace attn {

template <int DT, int DIM>
struct DqCfg {
  static_assert(DIM == 64 || DIM == 128, "deterministic dQ kernel is written for head dim 64 or 128");
  static constexpr int D = DIM;
  static constexpr int NBOX = D / 64;               // 64-element boxes per row
  static constexpr int TILE_B = 128 * D * 2;        // one 128-row tile
  static constexpr int BOX_B = 128 * 128;           // one 64-element box of 128 rows
  static constexpr int SBO = 1024;                  // 8 rows of 128 bytes
  static constexpr int NK = 3, NV = 2;              // ring stages
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 2 + 2 + 2 + 1;
  static constexpr int SMEM_BYTES = (2 + NK + NV) * TILE_B + NBAR * 8 + 16;   // base is 1024-aligned
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeded");
  static constexpr int NTHREADS = 384;
  // launch: 168 per thread; the load/MMA warpgroup keeps 88 and hands the
  // rest to the two compute warpgroups (each thread holds 64 S and 64 dP)
  static constexpr uint32_t kRegsCtl = 88, kRegsMath = 208;
  static_assert(128 * kRegsCtl + 256 * kRegsMath <= NTHREADS * 168, "register split");
  static constexpr int kRegsSplit = (128 * kRegsCtl + 256 * kRegsMath + NTHREADS - 1) / NTHREADS;   // per thread
  static constexpr uint32_t FMT = DT == kBF16 ? 1u : 0u;
  static constexpr uint32_t IDESC_SP = instr_desc(128, 128, FMT, FMT, 0, 0);   // A, B K-major
  static constexpr uint32_t IDESC_DQ = instr_desc(128, D, FMT, FMT, 0, 1);     // B (K) MN-major
  static constexpr uint32_t COL_S = 0, COL_DP = 128, COL_DQ = 256, COL_DS = 384;
};

template <int DT, int DIM>
__global__ void __launch_bounds__(384, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
              const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const BwdArgs a) {
  using C = DqCfg<DT, DIM>;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t dq_smem[];
  if (smem_u32(dq_smem) & 1023u) {
    if (threadIdx.x == 0 && a.status) atomicExch(a.status, kDevBadSmemAlign);
    return;
  }
  uint8_t* sQ = dq_smem;
  uint8_t* sdO = sQ + C::TILE_B;
  uint8_t* sK = sdO + C::TILE_B;                    // [NK][TILE_B]
  uint8_t* sV = sK + C::NK * C::TILE_B;             // [NV][TILE_B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + C::NV * C::TILE_B);
  uint64_t* q_full = bars;
  uint64_t* k_full = q_full + 1;                    // [NK]
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;               // [NV]
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* sp_full = v_empty + C::NV;              // S, dP ready
  uint64_t* sp_free = sp_full + 1;                  // S, dP in registers
  uint64_t* ds_ready = sp_free + 1;                 // [2]
  uint64_t* ds_free = ds_ready + 2;                 // [2]
  uint64_t* dq_final = ds_free + 2;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(dq_final + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.y;
  const int hkv = h / a.group;
  const bool packed = a.cu_seqlens != nullptr;
  int b, seq0, L;
  if (packed) {
    b = 0;
    seq0 = a.cu_seqlens[blockIdx.z];
    L = a.cu_seqlens[blockIdx.z + 1] - seq0;
  } else {
    b = blockIdx.z;
    seq0 = 0;
    L = a.N;
  }
  const int nqt = (L + 127) >> 7;
  // causal: the query tiles with the most KV tiles start first
  const int qt = a.causal ? static_cast<int>(gridDim.x - 1 - blockIdx.x) : static_cast<int>(blockIdx.x);
  if (qt >= nqt) return;   // whole CTA leaves before any set-up
  const int r0 = qt * 128, r1 = min(r0 + 128, L);
  const int klo = a.win_left < 0 ? 0 : max(0, r0 - a.win_left);
  const int khi = a.win_right < 0 ? L : min(L, r1 + a.win_right);   // exclusive
  const int kv0 = klo >> 7;
  const int nkv = ((khi + 127) >> 7) - kv0;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    mbar_init(sp_full, 1);
    mbar_init(sp_free, 256);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ds_ready[s], 256);
      mbar_init(&ds_free[s], 1);
    }
    mbar_init(dq_final, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_holder;
  const float kLog2e = 1.4426950408889634f;

  // Each role changes its register budget inside its own branch.
  if (warp < 4) {
  regs_dec<C::kRegsCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      const int qrow = seq0 + r0;
      mbar_arrive_expect_tx(q_full, 2 * C::TILE_B);
      for (int c = 0; c < C::NBOX; ++c) {
        if (packed) {
          tma_load_4d(sQ + c * C::BOX_B, &tmQ, q_full, c * 64, h, qrow, 0);
          tma_load_4d(sdO + c * C::BOX_B, &tmdO, q_full, c * 64, h, qrow, 0);
        } else {
          tma_load_4d(sQ + c * C::BOX_B, &tmQ, q_full, c * 64, qrow, h, b);
          tma_load_4d(sdO + c * C::BOX_B, &tmdO, q_full, c * 64, qrow, h, b);
        }
      }
      for (int j = 0; j < nkv; ++j) {
        const int krow = seq0 + (kv0 + j) * 128;
        const int sk = j % C::NK, sv = j % C::NV;
        if (!mbar_wait(&k_empty[sk], ((j / C::NK) & 1) ^ 1, a.status)) break;
        mbar_arrive_expect_tx(&k_full[sk], C::TILE_B);
        for (int c = 0; c < C::NBOX; ++c) {
          uint8_t* dst = sK + sk * C::TILE_B + c * C::BOX_B;
          if (packed) tma_load_4d(dst, &tmK, &k_full[sk], c * 64, hkv, krow, 0);
          else tma_load_4d(dst, &tmK, &k_full[sk], c * 64, krow, hkv, b);
        }
        if (!mbar_wait(&v_empty[sv], ((j / C::NV) & 1) ^ 1, a.status)) break;
        mbar_arrive_expect_tx(&v_full[sv], C::TILE_B);
        for (int c = 0; c < C::NBOX; ++c) {
          uint8_t* dst = sV + sv * C::TILE_B + c * C::BOX_B;
          if (packed) tma_load_4d(dst, &tmV, &v_full[sv], c * 64, hkv, krow, 0);
          else tma_load_4d(dst, &tmV, &v_full[sv], c * 64, krow, hkv, b);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA
    if (lane == 0) {
      const uint64_t dQ_k = smem_desc(smem_u32(sQ), 16, C::SBO, kSwizzle128);
      const uint64_t ddO_k = smem_desc(smem_u32(sdO), 16, C::SBO, kSwizzle128);
      const uint64_t dK_k = smem_desc(smem_u32(sK), 16, C::SBO, kSwizzle128);
      const uint64_t dV_k = smem_desc(smem_u32(sV), 16, C::SBO, kSwizzle128);
      const uint64_t dK_mn = smem_desc(smem_u32(sK), C::BOX_B, C::SBO, kSwizzle128);
      auto dadd = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
      // S(j) = Q K_j^T, dP(j) = dO V_j^T (K steps of 16 over the head dim)
      auto issue_sp = [&](int sk, int sv) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::BOX_B + (kk % 4) * 32;
          mma_ss<false>(tbase + C::COL_S, dadd(dQ_k, off), dadd(dK_k, sk * C::TILE_B + off), C::IDESC_SP, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::BOX_B + (kk % 4) * 32;
          mma_ss<false>(tbase + C::COL_DP, dadd(ddO_k, off), dadd(dV_k, sv * C::TILE_B + off), C::IDESC_SP, kk > 0);
        }
        mma_commit(sp_full);
      };
      // dQ += dS(j) K_j: dS from tensor memory (8 columns per 16 keys), K MN-major
      auto issue_dq = [&](int j) {
        const int sk = j % C::NK;
        const uint32_t ds_col = C::COL_DS + 64u * (j & 1);
#pragma unroll
        for (int kk = 0; kk < 128 / 16; ++kk) {
          mma_ts<false>(tbase + C::COL_DQ, tbase + ds_col + kk * 8, dadd(dK_mn, sk * C::TILE_B + kk * 2048),
                        C::IDESC_DQ, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ds_free[j & 1]);
        mma_commit(&k_empty[sk]);
      };
      bool ok = mbar_wait(q_full, 0, a.status);
      for (int j = 0; j < nkv && ok; ++j) {
        const int sk = j % C::NK, sv = j % C::NV;
        if (!(ok = mbar_wait(&k_full[sk], (j / C::NK) & 1, a.status))) break;
        if (!(ok = mbar_wait(&v_full[sv], (j / C::NV) & 1, a.status))) break;
        if (j > 0 && !(ok = mbar_wait(sp_free, (j - 1) & 1, a.status))) break;
        tc_fence_after();
        issue_sp(sk, sv);
        mma_commit(&v_empty[sv]);
        if (j > 0) {
          if (!(ok = mbar_wait(&ds_ready[(j - 1) & 1], ((j - 1) >> 1) & 1, a.status))) break;
          tc_fence_after();
          issue_dq(j - 1);
        }
      }
      if (ok && (ok = mbar_wait(&ds_ready[(nkv - 1) & 1], ((nkv - 1) >> 1) & 1, a.status))) {
        tc_fence_after();
        issue_dq(nkv - 1);
      }
      mma_commit(dq_final);
    }
    __syncwarp();
  }
  } else {
    regs_inc<C::kRegsMath>();
    // ------------------------------------------------------- dS and dQ out
    const int g = (warp - 4) >> 2;                  // keys 64g .. 64g + 63; dims 64g .. at the end
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int qi = r0 + row;                        // query position in the sequence
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const long long lrow = static_cast<long long>(b) * a.l_sb + static_cast<long long>(h) * a.l_sh + seq0;
    const bool qvalid = qi < L;
    const float nl = qvalid ? -a.lse[lrow + qi] * kLog2e : -INFINITY;   // -LSE in log2 units
    const float nd = qvalid ? -a.dvec[lrow + qi] : 0.f;                 // -D
    const float2 sl2v = make_float2(a.scale_log2, a.scale_log2), nlv = make_float2(nl, nl), ndv = make_float2(nd, nd);
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(sp_full, j & 1, a.status)))) break;
      tc_fence_after();
      uint32_t sv[64], dp[64];
      tmem_ld32(tbase + lane_off + C::COL_S + 64 * g, *reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      tmem_ld32(tbase + lane_off + C::COL_S + 64 * g + 32, *reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      tmem_ld32(tbase + lane_off + C::COL_DP + 64 * g, *reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      tmem_ld32(tbase + lane_off + C::COL_DP + 64 * g + 32, *reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tmem_wait_ld();
      reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&sv[0]));
      reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&sv[32]));
      reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&dp[0]));
      reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&dp[32]));
      tc_fence_before();
      mbar_arrive(sp_free);                         // S(j+1), dP(j+1) may now overwrite them
      // keys outside the sequence or the window give P = 0
      const int kb = (kv0 + j) * 128 + 64 * g;      // first key of this half
      if (kb + 64 > L || (a.win_right >= 0 && kb + 63 > qi + a.win_right) ||
          (a.win_left >= 0 && kb < qi - a.win_left)) {
        int hi = L - kb;                            // visible: lo <= c < hi
        if (a.win_right >= 0) hi = min(hi, qi + a.win_right - kb + 1);
        const int lo = a.win_left >= 0 ? qi - a.win_left - kb : 0;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= hi || c < lo) sv[c] = __float_as_uint(-INFINITY);
      }
      uint32_t ds[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        float2 x = ffma2(make_float2(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])), sl2v, nlv);
        const float2 p = make_float2(ex2(x.x), ex2(x.y));
        const float2 t = fadd2(make_float2(__uint_as_float(dp[2 * e]), __uint_as_float(dp[2 * e + 1])), ndv);
        const float2 gs = fmul2(p, t);
        ds[e] = DT == kBF16 ? pack_bf16x2(gs.x, gs.y) : pack_f16x2(gs.x, gs.y);
      }
      // dS buffer j % 2 was last read by dQ += dS(j-2) K_{j-2}
      if (j >= 2 && !(ok = __all_sync(0xffffffffu, mbar_wait(&ds_free[j & 1], ((j >> 1) & 1) ^ 1, a.status))))
        break;
      tc_fence_after();
      const uint32_t ds_col = tbase + lane_off + C::COL_DS + 64u * (j & 1) + 32 * g;
      tmem_st32(ds_col, ds);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&ds_ready[j & 1]);
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(dq_final, 0, a.status));
    tc_fence_after();
    if (ok && 64 * g < D) {   // dQ row qi, dims 64g .. 64g + 63, times scale
      const long long off = static_cast<long long>(b) * a.q_sb + static_cast<long long>(h) * a.q_sh +
                            static_cast<long long>(seq0 + qi) * a.q_sn + 64 * g;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        uint32_t v[32];
        tmem_ld32(tbase + lane_off + C::COL_DQ + 64 * g + 32 * c, v);
        tmem_wait_ld();
        reg_fence(v);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float x0 = __uint_as_float(v[2 * e]) * a.scale, x1 = __uint_as_float(v[2 * e + 1]) * a.scale;
          pk[e] = DT == kBF16 ? pack_bf16x2(x0, x1) : pack_f16x2(x0, x1);
        }
        if (qvalid) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dq) + off + 32 * c);
#pragma unroll
          for (int w = 0; w < 4; ++w) dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace attn
