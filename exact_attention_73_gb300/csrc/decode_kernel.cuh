// Persistent FP8 decode kernel over a block-quantised KV cache (split-KV).
//
// Method: FlashAttention-3 (zenmind.me summary) §3.2 Algorithm 1 in the FP8
// form of §3.5, run over one split of the cache's KV tiles per work item; a
// separate kernel combines the splits by their log-sum-exp weights.
//
// A work item is one (split, KV head, batch): the g = Hq / Hkv query heads of
// the KV group at the decoded position form one query tile (rows 0 .. g-1 of
// a 128-row MMA tile; the Q map views q as [B, Hkv, g, d]). The grid holds at
// most one CTA per SM and each CTA walks the items w = blockIdx.x,
// blockIdx.x + gridDim.x, ... . All roles walk the same items in the same
// order, so barrier phases follow from running counters: ri counts the items
// with at least one KV tile, tg the KV tiles before the current item. The K/V
// ring, the two score buffers and the two Q buffers run on across items, so
// the TMA loads of the next item stream while the current one drains and the
// cost of starting and draining a CTA is not paid once per item (which made
// high split counts slow with one CTA per item).
//
// Roles (256 threads): warp 0 loads Q (double-buffered per item) and K/V
// tiles (ring of NSLOT slots, order K0 K1 V0 K2 V1 ... per item); warp 1
// issues tcgen05.mma: S(j) = Q K_j^T into score buffer tg+j mod 2, O += P V_j
// with P read from tensor memory; warps 4-7 run the softmax (thread = row),
// write P over S, and at the end of an item write the FP32 partial O
// (normalised) and LSE of rows 0 .. g-1. The first O += P V of an item starts
// a fresh accumulator, after the softmax has read the previous item's O
// (barrier o_free).
#pragma once
#include <cmath>
#include <cstdint>
#include <cuda.h>

#include "fwd_kernel.cuh"

namespace attn {

template <int D>
struct DecCfg {
  using F = FwdCfg<kE4M3, D, 1>;
  static constexpr int QBUF = 2;                            // Q tiles in flight (items ri, ri+1)
  static constexpr int Q_B = F::TILE_B;
  static constexpr int NSLOT_RAW = (F::BUDGET - QBUF * Q_B) / F::TILE_B;
  static constexpr int NSLOT = NSLOT_RAW > 8 ? 8 : NSLOT_RAW;
  static_assert(NSLOT >= 3, "shared memory too small for the K/V ring");
  // q_full[2], q_empty[2], kv_full[NSLOT], kv_empty[NSLOT], s_full[2],
  // p_ready[2], o_done, o_final, o_free
  static constexpr int NBAR = 2 * QBUF + 2 * NSLOT + 4 + 3;
  static constexpr int SMEM_BYTES = 1024 + QBUF * Q_B + NSLOT * F::TILE_B + NBAR * 8 + 16;
  static constexpr int NTHREADS = 256;
};

struct DecItem {
  int b, hkv, split, L, kv0, nkv;   // nkv <= 0: the split lies past this sequence's cache
};

__device__ __forceinline__ DecItem dec_item(const FwdArgs& a, int w, int splits) {
  DecItem t;
  t.split = w % splits;
  const int r = w / splits;
  t.hkv = r % a.Hkv;
  t.b = r / a.Hkv;
  t.L = a.seqlens ? min(a.seqlens[t.b], a.N) : a.N;   // valid cache length, at most the cache
  t.kv0 = t.split * a.tiles_per_split;
  t.nkv = min((t.L + 127) >> 7, t.kv0 + a.tiles_per_split) - t.kv0;
  return t;
}

template <int D>
__global__ void __launch_bounds__(DecCfg<D>::NTHREADS, 1)
decode_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const FwdArgs a, int splits, int items) {
  using F = FwdCfg<kE4M3, D, 1>;
  using C = DecCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;                              // [QBUF] query tiles
  uint8_t* sKV = smem + C::QBUF * C::Q_B;          // [NSLOT] K or V tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::NSLOT * F::TILE_B);
  uint64_t* q_full = bars;                         // [QBUF]
  uint64_t* q_empty = q_full + C::QBUF;            // [QBUF] the S products of an item are done with its Q
  uint64_t* kv_full = q_empty + C::QBUF;           // [NSLOT]
  uint64_t* kv_empty = kv_full + C::NSLOT;         // [NSLOT]
  uint64_t* s_full = kv_empty + C::NSLOT;          // [2]
  uint64_t* p_ready = s_full + 2;                  // [2]
  uint64_t* o_done = p_ready + 2;                  // one phase per O += P V
  uint64_t* o_final = o_done + 1;                  // one phase per item
  uint64_t* o_free = o_final + 1;                  // one phase per item: O read by the softmax
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(o_free + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int i = 0; i < C::QBUF; ++i) {
      mbar_init(&q_full[i], 1);
      mbar_init(&q_empty[i], 1);
    }
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&p_ready[i], 128);
    }
    mbar_init(o_done, 1);
    mbar_init(o_final, 1);
    mbar_init(o_free, 128);
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

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int ri = 0;
      long long ig = 0;   // ring position of the next K/V tile
      bool ok = true;
      for (int w = blockIdx.x; w < items && ok; w += gridDim.x) {
        const DecItem t = dec_item(a, w, splits);
        if (t.nkv <= 0) continue;
        const int qb = ri & 1;
        if (ri >= 2 && !(ok = mbar_wait(&q_empty[qb], ((ri - 2) >> 1) & 1, a.status))) break;
        mbar_arrive_expect_tx(&q_full[qb], C::Q_B);
        for (int c = 0; c < F::NBOX; ++c)
          tma_load_4d(sQ + qb * C::Q_B + c * F::BOXT_B, &tmQ, &q_full[qb], c * F::BOX_E, 0, t.hkv, t.b);
        for (int it = 0; it < 2 * t.nkv; ++it) {
          const int slot = static_cast<int>(ig % C::NSLOT);
          if (!(ok = mbar_wait(&kv_empty[slot], static_cast<uint32_t>((ig / C::NSLOT) & 1) ^ 1, a.status))) break;
          mbar_arrive_expect_tx(&kv_full[slot], F::TILE_B);
          bool is_v;
          int jt;
          kv_item(1, it, t.nkv, is_v, jt);
          const CUtensorMap* m = is_v ? &tmV : &tmK;
          const int row = (t.kv0 + jt) * 128;
          for (int c = 0; c < F::NBOX; ++c)
            tma_load_4d(sKV + slot * F::TILE_B + c * F::BOXT_B, m, &kv_full[slot], c * F::BOX_E, row, t.hkv, t.b);
          ++ig;
        }
        ++ri;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t kv_addr = smem_u32(sKV);
      // S = Q K^T into score buffer sb
      auto issue_s = [&](int qb, int sb, int slot) {
#pragma unroll
        for (int kk = 0; kk < D / F::KSTEP_E; ++kk) {
          const uint32_t off = (kk * F::KSTEP_B / F::BOX_B) * F::BOXT_B + (kk * F::KSTEP_B) % F::BOX_B;
          const uint64_t ad = smem_desc(q_addr + qb * C::Q_B + off, 16, F::SBO, F::SWZ);
          const uint64_t bd = smem_desc(kv_addr + slot * F::TILE_B + off, 16, F::SBO, F::SWZ);
          mma_ss<true>(tbase + sb * 128, ad, bd, F::IDESC_S, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[sb]);
      };
      // O (+)= P V with P over S in score buffer sb; acc = false starts O afresh
      auto issue_pv = [&](int sb, int slot, bool acc) {
#pragma unroll
        for (int kk = 0; kk < 128 / F::KSTEP_E; ++kk) {
          const uint64_t bd = smem_desc(kv_addr + slot * F::TILE_B + kk * F::KSTEP_E * F::BOX_B,
                                        F::BOXT_B, F::SBO, F::SWZ);
          mma_ts<true>(tbase + F::O_COL, tbase + sb * 128 + kk * 8, bd, F::IDESC_O, (acc || kk > 0) ? 1u : 0u);
        }
      };
      auto kv_wait = [&](long long g) {
        return mbar_wait(&kv_full[g % C::NSLOT], static_cast<uint32_t>((g / C::NSLOT) & 1), a.status);
      };
      int ri = 0, tg = 0;
      long long ig = 0;   // ring position of the item's first K/V tile
      bool ok = true;
      for (int w = blockIdx.x; w < items && ok; w += gridDim.x) {
        const DecItem t = dec_item(a, w, splits);
        if (t.nkv <= 0) continue;
        const int qb = ri & 1;
        if (!(ok = mbar_wait(&q_full[qb], (ri >> 1) & 1, a.status))) break;
        // S(0), S(1): their buffers last held tiles tg-2 and tg-1, whose
        // O += P V were issued before (the tensor pipe runs in order)
        for (int j = 0; j < 2 && j < t.nkv; ++j) {
          const long long gk = ig + kv_index_k(1, j);
          if (!(ok = kv_wait(gk))) break;
          tc_fence_after();
          issue_s(qb, (tg + j) & 1, static_cast<int>(gk % C::NSLOT));
          mma_commit(&kv_empty[gk % C::NSLOT]);
        }
        // per step j: O += P(j) V_j, then S(j+2) into the buffer P(j) came from
        for (int j = 0; j < t.nkv && ok; ++j) {
          const int jg = tg + j, sb = jg & 1;
          const long long gv = ig + kv_index_v(1, j, t.nkv);
          if (!(ok = kv_wait(gv))) break;
          if (!(ok = mbar_wait(&p_ready[sb], (jg >> 1) & 1, a.status))) break;
          if (j == 0 && ri > 0 && !(ok = mbar_wait(o_free, (ri - 1) & 1, a.status))) break;
          tc_fence_after();
          issue_pv(sb, static_cast<int>(gv % C::NSLOT), j > 0);
          mma_commit(o_done);
          mma_commit(&kv_empty[gv % C::NSLOT]);
          if (j + 2 < t.nkv) {
            const long long gk = ig + kv_index_k(1, j + 2);
            if (!(ok = kv_wait(gk))) break;
            tc_fence_after();
            issue_s(qb, sb, static_cast<int>(gk % C::NSLOT));
            mma_commit(&kv_empty[gk % C::NSLOT]);
          }
        }
        if (!ok) break;
        mma_commit(&q_empty[qb]);
        mma_commit(o_final);
        tg += t.nkv;
        ig += 2 * t.nkv;
        ++ri;
      }
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------- softmax
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tO = tbase + lane_off + F::O_COL;
    // rows quarter*32 .. +31 hold real query heads only if quarter*32 < g; a
    // warp of padding rows skips the softmax and the epilogue (its rows of P
    // and O are never read) but keeps every barrier's arrival count, waiting
    // for each tile's S so that it never runs ahead by two phases
    const bool active = quarter * 32 < a.group;
    int ri = 0, tg = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < items && ok; w += gridDim.x) {
      const DecItem t = dec_item(a, w, splits);
      const long long prow0 = (static_cast<long long>(t.split) * a.batch + t.b) * a.Hq +
                              static_cast<long long>(t.hkv) * a.group;
      if (t.nkv <= 0) {   // a split past the cache: a neutral partial
        for (int i = threadIdx.x - 128; i < a.group * D; i += 128) a.o_part[prow0 * D + i] = 0.f;
        for (int i = threadIdx.x - 128; i < a.group; i += 128) a.lse_part[prow0 + i] = -INFINITY;
        continue;
      }
      const float q_fac = a.sq[static_cast<long long>(t.b) * a.Hkv + t.hkv];   // one factor per group
      const long long vs_base = (static_cast<long long>(t.b) * a.Hkv + t.hkv) * a.nblk + t.kv0;
      float m = -INFINITY;     // running max of x = S * scale * log2(e)
      float l = 0.f;           // running sum of exp2(x - m)
      int f_run = -1000;       // running max exponent of the V factors
      // the K and V block factors are fetched one KV step ahead
      float sk_next = a.sk[vs_base], sv_next = a.sv[vs_base];
      for (int j = 0; j < t.nkv; ++j) {
        const float sk_j = sk_next, sv_j = sv_next;
        if (j + 1 < t.nkv) {
          sk_next = a.sk[vs_base + j + 1];
          sv_next = a.sv[vs_base + j + 1];
        }
        const int jg = tg + j, sb = jg & 1;
        const uint32_t tS = tbase + lane_off + sb * 128;
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], (jg >> 1) & 1, a.status));
        if (!ok) break;
        if (!active) {
          mbar_arrive(&p_ready[sb]);
          continue;
        }
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        const int kb = (t.kv0 + j) * 128;
        if (kb + 128 > t.L) {   // keys past this sequence's cache length
          const int hi = t.L - kb;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= hi) sr[c] = __float_as_uint(-INFINITY);
        }
        const float mx = rowmax(sr);
        const float sl2 = a.scale_log2 * (q_fac * sk_j);
        const int f_j = pow2_exponent_of(sv_j);
        const int f_new = max(f_run, f_j);
        const float mxs = mx * sl2;
        const float m_new = (mxs > m + F::kTau) ? mxs : m;
        float corr = 1.f;
        if (m_new != m) corr = ex2(m - m_new);   // m = -inf gives 0
        float corr_o = corr;
        if (f_new != f_run) corr_o *= exp2i(max(f_run - f_new, -126));
        l *= corr;
        m = m_new;
        if (j > 0 && warp_any(corr_o != 1.f)) {   // O is final once O += P(j-1) V has completed
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(o_done, (jg - 1) & 1, a.status)))) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            tmem_ld32(tO + 32 * c, r);
            tmem_wait_ld();
            reg_fence(r);
#pragma unroll
            for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr_o);
            tmem_st32(tO + 32 * c, r);
          }
        }
        const float mu = (m == -INFINITY) ? 0.f : m;
        const float bias = -mu + static_cast<float>(F::kPShift + f_j - f_new);
        // p = exp2(s * sl2 + bias): packed FMA pairs, MUFU ex2, four packed
        // partial row sums; P~ rounded to E4M3, four per word, over S
        const float2 sl2v = make_float2(sl2, sl2), biasv = make_float2(bias, bias);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int i = 32 * c + 4 * e;
            float2 x01 = ffma2(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), sl2v, biasv);
            float2 x23 = ffma2(make_float2(__uint_as_float(sr[i + 2]), __uint_as_float(sr[i + 3])), sl2v, biasv);
            x01 = make_float2(ex2(x01.x), ex2(x01.y));
            x23 = make_float2(ex2(x23.x), ex2(x23.y));
            acc[e & 3] = fadd2(acc[e & 3], fadd2(x01, x23));
            pk[e] = pack_e4m3x4(x01.x, x01.y, x23.x, x23.y);
          }
          tmem_st8(tS + 8 * c, pk);
        }
        const float2 as = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
        l += (as.x + as.y) * exp2i(-(F::kPShift + f_j - f_new));
        f_run = f_new;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_ready[sb]);
      }
      if (!ok) break;
      if (!active) {   // no rows of this warp to write; o_final(ri) first, so that
                       // this arrival cannot count toward an earlier o_free phase
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(o_final, ri & 1, a.status)))) break;
        mbar_arrive(o_free);
        tg += t.nkv;
        ++ri;
        continue;
      }
      ok = __all_sync(0xffffffffu, mbar_wait(o_final, ri & 1, a.status));
      if (!ok) break;
      tc_fence_after();
      // rows 0 .. g-1: FP32 partial O (normalised) and LSE of this split; all
      // lanes load (the tensor-memory loads are collective), valid rows store
      float inv = 1.f / l;
      inv *= exp2i(f_run - F::kPShift);
      const bool prow_ok = row < a.group;
      const long long prow = prow0 + row;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + 32 * c, r);
        tmem_wait_ld();
        reg_fence(r);
        if (prow_ok) {
          float4* dst = reinterpret_cast<float4*>(a.o_part + prow * D + 32 * c);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            dst[v] = make_float4(__uint_as_float(r[4 * v]) * inv, __uint_as_float(r[4 * v + 1]) * inv,
                                 __uint_as_float(r[4 * v + 2]) * inv, __uint_as_float(r[4 * v + 3]) * inv);
        }
      }
      if (prow_ok) {
        const float lse2 = (m == -INFINITY ? 0.f : m) + __log2f(l);
        a.lse_part[prow] = lse2 * 0.69314718055994530942f;
      }
      tc_fence_before();
      mbar_arrive(o_free);   // the next item's first O += P V may overwrite O
      tg += t.nkv;
      ++ri;
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
