// Forward attention kernel for sm_103a (BF16 / FP16 / E4M3 operands).
//
// Method: FlashAttention-3 (zenmind.me summary) §3.2 Algorithm 1 — a tiled
// online softmax with running max m and running sum l; O is rescaled by
// exp(m_old - m_new) and divided by l at the end, LSE = m + log l. S and P
// stay on chip. §3.5 adds the FP8 variant (block scales folded into S).
//
// GB300 design (not the pages' Hopper layout):
//   * one CTA owns QT query tiles of 128 rows of one (batch, head);
//   * warp 0 issues TMA loads: Q once, then K_j and V_j into a ring of
//     NSLOT shared-memory slots guarded by full/empty mbarriers;
//   * warp 1 (one thread) issues tcgen05.mma: S_t = Q_t K_j^T into tensor
//     memory, then O_t += P_t V_j with P_t read straight from tensor memory;
//   * one warpgroup per query tile runs the softmax: it loads its S rows
//     from tensor memory (thread = row), applies the mask, updates m and l,
//     writes P (BF16/FP16/E4M3) back over S and rescales O in tensor memory
//     when the max moved by more than kTau (log2 units); the last step
//     normalises O and writes O and LSE.
//   With QT = 2 the tensor core computes S for one tile while the other
//   tile's softmax runs, the role the pages' ping-pong schedule plays.
//   Completion of S_t(j) implies completion of every earlier MMA of the CTA,
//   including O_t += P_t V_{j-1}, so O_t can be rescaled right then.
//   A CTA walks one or more units (QT query tiles of one head and batch or
//   sequence): over short rows the grid holds one CTA per SM and each walks
//   units round-robin, the next unit's loads and S products overlapping the
//   current unit's last products and epilogue.
#pragma once
#include <cmath>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace attn {

enum : int { kBF16 = 0, kFP16 = 1, kE4M3 = 2 };

struct FwdArgs {
  void* o;
  float* lse;
  long long o_sn, o_sh, o_sb;   // element strides of O: row, head, batch
  long long l_sh, l_sb;         // element strides of LSE: head, batch (row stride 1)
  int Hq, Hkv, group;           // group = Hq / Hkv
  int N;                        // dense sequence length
  const int* cu_seqlens;        // packed layout when non-null
  float scale_log2;             // scale * log2(e)
  int causal;                   // scheduling hint: window (-1, 0)
  int win_left, win_right;      // key j visible to query i iff i - left <= j <= i + right (-1: no bound)
  const float* sq;              // FP8 dequantisation factors per 128-row block
  const float* sk;
  const float* sv;
  int nblk;                     // blocks per (batch or packed sequence, head) in sq/sk/sv
  // decode over a KV cache (decode_kernel): items of (split, KV head, batch)
  const int* seqlens;           // valid cache length per sequence (null: N)
  int tiles_per_split;          // KV tiles per split
  int batch;                    // B
  float* o_part;                // [splits][B][Hq][D] FP32, normalised per split
  float* lse_part;              // [splits][B][Hq]
  int* status;
  // fwd_kernel: units of QT query tiles, ux query-tile groups x uy query
  // heads x uz batches (or packed sequences); the grid walks them.
  int ux, uy, uz;
};

template <int DT, int D, int QT>
struct FwdCfg {
  static constexpr bool kFp8 = DT == kE4M3;
  static constexpr int ESZ = kFp8 ? 1 : 2;
  static constexpr int ROW_B = D * ESZ;
  static constexpr int BOX_B = ROW_B < 128 ? ROW_B : 128;   // inner extent of one TMA box
  static constexpr int BOX_E = BOX_B / ESZ;
  static constexpr int NBOX = D / BOX_E;
  static constexpr int TILE_B = 128 * ROW_B;                // one 128-row tile
  static constexpr int BOXT_B = 128 * BOX_B;                // one box of 128 rows
  static constexpr uint32_t SWZ = BOX_B == 128 ? kSwizzle128 : kSwizzle64;
  static constexpr int SBO = 8 * BOX_B;                     // 8-row core-matrix group
  static constexpr int KSTEP_B = 32;                        // K bytes per MMA
  static constexpr int KSTEP_E = KSTEP_B / ESZ;
  static constexpr int Q_B = QT * TILE_B;
  static constexpr int BUDGET = 200 * 1024;
  static constexpr int NSLOT_RAW = (BUDGET - Q_B) / TILE_B;
  static constexpr int NSLOT = NSLOT_RAW > 8 ? 8 : NSLOT_RAW;
  static_assert(NSLOT >= 2, "shared memory too small for the K/V ring");
  // Score buffers in tensor memory: one per query tile, or two alternating
  // buffers when the CTA has a single query tile.
  static constexpr int NSB = QT == 1 ? 2 : QT;
  static constexpr int O_COL = NSB * 128;                   // O_t at O_COL + t * D
  static_assert(O_COL + QT * D <= 512, "tensor memory overflow");
  static constexpr int NTHREADS = 128 + 128 * QT;
  static constexpr uint32_t kRegsCtl = 96, kRegsSoft = 200;   // QT = 2 register split
  static_assert(QT != 2 || 128 * kRegsCtl + 256 * kRegsSoft <= 384 * 168, "register split");
  static constexpr int NBAR = 1 + 2 * NSLOT + 2 * NSB + 3;
  static constexpr int SMEM_BYTES = 1024 + Q_B + NSLOT * TILE_B + NBAR * 8 + 16;
  static constexpr uint32_t FMT = DT == kBF16 ? 1u : 0u;    // BF16=1, F16=0, E4M3=0
  static constexpr uint32_t IDESC_S = instr_desc(128, 128, FMT, FMT, 0, 0);
  static constexpr uint32_t IDESC_O = instr_desc(128, D, FMT, FMT, 0, 1);
  // Rescale threshold (log2 units): keep a stale max while exp2(x - m) <= 2^kTau,
  // so O in tensor memory is rescaled only when the max moves far. The exact
  // running max of Algorithm 1 (kTau = 0) would rescale O in most KV steps;
  // for FP8 it also rounds each row's largest entry of P~ exactly, so the
  // stale max costs a little accuracy there (bounded by one E4M3 step per
  // entry against the exact-max rounding).
  static constexpr float kTau = kFp8 ? 4.0f : 8.0f;
  // Power-of-two shift of P~ before its E4M3 rounding.
  static constexpr int kPShift = 4;   // P~ <= 2^kTau, so P~ * 2^kPShift <= 256 < 448
};

__device__ __forceinline__ int pow2_exponent_of(float x) {   // x an exact power of two
  return static_cast<int>((__float_as_uint(x) >> 23) & 0xFFu) - 127;
}
__device__ __forceinline__ float exp2i(int e) {               // exact 2^e, |e| < 127
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// Order of the K/V tiles through the shared-memory ring. Two-tile CTAs load
// K0 V0 K1 V1 ...; single-tile CTAs (two score buffers) consume K0 K1 V0 K2
// V1 K3 ... V(n-1) and load in that order, so K(j+2) never waits behind V(j+1).
__device__ __forceinline__ void kv_item(int qt, int it, int nkv, bool& is_v, int& j) {
  if (qt != 1) {
    is_v = it & 1;
    j = it >> 1;
    return;
  }
  if (nkv == 1) { is_v = it == 1; j = 0; return; }
  if (it < 2) { is_v = false; j = it; return; }
  if (it == 2 * nkv - 1) { is_v = true; j = nkv - 1; return; }
  const int r = it - 2;
  is_v = (r & 1) == 0;
  j = is_v ? (r >> 1) : (r >> 1) + 2;
}
__device__ __forceinline__ int kv_index_k(int qt, int j) { return qt != 1 ? 2 * j : (j < 2 ? j : 2 * j - 1); }
__device__ __forceinline__ int kv_index_v(int qt, int j, int nkv) {
  if (qt != 1) return 2 * j + 1;
  return nkv == 1 ? 1 : (j == nkv - 1 ? 2 * nkv - 1 : 2 + 2 * j);
}

// One unit of work: QT query tiles of one (batch or sequence, query head).
struct FwdUnit {
  int h, hkv, b, seq0, L, nqt, qt0, kv0, nkv;
  int fb;   // FP8 factors: batch, or packed sequence (factors [sequences][heads][blocks])
};

// The k-th unit of this CTA as a linear index over ux * uy * uz units (x
// fastest), or -1 past the end. Units are dealt round-robin over the grid;
// with causal masking (heavy-first order: work falls with the index) every
// other round runs backwards, so that each CTA's total stays even.
__device__ __forceinline__ int fwd_unit_of(const FwdArgs& a, int k) {
  const int P = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  const int lin = (a.causal && (k & 1)) ? k * P + (P - 1 - c) : k * P + c;
  return lin < a.ux * a.uy * a.uz ? lin : -1;
}

// Decode unit `lin`; false when it holds no query row (a packed sequence
// shorter than the longest one).
template <int QT>
__device__ __forceinline__ bool fwd_unit(const FwdArgs& a, int lin, FwdUnit& w) {
  int bx, by, bz;
  if (a.causal) {
    // the last query tiles have the most work: those of every (head, batch)
    // come first
    heavy_first_map(8, lin, a.ux, a.uy, a.uz, bx, by, bz);
  } else {
    bx = lin % a.ux;
    by = (lin / a.ux) % a.uy;
    bz = lin / a.ux / a.uy;
  }
  w.h = by;
  if (a.cu_seqlens != nullptr) {
    w.b = 0;
    w.seq0 = a.cu_seqlens[bz];
    w.L = a.cu_seqlens[bz + 1] - w.seq0;
  } else {
    w.b = bz;
    w.seq0 = 0;
    w.L = a.N;
  }
  w.nqt = (w.L + 127) >> 7;
  // causal: the units with the most KV tiles first
  const int cblk = a.causal ? a.ux - 1 - bx : bx;
  w.qt0 = cblk * QT;
  if (w.qt0 >= w.nqt) return false;
  // KV tiles that hold a key visible to some query row of the unit
  const int r0 = w.qt0 * 128, r1 = min((w.qt0 + QT) * 128, w.L);
  const int klo = a.win_left < 0 ? 0 : max(0, r0 - a.win_left);
  const int khi = a.win_right < 0 ? w.L : min(w.L, r1 + a.win_right);   // exclusive
  w.kv0 = klo >> 7;
  w.nkv = ((khi + 127) >> 7) - w.kv0;
  w.hkv = w.h / a.group;
  w.fb = bz;
  return true;
}

// kPersist: the grid is smaller than the unit count and each CTA walks its
// units; otherwise every CTA takes one unit and the unit loops below run
// once (known at compile time, so their bookkeeping folds away).
template <int DT, int D, int QT, bool kPersist>
__global__ void __launch_bounds__(FwdCfg<DT, D, QT>::NTHREADS, 1)
fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           const __grid_constant__ CUtensorMap tmV, const FwdArgs a) {
  using C = FwdCfg<DT, D, QT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = smem;
  uint8_t* sKV = smem + C::Q_B;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::NSLOT * C::TILE_B);
  uint64_t* q_full = bars;                         // one phase per unit
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + C::NSLOT;
  uint64_t* s_full = kv_empty + C::NSLOT;          // [NSB]
  uint64_t* p_ready = s_full + C::NSB;             // [NSB]
  uint64_t* o_final = p_ready + C::NSB;            // one phase per unit
  uint64_t* o_done = o_final + 1;                  // one phase per O += P V (single-tile CTAs)
  uint64_t* q_empty = o_done + 1;                  // the unit's products have read Q
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(q_empty + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const bool packed = a.cu_seqlens != nullptr;
  {   // a CTA whose units hold no query row leaves before any set-up
    bool any = false;
    FwdUnit w;
    for (int k = 0; !any; ++k) {
      const int lin = fwd_unit_of(a, k);
      if (lin < 0) break;
      any = fwd_unit<QT>(a, lin, w);
    }
    if (!any) return;
  }

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NSLOT; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int t = 0; t < C::NSB; ++t) {
      mbar_init(&s_full[t], 1);
      mbar_init(&p_ready[t], 128);
    }
    mbar_init(o_final, 1);
    mbar_init(o_done, 1);
    mbar_init(q_empty, 1);
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

  // Every role walks the same units in the same order. Barrier phases run on
  // across units: q_full, q_empty and o_final once per unit, s_full and
  // p_ready once per KV step, the ring's slots once per K or V tile.
  //
  // With two query tiles (384 threads, 168 registers each at launch) the
  // load/MMA warpgroup hands registers to the two softmax warpgroups; each
  // role changes its budget inside its own branch, so the compiler sizes
  // every role's code for the budget it runs with.
  if (warp < 4) {
  if constexpr (QT == 2) regs_dec<C::kRegsCtl>();
  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int kvit = 0, ui = 0;   // K/V tiles and units loaded before this unit
      bool ok = true;
      for (int k = 0; ok && (kPersist || k == 0); ++k) {
        const int lin = fwd_unit_of(a, k);
        if (lin < 0) break;
        FwdUnit w;
        if (!fwd_unit<QT>(a, lin, w)) continue;
        // K/V tile `it` of this unit into the ring
        auto load_kv = [&](int it) {
          const int slot = (kvit + it) % C::NSLOT;
          if (!mbar_wait(&kv_empty[slot], (((kvit + it) / C::NSLOT) & 1) ^ 1, a.status)) return false;
          mbar_arrive_expect_tx(&kv_full[slot], C::TILE_B);
          bool is_v;
          int jt;
          kv_item(QT, it, w.nkv, is_v, jt);
          const CUtensorMap* m = is_v ? &tmV : &tmK;
          const int row = w.seq0 + (w.kv0 + jt) * 128;
          for (int c = 0; c < C::NBOX; ++c) {
            uint8_t* dst = sKV + slot * C::TILE_B + c * C::BOXT_B;
            if (packed) tma_load_4d(dst, m, &kv_full[slot], c * C::BOX_E, w.hkv, row, 0);
            else tma_load_4d(dst, m, &kv_full[slot], c * C::BOX_E, row, w.hkv, w.b);
          }
          return true;
        };
        // after the first unit, the unit's first two K/V tiles go into slots
        // the previous unit has released while its last products (which
        // still read the Q buffer) run; the first unit loads Q first
        const int pre = ui > 0 ? min(2, 2 * w.nkv) : 0;
        for (int it = 0; it < pre && ok; ++it) ok = load_kv(it);
        if (ok && ui > 0) ok = mbar_wait(q_empty, (ui - 1) & 1, a.status);
        if (!ok) break;
        mbar_arrive_expect_tx(q_full, C::Q_B);
        for (int t = 0; t < QT; ++t) {
          const int row = w.seq0 + (w.qt0 + t) * 128;
          for (int c = 0; c < C::NBOX; ++c) {
            uint8_t* dst = sQ + t * C::TILE_B + c * C::BOXT_B;
            if (packed) tma_load_4d(dst, &tmQ, q_full, c * C::BOX_E, w.h, row, 0);
            else tma_load_4d(dst, &tmQ, q_full, c * C::BOX_E, row, w.h, w.b);
          }
        }
        for (int it = pre; it < 2 * w.nkv && ok; ++it) ok = load_kv(it);
        kvit += 2 * w.nkv;
        ++ui;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t q_addr = smem_u32(sQ);
      const uint32_t kv_addr = smem_u32(sKV);
      int kvb = 0, gs = 0, ui = 0;   // K/V tiles, KV steps and units consumed before this unit
      int nkv = 0;
      // S_t = Q_t K^T into score buffer sb
      auto issue_s = [&](int t, int sb, int slot) {
#pragma unroll
        for (int kk = 0; kk < D / C::KSTEP_E; ++kk) {
          const uint32_t off = (kk * C::KSTEP_B / C::BOX_B) * C::BOXT_B + (kk * C::KSTEP_B) % C::BOX_B;
          const uint64_t ad = smem_desc(q_addr + t * C::TILE_B + off, 16, C::SBO, C::SWZ);
          const uint64_t bd = smem_desc(kv_addr + slot * C::TILE_B + off, 16, C::SBO, C::SWZ);
          mma_ss<C::kFp8>(tbase + sb * 128, ad, bd, C::IDESC_S, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s_full[sb]);
      };
      // O_t += P V with P in score buffer sb
      auto issue_pv = [&](int t, int sb, int slot, int j) {
#pragma unroll
        for (int kk = 0; kk < 128 / C::KSTEP_E; ++kk) {
          const uint64_t bd = smem_desc(kv_addr + slot * C::TILE_B + kk * C::KSTEP_E * C::BOX_B,
                                        C::BOXT_B, C::SBO, C::SWZ);
          mma_ts<C::kFp8>(tbase + C::O_COL + t * D, tbase + sb * 128 + kk * 8, bd, C::IDESC_O,
                          (j > 0 || kk > 0) ? 1u : 0u);
        }
      };
      // K/V tile `it` of this unit
      auto kv_wait = [&](int it) {
        return mbar_wait(&kv_full[(kvb + it) % C::NSLOT], ((kvb + it) / C::NSLOT) & 1, a.status);
      };
      auto kv_slot = [&](int it) { return (kvb + it) % C::NSLOT; };
      bool ok = true;
      for (int k = 0; ok && (kPersist || k == 0); ++k) {
        const int lin = fwd_unit_of(a, k);
        if (lin < 0) break;
        FwdUnit w;
        if (!fwd_unit<QT>(a, lin, w)) continue;
        nkv = w.nkv;
        ok = mbar_wait(q_full, ui & 1, a.status) && kv_wait(0);
        if constexpr (QT == 1) {
          // One query tile, two score buffers (buffer of step j: (gs + j) & 1):
          // S(j+2) is issued right after PV(j), so the softmax of step j+1
          // overlaps PV(j) and S(j+2).
          if (ok) {
            tc_fence_after();
            issue_s(0, gs & 1, kv_slot(0));
            mma_commit(&kv_empty[kv_slot(0)]);
          }
          if (ok && nkv > 1) {
            const int itk1 = kv_index_k(1, 1);
            if ((ok = kv_wait(itk1))) {
              tc_fence_after();
              issue_s(0, (gs + 1) & 1, kv_slot(itk1));
              mma_commit(&kv_empty[kv_slot(itk1)]);
            }
          }
          for (int j = 0; j < nkv && ok; ++j) {
            const int sb = (gs + j) & 1;
            const int itv = kv_index_v(1, j, nkv), itk = j + 2 < nkv ? kv_index_k(1, j + 2) : 0;
            if (!(ok = kv_wait(itv))) break;
            if (!(ok = mbar_wait(&p_ready[sb], ((gs + j) >> 1) & 1, a.status))) break;
            tc_fence_after();
            issue_pv(0, sb, kv_slot(itv), j);
            mma_commit(o_done);
            mma_commit(&kv_empty[kv_slot(itv)]);
            if (j + 2 < nkv) {
              if (!(ok = kv_wait(itk))) break;
              tc_fence_after();
              issue_s(0, sb, kv_slot(itk));
              mma_commit(&kv_empty[kv_slot(itk)]);
            }
          }
        } else {
          // Issue order: S_t(0) for every tile, then per KV step j:
          //   PV_0(j), S_0(j+1), PV_1(j), S_1(j+1)
          // so the softmax of tile t for step j+1 overlaps the other tile's
          // PV(j) and S(j+1) (two GEMMs of slack).
          if (ok) {
            tc_fence_after();
            for (int t = 0; t < QT; ++t) issue_s(t, t, kv_slot(0));
            mma_commit(&kv_empty[kv_slot(0)]);
          }
          for (int j = 0; j < nkv && ok; ++j) {
            const int itv = 2 * j + 1, sv_ = kv_slot(itv);
            const int itk = 2 * j + 2, sk_ = kv_slot(itk);
            const bool next = j + 1 < nkv;
            if (!(ok = kv_wait(itv))) break;
            bool k_ready = false;
            for (int t = 0; t < QT && ok; ++t) {
              if (!(ok = mbar_wait(&p_ready[t], (gs + j) & 1, a.status))) break;
              tc_fence_after();
              issue_pv(t, t, sv_, j);
              if (next) {
                if (!k_ready) {                 // K(j+1) is needed only now
                  if (!(ok = kv_wait(itk))) break;
                  tc_fence_after();
                  k_ready = true;
                }
                issue_s(t, t, sk_);
              }
            }
            mma_commit(&kv_empty[sv_]);
            if (next && k_ready) mma_commit(&kv_empty[sk_]);
          }
        }
        if (!ok) break;
        mma_commit(o_final);
        // Q is released with the unit's last product: a commit inside the
        // KV loop right after the last S product would free it a step
        // earlier, but any extra work in that loop slows every step
        mma_commit(q_empty);
        kvb += 2 * nkv;
        gs += nkv;
        ++ui;
      }
    }
    __syncwarp();
  }
  } else {
    if constexpr (QT == 2) regs_inc<C::kRegsSoft>();
    // ------------------------------------------------------- softmax
    const int t = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tO = tbase + lane_off + C::O_COL + t * D;
    int gs = 0, ui = 0;   // KV steps and units before this unit
    bool ok = true;
    for (int k = 0; ok && (kPersist || k == 0); ++k) {
      const int lin = fwd_unit_of(a, k);
      if (lin < 0) break;
      FwdUnit w;
      if (!fwd_unit<QT>(a, lin, w)) continue;
      const int nkv = w.nkv, L = w.L, kv0 = w.kv0;
      const int qtile = w.qt0 + t;
      const int qrow = qtile * 128 + row;
      float m = -INFINITY;     // running max of x = S * scale * log2(e)
      float l = 0.f;           // running sum of exp2(x - m)
      int f_run = -1000;       // FP8: running max exponent of the V factors
      float q_fac = 1.f;
      long long vs_base = 0;
      if constexpr (C::kFp8) {
        q_fac = a.sq[(static_cast<long long>(w.fb) * a.Hq + w.h) * a.nblk + min(qtile, w.nqt - 1)];
        vs_base = (static_cast<long long>(w.fb) * a.Hkv + w.hkv) * a.nblk + kv0;
      }
      // FP8: the K and V block factors are fetched one KV step ahead, so their
      // global-load latency overlaps the wait for the next score tile.
      float sk_next = 1.f, sv_next = 1.f;
      if constexpr (C::kFp8) {
        sk_next = a.sk[vs_base];
        sv_next = a.sv[vs_base];
      }
      for (int j = 0; j < nkv; ++j) {
        const float sk_j = sk_next, sv_j = sv_next;
        if constexpr (C::kFp8) {
          if (j + 1 < nkv) {
            sk_next = a.sk[vs_base + j + 1];
            sv_next = a.sv[vs_base + j + 1];
          }
        }
        const int gj = gs + j;
        const int sb = QT == 1 ? (gj & 1) : t;              // score buffer of this step
        const uint32_t sphase = QT == 1 ? ((gj >> 1) & 1) : (gj & 1);
        const uint32_t tS = tbase + lane_off + sb * 128;
        ok = __all_sync(0xffffffffu, mbar_wait(&s_full[sb], sphase, a.status));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[128];
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c) reg_fence(*reinterpret_cast<uint32_t(*)[32]>(&sr[32 * c]));
        const int kb = (kv0 + j) * 128;
        // mask keys past the sequence and outside the window [qrow - left, qrow + right]
        if (kb + 128 > L || (a.win_right >= 0 && kb + 127 > qtile * 128 + a.win_right) ||
            (a.win_left >= 0 && kb < qtile * 128 + 127 - a.win_left)) {
          int hi = L - kb;                                             // visible: lo <= c < hi
          if (a.win_right >= 0) hi = min(hi, qrow + a.win_right - kb + 1);
          const int lo = a.win_left >= 0 ? qrow - a.win_left - kb : 0;
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= hi || c < lo) sr[c] = __float_as_uint(-INFINITY);
        }
        const float mx = rowmax(sr);
        float sl2 = a.scale_log2;
        int f_j = 0, f_new = 0;
        if constexpr (C::kFp8) {
          sl2 *= q_fac * sk_j;
          f_j = pow2_exponent_of(sv_j);
          f_new = max(f_run, f_j);
        }
        const float mxs = mx * sl2;
        const float m_new = (mxs > m + C::kTau) ? mxs : m;
        float corr = 1.f;
        if (m_new != m) corr = ex2(m - m_new);   // m = -inf gives 0
        float corr_o = corr;
        if constexpr (C::kFp8) {
          if (f_new != f_run) corr_o *= exp2i(max(f_run - f_new, -126));
        }
        l *= corr;
        m = m_new;
        if (j > 0 && warp_any(corr_o != 1.f)) {
          if constexpr (QT == 1) {   // PV(j-1) may still be running with two score buffers
            if (!(ok = __all_sync(0xffffffffu, mbar_wait(o_done, (gj - 1) & 1, a.status)))) break;
            tc_fence_after();
          }
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
        float bias = -mu;
        if constexpr (C::kFp8) bias += static_cast<float>(C::kPShift + f_j - f_new);
        // p = exp2(s * sl2 + bias): packed FMA pairs, MUFU ex2, four packed
        // partial row sums
        const float2 sl2v = make_float2(sl2, sl2), biasv = make_float2(bias, bias);
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if constexpr (C::kFp8) {
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
        } else {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int i = 32 * c + 2 * e;
              float2 x = ffma2(make_float2(__uint_as_float(sr[i]), __uint_as_float(sr[i + 1])), sl2v, biasv);
              x = make_float2(ex2(x.x), ex2(x.y));
              acc[e & 3] = fadd2(acc[e & 3], x);
              pk[e] = (DT == kBF16) ? pack_bf16x2(x.x, x.y) : pack_f16x2(x.x, x.y);
            }
            tmem_st16(tS + 16 * c, pk);
          }
        }
        const float2 a01 = fadd2(acc[0], acc[1]), a23 = fadd2(acc[2], acc[3]);
        const float2 as = fadd2(a01, a23);
        const float rs = as.x + as.y;
        if constexpr (C::kFp8) {
          l += rs * exp2i(-(C::kPShift + f_j - f_new));
          f_run = f_new;
        } else {
          l += rs;
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&p_ready[sb]);
      }
      // The next unit's O += P V overwrites O_t only after this warpgroup's
      // arrival on p_ready for that unit's first step, which follows these
      // tensor-memory reads.
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(o_final, ui & 1, a.status));
      tc_fence_after();
      if (!ok) break;
      float inv = 1.f / l;
      if constexpr (C::kFp8) inv *= exp2i(f_run - C::kPShift);
      const bool valid = qrow < L;
      const long long row_off = static_cast<long long>(w.b) * a.o_sb + static_cast<long long>(w.h) * a.o_sh +
                                static_cast<long long>(w.seq0 + qrow) * a.o_sn;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(tO + 32 * c, r);
        tmem_wait_ld();
        reg_fence(r);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float x0 = __uint_as_float(r[2 * e]) * inv;
          const float x1 = __uint_as_float(r[2 * e + 1]) * inv;
          pk[e] = (DT == kFP16) ? pack_f16x2(x0, x1) : pack_bf16x2(x0, x1);
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.o) + row_off + 32 * c);
#pragma unroll
          for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      if (valid) {
        const float lse2 = (m == -INFINITY ? 0.f : m) + __log2f(l);
        a.lse[static_cast<long long>(w.b) * a.l_sb + static_cast<long long>(w.h) * a.l_sh + w.seq0 + qrow] =
            lse2 * 0.69314718055994530942f;
      }
      gs += nkv;
      ++ui;
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
