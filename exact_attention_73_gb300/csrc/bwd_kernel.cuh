// Backward attention kernels for sm_103a (BF16 / FP16, head dim 64, 128 or 256).
//
// Method: FlashAttention-3 (zenmind.me summary) §3.1 backward chain with P
// recomputed from the forward's log-sum-exp, and §4 step 5 (paper App. B.1):
// a pre-kernel computes D = rowsum(dO o O); dQ partials of every KV block are
// added atomically into an FP32 accumulator, then converted.
//   P   = exp(scale * Q K^T - LSE)
//   dV += P^T dO,  dP = dO V^T,  dS = P o (dP - D)
//   dK += scale * dS^T Q,  dQ += scale * dS K
//
// GB300 design. One CTA owns one tile of 128 keys of one (batch, KV head) and
// loops over every query head of the group and every 64-row query tile that
// can see those keys, so dK and dV of the group accumulate in tensor memory
// and are written once (no atomics on dK/dV). Tensor memory (512 columns),
// with the score buffers doubled so that S^T/dP^T of the next query tile are
// computed while the current one is being turned into P^T/dS^T:
//   buffer X (X = 0, 1) at cols 128X: S^T [128 keys x 64 queries] at +0..63
//   and dP^T at +64..127. Once they are in registers, P^T and dS^T (BF16
//   pairs) and dQ^T [128 dims x 64 queries] (FP32, one N = 64 product) take
//   their place: for D = 128 at +0..31, +96..127 and +32..95; for D = 64 and
//   256 each group g (queries 32g..32g+31) writes P^T and dS^T over its own
//   S^T columns (+32g+0..15, +32g+16..31) and dQ^T replaces dP^T (+64..127).
//   dV [128 keys x D dims] from col 256, dK after it.
// Registers are split per warpgroup (setmaxnreg): load/MMA 88, dQ drain 88,
// each P^T/dS^T warpgroup 168 (launch: 128 for all 512 threads).
// Warp roles: warp 0 loads (TMA for K, V, Q_i, dO_i; plain loads for LSE and
// D), warp 1 issues tcgen05.mma, warps 4-7 and 12-15 turn S^T/dP^T into
// P^T/dS^T (one key per thread; the first group takes queries 0..31 of the
// tile, the second 32..63; for D = 128 they meet at a barrier between loading
// S^T/dP^T and writing P^T/dS^T, for D = 64 and 256 neither writes columns the
// other reads and they run independently) and also store dS^T to shared memory
// (double-buffered, 128-byte swizzle) for the dQ product, warps 8-11 drain
// dQ^T (one head-dim index per thread) into
// a [rows][D] FP32 tile in shared memory, which one thread adds into the
// global dQ accumulator with TMA reduce-adds.
// D = 64: dK and dV take 64 columns each; the dQ^T product keeps M = 128 with
// its A operand running from K into V (the next 64-dim box in shared memory),
// so tensor-memory lanes 64..127 hold V^T dS^T, which the drain ignores.
// D = 256: dK and dV of 128 keys at 256 dims would need all 512 columns, so
// two CTAs share a key tile and each owns half of the head dimensions of dK,
// dV and dQ (blockIdx.x = 2 * key tile + half); both compute the full S^T and
// dP^T (the contraction runs over all 256 dims). K and V of 256 dims leave
// room for one Q/dO stage only, so the products of one query tile are issued
// after the previous tile's, without overlap.
// Split walk (BwdArgs::nsplit = 2, clusters of two CTAs; the kSplit
// instance): both CTAs of a cluster own the same key tile and each walks
// half of its query tiles; at the end CTA 1 copies its dV and dK into CTA
// 0's shared memory (distributed shared memory) and CTA 0 writes the sums.
// The host uses it for the last, partly filled wave of grids without masks.
// The instance without kSplit carries none of that code; which instance
// runs the other grids is the host's choice per head dim (both compute the
// same values).
#pragma once
#include <cmath>
#include <cstdint>
#include <cuda.h>

#include "fwd_kernel.cuh"
#include "ptx.cuh"

namespace attn {

struct BwdArgs {
  const float* lse;         // natural-log LSE, strides l_sh, l_sb, row stride 1
  const float* dvec;        // D = rowsum(dO o O), same layout as lse
  float* dq_acc;            // FP32, layout of q (strides q_sn, q_sh, q_sb)
  void* dq;                 // dQ written directly (deterministic backward), layout of q
  void* dk;                 // layout of k (strides k_sn, k_sh, k_sb)
  void* dv;
  long long q_sn, q_sh, q_sb;
  long long k_sn, k_sh, k_sb;
  long long l_sh, l_sb;
  int Hq, Hkv, group, N;
  const int* cu_seqlens;
  float scale;
  float scale_log2;
  int causal;               // scheduling hint: window (-1, 0)
  int win_left, win_right;  // key j visible to query i iff i - left <= j <= i + right (-1: no bound)
  int* status;
  // Units are (key tile x DSPLIT, KV head, batch), x fastest, tiles_x of
  // them along x. tiles_x = 0: the grid is (tiles x DSPLIT, Hkv, batch or
  // sequences), one unit per CTA. tiles_x > 0: a 1-D grid, CTA blockIdx.x
  // taking part blockIdx.x % nsplit of the walk of unit unit0 + blockIdx.x /
  // nsplit (nsplit = 2 only in the kSplit instance, launched in clusters of
  // two).
  int tiles_x, unit0, nsplit;
  // persistent instance: the grid walks units blockIdx.x, + gridDim.x, ...
  // below `units` (tiles_x * Hkv * batch), in the linear order above
  int units;
};

// kP: the persistent walk's layout. At d = 64 it holds two K/V buffers, so
// the next unit's K and V load while the current unit runs; at d = 128 a
// second buffer would take the room of two of the four Q/dO stages, which
// measured far slower than what it hides (22 % at N = 512).
template <int DT, int D, bool kP = false>
struct BwdCfg {
  static_assert(D == 64 || D == 128 || D == 256, "backward kernel is written for head dim 64, 128 or 256");
  static constexpr int DSPLIT = D == 256 ? 2 : 1;   // CTAs per key tile (each owns DH dims of dK, dV, dQ)
  static constexpr int DH = D / DSPLIT;
  static constexpr int BR = 64;                     // query rows per iteration
  static constexpr int BC = 128;                    // keys per CTA
  static constexpr int NBOX = D / 64;               // 64-element (128-byte) boxes per row
  static constexpr int KV_B = BC * D * 2;           // K or V tile
  static constexpr int KV_BOX_B = BC * 128;
  static constexpr int Q_B = BR * D * 2;            // Q_i or dO_i tile
  static constexpr int Q_BOX_B = BR * 128;
  static constexpr int DS_B = BC * BR * 2;          // dS^T tile [128 keys][64 queries]
  // dS^T tiles in shared memory (the B operand of dQ^T). Head dim 64 has the
  // room for two, one per score buffer: tile g's dS^T then overwrites tile
  // g-2's, whose dQ^T was complete before tile g's S^T/dP^T were issued, so
  // the P^T/dS^T warps never wait for a product.
  static constexpr int NDS = D == 64 ? 2 : 1;
  static constexpr int NKV = kP && D == 64 ? 2 : 1;   // K/V buffers
  static constexpr int NQ = D == 64 ? 6 : (D == 128 ? 4 : 1);   // stages of the Q/dO ring
  static constexpr int LD_B = 2 * BR * 4;           // LSE*log2e and D for one tile
  static constexpr int DQ_ROWS = D == 64 ? BR : BR / 2;   // rows of dQ per reduce-add
  static constexpr int DQ_PARTS = BR / DQ_ROWS;            // reduce-adds per tile
  static constexpr int DQ_STAGE_B = DQ_ROWS * DH * 4;      // FP32 staging for one reduce-add
  // kv_full[NKV], q_full[NQ], q_empty[NQ], sp_full[2], ds_ready[2][2], dq_full, dq_empty, done,
  // kv_empty[NKV], acc_empty
  static constexpr int NBARS = 2 * NKV + 2 * NQ + 2 + 4 + 4;
  static constexpr int SMEM_BYTES =
      NKV * 2 * KV_B + NDS * DS_B + NQ * (2 * Q_B) + DQ_STAGE_B + NQ * LD_B + NBARS * 8 + 16;   // base is 1024-aligned
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA exceeded");
  // a split walk's hand-over of dV and dK ([2][BC][DH] FP32 from offset 0)
  // stays below the barriers
  static_assert(2 * BC * DH * 4 <= 2 * KV_B + NDS * DS_B + NQ * (2 * Q_B) + DQ_STAGE_B + NQ * LD_B, "hand-over area");
  static constexpr int NTHREADS = 512;
  // Registers: the launch gives 128 per thread (the whole register file);
  // the load/MMA warpgroup and the dQ drain warpgroup return part of theirs
  // so the two P^T/dS^T warpgroups, whose per-key work is a set of
  // independent exp2 chains, can keep all of them in flight.
  static constexpr uint32_t kRegsCtl = 88, kRegsDrain = 88, kRegsMath = 168;
  static_assert(128 * (kRegsCtl + kRegsDrain + 2 * kRegsMath) <= NTHREADS * 128, "register split");
  static constexpr int kRegsSplit = 128 * (kRegsCtl + kRegsDrain + 2 * kRegsMath) / NTHREADS;   // per thread
  static constexpr uint32_t FMT = DT == kBF16 ? 1u : 0u;
  static constexpr uint32_t IDESC_SP = instr_desc(128, BR, FMT, FMT, 0, 0);
  static constexpr uint32_t IDESC_KV = instr_desc(128, DH, FMT, FMT, 0, 1);
  static constexpr uint32_t IDESC_DQ = instr_desc(128, BR, FMT, FMT, 1, 1);   // M = 128 also for D = 64
  // within score buffer X (base 128X)
  // Score buffer layout. D = 64, 256: group g's P^T and dS^T go over its own
  // S^T columns (32g + 0..15 and 32g + 16..31) and dQ^T over dP^T, so neither
  // group writes columns the other still has to read and the groups run
  // independently. D = 128 (measured faster): P^T at +0..31, dQ^T at +32..95,
  // dS^T at +96..127, and the groups meet at a barrier between loading their
  // scores and overwriting them.
  static constexpr bool kOwnCols = D != 128;
  static constexpr uint32_t COL_S = 0, COL_DP = 64, COL_DQ = kOwnCols ? 64 : 32;
  // columns of P^T and dS^T for the 16 queries of K step kk, and of group g's writes
  __host__ __device__ static constexpr uint32_t col_p(int kk) { return kOwnCols ? 32 * (kk >> 1) + 8 * (kk & 1) : 8 * kk; }
  __host__ __device__ static constexpr uint32_t col_ds(int kk) { return kOwnCols ? col_p(kk) + 16 : 96 + 8 * kk; }
  static constexpr uint32_t COL_DV = 256, COL_DK = 256 + DH;
  static_assert(COL_DK + DH <= 512, "tensor memory overflow");
};

// Split walk: dV (offset 0) and dK (offset BC * DH floats) of part 1 go to
// part 0's shared memory as [BC keys][DH] FP32, 16-byte groups of each
// 32-column chunk swizzled by key % 8 so that a warp's 32 keys hit distinct
// banks. Key row `row` hands chunks c0 .. c1 - 1 from tensor memory `taddr`.
template <class C>
__device__ __forceinline__ void split_handover(const uint8_t* smem, uint32_t taddr, int row, int c0, int c1,
                                               int off) {
  const uint32_t dst = cluster_map(smem_u32(smem), 0) + 4u * static_cast<uint32_t>(off + row * C::DH);
#pragma unroll 1
  for (int c = c0; c < c1; ++c) {
    uint32_t v[32];
    tmem_ld32(taddr + 32 * c, v);
    tmem_wait_ld();
    reg_fence(v);
#pragma unroll
    for (int w = 0; w < 8; ++w)
      st_cluster_v4(dst + 4u * (32 * c + 4 * (w ^ (row & 7))), v[4 * w], v[4 * w + 1], v[4 * w + 2], v[4 * w + 3]);
  }
}
// Part 0: v (its own chunk c of key row `row`) += part 1's.
template <class C>
__device__ __forceinline__ void split_add(uint32_t (&v)[32], const float* part1, int row, int c) {
  const float* src = part1 + row * C::DH + 32 * c;
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float4 x = *reinterpret_cast<const float4*>(src + 4 * (w ^ (row & 7)));
    v[4 * w] = __float_as_uint(__uint_as_float(v[4 * w]) + x.x);
    v[4 * w + 1] = __float_as_uint(__uint_as_float(v[4 * w + 1]) + x.y);
    v[4 * w + 2] = __float_as_uint(__uint_as_float(v[4 * w + 2]) + x.z);
    v[4 * w + 3] = __float_as_uint(__uint_as_float(v[4 * w + 3]) + x.w);
  }
}

// kDQ = false: dK and dV only (the deterministic backward computes dQ in a
// separate query-stationary kernel); the dQ^T product, its drain and the
// reduce-adds are left out.
template <int DT, int D, bool kDQ = true, bool kSplit = false, bool kPersist = false>
__global__ void __launch_bounds__(512, 1)
bwd_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
           const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmdO,
           const __grid_constant__ CUtensorMap tmdQ, const BwdArgs a) {
  using C = BwdCfg<DT, D, kPersist>;
  static_assert(!kPersist || (!kSplit && C::DSPLIT == 1), "persistent walk: whole units, one CTA per key tile");
  // The layout uses all the shared memory it asks for, with no room to align
  // the base by hand: a base that is not 1024-byte aligned (needed by the
  // swizzled tiles) is reported and the CTA leaves before touching it.
  extern __shared__ __align__(1024) uint8_t bwd_smem[];
  // A split launch follows a 1-D grid of whole units (tiles_x > 0, nsplit =
  // 1) as its programmatic dependent: its clusters may take SMs as this
  // grid's last CTAs leave (it reads nothing this grid writes; dQ both only
  // add into). Every thread signals.
  if constexpr (!kSplit) {
    if (a.tiles_x > 0) grid_launch_dependents();
  }
  if (smem_u32(bwd_smem) & 1023u) {
    if (threadIdx.x == 0 && a.status) atomicExch(a.status, kDevBadSmemAlign);
    return;
  }
  uint8_t* smem = bwd_smem;
  uint8_t* sK = smem;                               // K/V buffer kb: sK + kb * 2 * KV_B, V after K
  uint8_t* sV = sK + C::KV_B;
  uint8_t* sDS = sK + C::NKV * 2 * C::KV_B;         // [NDS][DS_B], 128-byte swizzle
  uint8_t* sQ = sDS + C::NDS * C::DS_B;             // [NQ][Q_B]
  uint8_t* sdO = sQ + C::NQ * C::Q_B;               // [NQ][Q_B]
  float* sDQ = reinterpret_cast<float*>(sdO + C::NQ * C::Q_B);   // [DQ_ROWS][D] FP32
  float* sLD = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sDQ) + C::DQ_STAGE_B);   // [NQ][2*BR]
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sLD) + C::NQ * C::LD_B);
  uint64_t* kv_full = bars;                         // [NKV]
  uint64_t* q_full = bars + C::NKV;
  uint64_t* q_empty = q_full + C::NQ;
  uint64_t* sp_full = q_empty + C::NQ;             // [2], one per score buffer
  // P^T/dS^T ready. With independent groups (kOwnCols) one barrier per score
  // buffer and group, [buffer][group]: a group that runs a tile ahead of the
  // other arrives on the other buffer's barrier, never on this tile's. For
  // D = 128 the groups meet every tile and one barrier of 256 serves.
  uint64_t* ds_ready = sp_full + 2;
  uint64_t* dq_full = ds_ready + 4;
  uint64_t* dq_empty = dq_full + 1;
  uint64_t* done = dq_empty + 1;                    // one phase per unit
  uint64_t* kv_empty = done + 1;                    // [NKV] persistent: the unit's products have read K, V
  uint64_t* acc_empty = kv_empty + C::NKV;          // persistent: dV, dK read out of tensor memory
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(acc_empty + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nsplit = kSplit && a.tiles_x > 0 ? a.nsplit : 1;   // CTAs per unit
  int bx = blockIdx.x, by = blockIdx.y, bz = blockIdx.z, wp = 0;   // wp: this CTA's part of the walk
  if (kSplit && a.tiles_x > 0) {
    const int u = a.unit0 + static_cast<int>(blockIdx.x) / nsplit;
    wp = static_cast<int>(blockIdx.x) % nsplit;
    bx = u % a.tiles_x;
    by = (u / a.tiles_x) % a.Hkv;
    bz = u / a.tiles_x / a.Hkv;
  } else if (a.tiles_x > 0) {   // whole units from unit 0 (the instance without kSplit)
    bx = static_cast<int>(blockIdx.x) % a.tiles_x;
    by = static_cast<int>(blockIdx.x) / a.tiles_x % a.Hkv;
    bz = static_cast<int>(blockIdx.x) / a.tiles_x / a.Hkv;
  } else if (a.causal) {
    // with causal masking key tile 0 has the most work: heavy tiles start
    // first. Packed sequences run in blocks of 64 key tiles per (sequence,
    // KV head): fewer pairs at a time, so more of each pair's Q, dO and dQ
    // lines stay in L2 (a long sequence's are tens of MB).
    heavy_first_order(a.cu_seqlens != nullptr ? 64 : 16, bx, by, bz);
  }
  const bool packed = a.cu_seqlens != nullptr;
  // The unit: KV head, batch (or packed sequence), key tile j, head-dim part
  // dh; query tiles i0 .. i0 + per_head - 1 of each query head of the group
  int hkv, b, seq0, L, j, dh, i0, per_head, it_base, niter, rot;
  auto set_unit = [&](int ux, int uy, int uz) {
    hkv = uy;
    if (packed) {
      b = 0;
      seq0 = a.cu_seqlens[uz];
      L = a.cu_seqlens[uz + 1] - seq0;
    } else {
      b = uz;
      seq0 = 0;
      L = a.N;
    }
    j = ux / C::DSPLIT;             // key tile
    dh = ux % C::DSPLIT;            // which DH head dims of dK, dV, dQ this CTA owns
    // query tiles holding a query that sees a key of this tile
    const int klast = min(j * C::BC + C::BC, L) - 1;
    const int qlo = a.win_right < 0 ? 0 : max(0, j * C::BC - a.win_right);
    const int qhi = a.win_left < 0 ? L - 1 : min(L - 1, klast + a.win_left);
    i0 = qlo / C::BR;
    per_head = qhi / C::BR + 1 - i0;
    // this CTA's part of the walk over (query head, query tile): iterations
    // it_base .. it_base + niter - 1 of the group * per_head
    it_base = wp * (a.group * per_head) / nsplit;
    niter = (wp + 1) * (a.group * per_head) / nsplit - it_base;
    // Each key tile starts its walk at a different query tile, so the CTAs
    // of one head neither load the same Q/dO tile nor add into the same dQ
    // rows at the same moment.
    rot = j % per_head;
  };
  set_unit(bx, by, bz);
  if (j * C::BC >= L) return;
  // Persistent walk (dense rows without masks): unit k of this CTA is
  // blockIdx.x + k * gridDim.x while below a.units. Every unit has the same
  // query tiles (i0 = 0, per_head, niter); only the key tile, KV head and
  // batch change. Every role walks the same units, and the barrier phases
  // run on across them (counted in tiles g of the whole walk, or in units k).
  auto more_units = [&](int k) -> bool {
    return kPersist && static_cast<long long>(blockIdx.x) + static_cast<long long>(k) * gridDim.x < a.units;
  };
  // offset of key row `row` of unit k in dK and dV (dense layout), from the
  // unit index alone, so that the unit's coordinates need not stay live
  // through its tiles
  auto persist_key_off = [&](int k, int row) -> long long {
    const int ui = static_cast<int>(blockIdx.x + static_cast<unsigned>(k) * gridDim.x);
    const int uj = ui % a.tiles_x, uh = ui / a.tiles_x % a.Hkv, ub = ui / a.tiles_x / a.Hkv;
    return static_cast<long long>(ub) * a.k_sb + static_cast<long long>(uh) * a.k_sh +
           static_cast<long long>(uj * C::BC + row) * a.k_sn;
  };
  auto persist_key_row = [&](int k, int row) {
    return static_cast<int>(blockIdx.x + static_cast<unsigned>(k) * gridDim.x) % a.tiles_x * C::BC + row;
  };
  auto next_unit = [&](int k) -> bool {
    if constexpr (!kPersist) {
      return false;
    } else {
      if (!more_units(k)) return false;
      const int ui = static_cast<int>(blockIdx.x + static_cast<unsigned>(k) * gridDim.x);
      j = ui % a.tiles_x;
      hkv = ui / a.tiles_x % a.Hkv;
      b = ui / a.tiles_x / a.Hkv;
      rot = j % per_head;
      return true;
    }
  };
  // Query tile and head of local iteration it
  auto q_tile = [&](int it) {
    const int r = (it_base + it) % per_head + rot;
    return i0 + (r >= per_head ? r - per_head : r);
  };
  auto q_head = [&](int it) { return hkv * a.group + (it_base + it) / per_head; };

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmdO);
    tma_prefetch_desc(&tmdQ);
    for (int s = 0; s < C::NKV; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(&q_full[s], 2);   // TMA transaction + the LSE/D stores
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(&sp_full[0], 1);
    mbar_init(&sp_full[1], 1);
    if constexpr (C::kOwnCols) {
      for (int i = 0; i < 4; ++i) mbar_init(&ds_ready[i], 128);
    } else {
      mbar_init(&ds_ready[0], 256);
    }
    mbar_init(dq_full, 1);
    mbar_init(dq_empty, 128);
    mbar_init(done, 1);
    mbar_init(acc_empty, 384);   // the two P^T/dS^T groups (dV) and the drain warps (dK)
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
  if constexpr (kSplit) {
    if (nsplit == 1) grid_launch_dependents();   // as above, for this instance's own whole-unit grids
  }

  // Each role changes its register budget inside its own branch, so the
  // compiler sizes every role's code for the budget it runs with.
  if (warp < 4) {
  regs_dec<C::kRegsCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ loads
    int gt = 0;   // tiles of the earlier units
    for (int k = 0;; ++k) {
      const int kb = k % C::NKV;   // K/V buffer of unit k
      if (k > 0) {
        if (!next_unit(k)) break;
        // buffer kb was last read by unit k - NKV, whose last products must complete
        if (k >= C::NKV && !__all_sync(0xffffffffu, mbar_wait(&kv_empty[kb], (k / C::NKV - 1) & 1, a.status))) break;
      }
      const int krow = seq0 + j * C::BC;
      if (lane == 0) {
        uint8_t* bK = sK + kb * 2 * C::KV_B;
        uint8_t* bV = bK + C::KV_B;
        mbar_arrive_expect_tx(&kv_full[kb], 2 * C::KV_B);
        for (int c = 0; c < C::NBOX; ++c) {
          if (packed) {
            tma_load_4d(bK + c * C::KV_BOX_B, &tmK, &kv_full[kb], c * 64, hkv, krow, 0);
            tma_load_4d(bV + c * C::KV_BOX_B, &tmV, &kv_full[kb], c * 64, hkv, krow, 0);
          } else {
            tma_load_4d(bK + c * C::KV_BOX_B, &tmK, &kv_full[kb], c * 64, krow, hkv, b);
            tma_load_4d(bV + c * C::KV_BOX_B, &tmV, &kv_full[kb], c * 64, krow, hkv, b);
          }
        }
      }
      bool ok = true;
      for (int it = 0; it < niter; ++it) {
        const int g = gt + it;
        const int st = g % C::NQ;
        const int h = q_head(it);
        const int q0 = q_tile(it) * C::BR;
        // LSE and D of this tile are fetched before waiting for the stage (they
        // do not depend on it), so their latency hides behind that wait
        const long long lrow = static_cast<long long>(b) * a.l_sb + static_cast<long long>(h) * a.l_sh + seq0;
        float nl[C::BR / 32], nd[C::BR / 32];
  #pragma unroll
        for (int u = 0; u < C::BR / 32; ++u) {
          const int q = q0 + lane + 32 * u;
          const bool in = q < L;
          nl[u] = in ? -a.lse[lrow + q] * kLog2e : -INFINITY;    // -LSE in log2 units
          nd[u] = in ? -a.dvec[lrow + q] : 0.f;                  // -D
        }
        if (!__all_sync(0xffffffffu, mbar_wait(&q_empty[st], ((g / C::NQ) & 1) ^ 1, a.status))) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&q_full[st], 2 * C::Q_B);
          for (int c = 0; c < C::NBOX; ++c) {
            uint8_t* dq = sQ + st * C::Q_B + c * C::Q_BOX_B;
            uint8_t* dd = sdO + st * C::Q_B + c * C::Q_BOX_B;
            if (packed) {
              tma_load_4d(dq, &tmQ, &q_full[st], c * 64, h, seq0 + q0, 0);
              tma_load_4d(dd, &tmdO, &q_full[st], c * 64, h, seq0 + q0, 0);
            } else {
              tma_load_4d(dq, &tmQ, &q_full[st], c * 64, q0, h, b);
              tma_load_4d(dd, &tmdO, &q_full[st], c * 64, q0, h, b);
            }
          }
        }
        float* ld = sLD + st * 2 * C::BR;
  #pragma unroll
        for (int u = 0; u < C::BR / 32; ++u) {
          ld[lane + 32 * u] = nl[u];
          ld[C::BR + lane + 32 * u] = nd[u];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&q_full[st]);
        __syncwarp();
      }
      if (!ok || !kPersist) break;
      gt += niter;
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA
    // Order: SdP(0); per iteration it: SdP(it+1) into the other buffer, then
    // (after P^T/dS^T of it are ready) the two dQ^T halves, dV and dK of it.
    if (lane == 0) {
      // Descriptors are built once; a byte offset is added to the
      // start-address field (16-byte units) for each K step and stage.
      const uint64_t dK_kmaj = smem_desc(smem_u32(sK), 16, 1024, kSwizzle128);
      const uint64_t dV_kmaj = smem_desc(smem_u32(sV), 16, 1024, kSwizzle128);
      // K^T for this CTA's head dims (boxes of 64 dims, KV_BOX_B apart)
      const uint64_t dK_mn = smem_desc(smem_u32(sK) + dh * (C::DH / 64) * C::KV_BOX_B, C::KV_BOX_B, 1024,
                                       kSwizzle128);
      const uint64_t dQ0_kmaj = smem_desc(smem_u32(sQ), 16, 1024, kSwizzle128);
      const uint64_t ddO0_kmaj = smem_desc(smem_u32(sdO), 16, 1024, kSwizzle128);
      // Q_i and dO_i as MN-major B of dK and dV: this CTA's head dims only
      const uint32_t dh_off = dh * (C::DH / 64) * C::Q_BOX_B;
      const uint64_t dQ0_mn = smem_desc(smem_u32(sQ) + dh_off, C::Q_BOX_B, 1024, kSwizzle128);
      const uint64_t ddO0_mn = smem_desc(smem_u32(sdO) + dh_off, C::Q_BOX_B, 1024, kSwizzle128);
      const uint64_t dDS0_mn = smem_desc(smem_u32(sDS), C::DS_B, 1024, kSwizzle128);
      auto dadd = [](uint64_t d, uint32_t bytes) { return d + (bytes >> 4); };
      auto ds_wait = [&](int g) {   // P^T and dS^T of tile g are in tensor memory
        if constexpr (C::kOwnCols)
          return mbar_wait(&ds_ready[(g & 1) * 2], (g >> 1) & 1, a.status) &&
                 mbar_wait(&ds_ready[(g & 1) * 2 + 1], (g >> 1) & 1, a.status);
        else
          return mbar_wait(&ds_ready[0], g & 1, a.status);
      };
      // kvo: byte offset of the unit's K/V buffer
      auto issue_sdp = [&](int g, uint32_t kvo) {   // S^T = K Q^T and dP^T = V dO^T into buffer g % 2
        const uint32_t so = (g % C::NQ) * C::Q_B;
        const uint32_t xb = tbase + 128u * (g & 1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offk = kvo + (kk / 4) * C::KV_BOX_B + (kk % 4) * 32;
          const uint32_t offq = so + (kk / 4) * C::Q_BOX_B + (kk % 4) * 32;
          mma_ss<false>(xb + C::COL_S, dadd(dK_kmaj, offk), dadd(dQ0_kmaj, offq), C::IDESC_SP, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t offk = kvo + (kk / 4) * C::KV_BOX_B + (kk % 4) * 32;
          const uint32_t offq = so + (kk / 4) * C::Q_BOX_B + (kk % 4) * 32;
          mma_ss<false>(xb + C::COL_DP, dadd(dV_kmaj, offk), dadd(ddO0_kmaj, offq), C::IDESC_SP, kk > 0);
        }
        mma_commit(&sp_full[g & 1]);
      };
      // With several Q/dO stages dQ^T goes first, so the drain warps can read
      // it while dV and dK run and the next S^T/dP^T never waits for an empty
      // tensor pipe. With one stage the next tile's loads wait for the stage:
      // dV and dK (its last readers) go first and release it, and dQ^T runs
      // while the loads are in flight.
      // g: tile of the walk, it: tile of unit k (it = 0 starts dV and dK)
      auto issue_grads = [&](int g, int it, int k, uint32_t kvo) {
        const uint32_t xb = tbase + 128u * (g & 1);
        const uint32_t so = (g % C::NQ) * C::Q_B;
        auto issue_dq = [&]() {
          if constexpr (kDQ) {
#pragma unroll
            for (int kk = 0; kk < C::BC / 16; ++kk) {   // dQ^T = K^T dS^T, both MN-major
              mma_ss<false>(xb + C::COL_DQ, dadd(dK_mn, kvo + kk * 2048),
                            dadd(dDS0_mn, (C::NDS > 1 ? (g & 1) * C::DS_B : 0) + kk * 2048), C::IDESC_DQ, kk > 0);
            }
            mma_commit(dq_full);
          }
        };
        if constexpr (C::NQ > 1) issue_dq();
        // a persistent walk's next unit starts dV and dK once the previous
        // unit's have been read out of tensor memory
        if (kPersist && it == 0 && k > 0 && !mbar_wait(acc_empty, (k - 1) & 1, a.status)) return false;
#pragma unroll
        for (int kk = 0; kk < C::BR / 16; ++kk) {   // dV += P^T dO_i
          mma_ts<false>(tbase + C::COL_DV, xb + C::col_p(kk), dadd(ddO0_mn, so + kk * 2048), C::IDESC_KV,
                        (it > 0 || kk > 0) ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < C::BR / 16; ++kk) {   // dK += dS^T Q_i
          mma_ts<false>(tbase + C::COL_DK, xb + C::col_ds(kk), dadd(dQ0_mn, so + kk * 2048), C::IDESC_KV,
                        (it > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&q_empty[g % C::NQ]);
        if constexpr (C::NQ == 1) issue_dq();
        return true;
      };
      if constexpr (!kPersist) {
        bool ok = mbar_wait(kv_full, 0, a.status);
        if constexpr (C::NQ == 1) {
          // one Q/dO stage: tile it's products, then tile it+1's
          for (int it = 0; it < niter && ok; ++it) {
            if (!(ok = mbar_wait(&q_full[0], it & 1, a.status))) break;
            // buffer it%2 was last used by it-2, whose dQ^T was drained before it-1's
            if (kDQ && it > 0 && !(ok = mbar_wait(dq_empty, (it - 1) & 1, a.status))) break;
            tc_fence_after();
            issue_sdp(it, 0);
            if (!(ok = ds_wait(it))) break;
            tc_fence_after();
            issue_grads(it, it, 0, 0);
          }
        } else {
          ok = ok && mbar_wait(&q_full[0], 0, a.status);
          if (ok) {
            tc_fence_after();
            issue_sdp(0, 0);
          }
          for (int it = 0; it < niter && ok; ++it) {
            if (it + 1 < niter) {
              // buffer (it+1)%2 was last used by it-1: its dQ^T halves must be drained
              const int sn = (it + 1) % C::NQ;
              if (!(ok = mbar_wait(&q_full[sn], ((it + 1) / C::NQ) & 1, a.status))) break;
              if (kDQ && !(ok = mbar_wait(dq_empty, (it & 1) ^ 1, a.status))) break;
              tc_fence_after();
              issue_sdp(it + 1, 0);
            }
            if (!(ok = ds_wait(it))) break;
            // The drain warps wait on dq_full by parity. On the last tile there is
            // no S^T/dP^T issue (and no dq_empty wait) above, so wait here for the
            // drain of it-1: dq_full then never runs two phases ahead of them.
            if (kDQ && it + 1 >= niter && it > 0 && !(ok = mbar_wait(dq_empty, (it & 1) ^ 1, a.status))) break;
            tc_fence_after();
            issue_grads(it, it, 0, 0);
          }
        }
        mma_commit(done);
      } else {
        // Persistent walk (several Q/dO stages): tiles are counted over the
        // whole walk (g), so the order within a unit is the one above. With
        // two K/V buffers, at a unit's last tile the next unit's first
        // S^T/dP^T (from the other buffer) is issued before the last tile's
        // gradients, so its softmax overlaps them; with one, the next unit's
        // K and V load once the last products have read the buffer.
        static_assert(C::NQ > 1, "persistent walk with several Q/dO stages");
        constexpr bool kAhead = C::NKV > 1;
        int gt = 0;             // tiles of the earlier units
        bool ok = true;
        bool first_issued = false;   // this unit's first S^T/dP^T went out with the previous unit
        for (int k = 0; ok; ++k) {
          if (k > 0 && !more_units(k)) break;
          const uint32_t kvo = (k % C::NKV) * 2 * C::KV_B;
          const bool more = kAhead && more_units(k + 1);
          if (!first_issued) {
            ok = mbar_wait(&kv_full[k % C::NKV], (k / C::NKV) & 1, a.status) &&
                 mbar_wait(&q_full[gt % C::NQ], (gt / C::NQ) & 1, a.status);
            if (ok) {
              tc_fence_after();
              issue_sdp(gt, kvo);
            }
          }
          first_issued = false;
          for (int it = 0; it < niter && ok; ++it) {
            const int g = gt + it;
            const bool last = it + 1 >= niter;
            if (!last || more) {
              // tile g+1: this unit's next, or the next unit's first
              if (last && !(ok = mbar_wait(&kv_full[(k + 1) % C::NKV], ((k + 1) / C::NKV) & 1, a.status))) break;
              const int sn = (g + 1) % C::NQ;
              if (!(ok = mbar_wait(&q_full[sn], ((g + 1) / C::NQ) & 1, a.status))) break;
              // buffer (g+1)%2 was last used by g-1: its dQ^T halves must be drained
              if (kDQ && !(ok = mbar_wait(dq_empty, (g & 1) ^ 1, a.status))) break;
              tc_fence_after();
              issue_sdp(g + 1, last ? ((k + 1) % C::NKV) * 2 * C::KV_B : kvo);
              first_issued = last;
            }
            if (!(ok = ds_wait(g))) break;
            // a unit's last tile without the next unit's first products above:
            // as in the single-unit loop, the drain of g-1 first
            if (kDQ && last && !more && g > 0 && !(ok = mbar_wait(dq_empty, (g & 1) ^ 1, a.status))) break;
            tc_fence_after();
            ok = issue_grads(g, it, k, kvo);
          }
          mma_commit(done);
          mma_commit(&kv_empty[k % C::NKV]);
          gt += niter;
      }
      }
    }
    __syncwarp();
  }
  // the two barriers of the split-walk hand-over (see the dV and dK stores)
  if (kSplit && nsplit > 1) {
    __syncwarp();
    cluster_sync_all();
    cluster_sync_all();
  }
  } else if ((warp >= 4 && warp < 8) || warp >= 12) {
    regs_inc<C::kRegsMath>();
    // -------------------------------------------------- P^T and dS^T
    const int half = warp >= 12 ? 1 : 0;            // queries 32*half .. +31 of each tile
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;              // key row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float2 sl2v = make_float2(a.scale_log2, a.scale_log2);
    bool ok = true;
    bool dq_ok = true;   // the wait for the previous tile's dQ^T ended in time
    int gt = 0;          // tiles of the earlier units
    for (int k = 0;; ++k) {
      if (k > 0 && !next_unit(k)) break;
      const int kloc = j * C::BC + r;                 // key position in the sequence
      const bool kvalid = kloc < L;
      for (int it = 0; it < niter; ++it) {
        const int g = gt + it;
        const uint32_t xb = tbase + lane_off + 128u * (g & 1);
        uint8_t* ds_row = sDS + (C::NDS > 1 ? (g & 1) * C::DS_B : 0) + r * 128;
        const int st = g % C::NQ;
        // LSE and D of this stage (written by the load warp before it arrived
        // on q_full[st]) go to registers first: these shared-memory reads then
        // overlap the wait for S^T/dP^T instead of heading every exp2 chain
        // while the tensor core's operand reads keep shared memory busy.
        bool got = __all_sync(0xffffffffu, mbar_wait(&q_full[st], (g / C::NQ) & 1, a.status));
        float4 l4r[8], d4r[8];
        if (got) {
          const float* nlse = sLD + st * 2 * C::BR + 32 * half;     // -LSE * log2(e)
  #pragma unroll
          for (int e4 = 0; e4 < 8; ++e4) {
            l4r[e4] = *reinterpret_cast<const float4*>(nlse + 4 * e4);
            d4r[e4] = *reinterpret_cast<const float4*>(nlse + C::BR + 4 * e4);   // -D
          }
        }
        if (got) got = __all_sync(0xffffffffu, mbar_wait(&sp_full[g & 1], (g >> 1) & 1, a.status));
        got = got && dq_ok;   // a wait that ran out in the previous tile ends both groups here
        uint32_t sv[32], dp[32];
        if (got) {
          tc_fence_after();
          tmem_ld32(xb + C::COL_S + 32 * half, sv);
          tmem_ld32(xb + C::COL_DP + 32 * half, dp);
          tmem_wait_ld();
          reg_fence(sv);
          reg_fence(dp);
        }
        // D = 128: both groups have their scores in registers before either
        // overwrites columns the other reads; one decision for both groups
        if constexpr (!C::kOwnCols) ok = named_bar_and(2, 256, got);
        else ok = got;
        if (!ok) break;
        const int q0 = q_tile(it) * C::BR + 32 * half;
        // this key against queries q0 .. q0 + 31: outside the sequence or the window?
        const bool edge = kPersist ? !kvalid
                                   : !kvalid || (a.win_right >= 0 && kloc > q0 + a.win_right) ||
                                         (a.win_left >= 0 && kloc < q0 + 31 - a.win_left);
        uint32_t pp[16], dd[16];
  #pragma unroll
        for (int e4 = 0; e4 < 8; ++e4) {
          const float4 l4 = l4r[e4];
          const float4 d4 = d4r[e4];
          float2 x01 = ffma2(make_float2(__uint_as_float(sv[4 * e4]), __uint_as_float(sv[4 * e4 + 1])), sl2v,
                             make_float2(l4.x, l4.y));
          float2 x23 = ffma2(make_float2(__uint_as_float(sv[4 * e4 + 2]), __uint_as_float(sv[4 * e4 + 3])), sl2v,
                             make_float2(l4.z, l4.w));
          float p[4] = {ex2(x01.x), ex2(x01.y), ex2(x23.x), ex2(x23.y)};
          if (edge) {
  #pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int q = q0 + 4 * e4 + u;
              if (!kvalid || (a.win_right >= 0 && kloc > q + a.win_right) || (a.win_left >= 0 && kloc < q - a.win_left))
                p[u] = 0.f;
            }
          }
          const float2 t01 = fadd2(make_float2(__uint_as_float(dp[4 * e4]), __uint_as_float(dp[4 * e4 + 1])),
                                   make_float2(d4.x, d4.y));
          const float2 t23 = fadd2(make_float2(__uint_as_float(dp[4 * e4 + 2]), __uint_as_float(dp[4 * e4 + 3])),
                                   make_float2(d4.z, d4.w));
          const float2 g01 = fmul2(make_float2(p[0], p[1]), t01);
          const float2 g23 = fmul2(make_float2(p[2], p[3]), t23);
          if constexpr (DT == kBF16) {
            pp[2 * e4] = pack_bf16x2(p[0], p[1]);
            pp[2 * e4 + 1] = pack_bf16x2(p[2], p[3]);
            dd[2 * e4] = pack_bf16x2(g01.x, g01.y);
            dd[2 * e4 + 1] = pack_bf16x2(g23.x, g23.y);
          } else {
            pp[2 * e4] = pack_f16x2(p[0], p[1]);
            pp[2 * e4 + 1] = pack_f16x2(p[2], p[3]);
            dd[2 * e4] = pack_f16x2(g01.x, g01.y);
            dd[2 * e4 + 1] = pack_f16x2(g23.x, g23.y);
          }
        }
        tmem_st16(xb + C::col_p(2 * half), pp);
        tmem_st16(xb + C::col_ds(2 * half), dd);
        // dS^T row r, queries 32*half .. +31: 16-byte chunks 4*half .. +3 of a
        // 128-byte row, 128-byte swizzle (chunk ^= row % 8). A single dS^T
        // tile is read by dQ^T of the previous tile, which must be complete
        // first; waiting only here lets this tile's exponentials overlap it.
        // With two, this tile's buffer was last read by dQ^T of tile g-2,
        // drained before S^T/dP^T of this tile were issued.
        if constexpr (kDQ) {
          if (C::NDS == 1 && g > 0) dq_ok = __all_sync(0xffffffffu, mbar_wait(dq_full, (g - 1) & 1, a.status));
  #pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int chunk = (4 * half + c4) ^ (r & 7);
            *reinterpret_cast<uint4*>(ds_row + chunk * 16) =
                make_uint4(dd[4 * c4], dd[4 * c4 + 1], dd[4 * c4 + 2], dd[4 * c4 + 3]);
          }
        }
        tmem_wait_st();
        if constexpr (kDQ) fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(C::kOwnCols ? &ds_ready[(g & 1) * 2 + half] : &ds_ready[0]);
      }
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(done, k & 1, a.status));
      tc_fence_after();
      // dV rows, this CTA's columns, DH/2 per group. With a split walk part 1
      // hands its dV to part 0 (between the two cluster barriers, once both
      // parts' products are complete and part 0's shared memory is idle), and
      // part 0 stores the sum.
      const float* add = nullptr;
      if (kSplit && nsplit > 1) {
        cluster_sync_all();
        if (ok && wp == 1) split_handover<C>(smem, tbase + lane_off + C::COL_DV, r, half * (C::DH / 64),
                                             (half + 1) * (C::DH / 64), 0);
        cluster_sync_all();
        add = reinterpret_cast<const float*>(smem);
      }
      if (ok && wp == 0) {
        const long long off = kPersist ? persist_key_off(k, r)
                                       : static_cast<long long>(b) * a.k_sb + static_cast<long long>(hkv) * a.k_sh +
                                             static_cast<long long>(seq0 + kloc) * a.k_sn;
  #pragma unroll 1
        for (int c = half * (C::DH / 64); c < (half + 1) * (C::DH / 64); ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + C::COL_DV + 32 * c, v);
          tmem_wait_ld();
          reg_fence(v);
          if (kSplit && add) split_add<C>(v, add, r, c);
          uint32_t pk[16];
  #pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = (DT == kBF16) ? pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]))
                                  : pack_f16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
          if (kvalid) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dv) + off + dh * C::DH + 32 * c);
  #pragma unroll
            for (int w = 0; w < 4; ++w) dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
          }
        }
      }
      if constexpr (kPersist) {   // dV is read out: the next unit may start it
        tc_fence_before();
        mbar_arrive(acc_empty);
      }
      if (!ok || !kPersist) break;
      gt += niter;
    }
  } else {
    regs_dec<C::kRegsDrain>();
    // ---------------------------------------------------- dQ^T drain
    const int quarter = warp & 3;
    const int dim = quarter * 32 + lane;            // head-dim index = tensor-memory lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    bool ok = true;
    int gt = 0;   // tiles of the earlier units
    for (int k = 0;; ++k) {
      if (k > 0 && !next_unit(k)) break;
      for (int it = 0; it < (kDQ ? niter : 0); ++it) {
        const int g = gt + it;
        // one decision for all four drain warps, so none is left alone at the
        // named barriers below
        ok = named_bar_and(1, 128, __all_sync(0xffffffffu, mbar_wait(dq_full, g & 1, a.status)));
        if (!ok) break;
        tc_fence_after();
        uint32_t x0[32], x1[32];
        tmem_ld32(tbase + lane_off + 128u * (g & 1) + C::COL_DQ, x0);
        tmem_ld32(tbase + lane_off + 128u * (g & 1) + C::COL_DQ + 32, x1);
        tmem_wait_ld();
        reg_fence(x0);
        reg_fence(x1);
        tc_fence_before();
        mbar_arrive(dq_empty);
        const int h = q_head(it);
        const int q0 = q_tile(it) * C::BR;
        // reduce-adds of DQ_ROWS rows through one FP32 staging buffer; rows past
        // the sequence hold exact zeros (P = 0 there): for the dense layout the
        // map clips them, for the packed layout they add 0 to the next
        // sequence's rows
  #pragma unroll
        for (int part = 0; part < C::DQ_PARTS; ++part) {
          if (threadIdx.x == 256) bulk_wait_read_all();   // previous reduce-add has read the buffer
          named_bar_sync(1, 128);
          if (quarter * 32 < C::DH) {                     // D = 64: lanes 64..127 are not dQ
            // row q of the staging tile holds dQ of query q; lane l's value of
            // query q goes to word 32 * quarter + l of that row: four queries
            // per stmatrix, lane l addressing query +l/8, words +4(l%8) .. +3
            const uint32_t row = smem_u32(sDQ) + ((lane >> 3) * C::DH + quarter * 32 + 4 * (lane & 7)) * 4;
            if constexpr (C::DQ_PARTS == 2) {
              const uint32_t(&x)[32] = part == 0 ? x0 : x1;
  #pragma unroll
              for (int g = 0; g < 8; ++g)
                stmatrix_x4(row + 16 * g * C::DH, x[4 * g], x[4 * g + 1], x[4 * g + 2], x[4 * g + 3]);
            } else {
  #pragma unroll
              for (int g = 0; g < 8; ++g) {
                stmatrix_x4(row + 16 * g * C::DH, x0[4 * g], x0[4 * g + 1], x0[4 * g + 2], x0[4 * g + 3]);
                stmatrix_x4(row + 16 * (g + 8) * C::DH, x1[4 * g], x1[4 * g + 1], x1[4 * g + 2], x1[4 * g + 3]);
              }
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(1, 128);
          if (threadIdx.x == 256) {
            const int row = q0 + C::DQ_ROWS * part;
            if (packed) tma_reduce_add_4d(&tmdQ, sDQ, dh * C::DH, h, seq0 + row, 0);
            else tma_reduce_add_4d(&tmdQ, sDQ, dh * C::DH, row, h, b);
            bulk_commit();
          }
        }
      }
      if (!kPersist && threadIdx.x == 256) bulk_wait_all();
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(done, k & 1, a.status));
      tc_fence_after();
      // dK rows (here the lane indexes keys), times scale; a split walk's part 1
      // hands its dK to part 0 as for dV
      const float* add = nullptr;
      if (kSplit && nsplit > 1) {
        cluster_sync_all();
        if (ok && wp == 1) split_handover<C>(smem, tbase + lane_off + C::COL_DK, dim, 0, C::DH / 32, C::BC * C::DH);
        cluster_sync_all();
        add = reinterpret_cast<const float*>(smem) + C::BC * C::DH;
      }
      if (ok && wp == 0) {
        const int kloc = kPersist ? persist_key_row(k, dim) : j * C::BC + dim;
        const long long off = kPersist ? persist_key_off(k, dim)
                                       : static_cast<long long>(b) * a.k_sb + static_cast<long long>(hkv) * a.k_sh +
                                             static_cast<long long>(seq0 + kloc) * a.k_sn;
  #pragma unroll 1
        for (int c = 0; c < C::DH / 32; ++c) {
          uint32_t v[32];
          tmem_ld32(tbase + lane_off + C::COL_DK + 32 * c, v);
          tmem_wait_ld();
          reg_fence(v);
          if (kSplit && add) split_add<C>(v, add, dim, c);
          uint32_t pk[16];
  #pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float x0 = __uint_as_float(v[2 * e]) * a.scale, x1 = __uint_as_float(v[2 * e + 1]) * a.scale;
            pk[e] = (DT == kBF16) ? pack_bf16x2(x0, x1) : pack_f16x2(x0, x1);
          }
          if (kloc < L) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.dk) + off + dh * C::DH + 32 * c);
  #pragma unroll
            for (int w = 0; w < 4; ++w) dst[w] = make_uint4(pk[4 * w], pk[4 * w + 1], pk[4 * w + 2], pk[4 * w + 3]);
          }
        }
      }
      if constexpr (kPersist) {   // dK is read out: the next unit may start it
        tc_fence_before();
        mbar_arrive(acc_empty);
      }
      if (!ok || !kPersist) break;
      gt += niter;
    }
    if (kPersist && threadIdx.x == 256) bulk_wait_all();
  }
  // the split grid completes only after the grid it depends on, so work
  // queued after it (the dQ conversion) sees both grids' results
  if (kSplit && nsplit > 1) grid_wait_prerequisites();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// Launches of the kSplit instance (bwd_split.cu): with nsplit = 2, 2 * n CTAs
// in clusters of two over units a.unit0 .. a.unit0 + n - 1 (a.tiles_x units
// along x); with nsplit = 1, the grid `grid` of whole units.
template <int DT, int D, bool kDQ>
cudaError_t launch_bwd_split(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q, const CUtensorMap& d,
                             const CUtensorMap& dq, const BwdArgs& a, int n, dim3 grid, cudaStream_t st);

// Launch of the persistent instance (bwd_persist.cu; D = 64, 128, with dQ):
// `grid` CTAs walk units blockIdx.x, + grid, ... below a.units.
template <int DT, int D>
cudaError_t launch_bwd_persist(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                               const CUtensorMap& d, const CUtensorMap& dq, const BwdArgs& a, int grid,
                               cudaStream_t st);

}  // namespace attn
