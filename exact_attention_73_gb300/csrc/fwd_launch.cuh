// Launch helper for one forward instance.
#pragma once
#include "internal.h"

namespace attn {

// Longest rows (dense N or longest packed sequence) run persistent.
constexpr int kFwdPersistMaxRows = 2048;

// Two-tile instances over short rows run persistent: one CTA per SM walks
// the units, so one unit's epilogue overlaps the next unit's loads and S
// products; there a unit holds few KV steps and its set-up and epilogue
// weigh. The same holds for a window bounded on both sides whose span is
// short, however long the rows. Over long rows, and with causal masking
// (units of unequal work, which the hardware's dispatch in heavy-first
// order balances better than a fixed deal), each CTA takes one unit.
inline bool fwd_persistent(int qt, const FwdArgs& a, int rows) {
  if (qt != 2 || a.causal) return false;
  if (a.win_left < 0 && a.win_right < 0) return rows <= kFwdPersistMaxRows;
  return a.win_left >= 0 && a.win_right >= 0 && a.win_left + a.win_right + 256 <= kFwdPersistMaxRows;
}

template <int DT, int D, int QT, bool kPersist>
cudaError_t launch_fwd_grid(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v, const FwdArgs& u,
                            long long units, cudaStream_t st) {
  using C = FwdCfg<DT, D, QT>;
  auto kern = fwd_kernel<DT, D, QT, kPersist>;
  cudaError_t e = smem_attr_once<fwd_kernel<DT, D, QT, kPersist>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if constexpr (QT >= 2) {   // the role split must fit the registers of the launch
    constexpr int kSplit = (128 * C::kRegsCtl + 128 * QT * C::kRegsSoft + C::NTHREADS - 1) / C::NTHREADS;
    if ((e = reg_pool_once<fwd_kernel<DT, D, QT, kPersist>>(C::NTHREADS, kSplit)) != cudaSuccess) return e;
  }
  long long grid = units;
  if (kPersist) {
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (grid > sms) grid = sms;
  }
  kern<<<static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, st>>>(q, k, v, u);
  return cudaGetLastError();
}

template <int DT, int D, int QT>
cudaError_t launch_fwd_inst(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const FwdArgs& a, int rows, int gy, int gz, cudaStream_t st) {
  FwdArgs u = a;
  u.ux = (rows + 128 * QT - 1) / (128 * QT);
  u.uy = gy;
  u.uz = gz;
  const long long units = static_cast<long long>(u.ux) * gy * gz;
  if (units > INT32_MAX) return cudaErrorInvalidValue;
  if constexpr (QT == 2) {
    if (fwd_persistent(QT, a, rows)) return launch_fwd_grid<DT, D, QT, true>(q, k, v, u, units, st);
  }
  return launch_fwd_grid<DT, D, QT, false>(q, k, v, u, units, st);
}

}  // namespace attn
