// Launch helper for one forward instance.
#pragma once
#include "internal.h"

namespace attn {

template <int DT, int D, int QT>
cudaError_t launch_fwd_inst(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const FwdArgs& a, int rows, int gy, int gz, cudaStream_t st) {
  using C = FwdCfg<DT, D, QT>;
  auto kern = fwd_kernel<DT, D, QT>;
  cudaError_t e = smem_attr_once<fwd_kernel<DT, D, QT>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const dim3 grid((rows + 128 * QT - 1) / (128 * QT), gy, gz);
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, st>>>(q, k, v, a);
  return cudaGetLastError();
}

}  // namespace attn
