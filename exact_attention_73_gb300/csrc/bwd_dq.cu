// Launcher of the deterministic backward's dQ kernel (query-stationary).
#include "bwd_dq_kernel.cuh"
#include "ops.h"

namespace attn {

namespace {

template <int DT, int D>
cudaError_t launch(const CUtensorMap& q, const CUtensorMap& dout, const CUtensorMap& k, const CUtensorMap& v,
                   const BwdArgs& a, int max_len, int nz, cudaStream_t st) {
  using C = DqCfg<DT, D>;
  auto kern = bwd_dq_kernel<DT, D>;
  cudaError_t e = smem_attr_once<bwd_dq_kernel<DT, D>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if ((e = reg_pool_once<bwd_dq_kernel<DT, D>>(C::NTHREADS, C::kRegsSplit)) != cudaSuccess) return e;
  const dim3 grid((max_len + 127) / 128, a.Hq, nz);
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, st>>>(q, dout, k, v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(int dt, int d, const CUtensorMap& q, const CUtensorMap& dout, const CUtensorMap& k,
                          const CUtensorMap& v, const BwdArgs& a, int max_len, int nz, cudaStream_t st) {
  if (d == 64)
    return dt == kBF16 ? launch<kBF16, 64>(q, dout, k, v, a, max_len, nz, st)
                       : launch<kFP16, 64>(q, dout, k, v, a, max_len, nz, st);
  if (d == 128)
    return dt == kBF16 ? launch<kBF16, 128>(q, dout, k, v, a, max_len, nz, st)
                       : launch<kFP16, 128>(q, dout, k, v, a, max_len, nz, st);
  return cudaErrorInvalidValue;
}

}  // namespace attn
