// Launcher of the deterministic backward's dQ kernel (query-stationary).
#include "bwd_dq_kernel.cuh"
#include "ops.h"

namespace attn {

namespace {

template <int DT>
cudaError_t launch(const CUtensorMap& q, const CUtensorMap& dout, const CUtensorMap& k, const CUtensorMap& v,
                   const BwdArgs& a, int max_len, int nz, cudaStream_t st) {
  using C = DqCfg<DT>;
  auto kern = bwd_dq_kernel<DT>;
  cudaError_t e = smem_attr_once<bwd_dq_kernel<DT>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const dim3 grid((max_len + 127) / 128, a.Hq, nz);
  kern<<<grid, C::NTHREADS, C::SMEM_BYTES, st>>>(q, dout, k, v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dq(int dt, const CUtensorMap& q, const CUtensorMap& dout, const CUtensorMap& k,
                          const CUtensorMap& v, const BwdArgs& a, int max_len, int nz, cudaStream_t st) {
  return dt == kBF16 ? launch<kBF16>(q, dout, k, v, a, max_len, nz, st)
                     : launch<kFP16>(q, dout, k, v, a, max_len, nz, st);
}

}  // namespace attn
