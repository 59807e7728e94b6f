// Launches of the backward's persistent instance (one CTA per SM walking the
// units), in a translation unit of its own so that it compiles next to the
// other instances.
#include "bwd_kernel.cuh"
#include "launch_util.h"

namespace attn {

template <int DT, int D>
cudaError_t launch_bwd_persist(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                               const CUtensorMap& d, const CUtensorMap& dq, const BwdArgs& a, int grid,
                               cudaStream_t st) {
  using C = BwdCfg<DT, D, true>;
  cudaError_t e = smem_attr_once<bwd_kernel<DT, D, true, false, true>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if ((e = reg_pool_once<bwd_kernel<DT, D, true, false, true>>(C::NTHREADS, C::kRegsSplit)) != cudaSuccess) return e;
  bwd_kernel<DT, D, true, false, true><<<static_cast<unsigned>(grid), C::NTHREADS, C::SMEM_BYTES, st>>>(
      k, v, q, d, dq, a);
  return cudaGetLastError();
}

#define ATTN_BWD_PERSIST(DT, D)                                                                              \
  template cudaError_t launch_bwd_persist<DT, D>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,   \
                                                 const CUtensorMap&, const CUtensorMap&, const BwdArgs&, int, \
                                                 cudaStream_t);
ATTN_BWD_PERSIST(kBF16, 64)
ATTN_BWD_PERSIST(kFP16, 64)
ATTN_BWD_PERSIST(kBF16, 128)
ATTN_BWD_PERSIST(kFP16, 128)
#undef ATTN_BWD_PERSIST

}  // namespace attn
