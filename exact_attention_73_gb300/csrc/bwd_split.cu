// Launches of the backward's kSplit instance (two CTAs per unit in clusters
// of two, or whole units), in a translation unit of its own so that it
// compiles next to the other instance.
#include "bwd_kernel.cuh"
#include "launch_util.h"

namespace attn {

template <int DT, int D, bool kDQ>
cudaError_t launch_bwd_split(const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q, const CUtensorMap& d,
                             const CUtensorMap& dq, const BwdArgs& a, int n, dim3 grid, cudaStream_t st) {
  using C = BwdCfg<DT, D>;
  cudaError_t e = smem_attr_once<bwd_kernel<DT, D, kDQ, true>>(C::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  if ((e = reg_pool_once<bwd_kernel<DT, D, kDQ, true>>(C::NTHREADS, C::kRegsSplit)) != cudaSuccess) return e;
  if (a.nsplit == 1) {
    bwd_kernel<DT, D, kDQ, true><<<grid, C::NTHREADS, C::SMEM_BYTES, st>>>(k, v, q, d, dq, a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * n);
  cfg.blockDim = dim3(C::NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  // with whole units before it (a.unit0 > 0), a programmatic dependent of
  // their grid: it may start as that grid's last CTAs leave
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = a.unit0 > 0 ? 1 : 0;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, bwd_kernel<DT, D, kDQ, true>, k, v, q, d, dq, a);
}

#define ATTN_BWD_SPLIT(DT, D, DQ)                                                                            \
  template cudaError_t launch_bwd_split<DT, D, DQ>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&, \
                                                   const CUtensorMap&, const CUtensorMap&, const BwdArgs&, int, \
                                                   dim3, cudaStream_t);
ATTN_BWD_SPLIT(kBF16, 64, true)
ATTN_BWD_SPLIT(kFP16, 64, true)
ATTN_BWD_SPLIT(kBF16, 128, true)
ATTN_BWD_SPLIT(kFP16, 128, true)
ATTN_BWD_SPLIT(kBF16, 256, true)
ATTN_BWD_SPLIT(kFP16, 256, true)
ATTN_BWD_SPLIT(kBF16, 64, false)
ATTN_BWD_SPLIT(kFP16, 64, false)
ATTN_BWD_SPLIT(kBF16, 128, false)
ATTN_BWD_SPLIT(kFP16, 128, false)
#undef ATTN_BWD_SPLIT

}  // namespace attn
