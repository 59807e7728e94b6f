// Declarations shared by the library's translation units (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "fwd_kernel.cuh"
#include "launch_util.h"

namespace attn {

// Forward launchers, one per operand type; d selects the instance.
cudaError_t launch_fwd_bf16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const FwdArgs& a, int grid_x_rows, int gy, int gz, cudaStream_t st);
cudaError_t launch_fwd_fp16(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const FwdArgs& a, int grid_x_rows, int gy, int gz, cudaStream_t st);
cudaError_t launch_fwd_e4m3(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const FwdArgs& a, int grid_x_rows, int gy, int gz, cudaStream_t st);
// Keys per KV tile (rows of the K and V boxes) of the E4M3 forward instance
// for head dimension d; 0 for an unsupported d.
int fwd_e4m3_kv_rows(int d);

// Box width (elements) of the TMA maps a forward instance expects.
inline int fwd_box_elems(int dt, int d) {
  const int esz = dt == kE4M3 ? 1 : 2;
  const int row_b = d * esz;
  return (row_b < 128 ? row_b : 128) / esz;
}

}  // namespace attn
