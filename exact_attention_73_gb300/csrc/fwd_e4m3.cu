// Forward instances with e4m3 operands: d = 64 and 128 with two query tiles
// per CTA, d = 256 with one (tensor memory holds S and O for 512 columns);
// all with 128-key KV tiles.
#include "fwd_launch.cuh"

namespace attn {

cudaError_t launch_fwd_e4m3(int d, const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                            const FwdArgs& a, int rows, int gy, int gz, cudaStream_t st) {
  switch (d) {
    case 64: return launch_fwd_inst<kE4M3, 64, 2>(q, k, v, a, rows, gy, gz, st);
    case 128: return launch_fwd_inst<kE4M3, 128, 2>(q, k, v, a, rows, gy, gz, st);
    case 256: return launch_fwd_inst<kE4M3, 256, 1>(q, k, v, a, rows, gy, gz, st);
    default: return cudaErrorInvalidValue;
  }
}

int fwd_e4m3_kv_rows(int d) { return d == 64 || d == 128 || d == 256 ? 128 : 0; }

}  // namespace attn
