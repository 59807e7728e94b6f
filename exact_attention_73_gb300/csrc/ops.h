// Launchers of the non-attention kernels (quantiser, backward helpers).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/libattn.h"
#include "launch_util.h"

namespace attn {

attn_status device_context(int** status);

// Argument checks of the dense backward (pointers, alignment, shape, head
// dimension, GQA, dtype, workspace), all on the host before any device work.
attn_status bwd_check_dense(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, const void* dq, const void* dk, const void* dv, const void* ws,
                            size_t ws_bytes, int B, int Hq, int Hkv, int N, int d, attn_dtype dtype);

struct BwdArgs;
bool operand_map(CUtensorMap* m, const void* base, int dt, int d, bool packed, int B, int H, long long rows,
                 int box_rows);
cudaError_t launch_bwd_pre(int dt, int d, const void* o, const void* dout, float* dvec, float* dq_acc,
                           long long rows, int Hq, int T_tokens, int packed, cudaStream_t st);
cudaError_t launch_bwd_main(int dt, int d, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                            const CUtensorMap& dout, const CUtensorMap& dq_acc, const BwdArgs& a, int max_len, int nz,
                            cudaStream_t st);
// FP32 accumulator map (layout of the operands, no swizzle), boxes of box_e x box_rows.
bool accum_map(CUtensorMap* m, const float* base, int d, bool packed, int B, int H, long long rows, int box_rows,
               int box_e);
// Rows and head dims of the dQ accumulator per reduce-add of the main kernel
// (the box of its map).
int bwd_dq_rows(int d);
int bwd_dq_dims(int d);
cudaError_t launch_bwd_dkdv(int dt, int d, const CUtensorMap& k, const CUtensorMap& v, const CUtensorMap& q,
                            const CUtensorMap& dout, const BwdArgs& a, int max_len, int nz, cudaStream_t st);
cudaError_t launch_bwd_dq(int dt, int d, const CUtensorMap& q, const CUtensorMap& dout, const CUtensorMap& k,
                          const CUtensorMap& v, const BwdArgs& a, int max_len, int nz, cudaStream_t st);
cudaError_t launch_dq_convert(int dt, const float* acc, void* dq, long long n, float scale, cudaStream_t st);

// Block quantisation to E4M3 (see attn_quantize_fp8).
cudaError_t launch_quant_fp8(const void* x, int in_dt, uint8_t* x8, float* scales, int B, int H, int N, int d,
                             const int8_t* signs, float inv_sqrt_d, const float* rope_cos, const float* rope_sin,
                             cudaStream_t st);
// The same over packed [T, H, d] sequences, each blocked from its own first
// row; factors [nseq][H][ceil(max_len / 128)].
cudaError_t launch_quant_fp8_varlen(const void* x, int in_dt, uint8_t* x8, float* scales, const int* cu_seqlens,
                                    int nseq, int max_len, int H, int d, const int8_t* signs, float inv_sqrt_d,
                                    cudaStream_t st);

}  // namespace attn
