// Launchers of the non-attention kernels (quantiser, backward helpers).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/libattn.h"

namespace attn {

attn_status device_context(int** status);

// Block quantisation to E4M3 (see attn_quantize_fp8).
cudaError_t launch_quant_fp8(const void* x, int in_dt, uint8_t* x8, float* scales, int B, int H, int N, int d,
                             const int8_t* signs, float inv_sqrt_d, cudaStream_t st);

}  // namespace attn
