// Backward entry points: argument checks, workspace layout, launches.
#include <cstdint>

#include "../../include/libattn.h"
#include "bwd_kernel.cuh"
#include "ops.h"

namespace {

size_t round256(size_t x) { return (x + 255) / 256 * 256; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

attn_status check_common(const void* q, const void* k, const void* v, const void* o, const float* lse,
                         const void* dout, const void* dq, const void* dk, const void* dv, const void* ws,
                         size_t ws_bytes, size_t ws_need, int Hq, int Hkv, int d, attn_dtype dtype) {
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv || !ws) return ATTN_ERR_NULL;
  const void* ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv, ws};
  for (const void* p : ptrs)
    if (!aligned16(p)) return ATTN_ERR_ALIGN;
  if (Hq < 1 || Hkv < 1 || Hq > 65535) return ATTN_ERR_SHAPE;
  if (d != 64 && d != 128 && d != 256) return ATTN_ERR_HEADDIM;
  if (Hq % Hkv) return ATTN_ERR_GQA;
  if (dtype != ATTN_BF16 && dtype != ATTN_FP16) return ATTN_ERR_DTYPE;
  if (ws_bytes < ws_need) return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

constexpr float kLog2e = 1.4426950408889634f;

attn_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ATTN_OK;
  if (e == cudaErrorInvalidValue || e == cudaErrorLaunchOutOfResources) return ATTN_ERR_LAUNCH;
  return ATTN_ERR_CUDA;
}

// Dense when cu_seqlens is null (nz = B, rows per head = N = max_len);
// packed otherwise (nz = nseq, T tokens, longest sequence max_len).
attn_status run_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dout,
                    void* dq, void* dk, void* dv, void* ws, const int* cu_seqlens, int nz, int rows_or_T,
                    int max_len, int Hq, int Hkv, int d, float scale, int win_left, int win_right,
                    attn_dtype dtype, int* status, void* stream) {
  using namespace attn;
  const bool packed = cu_seqlens != nullptr;
  const int B = packed ? 1 : nz;
  const long long rows = static_cast<long long>(B) * Hq * rows_or_T;
  float* dq_acc = static_cast<float*>(ws);
  float* dvec = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + round256(static_cast<size_t>(rows) * d * 4));
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap tk, tv, tq, tdo, tdq;
  if (!operand_map(&tk, k, dtype, d, packed, B, Hkv, rows_or_T, 128) ||
      !operand_map(&tv, v, dtype, d, packed, B, Hkv, rows_or_T, 128) ||
      !operand_map(&tq, q, dtype, d, packed, B, Hq, rows_or_T, 64) ||
      !operand_map(&tdo, dout, dtype, d, packed, B, Hq, rows_or_T, 64) ||
      !accum_map(&tdq, dq_acc, d, packed, B, Hq, rows_or_T, bwd_dq_rows(d), bwd_dq_dims(d)))
    return ATTN_ERR_CUDA;
  BwdArgs a{};
  a.lse = lse;
  a.dvec = dvec;
  a.dq_acc = dq_acc;
  a.dk = dk;
  a.dv = dv;
  if (packed) {
    a.q_sn = static_cast<long long>(Hq) * d; a.q_sh = d; a.q_sb = 0;
    a.k_sn = static_cast<long long>(Hkv) * d; a.k_sh = d; a.k_sb = 0;
    a.l_sh = rows_or_T; a.l_sb = 0;
    a.N = 0;
  } else {
    a.q_sn = d; a.q_sh = static_cast<long long>(rows_or_T) * d; a.q_sb = static_cast<long long>(Hq) * rows_or_T * d;
    a.k_sn = d; a.k_sh = static_cast<long long>(rows_or_T) * d; a.k_sb = static_cast<long long>(Hkv) * rows_or_T * d;
    a.l_sh = rows_or_T; a.l_sb = static_cast<long long>(Hq) * rows_or_T;
    a.N = rows_or_T;
  }
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = Hq / Hkv;
  a.cu_seqlens = cu_seqlens;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.win_left = win_left;
  a.win_right = win_right;
  a.causal = (win_left < 0 && win_right == 0) ? 1 : 0;
  a.status = status;
  cudaError_t e = launch_bwd_pre(dtype, d, o, dout, dvec, dq_acc, rows, Hq, rows_or_T, packed ? 1 : 0, st);
  if (e == cudaSuccess) e = launch_bwd_main(dtype, d, tk, tv, tq, tdo, tdq, a, max_len, nz, st);
  if (e == cudaSuccess) e = launch_dq_convert(dtype, dq_acc, dq, rows * d, scale, st);
  return from_cuda(e);
}

// Deterministic backward, dense: D (no dQ accumulator), the key-stationary
// kernel for dK/dV without its dQ product, then the query-stationary dQ kernel.
attn_status run_bwd_det(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv, void* ws, int B, int N, int Hq, int Hkv,
                        int d, float scale, int win_left, int win_right, attn_dtype dtype, int* status,
                        void* stream) {
  using namespace attn;
  const long long rows = static_cast<long long>(B) * Hq * N;
  float* dvec = static_cast<float*>(ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CUtensorMap tk, tv, tq, tdo, tq128, tdo128;
  if (!operand_map(&tk, k, dtype, d, false, B, Hkv, N, 128) || !operand_map(&tv, v, dtype, d, false, B, Hkv, N, 128) ||
      !operand_map(&tq, q, dtype, d, false, B, Hq, N, 64) || !operand_map(&tdo, dout, dtype, d, false, B, Hq, N, 64) ||
      !operand_map(&tq128, q, dtype, d, false, B, Hq, N, 128) ||
      !operand_map(&tdo128, dout, dtype, d, false, B, Hq, N, 128))
    return ATTN_ERR_CUDA;
  BwdArgs a{};
  a.lse = lse;
  a.dvec = dvec;
  a.dq_acc = nullptr;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.q_sn = d; a.q_sh = static_cast<long long>(N) * d; a.q_sb = static_cast<long long>(Hq) * N * d;
  a.k_sn = d; a.k_sh = static_cast<long long>(N) * d; a.k_sb = static_cast<long long>(Hkv) * N * d;
  a.l_sh = N; a.l_sb = static_cast<long long>(Hq) * N;
  a.N = N;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.group = Hq / Hkv;
  a.cu_seqlens = nullptr;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.win_left = win_left;
  a.win_right = win_right;
  a.causal = (win_left < 0 && win_right == 0) ? 1 : 0;
  a.status = status;
  cudaError_t e = launch_bwd_pre(dtype, d, o, dout, dvec, nullptr, rows, Hq, N, 0, st);
  if (e == cudaSuccess) e = launch_bwd_dkdv(dtype, d, tk, tv, tq, tdo, a, N, B, st);
  if (e == cudaSuccess) e = launch_bwd_dq(dtype, d, tq128, tdo128, tk, tv, a, N, B, st);
  return from_cuda(e);
}

}  // namespace

extern "C" {

size_t attn_bwd_deterministic_workspace_size(int B, int Hq, int Hkv, int N, int d) {
  (void)Hkv;
  (void)d;
  if (B < 1 || Hq < 1 || N < 1) return 0;
  return round256(static_cast<size_t>(B) * Hq * N * 4);
}

attn_status attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                   const void* dout, void* dq, void* dk, void* dv, void* workspace,
                                   size_t ws_bytes, int B, int Hq, int Hkv, int N, int d, float scale,
                                   int window_left, int window_right, attn_dtype dtype, void* stream) {
  if (B < 1 || B > 65535 || N < 1 || window_left < -1 || window_right < -1) return ATTN_ERR_SHAPE;
  attn_status s = check_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, ws_bytes,
                               attn_bwd_deterministic_workspace_size(B, Hq, Hkv, N, d), Hq, Hkv, d, dtype);
  if (s != ATTN_OK) return s;
  if (d == 256) return ATTN_ERR_HEADDIM;   // the query-stationary dQ kernel is built for d = 64 and 128
  int* status;
  if ((s = attn::device_context(&status)) != ATTN_OK) return s;
  return run_bwd_det(q, k, v, o, lse, dout, dq, dk, dv, workspace, B, N, Hq, Hkv, d, scale, window_left,
                     window_right, dtype, status, stream);
}

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d) {
  (void)Hkv;
  if (B < 1 || Hq < 1 || N < 1 || d < 1) return 0;
  const size_t rows = static_cast<size_t>(B) * Hq * N;
  return round256(rows * d * 4) + round256(rows * 4);
}

size_t attn_bwd_varlen_workspace_size(int T, int Hq, int Hkv, int d) {
  return attn_bwd_workspace_size(1, Hq, Hkv, T, d);
}

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                     const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal, attn_dtype dtype,
                     void* stream) {
  attn_status s = attn::bwd_check_dense(q, k, v, o, lse, dout, dq, dk, dv, workspace, ws_bytes, B, Hq, Hkv, N, d,
                                        dtype);
  if (s != ATTN_OK) return s;
  int* status;
  if ((s = attn::device_context(&status)) != ATTN_OK) return s;
  return run_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, nullptr, B, N, N, Hq, Hkv, d, scale, -1,
                 causal ? 0 : -1, dtype, status, stream);
}

attn_status attn_bwd_window(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                            int B, int Hq, int Hkv, int N, int d, float scale, int window_left, int window_right,
                            attn_dtype dtype, void* stream) {
  if (B < 1 || B > 65535 || N < 1 || window_left < -1 || window_right < -1) return ATTN_ERR_SHAPE;
  attn_status s = check_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, ws_bytes,
                               attn_bwd_workspace_size(B, Hq, Hkv, N, d), Hq, Hkv, d, dtype);
  if (s != ATTN_OK) return s;
  int* status;
  if ((s = attn::device_context(&status)) != ATTN_OK) return s;
  return run_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, nullptr, B, N, N, Hq, Hkv, d, scale, window_left,
                 window_right, dtype, status, stream);
}

attn_status attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                            const int* cu_seqlens, int nseq, int T, int max_seqlen, int Hq, int Hkv, int d,
                            float scale, int causal, attn_dtype dtype, void* stream) {
  if (!cu_seqlens) return ATTN_ERR_NULL;
  if (!aligned16(cu_seqlens)) return ATTN_ERR_ALIGN;
  if (nseq < 1 || nseq > 65535 || T < 1 || max_seqlen < 1 || max_seqlen > T) return ATTN_ERR_SHAPE;
  attn_status s = check_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, ws_bytes,
                               attn_bwd_varlen_workspace_size(T, Hq, Hkv, d), Hq, Hkv, d, dtype);
  if (s != ATTN_OK) return s;
  int* status;
  if ((s = attn::device_context(&status)) != ATTN_OK) return s;
  return run_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, cu_seqlens, nseq, T, max_seqlen, Hq, Hkv, d, scale,
                 -1, causal ? 0 : -1, dtype, status, stream);
}

}  // extern "C"

namespace attn {

attn_status bwd_check_dense(const void* q, const void* k, const void* v, const void* o, const float* lse,
                            const void* dout, const void* dq, const void* dk, const void* dv, const void* ws,
                            size_t ws_bytes, int B, int Hq, int Hkv, int N, int d, attn_dtype dtype) {
  if (B < 1 || B > 65535 || N < 1) return ATTN_ERR_SHAPE;
  return check_common(q, k, v, o, lse, dout, dq, dk, dv, ws, ws_bytes, attn_bwd_workspace_size(B, Hq, Hkv, N, d),
                      Hq, Hkv, d, dtype);
}

}  // namespace attn
