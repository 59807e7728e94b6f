// Backward entry points: argument checks, workspace layout, launches.
#include <cstdint>

#include "../../include/libattn.h"
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

}  // namespace

extern "C" {

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
  if (B < 1 || B > 65535 || N < 1) return ATTN_ERR_SHAPE;
  attn_status s = check_common(q, k, v, o, lse, dout, dq, dk, dv, workspace, ws_bytes,
                               attn_bwd_workspace_size(B, Hq, Hkv, N, d), Hq, Hkv, d, dtype);
  if (s != ATTN_OK) return s;
  int* status;
  if ((s = attn::device_context(&status)) != ATTN_OK) return s;
  (void)scale; (void)causal; (void)stream;
  return ATTN_ERR_LAUNCH;
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
  (void)scale; (void)causal; (void)stream;
  return ATTN_ERR_LAUNCH;
}

}  // extern "C"
