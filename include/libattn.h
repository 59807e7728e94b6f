/*
 * libattn — exact fused scaled-dot-product attention for one NVIDIA GB300
 * (sm_103a). C ABI: plain device pointers, sizes and an opaque stream.
 *
 * What is computed (FlashAttention-3, zenmind.me summary of the paper):
 *   §3.1  S = scale * Q K^T, P = softmax(S) with the row max subtracted,
 *         O = P V; backward dV = P^T dO, dP = dO V^T, dS = P o (dP - D),
 *         dQ = scale dS K, dK = scale dS^T Q.
 *   §3.2  Algorithm 1: tiled online softmax with running max m and running
 *         sum l, O rescaled by exp(m_old - m_new); epilogue O / l and
 *         LSE = m + log(l). S and P never reach global memory.
 *   §3.5  FP8 (E4M3) forward: per-block power-of-two scales, FP32
 *         accumulation, optional random-sign Hadamard rotation of Q and K.
 *   §4 step 5 (paper App. B.1): D = rowsum(dO o O) before the backward;
 *         dQ partials are accumulated atomically in FP32.
 *   §3.2 / paper p.6: grouped-query attention by index mapping, K/V are
 *         not replicated in memory.
 *   guijiagi.com "Flash Attention 3 explained", practical notes: packed
 *         variable-length batches described by cu_seqlens.
 *
 * Conventions shared by every entry point
 *   - Dense tensors are contiguous [B, H, N, d] (d fastest). Packed tensors
 *     are contiguous [T, H, d] with cu_seqlens (int32, nseq + 1 entries,
 *     device memory) holding the exclusive prefix sum of the lengths.
 *   - d is 64, 128 or 256. Hq is a multiple of Hkv; query head h reads
 *     key/value head h / (Hq / Hkv).
 *   - causal: key j is visible to query i iff j <= i (positions counted
 *     inside each sequence; queries and keys have the same length).
 *   - LSE is float32, natural log: dense [B, Hq, N], packed [Hq, T].
 *   - All pointers are device pointers owned by the caller; the library
 *     never allocates or frees device memory and never synchronises.
 *     Every pointer must be 16-byte aligned.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Calls are asynchronous on it.
 *   - Arguments are checked before anything is launched; a failed check
 *     returns an error code and launches nothing. A CUDA error raised by a
 *     launch is returned as ATTN_ERR_CUDA.
 *   - CUDA graphs: the first call on a device probes it, and the first
 *     launch of each kernel instance raises its shared-memory limit; after
 *     that a call only encodes tensor maps on the host (passed by value in
 *     the kernel parameters) and enqueues kernels on `stream`, so it can be
 *     captured into a graph and replayed. Make one direct call with the same
 *     shapes and flags before capturing. A replay keeps the captured
 *     pointers, sizes and flags and reads the buffers' current contents
 *     (cu_seqlens and decode seqlens included). attn_get_device_status
 *     synchronises and cannot be captured.
 */
#ifndef LIBATTN_H
#define LIBATTN_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_BF16 = 0,
  ATTN_FP16 = 1,
  ATTN_E4M3 = 2
} attn_dtype;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL = 1,       /* a required pointer is NULL */
  ATTN_ERR_ALIGN = 2,      /* a pointer is not 16-byte aligned */
  ATTN_ERR_SHAPE = 3,      /* B, H, N, T, nseq or max_seqlen out of range */
  ATTN_ERR_HEADDIM = 4,    /* d not in {64, 128, 256} */
  ATTN_ERR_GQA = 5,        /* Hq is not a positive multiple of Hkv */
  ATTN_ERR_DTYPE = 6,      /* dtype not accepted by this entry point */
  ATTN_ERR_WORKSPACE = 7,  /* workspace NULL or smaller than the size query */
  ATTN_ERR_LAUNCH = 8,     /* kernel resources (shared memory, registers) not granted */
  ATTN_ERR_TIMEOUT = 9,    /* a device-side wait ran out (see status query) */
  ATTN_ERR_CUDA = 10,      /* CUDA runtime/driver error */
  ATTN_ERR_NODEVICE = 11   /* no sm_103 device is current */
} attn_status;

/* Human-readable name of a status code (static string). */
ATTN_API const char* attn_status_string(attn_status s);

/*
 * Forward, dense. Algorithm 1 (§3.2) with scale = alpha (§3.1).
 * q [B,Hq,N,d], k/v [B,Hkv,N,d] of `dtype` (ATTN_BF16 or ATTN_FP16);
 * o [B,Hq,N,d] same dtype (written); lse [B,Hq,N] float32 (written).
 */
ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                     attn_dtype dtype, void* stream);

/*
 * Forward, dense, sliding-window (local) attention (guijiagi.com, practical
 * notes: sliding-window attention). Arguments as attn_fwd, with the mask
 * given by a key window: key j is visible to query i iff
 * i - window_left <= j <= i + window_right; -1 means no bound on that side
 * (window (-1, 0) is causal, (-1, -1) full attention). Other negative values
 * return ATTN_ERR_SHAPE. Every window contains the diagonal, so each row sees
 * at least one key. KV tiles with no visible key are skipped.
 */
ATTN_API attn_status attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse,
                                     int B, int Hq, int Hkv, int N, int d, float scale, int window_left,
                                     int window_right, attn_dtype dtype, void* stream);

/*
 * Forward, packed variable length (guijiagi.com, practical notes).
 * q [T,Hq,d], k/v [T,Hkv,d], o [T,Hq,d], lse [Hq,T]; cu_seqlens int32 [nseq+1]
 * on the device; max_seqlen is the largest length (host value, >= 1; used to
 * size the grid). Every sequence must have length >= 1.
 */
ATTN_API attn_status attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                            const int* cu_seqlens, int nseq, int T, int max_seqlen,
                            int Hq, int Hkv, int d, float scale, int causal,
                            attn_dtype dtype, void* stream);

/*
 * Block quantisation to E4M3 (§3.5 block quantisation and incoherent
 * processing; m.xxqk.cn walkthrough §4.2 power-of-two scales).
 * x [B,H,N,d] of in_dtype (BF16/FP16) -> x8 [B,H,N,d] E4M3 codes (uint8) and
 * scales [B,H,ceil(N/128)] float32: for each 128-row block of one (b,h),
 * e = the largest integer with amax * 2^e <= 448, x8 = e4m3_rn_satfinite(x * 2^e),
 * scales = 2^-e (1 when the block is all zero).
 * hadamard_signs: NULL = no rotation; else int8 [d] of +-1 on the device, and
 * each row is first replaced by fp32(FWHT(signs o x) * fp32(1/sqrt(d))).
 */
ATTN_API attn_status attn_quantize_fp8(const void* x, attn_dtype in_dtype, void* x8, float* scales,
                              int B, int H, int N, int d, const int8_t* hadamard_signs,
                              void* stream);

/*
 * Fused producer: rotary position embedding, optional rotation and block
 * quantisation in one pass (§3.5: the paper fuses quantisation into the RoPE
 * step that produces Q and K). Arguments as
 * attn_quantize_fp8, plus rope_cos, rope_sin: float32 [N, d/2] device tables
 * (16-byte aligned; the caller chooses the frequencies, row n = position n).
 * Each row x at position n becomes, for i < d/2 with c = cos[n,i],
 * s = sin[n,i]: y_i = x_i c - x_{i+d/2} s, y_{i+d/2} = x_{i+d/2} c + x_i s
 * (rotate-half pairing; each product and sum rounded to float32 on its own),
 * then the optional sign + Hadamard rotation and the per-block E4M3
 * quantisation of attn_quantize_fp8. NULL tables return ATTN_ERR_NULL.
 */
ATTN_API attn_status attn_quantize_fp8_rope(const void* x, attn_dtype in_dtype, void* x8, float* scales,
                                            int B, int H, int N, int d, const float* rope_cos,
                                            const float* rope_sin, const int8_t* hadamard_signs, void* stream);

/*
 * FP8 forward, dense (§3.5). q8 [B,Hq,N,d], k8/v8 [B,Hkv,N,d] E4M3 codes;
 * sq [B,Hq,ceil(N/128)], sk/sv [B,Hkv,ceil(N/128)] float32 power-of-two
 * dequantisation factors from attn_quantize_fp8. o [B,Hq,N,d] BF16,
 * lse [B,Hq,N] float32. Both products accumulate in FP32. The running row
 * max is raised only when a tile's max exceeds it by more than 4 (log2
 * units), so P~ = exp2(x - m) <= 16; P~ is rounded to E4M3 as
 * e4m3(P~ * 2^(4 + f_j - F)) with sv_j = 2^f_j and F the running maximum of
 * f over the KV tiles seen (O rescaled when F grows). The KV tile holds
 * attn_fwd_fp8_kv_tile(d) keys; a tile that spans two 128-row blocks gives
 * each key its own block's factors and raises F to the larger exponent.
 */
ATTN_API attn_status attn_fwd_fp8(const void* q8, const void* k8, const void* v8,
                         const float* sq, const float* sk, const float* sv,
                         void* o, float* lse,
                         int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                         void* stream);

/*
 * FP8 forward with a key window (guijiagi.com, practical notes: sliding-window
 * attention): as attn_fwd_fp8 (same operands, factors, layouts and
 * arithmetic), with key j visible to query i iff
 * i - window_left <= j <= i + window_right; -1 leaves that side unbounded,
 * so (-1, 0) is attn_fwd_fp8 with causal = 1 and (-1, -1) without masking.
 * Every row sees at least its own key. ATTN_ERR_SHAPE for a bound below -1.
 */
ATTN_API attn_status attn_fwd_fp8_window(const void* q8, const void* k8, const void* v8,
                                         const float* sq, const float* sk, const float* sv,
                                         void* o, float* lse,
                                         int B, int Hq, int Hkv, int N, int d, float scale, int window_left,
                                         int window_right, void* stream);

/*
 * Block quantisation of packed sequences: x [T,H,d] (THD, as attn_fwd_varlen)
 * -> x8 [T,H,d] E4M3 codes and scales [nseq, H, ceil(max_seqlen/128)]
 * float32. Each sequence is blocked from its own first row (its last block
 * may be short), with the rule of attn_quantize_fp8 per block; block i of
 * sequence z, head h takes slot [z, h, i]; slots past a sequence's last
 * block are not written. cu_seqlens int32 [nseq+1] on the device and
 * max_seqlen as attn_fwd_varlen. Optional sign + Hadamard rotation as
 * attn_quantize_fp8 (no RoPE variant).
 */
ATTN_API attn_status attn_quantize_fp8_varlen(const void* x, attn_dtype in_dtype, void* x8, float* scales,
                                              const int* cu_seqlens, int nseq, int T, int max_seqlen, int H,
                                              int d, const int8_t* hadamard_signs, void* stream);

/*
 * FP8 forward over packed sequences: q8 [T,Hq,d], k8/v8 [T,Hkv,d] E4M3
 * codes and sq [nseq,Hq,ceil(max_seqlen/128)], sk/sv [nseq,Hkv,...]
 * factors from attn_quantize_fp8_varlen (same cu_seqlens and max_seqlen);
 * o [T,Hq,d] BF16, lse [Hq,T] float32. Arithmetic as attn_fwd_fp8 within
 * each sequence (every KV tile is one block of its sequence).
 */
ATTN_API attn_status attn_fwd_fp8_varlen(const void* q8, const void* k8, const void* v8,
                                         const float* sq, const float* sk, const float* sv,
                                         void* o, float* lse, const int* cu_seqlens, int nseq, int T,
                                         int max_seqlen, int Hq, int Hkv, int d, float scale, int causal,
                                         void* stream);

/*
 * Keys per KV tile of attn_fwd_fp8 for head dimension d (128 for d = 64,
 * 128, 256), 0 for an unsupported d. The stale running max and F move
 * once per KV tile (§3.2 Algorithm 1, Bc), so the E4M3 rounding of P~, and
 * with it the result's last bits, depends on this blocking. No device work.
 */
ATTN_API int attn_fwd_fp8_kv_tile(int d);

/* Bytes of workspace attn_decode_fp8 needs: per split, a float32 partial O
 * [B, Hq, d] and LSE [B, Hq], each area rounded up to 256 bytes. */
ATTN_API size_t attn_decode_fp8_workspace_size(int B, int Hq, int d, int num_splits);

/*
 * FP8 decode over a block-quantised KV cache, split-KV (§3.5 FP8 forward of
 * Algorithm 1 applied to one new token per sequence; the pages do not give a
 * decode kernel — this is the forward's split form). One query token per
 * sequence and query head:
 *   q8 [B, Hq, d] E4M3 codes and sq [B, Hkv] float32 power-of-two factors, one
 *   per KV group (quantise q viewed as [B, Hkv, g, d] with attn_quantize_fp8);
 *   k8, v8 [B, Hkv, Nmax, d] E4M3 cache, sk, sv [B, Hkv, ceil(Nmax/128)]
 *   factors (attn_quantize_fp8 of the cache);
 *   seqlens: int32 [B] on the device, valid cache length of each sequence
 *   (1 <= seqlens[b] <= Nmax), or NULL for Nmax everywhere;
 *   o [B, Hq, d] BF16 and lse [B, Hq] float32 (natural log) are written.
 * The cache's KV tiles are cut into num_splits runs of ceil(ceil(Nmax/128) /
 * num_splits) tiles (1 <= num_splits <= ceil(Nmax/128)); each run of each
 * (sequence, KV group) is one CTA computing the FP8 forward for the group's
 * g = Hq / Hkv query heads (g <= 128) from a fresh state, and a second kernel
 * combines the runs by their log-sum-exp weights (B * Hq <= 2^31 - 1, else
 * ATTN_ERR_SHAPE). Runs past a sequence's
 * length contribute nothing. workspace: attn_decode_fp8_workspace_size bytes.
 */
ATTN_API attn_status attn_decode_fp8(const void* q8, const float* sq, const void* k8, const void* v8,
                                     const float* sk, const float* sv, const int* seqlens, void* o, float* lse,
                                     void* workspace, size_t ws_bytes, int B, int Hq, int Hkv, int Nmax, int d,
                                     float scale, int num_splits, void* stream);

/* Bytes of device workspace attn_bwd needs: FP32 dQ accumulator [B,Hq,N,d]
 * plus D = rowsum(dO o O) [B,Hq,N], each rounded up to 256 bytes. */
ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int N, int d);

/*
 * Backward, dense (§3.1 backward chain; §4 step 5). Inputs q, k, v, o, dout of
 * `dtype` with the forward's shapes and lse from attn_fwd; outputs dq
 * [B,Hq,N,d], dk/dv [B,Hkv,N,d] of `dtype` (dk/dv sum over the query heads
 * of each group). P is recomputed from lse. workspace: device memory of at
 * least attn_bwd_workspace_size bytes, contents need not be initialised.
 * lse is treated as a non-differentiable output. Head dim d is 64, 128 or
 * 256 (other values return ATTN_ERR_HEADDIM; at 256 two CTAs share a key tile,
 * each owning half of the head dims). Kernels: D = rowsum(dO o O) with the
 * FP32 dQ accumulator cleared, the main kernel, the dQ conversion.
 */
ATTN_API attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const float* lse, const void* dout,
                     void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                     int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                     attn_dtype dtype, void* stream);

/*
 * Backward, dense, sliding window: arguments as attn_bwd with the key window
 * of attn_fwd_window (lse from attn_fwd_window with the same window).
 */
ATTN_API attn_status attn_bwd_window(const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dout,
                                     void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                     int B, int Hq, int Hkv, int N, int d, float scale, int window_left,
                                     int window_right, attn_dtype dtype, void* stream);

/* Bytes of device workspace attn_bwd_deterministic needs: D = rowsum(dO o O)
 * [B, Hq, N] float32, rounded up to 256 bytes (0 for sizes below 1). */
ATTN_API size_t attn_bwd_deterministic_workspace_size(int B, int Hq, int Hkv, int N, int d);

/*
 * Deterministic backward, dense (§3.1 backward chain; §4 step 5 computes
 * D first). Arguments as attn_bwd_window (window (-1, 0) = causal, (-1, -1)
 * = full), workspace of attn_bwd_deterministic_workspace_size bytes. The
 * pages accumulate dQ with atomic adds, whose order varies between runs; here
 * dK and dV come from the key-stationary kernel (its dQ product left out) and
 * dQ from a query-stationary kernel that recomputes S and dP per KV tile and
 * sums dS K over the KV tiles in increasing order inside one CTA. Every output
 * element has one writer and one summation order, so repeated calls with the
 * same inputs return identical bits. Costs three more GEMMs per tile pair
 * than attn_bwd (S and dP are computed twice). d must be 64 or 128
 * (ATTN_ERR_HEADDIM for 256).
 */
ATTN_API attn_status attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                                            const float* lse, const void* dout,
                                            void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                                            int B, int Hq, int Hkv, int N, int d, float scale, int window_left,
                                            int window_right, attn_dtype dtype, void* stream);

/* Size in bytes of the device array attn_bwd_noalloc uses as its workspace. */
#define ATTN_BWD_NOALLOC_MAX_BYTES (32u * 1024u * 1024u)

/*
 * Dense backward for callers that cannot allocate device memory. The pages
 * have no counterpart; it exists for callers such as a process whose device
 * memory is already reserved by another allocator (a framework's caching
 * pool), or a serving loop that must not allocate while running because
 * cudaMalloc/cudaFree can synchronise the device. Arguments and results are
 * those of attn_bwd without the workspace: the workspace is a library-owned
 * device array of ATTN_BWD_NOALLOC_MAX_BYTES, which every GPU that loads it
 * keeps until the process exits. A problem whose attn_bwd_workspace_size
 * exceeds that returns ATTN_ERR_WORKSPACE before any device work, and every
 * other argument error returns attn_bwd's code, also before any device work.
 * The first call on a device looks up the array's device address (do it
 * before any stream capture). Under lazy module loading (CUDA's default) that
 * first call is also when the driver reserves the array on the device, so it
 * can fail with ATTN_ERR_CUDA on a device that is already full: make one call
 * at start-up, before a memory pool reserves the device's memory. All calls
 * share the array: calls that overlap on the GPU race and must not be issued.
 * The entry point itself allocates and frees nothing.
 */
ATTN_API attn_status attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                      const float* lse, const void* dout,
                                      void* dq, void* dk, void* dv,
                                      int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                                      attn_dtype dtype, void* stream);

/* Workspace for attn_bwd_varlen: FP32 dQ [T,Hq,d] plus D [Hq,T]. */
ATTN_API size_t attn_bwd_varlen_workspace_size(int T, int Hq, int Hkv, int d);

/* Backward, packed variable length; layouts as attn_fwd_varlen. */
ATTN_API attn_status attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                            const float* lse, const void* dout,
                            void* dq, void* dk, void* dv, void* workspace, size_t ws_bytes,
                            const int* cu_seqlens, int nseq, int T, int max_seqlen,
                            int Hq, int Hkv, int d, float scale, int causal,
                            attn_dtype dtype, void* stream);

/*
 * Device status of the library's kernels on the current device: every wait
 * inside a kernel is bounded; one that runs out records ATTN_ERR_TIMEOUT in a
 * device word and the kernel returns early. This call synchronises `stream`,
 * reads the word, clears it and returns it (ATTN_OK when nothing happened).
 */
ATTN_API attn_status attn_get_device_status(void* stream);

/*
 * Diagnostic of the failure path; the pages have no counterpart. Launches one
 * warp that waits, with the kernels' own bounded wait and a limit of limit_ms
 * milliseconds (1..10000), on a barrier that nothing completes. The wait ends
 * on its own, records ATTN_ERR_TIMEOUT in the device status word and the
 * kernel returns: attn_get_device_status then reports ATTN_ERR_TIMEOUT once,
 * and the context stays usable. Asynchronous on `stream`.
 */
ATTN_API attn_status attn_selftest_wait_timeout(unsigned int limit_ms, void* stream);

/* Library version, e.g. "libattn 0.1 sm_103a". */
ATTN_API const char* attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBATTN_H */
