"""ctypes binding of libattn: the C entry points under the same names.

Argument marshalling only: tensors become device pointers and sizes, the
current torch stream becomes the stream handle, and a non-OK status raises
``AttnError``. Every step of the computation runs in the library's kernels;
there is no other code path. The library must have been built (``build()``);
loading fails loudly otherwise.
"""
from __future__ import annotations

import ctypes as C
import math
import os

import torch

from . import build as _build

_LIB = None

BF16, FP16, E4M3 = 0, 1, 2
STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_NULL", 2: "ATTN_ERR_ALIGN", 3: "ATTN_ERR_SHAPE", 4: "ATTN_ERR_HEADDIM",
          5: "ATTN_ERR_GQA", 6: "ATTN_ERR_DTYPE", 7: "ATTN_ERR_WORKSPACE", 8: "ATTN_ERR_LAUNCH",
          9: "ATTN_ERR_TIMEOUT", 10: "ATTN_ERR_CUDA", 11: "ATTN_ERR_NODEVICE"}
EXPORTS = ("attn_status_string", "attn_version", "attn_fwd", "attn_fwd_varlen", "attn_quantize_fp8",
           "attn_fwd_fp8", "attn_bwd_workspace_size", "attn_bwd", "attn_bwd_varlen_workspace_size",
           "attn_bwd_varlen", "attn_get_device_status", "attn_bwd_noalloc", "attn_selftest_wait_timeout",
           "attn_fwd_window", "attn_bwd_window", "attn_bwd_deterministic_workspace_size",
           "attn_bwd_deterministic", "attn_quantize_fp8_rope", "attn_decode_fp8_workspace_size",
           "attn_decode_fp8", "attn_fwd_fp8_kv_tile")


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)}")


_P, _I, _F, _Z = C.c_void_p, C.c_int, C.c_float, C.c_size_t
_SIGS = {
    "attn_status_string": ([_I], C.c_char_p),
    "attn_version": ([], C.c_char_p),
    "attn_fwd": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P], _I),
    "attn_fwd_varlen": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P], _I),
    "attn_quantize_fp8": ([_P, _I, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "attn_fwd_fp8": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P], _I),
    "attn_fwd_fp8_kv_tile": ([_I], _I),
    "attn_bwd_workspace_size": ([_I, _I, _I, _I, _I], _Z),
    "attn_bwd": ([_P] * 9 + [_P, _Z, _I, _I, _I, _I, _I, _F, _I, _I, _P], _I),
    "attn_bwd_varlen_workspace_size": ([_I, _I, _I, _I], _Z),
    "attn_bwd_varlen": ([_P] * 9 + [_P, _Z, _P, _I, _I, _I, _I, _I, _I, _F, _I, _I, _P], _I),
    "attn_get_device_status": ([_P], _I),
    "attn_selftest_wait_timeout": ([C.c_uint, _P], _I),
    "attn_bwd_noalloc": ([_P] * 9 + [_I, _I, _I, _I, _I, _F, _I, _I, _P], _I),
    "attn_fwd_window": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P], _I),
    "attn_bwd_window": ([_P] * 9 + [_P, _Z, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P], _I),
    "attn_bwd_deterministic_workspace_size": ([_I, _I, _I, _I, _I], _Z),
    "attn_quantize_fp8_rope": ([_P, _I, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "attn_decode_fp8_workspace_size": ([_I, _I, _I, _I], _Z),
    "attn_decode_fp8": ([_P] * 10 + [_Z, _I, _I, _I, _I, _I, _F, _I, _P], _I),
    "attn_bwd_deterministic": ([_P] * 9 + [_P, _Z, _I, _I, _I, _I, _I, _F, _I, _I, _I, _P], _I),
}


def load(build_if_missing: bool = True):
    """Load libattn.so from the package directory (building it first if asked)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise RuntimeError(f"libattn is not built ({_build.LIB} missing); run __graft_entry__.build()")
        _build.build()
    lib = C.CDLL(_build.LIB)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = lib
    return lib


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check(code, where):
    if code != 0:
        raise AttnError(code, where)


_DT = {torch.bfloat16: BF16, torch.float16: FP16}


def _dtype(t):
    if t.dtype not in _DT:
        raise TypeError(f"expected bf16 or fp16, got {t.dtype}")
    return _DT[t.dtype]


def attn_fwd(q, k, v, o, lse, scale=None, causal=False, stream=None):
    """Dense forward: q [B,Hq,N,d], k/v [B,Hkv,N,d], o like q, lse [B,Hq,N] fp32."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, scale,
                           int(bool(causal)), _dtype(q), _stream(stream)), "attn_fwd")


def attn_fwd_window(q, k, v, o, lse, window, scale=None, stream=None):
    """Dense forward with a key window (left, right): key j is visible to
    query i iff i - left <= j <= i + right; -1 means no bound on that side."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    left, right = (int(w) for w in window)
    _check(load().attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d, scale,
                                  left, right, _dtype(q), _stream(stream)), "attn_fwd_window")


def attn_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen, scale=None, causal=False, stream=None):
    """Packed forward: q [T,Hq,d], k/v [T,Hkv,d], o like q, lse [Hq,T]; cu_seqlens int32 on the device."""
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens),
                                  cu_seqlens.numel() - 1, T, int(max_seqlen), Hq, Hkv, d, scale,
                                  int(bool(causal)), _dtype(q), _stream(stream)), "attn_fwd_varlen")


def attn_quantize_fp8(x, x8, scales, hadamard_signs=None, stream=None):
    """x [B,H,N,d] bf16/fp16 -> x8 uint8 codes (same shape), scales [B,H,ceil(N/128)] fp32."""
    B, H, N, d = x.shape
    _check(load().attn_quantize_fp8(_ptr(x), _dtype(x), _ptr(x8), _ptr(scales), B, H, N, d,
                                    _ptr(hadamard_signs), _stream(stream)), "attn_quantize_fp8")


def attn_quantize_fp8_rope(x, x8, scales, rope_cos, rope_sin, hadamard_signs=None, stream=None):
    """RoPE (rotate-half, float32 cos/sin tables [N, d/2] on the device), then
    the optional rotation and block quantisation, in one pass."""
    B, H, N, d = x.shape
    _check(load().attn_quantize_fp8_rope(_ptr(x), _dtype(x), _ptr(x8), _ptr(scales), B, H, N, d, _ptr(rope_cos),
                                         _ptr(rope_sin), _ptr(hadamard_signs), _stream(stream)),
           "attn_quantize_fp8_rope")


def attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, scale=None, causal=False, stream=None):
    """FP8 forward on E4M3 codes (uint8) with block factors; o bf16, lse fp32."""
    B, Hq, N, d = q8.shape
    Hkv = k8.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(sq), _ptr(sk), _ptr(sv), _ptr(o), _ptr(lse),
                               B, Hq, Hkv, N, d, scale, int(bool(causal)), _stream(stream)), "attn_fwd_fp8")


def attn_fwd_fp8_kv_tile(d):
    """Keys per KV tile of attn_fwd_fp8 for head dimension d (0: unsupported)."""
    return load().attn_fwd_fp8_kv_tile(d)


def attn_decode_fp8_workspace_size(B, Hq, d, num_splits):
    return load().attn_decode_fp8_workspace_size(B, Hq, d, num_splits)


def attn_decode_fp8(q8, sq, k8, v8, sk, sv, o, lse, workspace, num_splits, seqlens=None, scale=None, stream=None):
    """One decoded token per sequence: q8 [B,Hq,d] codes, sq [B,Hkv]; cache k8/v8
    [B,Hkv,Nmax,d] with sk/sv [B,Hkv,ceil(Nmax/128)]; seqlens int32 [B] or None;
    o [B,Hq,d] bf16, lse [B,Hq]."""
    B, Hq, d = q8.shape
    _, Hkv, Nmax, _ = k8.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_decode_fp8(_ptr(q8), _ptr(sq), _ptr(k8), _ptr(v8), _ptr(sk), _ptr(sv), _ptr(seqlens), _ptr(o),
                                  _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  B, Hq, Hkv, Nmax, d, scale, int(num_splits), _stream(stream)), "attn_decode_fp8")


def attn_bwd_workspace_size(B, Hq, Hkv, N, d):
    return int(load().attn_bwd_workspace_size(B, Hq, Hkv, N, d))


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, scale=None, causal=False, stream=None):
    """Dense backward; workspace is a byte tensor of at least attn_bwd_workspace_size bytes."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                           _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                           B, Hq, Hkv, N, d, scale, int(bool(causal)), _dtype(q), _stream(stream)), "attn_bwd")


def attn_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, workspace, window, scale=None, stream=None):
    """Dense backward with the key window of attn_fwd_window."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    left, right = (int(w) for w in window)
    _check(load().attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                  _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  B, Hq, Hkv, N, d, scale, left, right, _dtype(q), _stream(stream)),
           "attn_bwd_window")


def attn_bwd_deterministic_workspace_size(B, Hq, Hkv, N, d):
    return load().attn_bwd_deterministic_workspace_size(B, Hq, Hkv, N, d)


def attn_bwd_deterministic(q, k, v, o, lse, dout, dq, dk, dv, workspace, window=(-1, -1), causal=False,
                           scale=None, stream=None):
    """Dense backward with one writer and one summation order per output
    element (identical bits on every call); window as attn_fwd_window, and
    causal=True means the window (-1, 0)."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    left, right = (int(w) for w in window)
    if causal:
        right = 0 if right < 0 else min(right, 0)
    _check(load().attn_bwd_deterministic(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
                                         _ptr(dk), _ptr(dv), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         B, Hq, Hkv, N, d, scale, left, right, _dtype(q), _stream(stream)),
           "attn_bwd_deterministic")


def attn_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, scale=None, causal=False, stream=None):
    """Dense backward with the library's own fixed device workspace (no allocation).

    For callers that cannot allocate device memory; see include/libattn.h.
    Calls that overlap on the GPU share that workspace and must not be issued.
    """
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                   _ptr(dv), B, Hq, Hkv, N, d, scale, int(bool(causal)), _dtype(q),
                                   _stream(stream)), "attn_bwd_noalloc")


def attn_bwd_varlen_workspace_size(T, Hq, Hkv, d):
    return int(load().attn_bwd_varlen_workspace_size(T, Hq, Hkv, d))


def attn_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, workspace, cu_seqlens, max_seqlen, scale=None,
                    causal=False, stream=None):
    T, Hq, d = q.shape
    Hkv = k.shape[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
                                  _ptr(dv), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, int(max_seqlen), Hq, Hkv, d, scale,
                                  int(bool(causal)), _dtype(q), _stream(stream)), "attn_bwd_varlen")


def attn_get_device_status(stream=None):
    return int(load().attn_get_device_status(_stream(stream)))


def attn_selftest_wait_timeout(limit_ms, stream=None):
    """Launch a warp whose bounded wait runs out after limit_ms (failure-path check)."""
    _check(load().attn_selftest_wait_timeout(int(limit_ms), _stream(stream)), "attn_selftest_wait_timeout")


def attn_status_string(code):
    return load().attn_status_string(int(code)).decode()


def attn_version():
    return load().attn_version().decode()
