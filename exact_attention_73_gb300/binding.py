"""ctypes binding of libattn: the C entry points under the same names.

Argument marshalling only: tensors become device pointers and sizes (after a
check that each is a contiguous GPU tensor of the documented element type and
count, since the C ABI cannot see strides), the current torch stream becomes
the stream handle, and a non-OK status raises ``AttnError``. Every step of the computation runs in the library's kernels;
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
           "attn_decode_fp8", "attn_fwd_fp8_kv_tile", "attn_quantize_fp8_varlen", "attn_fwd_fp8_varlen",
           "attn_fwd_fp8_window")


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
    "attn_fwd_fp8_window": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P], _I),
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
    "attn_quantize_fp8_varlen": ([_P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "attn_fwd_fp8_varlen": ([_P] * 9 + [_I, _I, _I, _I, _I, _I, _F, _I, _P], _I),
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


# The C ABI sees only pointers, so the layout its kernels assume is checked
# here: every tensor handed to the library is a contiguous tensor on the GPU
# with the documented number of elements and element type. A mismatch would
# otherwise make a kernel read or write past the end of a buffer.
_DEVICE_TYPE = "cuda"


def _ptr(t, name="tensor", numel=None, dtype=None, shape=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.device.type != _DEVICE_TYPE:
        raise ValueError(f"{name} must be a {_DEVICE_TYPE} tensor, not on {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (the library reads it as a dense array)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must hold {numel} elements, got {t.numel()}")
    return C.c_void_p(t.data_ptr())


def _dims(t, name, n):
    if not isinstance(t, torch.Tensor) or t.dim() != n:
        raise ValueError(f"{name} must be a {n}-D tensor")
    return tuple(t.shape)


def _nb(n):
    return (n + 127) // 128


def _bwd_ptrs(q, k, v, o, lse, dout, dq, dk, dv):
    """Pointers of a dense backward call: q [B,Hq,N,d], k/v [B,Hkv,N,d], o, dout,
    dq like q, dk/dv like k (all of q's type), lse [B,Hq,N] float32."""
    B, Hq, N, d = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    dt = q.dtype
    kv = (B, Hkv, N, d)
    return [_ptr(q, "q"), _ptr(k, "k", dtype=dt, shape=kv), _ptr(v, "v", dtype=dt, shape=kv),
            _ptr(o, "o", q.numel(), dt), _ptr(lse, "lse", B * Hq * N, torch.float32),
            _ptr(dout, "dout", q.numel(), dt), _ptr(dq, "dq", q.numel(), dt), _ptr(dk, "dk", k.numel(), dt),
            _ptr(dv, "dv", k.numel(), dt)]


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


def _fwd_ptrs(q, k, v, o, lse):
    """Pointers of a dense forward call: q [B,Hq,N,d], k/v [B,Hkv,N,d] of q's
    type, o like q, lse [B,Hq,N] float32."""
    B, Hq, N, d = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    kv = (B, Hkv, N, d)
    return [_ptr(q, "q"), _ptr(k, "k", dtype=q.dtype, shape=kv), _ptr(v, "v", dtype=q.dtype, shape=kv),
            _ptr(o, "o", q.numel(), q.dtype), _ptr(lse, "lse", B * Hq * N, torch.float32)]


def attn_fwd(q, k, v, o, lse, scale=None, causal=False, stream=None):
    """Dense forward: q [B,Hq,N,d], k/v [B,Hkv,N,d], o like q, lse [B,Hq,N] fp32."""
    B, Hq, N, d = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_fwd(*_fwd_ptrs(q, k, v, o, lse), B, Hq, Hkv, N, d, scale,
                           int(bool(causal)), _dtype(q), _stream(stream)), "attn_fwd")


def attn_fwd_window(q, k, v, o, lse, window, scale=None, stream=None):
    """Dense forward with a key window (left, right): key j is visible to
    query i iff i - left <= j <= i + right; -1 means no bound on that side."""
    B, Hq, N, d = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    left, right = (int(w) for w in window)
    _check(load().attn_fwd_window(*_fwd_ptrs(q, k, v, o, lse), B, Hq, Hkv, N, d, scale,
                                  left, right, _dtype(q), _stream(stream)), "attn_fwd_window")


def attn_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen, scale=None, causal=False, stream=None):
    """Packed forward: q [T,Hq,d], k/v [T,Hkv,d], o like q, lse [Hq,T]; cu_seqlens int32 on the device."""
    T, Hq, d = _dims(q, "q", 3)
    Hkv = _dims(k, "k", 3)[1]
    kv = (T, Hkv, d)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_fwd_varlen(_ptr(q, "q"), _ptr(k, "k", dtype=q.dtype, shape=kv),
                                  _ptr(v, "v", dtype=q.dtype, shape=kv), _ptr(o, "o", q.numel(), q.dtype),
                                  _ptr(lse, "lse", Hq * T, torch.float32),
                                  _ptr(cu_seqlens, "cu_seqlens", dtype=torch.int32),
                                  cu_seqlens.numel() - 1, T, int(max_seqlen), Hq, Hkv, d, scale,
                                  int(bool(causal)), _dtype(q), _stream(stream)), "attn_fwd_varlen")


def attn_quantize_fp8_varlen(x, x8, scales, cu_seqlens, max_seqlen, hadamard_signs=None, stream=None):
    """x [T,H,d] bf16/fp16 -> x8 uint8 codes (same shape), scales [nseq, H, ceil(max_seqlen/128)] fp32;
    each sequence is blocked from its own first row."""
    T, H, d = _dims(x, "x", 3)
    nseq = cu_seqlens.numel() - 1
    _check(load().attn_quantize_fp8_varlen(_ptr(x, "x"), _dtype(x), _ptr(x8, "x8", x.numel(), torch.uint8),
                                           _ptr(scales, "scales", nseq * H * _nb(int(max_seqlen)), torch.float32),
                                           _ptr(cu_seqlens, "cu_seqlens", dtype=torch.int32), nseq, T,
                                           int(max_seqlen), H, d,
                                           _ptr(hadamard_signs, "hadamard_signs", d, torch.int8), _stream(stream)),
           "attn_quantize_fp8_varlen")


def attn_fwd_fp8_varlen(q8, k8, v8, sq, sk, sv, o, lse, cu_seqlens, max_seqlen, scale=None, causal=False,
                        stream=None):
    """Packed FP8 forward: q8 [T,Hq,d], k8/v8 [T,Hkv,d] codes, sq [nseq,Hq,nb], sk/sv [nseq,Hkv,nb]
    (nb = ceil(max_seqlen/128)); o [T,Hq,d] bf16, lse [Hq,T] fp32."""
    T, Hq, d = _dims(q8, "q8", 3)
    Hkv = _dims(k8, "k8", 3)[1]
    kv = (T, Hkv, d)
    u8, f32 = torch.uint8, torch.float32
    nseq = cu_seqlens.numel() - 1
    nb = _nb(int(max_seqlen))
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_fwd_fp8_varlen(_ptr(q8, "q8", dtype=u8), _ptr(k8, "k8", dtype=u8, shape=kv),
                                      _ptr(v8, "v8", dtype=u8, shape=kv), _ptr(sq, "sq", nseq * Hq * nb, f32),
                                      _ptr(sk, "sk", nseq * Hkv * nb, f32), _ptr(sv, "sv", nseq * Hkv * nb, f32),
                                      _ptr(o, "o", q8.numel(), torch.bfloat16), _ptr(lse, "lse", Hq * T, f32),
                                      _ptr(cu_seqlens, "cu_seqlens", dtype=torch.int32), nseq, T,
                                      int(max_seqlen), Hq, Hkv, d, scale, int(bool(causal)), _stream(stream)),
           "attn_fwd_fp8_varlen")


def attn_quantize_fp8(x, x8, scales, hadamard_signs=None, stream=None):
    """x [B,H,N,d] bf16/fp16 -> x8 uint8 codes (same shape), scales [B,H,ceil(N/128)] fp32."""
    B, H, N, d = _dims(x, "x", 4)
    _check(load().attn_quantize_fp8(_ptr(x, "x"), _dtype(x), _ptr(x8, "x8", x.numel(), torch.uint8),
                                    _ptr(scales, "scales", B * H * _nb(N), torch.float32), B, H, N, d,
                                    _ptr(hadamard_signs, "hadamard_signs", d, torch.int8), _stream(stream)),
           "attn_quantize_fp8")


def attn_quantize_fp8_rope(x, x8, scales, rope_cos, rope_sin, hadamard_signs=None, stream=None):
    """RoPE (rotate-half, float32 cos/sin tables [N, d/2] on the device), then
    the optional rotation and block quantisation, in one pass."""
    B, H, N, d = _dims(x, "x", 4)
    _check(load().attn_quantize_fp8_rope(_ptr(x, "x"), _dtype(x), _ptr(x8, "x8", x.numel(), torch.uint8),
                                         _ptr(scales, "scales", B * H * _nb(N), torch.float32), B, H, N, d,
                                         _ptr(rope_cos, "rope_cos", N * (d // 2), torch.float32),
                                         _ptr(rope_sin, "rope_sin", N * (d // 2), torch.float32),
                                         _ptr(hadamard_signs, "hadamard_signs", d, torch.int8), _stream(stream)),
           "attn_quantize_fp8_rope")


def _fp8_ptrs(q8, k8, v8, sq, sk, sv, o, lse):
    """Checked pointers of a dense FP8 forward and its sizes (B, Hq, Hkv, N, d)."""
    B, Hq, N, d = _dims(q8, "q8", 4)
    Hkv = _dims(k8, "k8", 4)[1]
    kv = (B, Hkv, N, d)
    u8, f32 = torch.uint8, torch.float32
    ptrs = (_ptr(q8, "q8", dtype=u8), _ptr(k8, "k8", dtype=u8, shape=kv), _ptr(v8, "v8", dtype=u8, shape=kv),
            _ptr(sq, "sq", B * Hq * _nb(N), f32), _ptr(sk, "sk", B * Hkv * _nb(N), f32),
            _ptr(sv, "sv", B * Hkv * _nb(N), f32), _ptr(o, "o", q8.numel(), torch.bfloat16),
            _ptr(lse, "lse", B * Hq * N, f32))
    return ptrs, (B, Hq, Hkv, N, d)


def attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, scale=None, causal=False, stream=None):
    """FP8 forward on E4M3 codes (uint8) with block factors; o bf16, lse fp32."""
    ptrs, dims = _fp8_ptrs(q8, k8, v8, sq, sk, sv, o, lse)
    d = dims[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_fwd_fp8(*ptrs, *dims, scale, int(bool(causal)), _stream(stream)), "attn_fwd_fp8")


def attn_fwd_fp8_window(q8, k8, v8, sq, sk, sv, o, lse, window, scale=None, stream=None):
    """FP8 forward with a key window (left, right), as attn_fwd_window."""
    ptrs, dims = _fp8_ptrs(q8, k8, v8, sq, sk, sv, o, lse)
    d = dims[-1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    left, right = (int(w) for w in window)
    _check(load().attn_fwd_fp8_window(*ptrs, *dims, scale, left, right, _stream(stream)), "attn_fwd_fp8_window")


def attn_fwd_fp8_kv_tile(d):
    """Keys per KV tile of attn_fwd_fp8 for head dimension d (0: unsupported)."""
    return load().attn_fwd_fp8_kv_tile(d)


def attn_decode_fp8_workspace_size(B, Hq, d, num_splits):
    return load().attn_decode_fp8_workspace_size(B, Hq, d, num_splits)


def attn_decode_fp8(q8, sq, k8, v8, sk, sv, o, lse, workspace, num_splits, seqlens=None, scale=None, stream=None):
    """One decoded token per sequence: q8 [B,Hq,d] codes, sq [B,Hkv]; cache k8/v8
    [B,Hkv,Nmax,d] with sk/sv [B,Hkv,ceil(Nmax/128)]; seqlens int32 [B] or None;
    o [B,Hq,d] bf16, lse [B,Hq]."""
    B, Hq, d = _dims(q8, "q8", 3)
    Hkv, Nmax = _dims(k8, "k8", 4)[1:3]
    kv = (B, Hkv, Nmax, d)
    u8, f32 = torch.uint8, torch.float32
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_decode_fp8(_ptr(q8, "q8", dtype=u8), _ptr(sq, "sq", B * Hkv, f32),
                                  _ptr(k8, "k8", dtype=u8, shape=kv), _ptr(v8, "v8", dtype=u8, shape=kv),
                                  _ptr(sk, "sk", B * Hkv * _nb(Nmax), f32), _ptr(sv, "sv", B * Hkv * _nb(Nmax), f32),
                                  _ptr(seqlens, "seqlens", B, torch.int32), _ptr(o, "o", B * Hq * d, torch.bfloat16),
                                  _ptr(lse, "lse", B * Hq, f32), _ptr(workspace, "workspace"),
                                  workspace.numel() * workspace.element_size(),
                                  B, Hq, Hkv, Nmax, d, scale, int(num_splits), _stream(stream)), "attn_decode_fp8")


def attn_bwd_workspace_size(B, Hq, Hkv, N, d):
    return int(load().attn_bwd_workspace_size(B, Hq, Hkv, N, d))


def attn_bwd(q, k, v, o, lse, dout, dq, dk, dv, workspace, scale=None, causal=False, stream=None):
    """Dense backward; workspace is a byte tensor of at least attn_bwd_workspace_size bytes."""
    B, Hq, N, d = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_bwd(*_bwd_ptrs(q, k, v, o, lse, dout, dq, dk, dv), _ptr(workspace, "workspace"),
                           workspace.numel() * workspace.element_size(),
                           B, Hq, Hkv, N, d, scale, int(bool(causal)), _dtype(q), _stream(stream)), "attn_bwd")


def attn_bwd_window(q, k, v, o, lse, dout, dq, dk, dv, workspace, window, scale=None, stream=None):
    """Dense backward with the key window of attn_fwd_window."""
    B, Hq, N, d = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    left, right = (int(w) for w in window)
    _check(load().attn_bwd_window(*_bwd_ptrs(q, k, v, o, lse, dout, dq, dk, dv), _ptr(workspace, "workspace"),
                                  workspace.numel() * workspace.element_size(),
                                  B, Hq, Hkv, N, d, scale, left, right, _dtype(q), _stream(stream)),
           "attn_bwd_window")


def attn_bwd_deterministic_workspace_size(B, Hq, Hkv, N, d):
    return load().attn_bwd_deterministic_workspace_size(B, Hq, Hkv, N, d)


def attn_bwd_deterministic(q, k, v, o, lse, dout, dq, dk, dv, workspace, window=(-1, -1), causal=False,
                           scale=None, stream=None):
    """Dense backward with one writer and one summation order per output
    element (identical bits on every call); window as attn_fwd_window, and
    causal=True means the window (-1, 0)."""
    B, Hq, N, d = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    left, right = (int(w) for w in window)
    if causal:
        right = 0 if right < 0 else min(right, 0)
    _check(load().attn_bwd_deterministic(*_bwd_ptrs(q, k, v, o, lse, dout, dq, dk, dv), _ptr(workspace, "workspace"),
                                         workspace.numel() * workspace.element_size(),
                                         B, Hq, Hkv, N, d, scale, left, right, _dtype(q), _stream(stream)),
           "attn_bwd_deterministic")


def attn_bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, scale=None, causal=False, stream=None):
    """Dense backward with the library's own fixed device workspace (no allocation).

    For callers that cannot allocate device memory; see include/libattn.h.
    Calls that overlap on the GPU share that workspace and must not be issued.
    """
    B, Hq, N, d = _dims(q, "q", 4)
    Hkv = _dims(k, "k", 4)[1]
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_bwd_noalloc(*_bwd_ptrs(q, k, v, o, lse, dout, dq, dk, dv), B, Hq, Hkv, N, d, scale,
                                   int(bool(causal)), _dtype(q), _stream(stream)), "attn_bwd_noalloc")


def attn_bwd_varlen_workspace_size(T, Hq, Hkv, d):
    return int(load().attn_bwd_varlen_workspace_size(T, Hq, Hkv, d))


def attn_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, workspace, cu_seqlens, max_seqlen, scale=None,
                    causal=False, stream=None):
    T, Hq, d = _dims(q, "q", 3)
    Hkv = _dims(k, "k", 3)[1]
    kv, dt = (T, Hkv, d), q.dtype
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    _check(load().attn_bwd_varlen(_ptr(q, "q"), _ptr(k, "k", dtype=dt, shape=kv), _ptr(v, "v", dtype=dt, shape=kv),
                                  _ptr(o, "o", q.numel(), dt), _ptr(lse, "lse", Hq * T, torch.float32),
                                  _ptr(dout, "dout", q.numel(), dt), _ptr(dq, "dq", q.numel(), dt),
                                  _ptr(dk, "dk", k.numel(), dt), _ptr(dv, "dv", k.numel(), dt),
                                  _ptr(workspace, "workspace"), workspace.numel() * workspace.element_size(),
                                  _ptr(cu_seqlens, "cu_seqlens", dtype=torch.int32), cu_seqlens.numel() - 1, T,
                                  int(max_seqlen), Hq, Hkv, d, scale, int(bool(causal)), _dtype(q), _stream(stream)),
           "attn_bwd_varlen")


def attn_get_device_status(stream=None):
    return int(load().attn_get_device_status(_stream(stream)))


def attn_selftest_wait_timeout(limit_ms, stream=None):
    """Launch a warp whose bounded wait runs out after limit_ms (failure-path check)."""
    _check(load().attn_selftest_wait_timeout(int(limit_ms), _stream(stream)), "attn_selftest_wait_timeout")


def attn_status_string(code):
    return load().attn_status_string(int(code)).decode()


def attn_version():
    return load().attn_version().decode()
