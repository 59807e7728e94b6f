"""The Python binding's tensor checks (CPU only).

The C ABI receives bare pointers, so the binding checks every tensor it hands
over: on the GPU, contiguous, of the documented element type and element
count. These tests replay the calls that the GPU tests, the benchmark and
smoke() make (same shapes and types, on CPU tensors, with the device check
pointed at the CPU and a stand-in library that records the call), and check
that tensors a kernel would read or write out of bounds are refused before
the library is called.
"""
import types

import pytest
import torch

from exact_attention_73_gb300 import binding as L

STREAM = types.SimpleNamespace(cuda_stream=0)
BF, FP, U8, F32, I32 = torch.bfloat16, torch.float16, torch.uint8, torch.float32, torch.int32


class _Lib:
    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        def call(*args):
            self.calls.append(name)
            return 0
        return call


@pytest.fixture
def lib(monkeypatch):
    fake = _Lib()
    monkeypatch.setattr(L, "_DEVICE_TYPE", "cpu")
    monkeypatch.setattr(L, "load", lambda build_if_missing=True: fake)
    return fake


def z(*shape, dtype=BF):
    return torch.zeros(shape, dtype=dtype)


def dense(dtype=BF, B=1, Hq=4, Hkv=2, N=300, d=128):
    q, k, v = z(B, Hq, N, d, dtype=dtype), z(B, Hkv, N, d, dtype=dtype), z(B, Hkv, N, d, dtype=dtype)
    return q, k, v, torch.empty_like(q), z(B, Hq, N, dtype=F32)


@pytest.mark.parametrize("dtype", [BF, FP])
def test_dense_calls_of_the_tests_pass(lib, dtype):
    q, k, v, o, lse = dense(dtype)
    do, dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = z(1024, dtype=U8)
    L.attn_fwd(q, k, v, o, lse, causal=True, stream=STREAM)
    L.attn_fwd_window(q, k, v, o, lse, (64, 0), stream=STREAM)
    L.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, causal=True, stream=STREAM)
    L.attn_bwd_window(q, k, v, o, lse, do, dq, dk, dv, ws, (100, 7), stream=STREAM)
    L.attn_bwd_deterministic(q, k, v, o, lse, do, dq, dk, dv, ws, window=(64, 0), stream=STREAM)
    L.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, causal=True, stream=STREAM)
    assert lib.calls == ["attn_fwd", "attn_fwd_window", "attn_bwd", "attn_bwd_window", "attn_bwd_deterministic",
                         "attn_bwd_noalloc"]


def test_varlen_calls_of_the_tests_pass(lib):
    T, Hq, Hkv, d = 1000, 4, 2, 128
    q, k, v = z(T, Hq, d), z(T, Hkv, d), z(T, Hkv, d)
    o, do, dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q), torch.empty_like(k), \
        torch.empty_like(v)
    lse = z(Hq, T, dtype=F32)
    cu = torch.tensor([0, 300, 1000], dtype=I32)
    L.attn_fwd_varlen(q, k, v, o, lse, cu, 700, causal=True, stream=STREAM)
    L.attn_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, z(64, dtype=U8), cu, 700, causal=True, stream=STREAM)
    assert lib.calls == ["attn_fwd_varlen", "attn_bwd_varlen"]


def test_fp8_calls_of_the_tests_pass(lib):
    B, Hq, Hkv, N, d = 1, 4, 2, 700, 128
    nb = 6
    signs = z(d, dtype=torch.int8)
    x = z(B, Hq, N, d)
    L.attn_quantize_fp8(x, z(B, Hq, N, d, dtype=U8), z(B, Hq, nb, dtype=F32), signs, stream=STREAM)
    L.attn_quantize_fp8(x, z(B, Hq, N, d, dtype=U8), z(B, Hq, nb, dtype=F32), stream=STREAM)
    cos = z(N, d // 2, dtype=F32)
    L.attn_quantize_fp8_rope(x, z(B, Hq, N, d, dtype=U8), z(B, Hq, nb, dtype=F32), cos, cos, signs, stream=STREAM)
    # the decode's query quantisation: g = 4 rows per KV group, one factor each
    L.attn_quantize_fp8(z(B, 2, 4, d), z(B, 2, 4, d, dtype=U8), z(B, 2, 1, dtype=F32), signs, stream=STREAM)
    L.attn_fwd_fp8(z(B, Hq, N, d, dtype=U8), z(B, Hkv, N, d, dtype=U8), z(B, Hkv, N, d, dtype=U8),
                   z(B, Hq, nb, dtype=F32), z(B, Hkv, nb, dtype=F32), z(B, Hkv, nb, dtype=F32), z(B, Hq, N, d),
                   z(B, Hq, N, dtype=F32), causal=True, stream=STREAM)
    L.attn_fwd_fp8_window(z(B, Hq, N, d, dtype=U8), z(B, Hkv, N, d, dtype=U8), z(B, Hkv, N, d, dtype=U8),
                          z(B, Hq, nb, dtype=F32), z(B, Hkv, nb, dtype=F32), z(B, Hkv, nb, dtype=F32),
                          z(B, Hq, N, d), z(B, Hq, N, dtype=F32), (130, 5), stream=STREAM)
    assert lib.calls == ["attn_quantize_fp8"] * 2 + ["attn_quantize_fp8_rope", "attn_quantize_fp8", "attn_fwd_fp8",
                         "attn_fwd_fp8_window"]
    # the window call refuses what the plain one refuses: a short factor array
    with pytest.raises(ValueError):
        L.attn_fwd_fp8_window(z(B, Hq, N, d, dtype=U8), z(B, Hkv, N, d, dtype=U8), z(B, Hkv, N, d, dtype=U8),
                              z(B, Hq, nb - 1, dtype=F32), z(B, Hkv, nb, dtype=F32), z(B, Hkv, nb, dtype=F32),
                              z(B, Hq, N, d), z(B, Hq, N, dtype=F32), (130, 5), stream=STREAM)


@pytest.mark.parametrize("with_lengths", [False, True])
def test_decode_call_of_the_tests_passes(lib, with_lengths):
    B, Hq, Hkv, Nmax, d = 4, 32, 8, 600, 128
    seqlens = torch.tensor([600, 1, 129, 300], dtype=I32) if with_lengths else None
    L.attn_decode_fp8(z(B, Hq, d, dtype=U8), z(B, Hkv, dtype=F32), z(B, Hkv, Nmax, d, dtype=U8),
                      z(B, Hkv, Nmax, d, dtype=U8), z(B, Hkv, 5, dtype=F32), z(B, Hkv, 5, dtype=F32), z(B, Hq, d),
                      z(B, Hq, dtype=F32), z(4096, dtype=U8), 2, seqlens=seqlens, stream=STREAM)
    assert lib.calls == ["attn_decode_fp8"]


def test_layout_errors_are_refused_before_the_library(lib):
    q, k, v, o, lse = dense()
    bad = [
        (ValueError, "contiguous", lambda: L.attn_fwd(q.transpose(2, 3).contiguous().transpose(2, 3), k, v, o, lse,
                                                      stream=STREAM)),
        (TypeError, "must be torch.bfloat16", lambda: L.attn_fwd(q, k, v, o.float(), lse, stream=STREAM)),
        (TypeError, "must be torch.float32", lambda: L.attn_fwd(q, k, v, o, lse.double(), stream=STREAM)),
        (ValueError, "elements", lambda: L.attn_fwd(q, k, v, o, lse[:, :, :10].contiguous(), stream=STREAM)),
        (ValueError, "shape", lambda: L.attn_fwd(q, k.transpose(1, 2).contiguous(), v, o, lse, stream=STREAM)),
        (TypeError, "must be torch.bfloat16", lambda: L.attn_fwd(q, k.half(), v, o, lse, stream=STREAM)),
        (ValueError, "4-D", lambda: L.attn_fwd(q[0], k, v, o, lse, stream=STREAM)),
        (ValueError, "elements", lambda: L.attn_bwd(q, k, v, o, lse, q, q, k[:, :1].contiguous(), v, z(64, dtype=U8),
                                                    stream=STREAM)),
        (ValueError, "elements", lambda: L.attn_quantize_fp8(q, z(1, 4, 300, 128, dtype=U8), z(1, 4, 2, dtype=F32),
                                                             stream=STREAM)),
        (ValueError, "elements", lambda: L.attn_quantize_fp8(q, z(1, 4, 300, 128, dtype=U8), z(1, 4, 3, dtype=F32),
                                                             z(64, dtype=torch.int8), stream=STREAM)),
        (TypeError, "must be torch.uint8", lambda: L.attn_quantize_fp8(q, z(1, 4, 300, 128, dtype=torch.int8),
                                                                      z(1, 4, 3, dtype=F32), stream=STREAM)),
        (TypeError, "must be torch.int32", lambda: L.attn_fwd_varlen(z(300, 4, 128), z(300, 2, 128), z(300, 2, 128),
                                                                    z(300, 4, 128), z(4, 300, dtype=F32),
                                                                    torch.tensor([0, 300]), 300, stream=STREAM)),
        (TypeError, "must be torch.int32", lambda: L.attn_decode_fp8(
            z(1, 4, 128, dtype=U8), z(1, 2, dtype=F32), z(1, 2, 200, 128, dtype=U8), z(1, 2, 200, 128, dtype=U8),
            z(1, 2, 2, dtype=F32), z(1, 2, 2, dtype=F32), z(1, 4, 128), z(1, 4, dtype=F32), z(64, dtype=U8), 1,
            seqlens=torch.tensor([200]), stream=STREAM)),
        (TypeError, "expected a torch.Tensor", lambda: L.attn_fwd(q, k, v, o, lse.numpy(), stream=STREAM)),
    ]
    for err, text, call in bad:
        with pytest.raises(err, match=text):
            call()
    assert lib.calls == []


def test_host_tensors_are_refused_on_the_real_device_check(monkeypatch):
    fake = _Lib()
    monkeypatch.setattr(L, "load", lambda build_if_missing=True: fake)
    q, k, v, o, lse = dense()
    with pytest.raises(ValueError, match="must be a cuda tensor"):
        L.attn_fwd(q, k, v, o, lse, stream=STREAM)
    assert fake.calls == []
