"""Guard canaries: every entry point writes its outputs and nothing next to
them (GPU only).

Each output (and each workspace) is a view into the middle of a larger buffer
whose margins hold a sentinel value; after the call the margins must still
hold it, the interior must have been written, and, for the kernels whose
result does not depend on the order of atomic additions, a second call into
fresh buffers must give the same bits. Shapes are ragged (lengths that are not
multiples of 128, GQA groups) so that the edge tiles are exercised.
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_73_gb300 import binding as L
from exact_attention_73_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
PAD = 4096                     # elements on each side (a multiple of 16 bytes for every type)
SENTINEL = {torch.bfloat16: -7.0, torch.float16: -7.0, torch.float32: -7.0, torch.uint8: 0x5A}


def padded(shape, dtype):
    """(buffer, view): the view is a contiguous tensor of `shape` in the middle
    of the buffer; the margins hold the sentinel, a floating-point interior
    starts as NaN so that an element left unwritten shows."""
    n = math.prod(shape)
    buf = torch.full((PAD + n + PAD,), SENTINEL[dtype], dtype=dtype, device=DEV)
    view = buf[PAD:PAD + n].view(shape)
    if dtype.is_floating_point:
        view.fill_(float("nan"))
    return buf, view


def margins_intact(buf):
    s = SENTINEL[buf.dtype]
    return bool((buf[:PAD] == s).all()) and bool((buf[-PAD:] == s).all())


def check(bufs, outs):
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    for name, buf in bufs.items():
        assert margins_intact(buf), f"{name}: a margin was overwritten"
    for name, t in outs.items():
        if t.dtype == torch.uint8:
            continue
        assert torch.isfinite(t.float()).all(), f"{name}: not written everywhere"


def dense_inputs(seed, B=1, Hq=4, Hkv=2, N=300, d=128, dtype="bf16"):
    q, k, v, do = inputs.normal(seed, [(B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d), (B, Hq, N, d)], dtype=dtype)
    return [x.to(DEV) for x in (q, k, v, do)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("window", [None, (-1, 0), (64, 0)])
def test_forward(dtype, window):
    q, k, v, _ = dense_inputs(700, dtype=dtype)
    B, Hq, N, d = q.shape
    ob, o = padded(q.shape, q.dtype)
    lb, lse = padded((B, Hq, N), torch.float32)
    call = (lambda o_, l_: L.attn_fwd(q, k, v, o_, l_)) if window is None else \
        (lambda o_, l_: L.attn_fwd_window(q, k, v, o_, l_, window))
    call(o, lse)
    check({"o": ob, "lse": lb}, {"o": o, "lse": lse})
    o2, l2 = torch.empty_like(o), torch.empty_like(lse)
    call(o2, l2)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("kind,d", [("fused", 128), ("window", 128), ("deterministic", 128), ("noalloc", 128),
                                    ("fused", 64), ("window", 64), ("deterministic", 64), ("noalloc", 64),
                                    ("fused", 256), ("window", 256)])
def test_backward(kind, d):
    q, k, v, do = dense_inputs(701, d=d)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    o, lse = torch.empty_like(q), torch.empty((B, Hq, N), device=DEV)
    L.attn_fwd(q, k, v, o, lse, causal=True)
    bufs, outs = {}, {}
    for name, like in (("dq", q), ("dk", k), ("dv", v)):
        bufs[name], outs[name] = padded(like.shape, like.dtype)
    if kind != "noalloc":
        wsize = (L.attn_bwd_deterministic_workspace_size if kind == "deterministic" else L.attn_bwd_workspace_size)(
            B, Hq, Hkv, N, d)
        bufs["workspace"], ws = padded((wsize,), torch.uint8)
    dq, dk, dv = outs["dq"], outs["dk"], outs["dv"]
    if kind == "fused":
        L.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, causal=True)
    elif kind == "window":
        L.attn_bwd_window(q, k, v, o, lse, do, dq, dk, dv, ws, (-1, 0))
    elif kind == "deterministic":
        L.attn_bwd_deterministic(q, k, v, o, lse, do, dq, dk, dv, ws, causal=True)
    else:
        L.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, causal=True)
    check(bufs, outs)
    # dK and dV have one writer and one summation order per element: every
    # variant gives the fused backward's bits
    dq2, dk2, dv2 = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    ws2 = torch.empty((L.attn_bwd_workspace_size(B, Hq, Hkv, N, d),), dtype=torch.uint8, device=DEV)
    L.attn_bwd(q, k, v, o, lse, do, dq2, dk2, dv2, ws2, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)


@pytest.mark.parametrize("d", [64, 128])
def test_persistent_walks(d):
    """The persistent walks (more units than SMs over short rows: the forward
    without masks and with a short two-sided window, the backward without
    masks), ragged rows, GQA: margins untouched, every element written."""
    q, k, v, do = dense_inputs(702, B=24, Hq=8, Hkv=4, N=200, d=d)
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert (N + 127) // 128 * Hkv * B > sms and (N + 255) // 256 * Hq * B > sms
    for window in ((30, 50), None):   # the backward takes the unmasked forward's O and LSE
        ob, o = padded(q.shape, q.dtype)
        lb, lse = padded((B, Hq, N), torch.float32)
        if window is None:
            L.attn_fwd(q, k, v, o, lse)
        else:
            L.attn_fwd_window(q, k, v, o, lse, window)
        check({"o": ob, "lse": lb}, {"o": o, "lse": lse})
    bufs, outs = {}, {}
    for name, like in (("dq", q), ("dk", k), ("dv", v)):
        bufs[name], outs[name] = padded(like.shape, like.dtype)
    bufs["workspace"], ws = padded((L.attn_bwd_workspace_size(B, Hq, Hkv, N, d),), torch.uint8)
    L.attn_bwd(q, k, v, o, lse, do, outs["dq"], outs["dk"], outs["dv"], ws)
    check(bufs, outs)


def test_varlen_forward_and_backward():
    lens = [1, 127, 300, 5, 129]
    cu = inputs.cu_seqlens(lens).to(DEV)
    T, Hq, Hkv, d = int(sum(lens)), 4, 2, 128
    q, k, v, do = (x.to(DEV) for x in inputs.normal(702, [(T, Hq, d), (T, Hkv, d), (T, Hkv, d), (T, Hq, d)]))
    ob, o = padded(q.shape, q.dtype)
    lb, lse = padded((Hq, T), torch.float32)
    L.attn_fwd_varlen(q, k, v, o, lse, cu, max(lens), causal=True)
    check({"o": ob, "lse": lb}, {"o": o, "lse": lse})
    bufs, outs = {}, {}
    for name, like in (("dq", q), ("dk", k), ("dv", v)):
        bufs[name], outs[name] = padded(like.shape, like.dtype)
    bufs["workspace"], ws = padded((L.attn_bwd_varlen_workspace_size(T, Hq, Hkv, d),), torch.uint8)
    L.attn_bwd_varlen(q, k, v, o, lse, do, outs["dq"], outs["dk"], outs["dv"], ws, cu, max(lens), causal=True)
    check(bufs, outs)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("rope", [False, True])
def test_quantiser(d, rope):
    (x,) = inputs.outliers(703, [(2, 3, 300, d)])
    x = x.to(DEV)
    B, H, N, _ = x.shape
    signs = inputs.random_signs(4, d).to(DEV)
    cb, codes = padded(x.shape, torch.uint8)
    sb, scales = padded((B, H, (N + 127) // 128), torch.float32)
    if rope:
        ang = torch.arange(N, dtype=torch.float64)[:, None] * 10000.0 ** (-2.0 * torch.arange(d // 2) / d)[None, :]
        cos, sin = (t.to(torch.float32).to(DEV).contiguous() for t in (torch.cos(ang), torch.sin(ang)))
        L.attn_quantize_fp8_rope(x, codes, scales, cos, sin, signs)
    else:
        L.attn_quantize_fp8(x, codes, scales, signs)
    check({"codes": cb, "scales": sb}, {"scales": scales})
    # the codes are compared with a call into fresh buffers (the quantiser is exact)
    c2, s2 = torch.empty_like(codes), torch.empty_like(scales)
    if rope:
        L.attn_quantize_fp8_rope(x, c2, s2, cos, sin, signs)
    else:
        L.attn_quantize_fp8(x, c2, s2, signs)
    torch.cuda.synchronize()
    assert torch.equal(codes, c2) and torch.equal(scales, s2)


def _fp8_operands(seed, shapes):
    """Block-quantised E4M3 codes and factors of seeded outlier inputs of the given shapes."""
    out = []
    for x in (t.to(DEV) for t in inputs.outliers(seed, shapes)):
        x8 = torch.empty(x.shape, dtype=torch.uint8, device=DEV)
        sc = torch.empty((x.shape[0], x.shape[1], (x.shape[2] + 127) // 128), device=DEV)
        L.attn_quantize_fp8(x, x8, sc)
        out.append((x8, sc))
    return out


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True])
def test_fp8_forward(d, causal):
    B, Hq, Hkv, N = 1, 4, 2, 300
    (q8, sq), (k8, sk), (v8, sv) = _fp8_operands(704, [(B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d)])
    ob, o = padded((B, Hq, N, d), torch.bfloat16)
    lb, lse = padded((B, Hq, N), torch.float32)
    L.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, causal=causal)
    check({"o": ob, "lse": lb}, {"o": o, "lse": lse})
    o2, l2 = torch.empty_like(o), torch.empty_like(lse)
    L.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o2, l2, causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("window", [(30, 50), (200, 0)])
def test_fp8_forward_window(d, window):
    B, Hq, Hkv, N = 1, 4, 2, 300
    (q8, sq), (k8, sk), (v8, sv) = _fp8_operands(705, [(B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d)])
    ob, o = padded((B, Hq, N, d), torch.bfloat16)
    lb, lse = padded((B, Hq, N), torch.float32)
    L.attn_fwd_fp8_window(q8, k8, v8, sq, sk, sv, o, lse, window)
    check({"o": ob, "lse": lb}, {"o": o, "lse": lse})


@pytest.mark.parametrize("splits", [1, 3])
def test_fp8_decode(splits):
    B, Hq, Hkv, Nmax, d = 3, 16, 4, 500, 128
    g = Hq // Hkv
    (k8, sk), (v8, sv) = _fp8_operands(705, [(B, Hkv, Nmax, d)] * 2)
    (q,) = inputs.outliers(706, [(B, Hq, d)])
    q8 = torch.empty((B, Hq, d), dtype=torch.uint8, device=DEV)
    sq3 = torch.empty((B, Hkv, 1), device=DEV)
    L.attn_quantize_fp8(q.to(DEV).view(B, Hkv, g, d), q8.view(B, Hkv, g, d), sq3)
    sq = sq3[:, :, 0].contiguous()
    ob, o = padded((B, Hq, d), torch.bfloat16)
    lb, lse = padded((B, Hq), torch.float32)
    wb, ws = padded((L.attn_decode_fp8_workspace_size(B, Hq, d, splits),), torch.uint8)
    seqlens = torch.tensor([500, 1, 260], dtype=torch.int32, device=DEV)
    L.attn_decode_fp8(q8, sq, k8, v8, sk, sv, o, lse, ws, splits, seqlens=seqlens)
    check({"o": ob, "lse": lb, "workspace": wb}, {"o": o, "lse": lse})
    o2, l2 = torch.empty_like(o), torch.empty_like(lse)
    ws2 = torch.empty_like(ws)
    L.attn_decode_fp8(q8, sq, k8, v8, sk, sv, o2, l2, ws2, splits, seqlens=seqlens)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    assert np.isfinite(lse.cpu().numpy()).all()
