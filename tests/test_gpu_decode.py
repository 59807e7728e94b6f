"""FP8 decode over a block-quantised KV cache (split-KV): the CUDA library
against the oracle's split decode emulation and against float64 attention of
the unquantised inputs (GPU only).

Tolerances: those of the FP8 forward against its emulation (RMS <= 2e-3,
99.9th percentile <= 1e-2, max <= 1e-1 on O; |dLSE| <= 1e-3). Against exact
attention of the bf16 inputs, the error is that of the method (E4M3 operands
and P~, measured by the emulation itself) plus the kernel's arithmetic: RMS
at most the emulation's RMS error + 2e-3, and |dLSE| at most the emulation's
|dLSE| + 1e-3 (quantising q and k moves every score, hence the LSE).
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_73_gb300 import binding as L
from exact_attention_73_gb300 import inputs
from oracle import attention as A
from oracle import fp8 as F

pytestmark = pytest.mark.gpu


def quantize(x, signs=None):
    """x [B, H, N, d] bf16 on the device -> codes, factors [B, H, ceil(N/128)]."""
    B, H, N, d = x.shape
    x8 = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    sc = torch.empty((B, H, (N + 127) // 128), device="cuda")
    L.attn_quantize_fp8(x, x8, sc, signs)
    return x8, sc


def run_case(B, Hq, Hkv, nmax, d, lens, splits, seed):
    g = Hq // Hkv
    (q,) = inputs.outliers(seed, [(B, Hq, d)])
    k, v = inputs.outliers(seed + 1, [(B, Hkv, nmax, d)] * 2)
    signs = inputs.random_signs(seed + 2, d).cuda()
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    q8, sq = quantize(qd.view(B, Hkv, g, d), signs)   # one factor per KV group
    k8, sk = quantize(kd, signs)
    v8, sv = quantize(vd)
    sq = sq[:, :, 0].contiguous()
    o = torch.full((B, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, Hq), float("nan"), device="cuda")
    ws = torch.empty((L.attn_decode_fp8_workspace_size(B, Hq, d, splits),), dtype=torch.uint8, device="cuda")
    seqlens = torch.tensor(lens, dtype=torch.int32, device="cuda")
    L.attn_decode_fp8(q8.view(B, Hq, d), sq, k8, v8, sk, sv, o, lse, ws, splits, seqlens=seqlens)
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    ntiles = (nmax + 127) // 128
    tps = -(-ntiles // splits)
    # the oracle quantises the same seeded inputs itself; the GPU's codes must equal its own
    s = signs.cpu().numpy()
    rq8, rsq = F.quantize_blocks(q.view(B, Hkv, g, d), s)
    rk8, rsk = F.quantize_blocks(k, s)
    rv8, rsv = F.quantize_blocks(v)
    rsq = rsq[:, :, 0]
    for name, a, b in (("q8", q8.view(B, Hkv, g, d), rq8), ("sq", sq, rsq), ("k8", k8, rk8), ("sk", sk, rsk),
                       ("v8", v8, rv8), ("sv", sv, rsv)):
        assert np.array_equal(a.cpu().numpy(), b), name
    # the emulation of the kernel's bookkeeping (stale running max)
    o_ref, lse_ref = F.decode_fp8(rq8, rsq, rk8, rv8, rsk, rsv, lens, d ** -0.5, tps, tau=F.STALE_MAX_TAU)
    return o.double().cpu().numpy().reshape(B, Hkv, g, d), lse.cpu().numpy().reshape(B, Hkv, g), o_ref, lse_ref, \
        (q, k, v)


def check_vs_emulation(o, o_ref):
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all()
    assert math.sqrt((err ** 2).mean()) <= 2e-3, math.sqrt((err ** 2).mean())
    assert np.quantile(err, 0.999) <= 1e-2, np.quantile(err, 0.999)
    assert err.max() <= 1e-1, err.max()


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("heads", [(8, 8), (8, 2), (32, 4)])
@pytest.mark.parametrize("splits", [1, 2, 4])
def test_decode_matches_split_emulation(d, heads, splits):
    Hq, Hkv = heads
    nmax = 600
    lens = [600, 1, 129, 300]            # full, one key, one tile plus one, a split boundary
    o, lse, o_ref, lse_ref, _ = run_case(4, Hq, Hkv, nmax, d, lens, splits, 500 + d + Hq + splits)
    check_vs_emulation(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= 1e-3


def test_decode_accuracy_against_exact_attention():
    B, Hq, Hkv, nmax, d = 2, 16, 2, 3000, 128
    lens = [3000, 1777]
    o, lse, o_emu, lse_emu, (q, k, v) = run_case(B, Hq, Hkv, nmax, d, lens, 8, 77)
    g = Hq // Hkv
    rms = lambda x: math.sqrt((x ** 2).mean())
    for b in range(B):
        for kv in range(Hkv):
            n = lens[b]
            ro, rl, _ = A.head_forward(q[b, kv * g:(kv + 1) * g], k[b, kv, :n], v[b, kv, :n], d ** -0.5, False)
            assert rms(o[b, kv] - ro) <= rms(o_emu[b, kv] - ro) + 2e-3, (rms(o[b, kv] - ro), rms(o_emu[b, kv] - ro))
            assert (np.abs(lse[b, kv] - rl) - np.abs(lse_emu[b, kv] - rl)).max() <= 1e-3


def test_decode_without_seqlens_uses_the_whole_cache():
    B, Hq, Hkv, nmax, d = 1, 4, 4, 256, 64
    (q,) = inputs.normal(90, [(B, Hq, d)])
    k, v = inputs.normal(91, [(B, Hkv, nmax, d)] * 2)
    q8, sq = quantize(q.cuda().view(B, Hkv, 1, d))
    k8, sk = quantize(k.cuda())
    v8, sv = quantize(v.cuda())
    sq = sq[:, :, 0].contiguous()
    outs = []
    for seqlens in (None, torch.full((B,), nmax, dtype=torch.int32, device="cuda")):
        o = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, Hq), device="cuda")
        ws = torch.empty((L.attn_decode_fp8_workspace_size(B, Hq, d, 2),), dtype=torch.uint8, device="cuda")
        L.attn_decode_fp8(q8.view(B, Hq, d), sq, k8, v8, sk, sv, o, lse, ws, 2, seqlens=seqlens)
        torch.cuda.synchronize()
        outs.append((o, lse))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_decode_more_items_than_sms():
    """480 (split, KV head, batch) items: each CTA of the persistent kernel
    walks several, across items of different lengths and empty splits (the
    K/V ring, score buffers and Q buffers run on from one item to the next)."""
    B, Hq, Hkv, nmax, d, splits = 20, 16, 8, 384, 128, 3
    rng = np.random.default_rng(81)
    lens = [int(x) for x in rng.integers(1, nmax + 1, B)]
    lens[0], lens[1] = nmax, 1
    o, lse, o_ref, lse_ref, _ = run_case(B, Hq, Hkv, nmax, d, lens, splits, 910)
    check_vs_emulation(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= 1e-3


@pytest.mark.parametrize("d", [64, 128])
def test_decode_largest_group(d):
    """g = 128 query heads per KV head: every row of the 128-row query tile is real."""
    lens = [500, 130]
    o, lse, o_ref, lse_ref, _ = run_case(2, 128, 1, 500, d, lens, 2, 920 + d)
    check_vs_emulation(o, o_ref)
    assert np.abs(lse - lse_ref).max() <= 1e-3
