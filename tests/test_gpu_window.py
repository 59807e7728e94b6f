"""Sliding-window (local) attention: the CUDA library against the float64
oracle (GPU only).

Key j is visible to query i iff i - left <= j <= i + right (-1: no bound).
Tolerances are those of the dense forward and backward tests: RMS <= 2e-3,
max |dLSE| <= 1e-3, relative RMS <= 1e-2 for dQ, dK, dV, and
max (|dO| - 2^-8 |O_ref|) <= 1e-2. The relative term matters here: a narrow
window averages few values, so |O| reaches 2-3, where rounding O to bf16
(2^-9 relative) and P to bf16 (2^-9 relative per term) exceed 1e-2 absolute.
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_73_gb300 import binding as L
from exact_attention_73_gb300 import inputs
from oracle import attention as A

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "fp16": torch.float16}

# windows around the 128-wide tiles: inside one tile, exactly one tile, just
# past a tile boundary, one-sided, two-sided, and wider than the sequence
WINDOWS = [(0, 0), (3, 0), (127, 0), (128, 0), (130, 5), (-1, 40), (64, 64), (300, -1), (5000, 5000)]


def check_o_lse(o, lse, o_ref, lse_ref, tag):
    o = o.double().cpu().numpy() if hasattr(o, "cpu") else o
    lse = lse.double().cpu().numpy() if hasattr(lse, "cpu") else lse
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all(), tag
    assert (err - 2.0 ** -8 * np.abs(o_ref)).max() <= 1e-2, (tag, err.max())
    assert math.sqrt((err ** 2).mean()) <= 2e-3, (tag, math.sqrt((err ** 2).mean()))
    assert np.abs(lse - lse_ref).max() <= 1e-3, (tag, np.abs(lse - lse_ref).max())


def rel_rms(x, ref):
    x = x.double().cpu().numpy() if hasattr(x, "cpu") else x
    assert np.isfinite(x).all()
    denom = max(float(np.linalg.norm(ref)), 1e-3 * np.sqrt(ref.size))
    return float(np.linalg.norm(x - ref) / denom)


def run_fwd(q, k, v, window):
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    B, Hq, N, d = q.shape
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((B, Hq, N), float("nan"), device="cuda")
    L.attn_fwd_window(qd, kd, vd, o, lse, window)
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    return o, lse


@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("n", [200, 1000])
def test_forward_window(window, d, n):
    q, k, v = inputs.normal(300 + d + n, [(2, 4, n, d), (2, 2, n, d), (2, 2, n, d)])
    o, lse = run_fwd(q, k, v, window)
    o_ref, lse_ref = A.forward(q, k, v, d ** -0.5, False, window)
    check_o_lse(o, lse, o_ref, lse_ref, f"d{d} n{n} w{window}")


def test_forward_window_fp16():
    q, k, v = inputs.normal(310, [(1, 2, 700, 128)] * 3, dtype="fp16")
    o, lse = run_fwd(q, k, v, (90, 10))
    o_ref, lse_ref = A.forward(q, k, v, 128 ** -0.5, False, (90, 10))
    check_o_lse(o, lse, o_ref, lse_ref, "fp16")


def test_causal_window_equals_causal_entry_point():
    q, k, v = inputs.normal(311, [(1, 4, 777, 128), (1, 2, 777, 128), (1, 2, 777, 128)])
    o1, l1 = run_fwd(q, k, v, (-1, 0))
    o2 = torch.empty_like(o1)
    l2 = torch.empty_like(l1)
    L.attn_fwd(q.cuda(), k.cuda(), v.cuda(), o2, l2, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def run_bwd(q, k, v, do, window):
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    B, Hq, N, d = q.shape
    o, lse = run_fwd(q, k, v, window)
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    ws = torch.full((L.attn_bwd_workspace_size(B, Hq, k.shape[1], N, d),), 255, dtype=torch.uint8, device="cuda")
    L.attn_bwd_window(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, window)
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    return dq.cpu(), dk.cpu(), dv.cpu()


@pytest.mark.parametrize("window", WINDOWS)
@pytest.mark.parametrize("n", [200, 700])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_backward_window(window, n, d):
    q, k, v, do = inputs.normal(320 + n, [(2, 4, n, d), (2, 2, n, d), (2, 2, n, d), (2, 4, n, d)])
    got = run_bwd(q, k, v, do, window)
    ref = A.backward(q, k, v, do, d ** -0.5, False, window)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert rel_rms(g, r) <= 1e-2, (name, window, rel_rms(g, r))


@pytest.mark.parametrize("window", [(200, 300), (0, 0), (1000, 700)])
def test_forward_window_persistent_walk(window):
    """A window bounded on both sides with a short span runs the persistent
    forward walk (one CTA per SM taking several units); B=4, H=16, N=2000
    is 512 units of two query tiles. Against the oracle on four heads."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H, n, d = 4, 16, 2000, 128
    assert (n + 255) // 256 * H * B > sms
    q, k, v = inputs.normal(71, [(B, H, n, d)] * 3)
    o, lse = run_fwd(q, k, v, window)
    o, lse = o.cpu(), lse.cpu()
    for b, h in ((0, 0), (1, 5), (2, 11), (3, 15)):
        sel = lambda x: x[b:b + 1, h:h + 1]
        o_ref, lse_ref = A.forward(sel(q), sel(k), sel(v), d ** -0.5, False, window)
        check_o_lse(sel(o), sel(lse), o_ref, lse_ref, f"b{b} h{h} w{window}")


@pytest.mark.slow
def test_window_config_sampled():
    """B=1, H=16, N=16384, d=128, window (1024, 0): sampled rows of three heads
    against the oracle's per-row forward; the backward on one head of a
    2048-token slice of the same data against the full oracle backward."""
    n, window = 16384, (1024, 0)
    q, k, v = inputs.normal(6, [(1, 16, n, 128)] * 3)
    o, lse = run_fwd(q, k, v, window)
    o, lse = o.cpu(), lse.cpu()
    rng = np.random.default_rng(61)
    for h in (0, 7, 15):
        rows = np.unique(np.concatenate([rng.choice(n, 40, replace=False), [0, 1023, 1024, 1025, n - 1]]))
        o_ref, lse_ref = A.forward_rows(q[0, h], k[0, h], v[0, h], rows, 128 ** -0.5, False, window)
        check_o_lse(o[0, h, rows], lse[0, h, rows], o_ref, lse_ref, f"h{h}")
    m = 2048
    qs, ks, vs = (x[:, :2, :m].contiguous() for x in (q, k, v))
    do = inputs.normal(62, [(1, 2, m, 128)])[0]
    got = run_bwd(qs, ks, vs, do, window)
    ref = A.backward(qs, ks, vs, do, 128 ** -0.5, False, window)
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert rel_rms(g, r) <= 1e-2, (name, rel_rms(g, r))


def _fp8_window_case(seed, b, hq, hkv, n, d, rotate):
    """Seeded outlier inputs quantised on the GPU and by the oracle (codes and
    factors checked bit for bit); returns the GPU codes and the oracle's."""
    from oracle import fp8 as F
    q, k, v = inputs.outliers(seed, [(b, hq, n, d), (b, hkv, n, d), (b, hkv, n, d)])
    signs = inputs.random_signs(4, d) if rotate else None
    nb = (n + 127) // 128

    def quant(x, s):
        x8 = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty(x.shape[:2] + (nb,), dtype=torch.float32, device="cuda")
        L.attn_quantize_fp8(x.cuda(), x8, sc, None if s is None else s.cuda())
        return x8, sc

    gpu = (quant(q, signs), quant(k, signs), quant(v, None))
    s_np = None if signs is None else signs.numpy()
    ref = (F.quantize_blocks(q, s_np), F.quantize_blocks(k, s_np), F.quantize_blocks(v))
    for (c_ref, f_ref), (c_gpu, f_gpu) in zip(ref, gpu):
        assert np.array_equal(c_gpu.cpu().numpy(), c_ref)
        assert np.array_equal(f_gpu.cpu().numpy(), f_ref)
    return gpu, ref


@pytest.mark.parametrize("window", [(0, 0), (127, 0), (130, 5), (-1, 40), (64, 64), (300, -1)])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("n", [200, 700])
def test_fp8_forward_window(window, d, n):
    """attn_fwd_fp8_window against the oracle's FP8 emulation with the same
    window, stale-max rule and KV tile (the tolerances of the dense FP8
    tests: RMS 2e-3, 99.9th percentile 1e-2, max 1e-1; LSE 1e-3)."""
    from oracle import fp8 as F
    b, hq, hkv = 1, 4, 2
    (q8g, k8g, v8g), ref = _fp8_window_case(40 + d + n, b, hq, hkv, n, d, rotate=(d != 256))
    o = torch.full((b, hq, n, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((b, hq, n), float("nan"), device="cuda")
    L.attn_fwd_fp8_window(q8g[0], k8g[0], v8g[0], q8g[1], k8g[1], v8g[1], o, lse, window)
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    codes = (ref[0][0], ref[1][0], ref[2][0], ref[0][1], ref[1][1], ref[2][1])
    o_ref, lse_ref = F.attention_fp8(*codes, d ** -0.5, tau=F.STALE_MAX_TAU, kv_tile=L.attn_fwd_fp8_kv_tile(d),
                                     window=window)
    err = np.abs(o.cpu().double().numpy() - o_ref)
    tag = f"d{d} n{n} w{window}"
    assert math.sqrt((err ** 2).mean()) <= 2e-3, tag
    assert np.quantile(err, 0.999) <= 1e-2, tag
    assert err.max() <= 1e-1, tag
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= 1e-3, tag


def test_fp8_window_special_cases_are_the_dense_entry_point():
    """The window (-1, 0) is attn_fwd_fp8 with causal masking and (-1, -1)
    attn_fwd_fp8 without: the same kernel with the same bounds, bit for bit."""
    b, hq, hkv, n, d = 2, 4, 2, 333, 128
    (q8g, k8g, v8g), _ = _fp8_window_case(55, b, hq, hkv, n, d, rotate=True)
    args = (q8g[0], k8g[0], v8g[0], q8g[1], k8g[1], v8g[1])
    for window, causal in (((-1, 0), True), ((-1, -1), False)):
        o1 = torch.empty((b, hq, n, d), dtype=torch.bfloat16, device="cuda")
        o2, l1, l2 = torch.empty_like(o1), torch.empty((b, hq, n), device="cuda"), torch.empty((b, hq, n), device="cuda")
        L.attn_fwd_fp8_window(*args, o1, l1, window)
        L.attn_fwd_fp8(*args, o2, l2, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2), window
