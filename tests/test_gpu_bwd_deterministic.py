"""Deterministic backward: parity with the float64 oracle and bit-identical
repeats (GPU only).

Tolerance: relative RMS <= 1e-2 for dQ, dK and dV, as for attn_bwd. dK and dV
come from the same key-stationary kernel as attn_bwd (its dQ product left
out), so they must equal attn_bwd's bit for bit; dQ comes from the
query-stationary kernel and must not change between calls.
"""
import numpy as np
import pytest
import torch

from exact_attention_73_gb300 import binding as L
from exact_attention_73_gb300 import inputs
from oracle import attention as A

pytestmark = pytest.mark.gpu


def rel_rms(x, ref):
    x = x.double().cpu().numpy() if hasattr(x, "cpu") else x
    assert np.isfinite(x).all()
    denom = max(float(np.linalg.norm(ref)), 1e-3 * np.sqrt(ref.size))
    return float(np.linalg.norm(x - ref) / denom)


def forward(qd, kd, vd, window):
    B, Hq, N, d = qd.shape
    o = torch.empty_like(qd)
    lse = torch.empty((B, Hq, N), device="cuda")
    L.attn_fwd_window(qd, kd, vd, o, lse, window)
    return o, lse


def run_det(qd, kd, vd, dod, o, lse, window):
    B, Hq, N, d = qd.shape
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    ws = torch.full((L.attn_bwd_deterministic_workspace_size(B, Hq, kd.shape[1], N, d),), 255,
                    dtype=torch.uint8, device="cuda")
    L.attn_bwd_deterministic(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, window=window)
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    return dq, dk, dv


def run_fused(qd, kd, vd, dod, o, lse, window):
    B, Hq, N, d = qd.shape
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty((L.attn_bwd_workspace_size(B, Hq, kd.shape[1], N, d),), dtype=torch.uint8, device="cuda")
    L.attn_bwd_window(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, window)
    torch.cuda.synchronize()
    return dq, dk, dv


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("window", [(-1, -1), (-1, 0), (100, 7)])
@pytest.mark.parametrize("n", [1, 64, 200, 640, 1000])
@pytest.mark.parametrize("d", [64, 128])
def test_parity_and_repeats(dtype, window, n, d):
    q, k, v, do = inputs.normal(400 + n + d, [(2, 4, n, d), (2, 2, n, d), (2, 2, n, d), (2, 4, n, d)],
                                dtype=dtype)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = forward(qd, kd, vd, window)
    a = run_det(qd, kd, vd, dod, o, lse, window)
    ref = A.backward(q, k, v, do, d ** -0.5, False, window)
    for name, g, r in zip(("dQ", "dK", "dV"), a, ref):
        assert rel_rms(g.cpu(), r) <= 1e-2, (name, rel_rms(g.cpu(), r))
    b = run_det(qd, kd, vd, dod, o, lse, window)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    f = run_fused(qd, kd, vd, dod, o, lse, window)
    assert torch.equal(a[1], f[1]) and torch.equal(a[2], f[2])


def test_causal_flag_is_the_causal_window():
    q, k, v, do = inputs.normal(410, [(1, 2, 333, 128)] * 4)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = forward(qd, kd, vd, (-1, 0))
    a = run_det(qd, kd, vd, dod, o, lse, (-1, 0))
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty((L.attn_bwd_deterministic_workspace_size(1, 2, 2, 333, 128),), dtype=torch.uint8,
                     device="cuda")
    L.attn_bwd_deterministic(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, causal=True)
    torch.cuda.synchronize()
    for x, y in zip(a, (dq, dk, dv)):
        assert torch.equal(x, y)


@pytest.mark.slow
def test_gqa_config_sampled_heads_and_repeats():
    """B=2, Hq=32, Hkv=8, N=8192, d=128, causal: two full calls agree bit for
    bit; the oracle checks two KV groups (each with its four query heads)."""
    q, k, v, do = inputs.normal(2, [(2, 32, 8192, 128), (2, 8, 8192, 128), (2, 8, 8192, 128),
                                    (2, 32, 8192, 128)])
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = forward(qd, kd, vd, (-1, 0))
    a = run_det(qd, kd, vd, dod, o, lse, (-1, 0))
    b = run_det(qd, kd, vd, dod, o, lse, (-1, 0))
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    dq, dk, dv = (x.cpu() for x in a)
    for (bb, g) in [(0, 0), (1, 7)]:
        hs = slice(4 * g, 4 * g + 4)
        ref = A.backward(q[bb:bb + 1, hs], k[bb:bb + 1, g:g + 1], v[bb:bb + 1, g:g + 1], do[bb:bb + 1, hs],
                         128 ** -0.5, True)
        for name, got, r in zip(("dQ", "dK", "dV"),
                                (dq[bb:bb + 1, hs], dk[bb:bb + 1, g:g + 1], dv[bb:bb + 1, g:g + 1]), ref):
            assert rel_rms(got, r) <= 1e-2, (name, bb, g, rel_rms(got, r))
