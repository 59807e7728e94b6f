"""Random shapes against the float64 oracle (GPU only).

Seeded draws over what the other tests fix one at a time: batch, query and
KV heads (GQA groups 1..4), sequence length 1..700, head dim 64/128/256,
dtype, causal, a random key window, and packed sequences; each case runs the
forward and the backward through the public API (dense, window or varlen
entry point) and compares O, LSE, dQ, dK and dV with the oracle at the
tolerances of the dedicated tests.
"""
import math

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


def check_fwd(o, lse, o_ref, lse_ref, tag, packed=False):
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    vis = np.isfinite(lse_ref)   # rows with at least one visible key
    err = np.abs(o - o_ref)[vis.T if packed else vis]   # packed: O [T, H, d], LSE [H, T]
    assert err.max() <= 1e-2, (tag, err.max())
    assert math.sqrt((err ** 2).mean()) <= 2e-3, tag
    assert np.abs(lse - lse_ref)[vis].max() <= 1e-3, tag


def draw(seed):
    rng = np.random.default_rng(seed)
    hkv = int(rng.integers(1, 4))
    g = int(rng.choice([1, 2, 4]))
    d = int(rng.choice([64, 128, 256]))
    kind = str(rng.choice(["dense", "window", "varlen"]))
    causal = bool(rng.integers(0, 2))
    dtype = str(rng.choice(["bf16", "fp16"]))
    if kind == "varlen":
        lens = [int(x) for x in rng.integers(1, 400, size=int(rng.integers(1, 5)))]
        return dict(kind=kind, hkv=hkv, hq=hkv * g, d=d, causal=causal, dtype=dtype, lens=lens)
    n = int(rng.integers(1, 700))
    b = int(rng.integers(1, 3))
    window = None
    if kind == "window":
        # left bound -1 or 0..n, right bound -1 or 0..n; at least one bounded
        left = int(rng.choice([-1, int(rng.integers(0, n + 1))]))
        right = int(rng.integers(0, n + 1)) if left < 0 else int(rng.choice([-1, int(rng.integers(0, n + 1))]))
        window = (left, right)
    return dict(kind=kind, hkv=hkv, hq=hkv * g, d=d, causal=causal, dtype=dtype, n=n, b=b, window=window)


@pytest.mark.parametrize("seed", range(48))
def test_random_case(seed):
    c = draw(1000 + seed)
    tag = str(c)
    d, hq, hkv = c["d"], c["hq"], c["hkv"]
    scale = d ** -0.5
    if c["kind"] == "varlen":
        lens = c["lens"]
        cu = inputs.cu_seqlens(lens)
        T = int(cu[-1])
        q, k, v, do = inputs.normal(seed, [(T, hq, d), (T, hkv, d), (T, hkv, d), (T, hq, d)], dtype=c["dtype"])
        qd, kd, vd, dod, cud = (x.cuda() for x in (q, k, v, do, cu))
        o = torch.full_like(qd, float("nan"))
        lse = torch.full((hq, T), float("nan"), device="cuda")
        L.attn_fwd_varlen(qd, kd, vd, o, lse, cud, max(lens), causal=c["causal"])
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        ws = torch.empty((L.attn_bwd_varlen_workspace_size(T, hq, hkv, d),), dtype=torch.uint8, device="cuda")
        L.attn_bwd_varlen(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, cud, max(lens), causal=c["causal"])
        torch.cuda.synchronize()
        assert L.attn_get_device_status() == 0
        o_ref, lse_ref = A.forward_varlen(q, k, v, cu.numpy(), scale, c["causal"])
        check_fwd(o, lse, o_ref, lse_ref, tag, packed=True)
        ref = A.backward_varlen(q, k, v, do, cu.numpy(), scale, c["causal"])
    else:
        b, n = c["b"], c["n"]
        q, k, v, do = inputs.normal(seed, [(b, hq, n, d), (b, hkv, n, d), (b, hkv, n, d), (b, hq, n, d)],
                                    dtype=c["dtype"])
        qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
        o = torch.full_like(qd, float("nan"))
        lse = torch.full((b, hq, n), float("nan"), device="cuda")
        ws = torch.empty((L.attn_bwd_workspace_size(b, hq, hkv, n, d),), dtype=torch.uint8, device="cuda")
        dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
        if c["kind"] == "window":
            L.attn_fwd_window(qd, kd, vd, o, lse, c["window"])
            L.attn_bwd_window(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, c["window"])
            args = (False, c["window"])
        else:
            L.attn_fwd(qd, kd, vd, o, lse, causal=c["causal"])
            L.attn_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, causal=c["causal"])
            args = (c["causal"], None)
        torch.cuda.synchronize()
        assert L.attn_get_device_status() == 0
        o_ref, lse_ref = A.forward(q, k, v, scale, *args)
        check_fwd(o, lse, o_ref, lse_ref, tag)
        ref = A.backward(q, k, v, do, scale, *args)
    for name, g_, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
        assert rel_rms(g_, r) <= 1e-2, (name, rel_rms(g_, r), tag)
