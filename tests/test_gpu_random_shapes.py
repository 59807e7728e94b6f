"""Random shapes against the float64 oracle (GPU only).

Seeded draws over what the other tests fix one at a time: batch, query and
KV heads (GQA groups 1..4), sequence length 1..700, head dim 64/128/256,
dtype, causal, a random key window, and packed sequences; each case runs the
forward and the backward through the public API (dense, window or varlen
entry point) and compares O, LSE, dQ, dK and dV with the oracle at the
tolerances of the dedicated tests. A second sweep does the same for the
FP8 quantiser and forward on dense shapes (codes bit-exact, O against the
oracle's FP8 emulation).
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


@pytest.mark.parametrize("seed", range(16))
def test_random_fp8_case(seed):
    """FP8 forward (GPU quantiser, Q and K rotated half of the time) on
    random dense shapes: codes and factors bit-exact against the oracle's
    quantisation, O within the tolerances of the stale-max emulation, LSE
    within 1e-3."""
    from oracle import fp8 as F
    rng = np.random.default_rng(2000 + seed)
    hkv = int(rng.integers(1, 4))
    hq = hkv * int(rng.choice([1, 2, 4]))
    d = int(rng.choice([64, 128, 256]))
    n = int(rng.integers(1, 600))
    b = int(rng.integers(1, 3))
    causal = bool(rng.integers(0, 2))
    rotate = bool(rng.integers(0, 2))
    tag = dict(hq=hq, hkv=hkv, d=d, n=n, b=b, causal=causal, rotate=rotate)
    q, k, v = inputs.outliers(seed, [(b, hq, n, d), (b, hkv, n, d), (b, hkv, n, d)])
    signs = inputs.random_signs(4, d) if rotate else None
    nb = (n + 127) // 128

    def quant(x, s):
        x8 = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty(x.shape[:2] + (nb,), dtype=torch.float32, device="cuda")
        L.attn_quantize_fp8(x.cuda(), x8, sc, None if s is None else s.cuda())
        return x8, sc

    (q8, sq), (k8, sk), (v8, sv) = quant(q, signs), quant(k, signs), quant(v, None)
    o = torch.full((b, hq, n, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((b, hq, n), float("nan"), device="cuda")
    L.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse, causal=causal)
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    s_np = None if signs is None else signs.numpy()
    ref = (F.quantize_blocks(q, s_np), F.quantize_blocks(k, s_np), F.quantize_blocks(v))
    for (c_ref, f_ref), (c_gpu, f_gpu) in zip(ref, ((q8, sq), (k8, sk), (v8, sv))):
        assert np.array_equal(c_gpu.cpu().numpy(), c_ref), tag
        assert np.array_equal(f_gpu.cpu().numpy(), f_ref), tag
    codes = (ref[0][0], ref[1][0], ref[2][0], ref[0][1], ref[1][1], ref[2][1])
    o_ref, lse_ref = F.attention_fp8(*codes, d ** -0.5, causal, tau=F.STALE_MAX_TAU,
                                     kv_tile=L.attn_fwd_fp8_kv_tile(d))
    err = np.abs(o.cpu().double().numpy() - o_ref)
    assert math.sqrt((err ** 2).mean()) <= 2e-3, tag
    assert np.quantile(err, 0.999) <= 1e-2, tag
    assert err.max() <= 1e-1, tag
    assert np.abs(lse.cpu().double().numpy() - lse_ref).max() <= 1e-3, tag


@pytest.mark.parametrize("seed", range(8))
def test_random_persistent_case(seed):
    """Random shapes with more units than SMs over short rows, so the
    persistent walks run (the forward unmasked or with a short two-sided
    window, the backward unmasked): batch 12..48, GQA groups 1..4, length
    1..768, head dim 64/128, BF16/FP16. Forward and backward through the
    public API; two (batch, KV group) slices against the oracle."""
    rng = np.random.default_rng(3000 + seed)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    d = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4]))
    hkv = int(rng.integers(2, 5))
    n = int(rng.integers(1, 769))
    b = max(int(rng.integers(12, 49)), sms // ((n + 127) // 128 * hkv) + 1)
    window = None if rng.integers(0, 2) else (int(rng.integers(0, 600)), int(rng.integers(0, 600)))
    dtype = str(rng.choice(["bf16", "fp16"]))
    hq = hkv * g
    tag = dict(b=b, hq=hq, hkv=hkv, n=n, d=d, window=window, dtype=dtype)
    q, k, v, do = inputs.normal(seed, [(b, hq, n, d), (b, hkv, n, d), (b, hkv, n, d), (b, hq, n, d)], dtype=dtype)
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o = torch.full_like(qd, float("nan"))
    lse = torch.full((b, hq, n), float("nan"), device="cuda")
    if window is None:
        L.attn_fwd(qd, kd, vd, o, lse)
    else:
        L.attn_fwd_window(qd, kd, vd, o, lse, window)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty((L.attn_bwd_workspace_size(b, hq, hkv, n, d),), dtype=torch.uint8, device="cuda")
    if window is None:
        L.attn_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, ws)
    else:
        L.attn_bwd_window(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, window)
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    o, lse, dq, dk, dv = (x.cpu() for x in (o, lse, dq, dk, dv))
    args = (False, window)
    for bi, gi in ((0, 0), (b - 1, hkv - 1)):
        qs, dos = q[bi:bi + 1, gi * g:(gi + 1) * g], do[bi:bi + 1, gi * g:(gi + 1) * g]
        ks, vs = k[bi:bi + 1, gi:gi + 1], v[bi:bi + 1, gi:gi + 1]
        o_ref, lse_ref = A.forward(qs, ks, vs, d ** -0.5, *args)
        check_fwd(o[bi:bi + 1, gi * g:(gi + 1) * g], lse[bi:bi + 1, gi * g:(gi + 1) * g], o_ref, lse_ref, tag)
        ref = A.backward(qs, ks, vs, dos, d ** -0.5, *args)
        got = (dq[bi:bi + 1, gi * g:(gi + 1) * g], dk[bi:bi + 1, gi:gi + 1], dv[bi:bi + 1, gi:gi + 1])
        for name, g_, r in zip(("dQ", "dK", "dV"), got, ref):
            assert rel_rms(g_, r) <= 1e-2, (name, rel_rms(g_, r), tag)
