"""Parity in the benchmark's own step configuration (GPU only).

B=2, H=16, N=8192, d=128, non-causal, the benchmark's seeded N(0,1) inputs
(Q, K, V, dO drawn in that order from seed 1; rotation signs from seed 4):
the full-size GPU backward, and the full-size FP8 forward after the GPU
quantiser, each checked on sampled heads against the oracle. (The BF16
forward on these inputs is covered by the full-size sweep test.)
Tolerances as elsewhere: relative RMS <= 1e-2 per gradient; FP8 forward
RMS <= 1.5e-2 against float64 attention of the unquantised inputs, and within
the emulation tolerances of the oracle's FP8 emulation.
"""
import math

import numpy as np
import pytest
import torch

from exact_attention_73_gb300 import binding as L
from exact_attention_73_gb300 import inputs
from oracle import attention as A
from oracle import fp8 as F

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

B, H, N, D = 2, 16, 8192, 128
HEADS = [(0, 0), (1, 15)]


def bench_inputs():
    return inputs.normal(1, [(B, H, N, D)] * 4)


def rel_rms(x, ref):
    x = x.double().numpy()
    assert np.isfinite(x).all()
    return float(np.linalg.norm(x - ref) / np.linalg.norm(ref))


def test_backward_sampled_heads():
    q, k, v, do = bench_inputs()
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    o, lse = torch.empty_like(qd), torch.empty((B, H, N), device="cuda")
    L.attn_fwd(qd, kd, vd, o, lse)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty((L.attn_bwd_workspace_size(B, H, H, N, D),), dtype=torch.uint8, device="cuda")
    L.attn_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, ws)
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    for b, h in HEADS:
        one = lambda x: x[b:b + 1, h:h + 1]
        ref = A.backward(one(q), one(k), one(v), one(do), D ** -0.5, False)
        for name, got, r in zip(("dQ", "dK", "dV"), (one(dq), one(dk), one(dv)), ref):
            assert rel_rms(got, r) <= 1e-2, (name, b, h, rel_rms(got, r))


def test_fp8_forward_sampled_heads():
    q, k, v, _ = bench_inputs()
    signs = inputs.random_signs(4, D)
    nb = (N + 127) // 128
    dev = [x.cuda() for x in (q, k, v)]
    codes = []
    for x, s in zip(dev, (signs, signs, None)):
        x8 = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty((B, H, nb), device="cuda")
        L.attn_quantize_fp8(x, x8, sc, None if s is None else s.cuda())
        codes.append((x8, sc))
    (q8, sq), (k8, sk), (v8, sv) = codes
    o = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, N), float("nan"), device="cuda")
    L.attn_fwd_fp8(q8, k8, v8, sq, sk, sv, o, lse)
    torch.cuda.synchronize()
    assert L.attn_get_device_status() == 0
    o = o.cpu().double().numpy()
    rows = np.unique(np.concatenate([np.random.default_rng(11).choice(N, 48, replace=False), [0, 127, 128, N - 1]]))
    for b, h in HEADS:
        one = lambda x: x[b:b + 1, h:h + 1]
        # the oracle quantises the head itself; the GPU's codes and factors must equal its own
        mine = [F.quantize_blocks(one(q), signs.numpy()), F.quantize_blocks(one(k), signs.numpy()),
                F.quantize_blocks(one(v))]
        for (c, f), (g8, gs) in zip(mine, codes):
            assert np.array_equal(one(g8).cpu().numpy(), c) and np.array_equal(one(gs).cpu().numpy(), f)
        (rq8, rsq), (rk8, rsk), (rv8, rsv) = mine
        emu, _ = F.attention_fp8(rq8, rk8, rv8, rsq, rsk, rsv, D ** -0.5, rows=rows, tau=F.STALE_MAX_TAU,
                                 kv_tile=L.attn_fwd_fp8_kv_tile(D))
        exact, _ = A.forward_rows(q[b, h], k[b, h], v[b, h], rows, D ** -0.5)
        got = o[b, h, rows]
        err_emu = np.abs(got - emu[0, 0, rows])
        assert math.sqrt((err_emu ** 2).mean()) <= 2e-3 and np.quantile(err_emu, 0.999) <= 1e-2 \
            and err_emu.max() <= 1e-1, (b, h, err_emu.max())
        assert math.sqrt(((got - exact) ** 2).mean()) <= 1.5e-2
