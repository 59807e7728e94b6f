"""Failure path of the kernels' bounded waits (GPU), without a fault or a hang.

A warp waits on a barrier that nothing completes; its bounded wait must end by
itself, the device status must read ATTN_ERR_TIMEOUT exactly once, and the
context must stay usable for an ordinary forward pass afterwards.
"""
import time

import numpy as np
import pytest
import torch

from exact_attention_73_gb300 import binding as L
from exact_attention_73_gb300 import inputs
from oracle import attention as A

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_is_reported_and_cleared(lib):
    assert L.attn_get_device_status() == 0
    t0 = time.perf_counter()
    L.attn_selftest_wait_timeout(200)
    assert L.attn_get_device_status() == 9          # ATTN_ERR_TIMEOUT
    assert time.perf_counter() - t0 >= 0.2          # the wait lasted at least its limit
    assert L.attn_get_device_status() == 0          # read once, then cleared
    # the context is still usable
    q, k, v = inputs.normal(3, [(1, 2, 200, 128)] * 3)
    qd, kd, vd = (x.cuda() for x in (q, k, v))
    o = torch.empty_like(qd)
    lse = torch.empty((1, 2, 200), device="cuda")
    L.attn_fwd(qd, kd, vd, o, lse, causal=True)
    torch.cuda.synchronize()
    o_ref, _ = A.forward(q, k, v, 128 ** -0.5, True)
    assert np.abs(o.double().cpu().numpy() - o_ref).max() <= 1e-2
    assert L.attn_get_device_status() == 0


def test_limit_is_checked(lib):
    with pytest.raises(L.AttnError):
        L.attn_selftest_wait_timeout(0)
