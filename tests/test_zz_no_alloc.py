"""attn_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc for attn_bwd's workspace: their device
memory is already held by another allocator, or they must not allocate while
running. attn_bwd_noalloc uses a fixed array owned by the library instead.
These tests check, through the C ABI, that it returns what attn_bwd returns
with a caller-provided workspace, on two calls in a row (the shared array keeps
the previous call's contents, so the second call also checks that nothing
carries over), and that oversized problems are refused.
The test session runs this file last (tests/conftest.py orders it after
every other file), so a run that stops at its first failure has already run
every other test when one of these fails.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from exact_attention_73_gb300 import binding as L
from exact_attention_73_gb300 import inputs

MAX_BYTES = 32 * 1024 * 1024


def rel_rms(x, ref):
    x = x.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    assert np.isfinite(x).all()
    denom = max(float(np.linalg.norm(ref)), 1e-3 * np.sqrt(ref.size))
    return float(np.linalg.norm(x - ref) / denom)


def _case(seed, B, Hq, Hkv, N, causal):
    d = 128
    q, k, v, do = (x.cuda() for x in inputs.normal(seed, [(B, Hq, N, d), (B, Hkv, N, d), (B, Hkv, N, d),
                                                           (B, Hq, N, d)]))
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, N), device="cuda")
    L.attn_fwd(q, k, v, o, lse, causal=causal)
    ref = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    ws = torch.empty((L.attn_bwd_workspace_size(B, Hq, Hkv, N, d),), dtype=torch.uint8, device="cuda")
    L.attn_bwd(q, k, v, o, lse, do, *ref, ws, causal=causal)
    return (q, k, v, o, lse, do), ref


@pytest.mark.gpu
def test_noalloc_backward_matches_workspace_backward_on_two_calls():
    # the last case needs 33,552,384 of the array's 33,554,432 bytes
    cases = [(31, 1, 4, 2, 1000, True), (32, 1, 8, 4, 4096, False), (33, 1, 16, 4, 4064, True)]
    for seed, B, Hq, Hkv, N, causal in cases:
        assert L.attn_bwd_workspace_size(B, Hq, Hkv, N, 128) <= MAX_BYTES
        args, ref = _case(seed, B, Hq, Hkv, N, causal)
        got = [torch.full_like(x, float("nan")) for x in ref]
        L.attn_bwd_noalloc(*args, *got, causal=causal)
        torch.cuda.synchronize()
        assert L.attn_get_device_status() == 0
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert rel_rms(g, r) <= 1e-2, (name, seed, rel_rms(g, r))


@pytest.mark.gpu
def test_noalloc_refuses_oversized_problem_on_a_gpu():
    """Where the array is actually loaded: a problem one row too large for it
    is refused with ATTN_ERR_WORKSPACE before any device work (the pointers
    are aligned stand-ins that are never dereferenced)."""
    lib = L.load()
    P = C.c_void_p
    args = [P(256)] * 9
    assert L.attn_bwd_workspace_size(1, 16, 4, 4065, 128) > MAX_BYTES
    assert lib.attn_bwd_noalloc(*args, 1, 16, 4, 4065, 128, 0.1, 1, 0, None) == 7
    assert lib.attn_bwd_noalloc(*args, 2, 32, 8, 8192, 128, 0.1, 1, 0, None) == 7
    assert L.attn_get_device_status() == 0


@pytest.mark.skipif(torch.cuda.is_available(), reason="argument check only, run where no GPU is present")
def test_noalloc_refuses_problems_larger_than_its_array():
    lib = L.load()
    P = C.c_void_p
    args = [P(16)] * 9
    # 2 x 32 heads x 8192 rows x 128 dims of FP32 accumulator is far above 32 MiB
    assert lib.attn_bwd_noalloc(*args, 2, 32, 8, 8192, 128, 0.1, 1, 0, None) == 7   # ATTN_ERR_WORKSPACE
    assert lib.attn_bwd_noalloc(None, *args[1:], 1, 2, 1, 8, 128, 0.1, 0, 0, None) == 1
    # the other argument errors, as attn_bwd reports them, before the array is looked up
    assert lib.attn_bwd_noalloc(*args, 1, 2, 1, 0, 128, 0.1, 0, 0, None) == 3         # N = 0
    assert lib.attn_bwd_noalloc(P(20), *args[1:], 1, 2, 1, 8, 128, 0.1, 0, 0, None) == 2
    assert lib.attn_bwd_noalloc(*args, 1, 2, 1, 8, 96, 0.1, 0, 0, None) == 4          # d = 64, 128 or 256
    assert lib.attn_bwd_noalloc(*args, 1, 3, 2, 8, 128, 0.1, 0, 0, None) == 5
    assert lib.attn_bwd_noalloc(*args, 1, 2, 1, 8, 128, 0.1, 0, 2, None) == 6         # E4M3 has no backward
    assert lib.attn_bwd_noalloc(*args, 1, 2, 1, 8, 128, 0.1, 0, 0, None) == 11        # valid: no device here
