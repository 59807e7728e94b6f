"""Pins for the float64 attention oracle (CPU only).

Each check fixes the oracle to something other than itself: closed forms,
invariants of softmax attention, a tiled re-derivation of Algorithm 1, a
library routine, finite differences and a hand-derived worked example.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def rnd(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_mean_of_visible_values(causal):
    n, d = 37, 8
    v = rnd(1, 1, 1, n, d)
    k = rnd(2, 1, 1, n, d)
    q = np.zeros((1, 1, n, d))
    o, lse = A.forward(q, k, v, 0.3, causal)
    for i in range(n):
        vis = i + 1 if causal else n
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :vis].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(lse[0, 0, i] - math.log(vis)) < 1e-13


def test_causal_first_row_is_first_value():
    q, k, v = rnd(3, 1, 2, 9, 4), rnd(4, 1, 2, 9, 4), rnd(5, 1, 2, 9, 4)
    o, lse = A.forward(q, k, v, 0.7, True)
    np.testing.assert_array_equal(o[0, :, 0], v[0, :, 0])
    np.testing.assert_allclose(lse[0, :, 0], 0.7 * (q[0, :, 0] * k[0, :, 0]).sum(-1), rtol=1e-15)


def test_one_hot_query_selects_one_value_row():
    n, d, c, delta = 16, 8, 10.0, 6.0
    k = rnd(6, n, d) * 0.1
    jstar, axis = 11, 3
    k[jstar, axis] += delta
    q = np.zeros((n, d))
    q[:, axis] = c
    v = rnd(7, n, d)
    o, _, p = A.head_forward(q, k, v, 1.0, False)   # c * delta = 60 >= 50
    # every other key trails by c * delta - noise > 50, so its weight is < e^-50
    np.testing.assert_allclose(o, np.broadcast_to(v[jstar], o.shape), rtol=0, atol=n * np.exp(-50.0) * np.abs(v).max())


def test_probability_rows_sum_to_one():
    _, _, p = A.head_forward(rnd(8, 20, 6), rnd(9, 20, 6), rnd(10, 20, 6), 0.5, True)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    assert np.all(np.triu(p, 1) == 0.0)


def test_key_shift_changes_only_lse():
    q, k, v = rnd(11, 12, 5), rnd(12, 12, 5), rnd(13, 12, 5)
    u = rnd(14, 5)
    o1, l1, _ = A.head_forward(q, k, v, 0.4, False)
    o2, l2, _ = A.head_forward(q, k + u, v, 0.4, False)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(l2 - l1, 0.4 * q @ u, atol=1e-13)


def test_joint_key_value_permutation_noncausal():
    q, k, v = rnd(15, 10, 4), rnd(16, 10, 4), rnd(17, 10, 4)
    perm = np.random.default_rng(0).permutation(10)
    o1, l1, _ = A.head_forward(q, k, v, 0.9, False)
    o2, l2, _ = A.head_forward(q, k[perm], v[perm], 0.9, False)
    np.testing.assert_allclose(o2, o1, atol=1e-14)
    np.testing.assert_allclose(l2, l1, atol=1e-14)


def test_worked_example_two_tokens():
    g = json.load(open(os.path.join(GOLD, "two_token_closed_form.json")))
    q, k, v, do = (np.array(g[x])[None, None] for x in ("q", "k", "v", "dO"))
    ln = {"ln 4": math.log(4), "ln 2": math.log(2), "0": 0.0}
    for causal, key in ((False, "noncausal"), (True, "causal")):
        o, lse = A.forward(q, k, v, 1.0, causal)
        np.testing.assert_allclose(o[0, 0], g[key]["O"], atol=1e-15)
        np.testing.assert_allclose(lse[0, 0], [ln[s] for s in g[key]["LSE_exact"]], atol=1e-15)
        dq, dk, dv = A.backward(q, k, v, do, 1.0, causal)
        np.testing.assert_allclose(dq[0, 0], g[key]["dQ"], atol=1e-15)
        np.testing.assert_allclose(dk[0, 0] / math.log(3), g[key]["dK_over_ln3"], atol=1e-15)
        np.testing.assert_allclose(dv[0, 0], g[key]["dV"], atol=1e-15)


# ------------------------------------------------ independent re-derivations

def _tiled_online(q, k, v, scale, causal, bc):
    """Algorithm 1 of the pages (running max m, running sum l, rescaled O),
    written independently of the oracle, one KV block of bc keys at a time."""
    nq, d = q.shape
    m = np.full(nq, -np.inf)
    l = np.zeros(nq)
    o = np.zeros((nq, v.shape[1]))
    for j0 in range(0, k.shape[0], bc):
        kb, vb = k[j0:j0 + bc], v[j0:j0 + bc]
        s = scale * q @ kb.T
        if causal:
            s[np.arange(j0, j0 + len(kb))[None, :] > np.arange(nq)[:, None]] = -np.inf
        m_new = np.maximum(m, s.max(axis=1))
        safe = np.where(np.isinf(m_new), 0.0, m_new)
        pt = np.exp(s - safe[:, None])
        a = np.exp(m - safe)
        l = a * l + pt.sum(axis=1)
        o = a[:, None] * o + pt @ vb
        m = m_new
    return o / l[:, None], m + np.log(l)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("bc", [1, 7, 64])
def test_matches_online_softmax_rederivation(causal, bc):
    q, k, v = rnd(20, 70, 16), rnd(21, 70, 16), rnd(22, 70, 16)
    o, lse, _ = A.head_forward(q, k, v, 0.25, causal)
    o2, lse2 = _tiled_online(q, k, v, 0.25, causal, bc)
    np.testing.assert_allclose(o, o2, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, lse2, atol=1e-12, rtol=0)


@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa_float64(causal):
    q, k, v = (torch.from_numpy(rnd(s, 2, 4, 33, 8)) for s in (30, 31, 32))
    k2, v2 = k[:, :2], v[:, :2]
    o, _ = A.forward(q, k2, v2, 0.35, causal)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k2.repeat_interleave(2, 1), v2.repeat_interleave(2, 1), is_causal=causal, scale=0.35)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12, rtol=0)


def test_gqa_equals_mha_with_replicated_kv():
    q, k, v = rnd(40, 1, 6, 12, 4), rnd(41, 1, 2, 12, 4), rnd(42, 1, 2, 12, 4)
    o1, l1 = A.forward(q, k, v, 0.5, True)
    o2, l2 = A.forward(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), 0.5, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    do = rnd(43, 1, 6, 12, 4)
    dq1, dk1, dv1 = A.backward(q, k, v, do, 0.5, True)
    dq2, dk2, dv2 = A.backward(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), do, 0.5, True)
    np.testing.assert_allclose(dq1, dq2, atol=1e-14)
    np.testing.assert_allclose(dk1, dk2.reshape(1, 2, 3, 12, 4).sum(2), atol=1e-14)
    np.testing.assert_allclose(dv1, dv2.reshape(1, 2, 3, 12, 4).sum(2), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_equals_dense_per_sequence(causal):
    lens = [5, 17, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    t = cu[-1]
    q, k, v, do = rnd(50, t, 4, 8), rnd(51, t, 2, 8), rnd(52, t, 2, 8), rnd(53, t, 4, 8)
    o, lse = A.forward_varlen(q, k, v, cu, 0.3, causal)
    dq, dk, dv = A.backward_varlen(q, k, v, do, cu, 0.3, causal)
    for s in range(len(lens)):
        a, e = cu[s], cu[s + 1]
        tr = lambda x: x[a:e].transpose(1, 0, 2)[None]
        o2, l2 = A.forward(tr(q), tr(k), tr(v), 0.3, causal)
        np.testing.assert_allclose(o[a:e], o2[0].transpose(1, 0, 2), atol=1e-14)
        np.testing.assert_allclose(lse[:, a:e], l2[0], atol=1e-14)
        g = A.backward(tr(q), tr(k), tr(v), tr(do), 0.3, causal)
        for got, ref in zip((dq, dk, dv), g):
            np.testing.assert_allclose(got[a:e], ref[0].transpose(1, 0, 2), atol=1e-13)


def test_forward_rows_matches_full():
    q, k, v = rnd(60, 50, 8), rnd(61, 50, 8), rnd(62, 50, 8)
    for causal in (False, True):
        o, lse, _ = A.head_forward(q, k, v, 0.2, causal)
        rows = [0, 7, 31, 49]
        o2, l2 = A.forward_rows(q, k, v, rows, 0.2, causal)
        np.testing.assert_allclose(o2, o[rows], atol=1e-14)
        np.testing.assert_allclose(l2, lse[rows], atol=1e-14)


# ------------------------------------------------------------------ backward

@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_central_differences(causal):
    n, d, scale, h = 9, 5, 0.6, 1e-6
    q, k, v, do = rnd(70, n, d), rnd(71, n, d), rnd(72, n, d), rnd(73, n, d)
    dq, dk, dv = A.head_backward(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        return (A.head_forward(qq, kk, vv, scale, causal)[0] * do).sum()

    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(grad.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            num[idx] = (up - loss(*args)) / (2 * h)
        rel = np.linalg.norm(num - grad) / np.linalg.norm(grad)
        assert rel < 1e-6, (which, rel)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd_float64(causal):
    q, k, v, do = (torch.from_numpy(rnd(s, 1, 4, 21, 6)) for s in (80, 81, 82, 83))
    k, v = k[:, :2].clone(), v[:, :2].clone()
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(2, 1), vt.repeat_interleave(2, 1), is_causal=causal, scale=0.45)
    o.backward(do)
    dq, dk, dv = A.backward(q, k, v, do, 0.45, causal)
    for got, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        np.testing.assert_allclose(got, ref.numpy(), atol=1e-12, rtol=0)


def test_backward_invariants():
    q, k, v, do = rnd(90, 30, 8), rnd(91, 30, 8), rnd(92, 30, 8), rnd(93, 30, 8)
    for causal in (False, True):
        dq, dk, dv = A.head_backward(q, k, v, do, 0.3, causal)
        # every row of dS sums to zero, so the key gradients sum to zero
        np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
        # every row of P sums to one, so the value gradients sum to sum(dO)
        np.testing.assert_allclose(dv.sum(axis=0), do.sum(axis=0), atol=1e-12)


# --------------------------------------------------------- planted mistakes

def test_pins_catch_planted_mistakes():
    """Plant plausible bugs in the oracle (on the CPU) and check a pin fails."""
    good = A.head_forward
    q, k, v = rnd(100, 24, 8), rnd(101, 24, 8), rnd(102, 24, 8)
    ref = _tiled_online(q, k, v, 0.3, True, 5)

    def no_max(q, k, v, scale, causal):          # LSE off by a constant
        o, lse, p = good(q, k, v, scale, causal)
        return o, lse - 1e-3, p

    def transposed(q, k, v, scale, causal):      # causal mask on the wrong side
        o, lse, p = good(q[::-1], k[::-1], v[::-1], scale, causal)
        return o[::-1], lse[::-1], p

    def no_scale(q, k, v, scale, causal):
        return good(q, k, v, 1.0, causal)

    for bad in (no_max, transposed, no_scale):
        o, lse, _ = bad(q, k, v, 0.3, True)
        assert not (np.allclose(o, ref[0], atol=1e-12) and np.allclose(lse, ref[1], atol=1e-12)), bad.__name__

    def dropped_d(q, k, v, do, scale, causal):   # dS = P o dP without the rowsum term
        o, _, p = good(q, k, v, scale, causal)
        ds = p * (do @ v.T)
        return scale * ds @ k, scale * ds.T @ q, p.T @ do
    dq, dk, dv = dropped_d(q, k, v, rnd(103, 24, 8), 0.3, False)
    assert abs(dk.sum(axis=0)).max() > 1e-6


# ------------------------------------------------------------ sliding window

WINDOWS = [(3, 0), (2, 5), (0, 4), (7, -1), (-1, 2), (0, 0), (1, 1)]


def _mask_loops(n, left, right):
    """Visibility written as explicit loops (independent of the oracle's)."""
    m = np.zeros((n, n), dtype=bool)
    for i in range(n):
        for j in range(n):
            ok = True
            if right >= 0 and j > i + right:
                ok = False
            if left >= 0 and j < i - left:
                ok = False
            m[i, j] = ok
    return m


def test_window_zero_selects_own_value():
    """Window (0, 0): every query sees only its own key, so O = V, LSE = s_ii."""
    q, k, v = rnd(110, 1, 2, 19, 6), rnd(111, 1, 2, 19, 6), rnd(112, 1, 2, 19, 6)
    o, lse = A.forward(q, k, v, 0.4, False, (0, 0))
    np.testing.assert_allclose(o, v, atol=1e-14, rtol=0)
    np.testing.assert_allclose(lse, 0.4 * (q * k).sum(-1), atol=1e-14, rtol=0)


def test_window_brute_force_rows():
    n, d, scale = 11, 3, 0.7
    q, k, v = rnd(113, n, d), rnd(114, n, d), rnd(115, n, d)
    for left, right in WINDOWS:
        o, lse, _ = A.head_forward(q, k, v, scale, False, (left, right))
        for i in range(n):
            keys = [j for j in range(n) if (right < 0 or j <= i + right) and (left < 0 or j >= i - left)]
            s = [scale * sum(q[i, t] * k[j, t] for t in range(d)) for j in keys]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            tot = sum(e)
            ref = [sum(e[a] * v[j, t] for a, j in enumerate(keys)) / tot for t in range(d)]
            np.testing.assert_allclose(o[i], ref, atol=1e-13, rtol=0)
            assert abs(lse[i] - (mx + math.log(tot))) < 1e-13


@pytest.mark.parametrize("window", WINDOWS)
def test_window_matches_torch_sdpa_masked(window):
    n = 23
    q, k, v, do = (torch.from_numpy(rnd(s, 1, 4, n, 5)) for s in (116, 117, 118, 119))
    k, v = k[:, :2].clone(), v[:, :2].clone()
    mask = torch.from_numpy(_mask_loops(n, *window))
    qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, kt.repeat_interleave(2, 1), vt.repeat_interleave(2, 1), attn_mask=mask, scale=0.55)
    ref.backward(do)
    o, _ = A.forward(q, k, v, 0.55, False, window)
    np.testing.assert_allclose(o, ref.detach().numpy(), atol=1e-12, rtol=0)
    dq, dk, dv = A.backward(q, k, v, do, 0.55, False, window)
    for got, g in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
        np.testing.assert_allclose(got, g.numpy(), atol=1e-12, rtol=0)


def test_window_limits():
    """A window wider than the sequence is full attention; (n, 0) is causal;
    causal given with a window caps the window's right bound at 0."""
    q, k, v = rnd(120, 1, 1, 17, 4), rnd(121, 1, 1, 17, 4), rnd(122, 1, 1, 17, 4)
    full = A.forward(q, k, v, 0.3, False)
    causal = A.forward(q, k, v, 0.3, True)
    for got, ref in ((A.forward(q, k, v, 0.3, False, (17, 17)), full),
                     (A.forward(q, k, v, 0.3, False, (40, 0)), causal),
                     (A.forward(q, k, v, 0.3, True, (-1, 5)), causal)):
        np.testing.assert_array_equal(got[0], ref[0])
        np.testing.assert_array_equal(got[1], ref[1])
    with pytest.raises(ValueError):
        A.forward(q, k, v, 0.3, False, (-2, 0))


def test_window_backward_central_differences():
    n, d, scale, h = 9, 4, 0.6, 1e-6
    q, k, v, do = rnd(123, n, d), rnd(124, n, d), rnd(125, n, d), rnd(126, n, d)
    window = (2, 1)
    dq, dk, dv = A.head_backward(q, k, v, do, scale, False, window)

    def loss(qq, kk, vv):
        return (A.head_forward(qq, kk, vv, scale, False, window)[0] * do).sum()

    for which, grad in ((0, dq), (1, dk), (2, dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(grad.shape):
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            up = loss(*args)
            args[which][idx] -= 2 * h
            num[idx] = (up - loss(*args)) / (2 * h)
        assert np.linalg.norm(num - grad) / np.linalg.norm(grad) < 1e-6, which


def test_window_forward_rows_matches_full():
    q, k, v = rnd(127, 40, 6), rnd(128, 40, 6), rnd(129, 40, 6)
    for window in WINDOWS:
        o, lse, _ = A.head_forward(q, k, v, 0.25, False, window)
        rows = [0, 1, 13, 38, 39]
        o2, l2 = A.forward_rows(q, k, v, rows, 0.25, False, window)
        np.testing.assert_allclose(o2, o[rows], atol=1e-14)
        np.testing.assert_allclose(l2, lse[rows], atol=1e-14)


def test_window_pins_catch_off_by_one():
    """Plant an off-by-one in the window's left bound (on the CPU): the
    brute-force rows must disagree."""
    good = A.visible

    def shifted(nq, nk, causal, window=None):
        left, right = A.window_bounds(causal, window)
        return good(nq, nk, causal, (left + 1 if left >= 0 else left, right))

    q, k, v = rnd(130, 10, 3), rnd(131, 10, 3), rnd(132, 10, 3)
    ref, _, _ = A.head_forward(q, k, v, 0.5, False, (2, 0))
    A.visible = shifted
    try:
        bad, _, _ = A.head_forward(q, k, v, 0.5, False, (2, 0))
    finally:
        A.visible = good
    assert not np.allclose(bad, ref, atol=1e-12)


# ------------------------------------------------------- property-based check

def test_random_problems_match_torch_float64():
    """Random small problems (batch, KV heads, GQA group, length, head dim,
    scale, causal flag and window): the oracle's O, LSE and gradients equal
    torch's float64 SDPA with an explicit mask built by loops, its autograd,
    and torch.logsumexp of the masked scores, to 1e-12."""
    hyp = pytest.importorskip("hypothesis")
    st = hyp.strategies

    @hyp.settings(max_examples=40, deadline=None, derandomize=True)
    @hyp.given(b=st.integers(1, 2), hkv=st.integers(1, 2), g=st.integers(1, 3), n=st.integers(1, 40),
               d=st.integers(1, 9), scale=st.floats(0.05, 2.0), causal=st.booleans(),
               left=st.integers(-1, 12), right=st.integers(-1, 12), seed=st.integers(0, 10 ** 6))
    def check(b, hkv, g, n, d, scale, causal, left, right, seed):
        rng = np.random.default_rng(seed)
        q = torch.from_numpy(rng.standard_normal((b, hkv * g, n, d)))
        k, v = (torch.from_numpy(rng.standard_normal((b, hkv, n, d))) for _ in range(2))
        do = torch.from_numpy(rng.standard_normal((b, hkv * g, n, d)))
        r = right if not causal else (0 if right < 0 else min(right, 0))
        mask = torch.from_numpy(_mask_loops(n, left, r))
        qt, kt, vt = (x.clone().requires_grad_(True) for x in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt, kt.repeat_interleave(g, 1), vt.repeat_interleave(g, 1), attn_mask=mask, scale=scale)
        ref.backward(do)
        s = scale * q @ k.repeat_interleave(g, 1).transpose(-1, -2)
        lse_ref = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
        o, lse = A.forward(q, k, v, scale, causal, (left, right))
        np.testing.assert_allclose(o, ref.detach().numpy(), atol=1e-12, rtol=0)
        np.testing.assert_allclose(lse, lse_ref.numpy(), atol=1e-12, rtol=0)
        for got, want in zip(A.backward(q, k, v, do, scale, causal, (left, right)), (qt.grad, kt.grad, vt.grad)):
            np.testing.assert_allclose(got, want.numpy(), atol=1e-11, rtol=0)

    check()
