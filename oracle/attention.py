"""Plain float64 attention: the definition written out (test infrastructure only).

Sources (FlashAttention-3, zenmind.me summary of the paper):
* §3.1 (paper §2.1): S = alpha * Q K^T, P = softmax(S) with the row maximum
  subtracted, O = P V; backward chain dV = P^T dO, dP = dO V^T,
  dS = dsoftmax(dP), dQ = alpha dS K, dK = alpha dS^T Q.
* §3.2 (Algorithm 1, epilogue): the log-sum-exp L_i = m_i + log(l_i).
* §4 step 5 (paper App. B.1): D = rowsum(dO o O), so dS = P o (dP - D).
* §3.2 / §4 step 1 (paper p.6): MQA/GQA re-indexes heads; K/V are not copied.
* Variable length (guijiagi.com "Flash Attention 3 explained", practical
  notes): sequences are concatenated along one token axis, with boundaries in
  cu_seqlens and no padding.
* Sliding-window (local) attention (same page, practical notes): each query
  sees only the keys within a fixed distance of its own position.

Readings where the pages are silent: dense tensors are [B, H, N, d]; packed
tensors are [T, H, d] with LSE [H, T]; causal means key j is visible to query
i iff j <= i (queries and keys have the same length); query head h reads
key/value head h // (Hq / Hkv); LSE is the natural log. A window
(left, right) makes key j visible to query i iff i - left <= j <= i + right,
a negative bound meaning no limit on that side; causal is the window (-1, 0)
and, given together with a window, caps its right bound at 0.
The softmax is the naive two-pass form: pass 1 takes the row max, pass 2 the
exponentials, their sum and the normalised product with V.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    """Any array-like (numpy or a CPU torch tensor) as a float64 numpy array."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.asarray(x, dtype=np.float64)


def window_bounds(causal, window=None):
    """(left, right) key-distance bounds; -1 means unbounded on that side."""
    left, right = (-1, -1) if window is None else (int(window[0]), int(window[1]))
    if left < -1 or right < -1:
        raise ValueError("window bounds must be -1 (unbounded) or >= 0")
    if causal:
        right = 0 if right < 0 else min(right, 0)
    return left, right


def visible(nq, nk, causal, window=None):
    """Boolean [nq, nk]: key j visible to query i (positions counted from 0)."""
    left, right = window_bounds(causal, window)
    i = np.arange(nq)[:, None]
    j = np.arange(nk)[None, :]
    vis = np.ones((nq, nk), dtype=bool)
    if right >= 0:
        vis &= j <= i + right
    if left >= 0:
        vis &= j >= i - left
    return vis


def head_forward(q, k, v, scale, causal, window=None):
    """One head: q [Nq, d], k/v [Nk, d] -> (O [Nq, d], LSE [Nq], P [Nq, Nk])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    s = scale * (q @ k.T)
    s = np.where(visible(*s.shape, causal, window), s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=1, keepdims=True)
    p = e / l
    return p @ v, (m + np.log(l))[:, 0], p


def head_backward(q, k, v, do, scale, causal, window=None):
    """One head: gradients (dQ, dK, dV) of sum(dO o O) through head_forward."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    o, _, p = head_forward(q, k, v, scale, causal, window)
    dv = p.T @ do
    dp = do @ v.T
    d_row = (do * o).sum(axis=1, keepdims=True)
    ds = p * (dp - d_row)
    dq = scale * (ds @ k)
    dk = scale * (ds.T @ q)
    return dq, dk, dv


def _group(hq, hkv):
    if hkv <= 0 or hq % hkv:
        raise ValueError("Hq must be a positive multiple of Hkv")
    return hq // hkv


def forward(q, k, v, scale, causal=False, window=None):
    """Dense [B, Hq, N, d] / [B, Hkv, N, d] -> (O [B, Hq, N, d], LSE [B, Hq, N])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    b_, hq, n, d = q.shape
    g = _group(hq, k.shape[1])
    o = np.empty((b_, hq, n, v.shape[-1]))
    lse = np.empty((b_, hq, n))
    for b in range(b_):
        for h in range(hq):
            o[b, h], lse[b, h], _ = head_forward(q[b, h], k[b, h // g], v[b, h // g], scale, causal, window)
    return o, lse


def backward(q, k, v, do, scale, causal=False, window=None):
    """Dense gradients; dK/dV of a KV head sum over the query heads that read it."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    b_, hq, n, d = q.shape
    g = _group(hq, k.shape[1])
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for b in range(b_):
        for h in range(hq):
            a, bb, c = head_backward(q[b, h], k[b, h // g], v[b, h // g], do[b, h], scale, causal, window)
            dq[b, h] = a
            dk[b, h // g] += bb
            dv[b, h // g] += c
    return dq, dk, dv


def forward_rows(q_head, k_head, v_head, rows, scale, causal=False, window=None):
    """O and LSE of selected query rows of one head, each row on its own.

    Used to check full-size outputs at sampled positions.
    """
    q_head, k_head, v_head = _f64(q_head), _f64(k_head), _f64(v_head)
    o = np.empty((len(rows), v_head.shape[-1]))
    lse = np.empty(len(rows))
    left, right = window_bounds(causal, window)
    for r, i in enumerate(rows):
        s = scale * (k_head @ q_head[i])
        if right >= 0:
            s[i + right + 1:] = -np.inf
        if left >= 0:
            s[:max(i - left, 0)] = -np.inf
        m = s.max()
        e = np.exp(s - m)
        l = e.sum()
        o[r] = (e / l) @ v_head
        lse[r] = m + np.log(l)
    return o, lse


def _check_cu(cu, total):
    cu = np.asarray(cu, dtype=np.int64)
    if cu[0] != 0 or cu[-1] != total or np.any(np.diff(cu) <= 0):
        raise ValueError("cu_seqlens must start at 0, rise strictly and end at T")
    return cu


def forward_varlen(q, k, v, cu, scale, causal=False):
    """Packed [T, Hq, d] -> (O [T, Hq, d], LSE [Hq, T]); attention stays inside each sequence."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    t, hq, d = q.shape
    g = _group(hq, k.shape[1])
    cu = _check_cu(cu, t)
    o = np.empty((t, hq, v.shape[-1]))
    lse = np.empty((hq, t))
    for s in range(len(cu) - 1):
        a, e = cu[s], cu[s + 1]
        for h in range(hq):
            o[a:e, h], lse[h, a:e], _ = head_forward(q[a:e, h], k[a:e, h // g], v[a:e, h // g], scale, causal)
    return o, lse


def backward_varlen(q, k, v, do, cu, scale, causal=False):
    """Packed-layout gradients, sequence by sequence."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    t, hq, d = q.shape
    g = _group(hq, k.shape[1])
    cu = _check_cu(cu, t)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for s in range(len(cu) - 1):
        a, e = cu[s], cu[s + 1]
        for h in range(hq):
            x, y, z = head_backward(q[a:e, h], k[a:e, h // g], v[a:e, h // g], do[a:e, h], scale, causal)
            dq[a:e, h] = x
            dk[a:e, h // g] += y
            dv[a:e, h // g] += z
    return dq, dk, dv
