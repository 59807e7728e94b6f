"""FP8 (E4M3) block quantisation and FP8 attention, written out plainly.

Test infrastructure only. Sources (FlashAttention-3, zenmind.me summary):
* §3.5 "block quantisation" (paper §3.3): one scale per Br x d block of Q and
  per Bc x d block of K and V instead of one per tensor; the S block is
  rescaled by the product of its Q and K scales.
* §3.5 "incoherent processing" (paper §3.3): Q and K are multiplied by
  M = diag(random signs) * Hadamard before quantisation, so (QM)(KM)^T = QK^T.
* §3.2 Algorithm 1: the tiled online softmax that the FP8 forward follows.
* m.xxqk.cn FA3 walkthrough §4.1-4.2: E4M3 operands, FP32 accumulation,
  power-of-two scale factors.
* §3.5 / guijiagi.com practical notes: quantisation is fused into the rotary
  position embedding (RoPE) step that produces Q and K.

Readings (the pages leave these open):
* E4M3 is the OCP "e4m3fn" format: bias 7, largest finite 448, no infinity,
  NaN = S.1111.111. Encoding rounds to nearest even and saturates to +-448.
* Block = 128 rows of one (batch, head); scale e = the largest integer with
  amax * 2^e <= 448; the stored dequantisation factor is 2^-e (1 if amax = 0).
* The rotation is y = fp32(FWHT_fp32(sigma o x) * fp32(1/sqrt(d))), with the
  fast Walsh-Hadamard transform taken in the textbook radix-2 order (stride
  1, 2, 4, ...), every add and subtract rounded to float32. Sylvester order.
* The running max m is the one of Algorithm 1: m_new = max(m_old, rowmax S_j)
  at every KV tile (``tau = 0``, the default). ``tau > 0`` selects the
  stale-max variant (STALE_MAX_TAU): m is raised only when a tile's row max
  exceeds it by more than tau log2 units, so P~ = exp(S - m) <= 2^tau and O
  is rescaled less often. Both give the same result in exact arithmetic; they
  differ only in which values are rounded to E4M3, by at most one E4M3 step
  per entry of P~ (half a step on each side, see ``half_step``).
* The V factor of KV tile j, sv_j = 2^f_j, is folded into P~ before its
  E4M3 rounding, relative to F, the running maximum of f over the tiles seen
  so far: P~ enters the second product as e4m3(P~ * 2^(4 + f_j - F)), and
  the accumulated O is multiplied by 2^(F_old - F_new) whenever F grows (the
  same correction as for the running row max m). The rounded value lies in
  (0, 2^(4 + tau)]. At the end O = O_acc * 2^(F - 4) / l; l sums the
  unrounded P~.
  The KV tile (Bc keys) need not equal the quantisation block: a tile that
  spans two blocks gives each key its own block's K and V factors, and F is
  raised once per tile, to the largest f among the tile's keys.
* Decode over a KV cache: the g query heads of one KV group at the decoded
  position are one block of g query rows with one factor; the cache keys are
  split into runs of whole 128-key tiles, each run is processed as Algorithm 1
  from a fresh state (m = -inf, l = 0, F = -inf), and the runs are combined
  exactly by their log-sum-exp weights (the split-KV form of the forward).
* RoPE uses the rotate-half pairing (i, i + d/2), i < d/2: for the row at
  position n, with c = cos[n, i] and s = sin[n, i] from caller-supplied float32
  tables [N, d/2], y_i = x_i c - x_{i+d/2} s and y_{i+d/2} = x_{i+d/2} c + x_i s,
  each product and the sum rounded to float32 separately (no fused multiply-
  add). The producer order is RoPE, then the optional rotation, then the block
  quantisation; V is not rotated.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
BLOCK = 128
# Stale-max variant of the running max (log2 units): m moves only when a
# tile's row max exceeds it by more than this. Not the pages' rule (tau = 0);
# it changes which values are rounded to E4M3, not the exact result.
STALE_MAX_TAU = 4.0


def e4m3_decode(codes):
    """uint8 codes -> float64 values."""
    c = np.asarray(codes).astype(np.int64)
    sign = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(sign == 1, -mag, mag)


def e4m3_encode(x):
    """float values -> uint8 codes, round to nearest even, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    nan = np.isnan(x)
    neg = np.signbit(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), E4M3_MAX)
    mant, ex = np.frexp(a)                     # a = mant * 2^ex, mant in [0.5, 1)
    e = ex - 1                                  # a = (2 mant) * 2^e
    q_norm = np.rint((2.0 * mant - 1.0) * 8.0)  # exact products, ties to even
    carry = q_norm == 8
    e = np.where(carry, e + 1, e)
    q_norm = np.where(carry, 0, q_norm)
    code_norm = ((e + 7) << 3) + q_norm.astype(np.int64)
    q_sub = np.rint(a / 2.0 ** -9).astype(np.int64)   # subnormal step 2^-9
    code = np.where(a < 2.0 ** -6, q_sub, code_norm)
    code = code + np.where(neg, 128, 0)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


def half_step(x):
    """Largest rounding error of e4m3_encode at x >= 0 (below saturation):
    half the spacing of the E4M3 grid in the binade of x, 2^(e - 4) for
    x in [2^e, 2^(e+1)) with e >= -6, and 2^-10 in the subnormal range."""
    x = np.asarray(x, dtype=np.float64)
    _, ex = np.frexp(np.where(x > 0, x, 1.0))     # x = mant * 2^ex, mant in [0.5, 1)
    return np.where(x >= 2.0 ** -6, np.exp2(ex - 5.0), 2.0 ** -10)


def pow2_exponent(amax):
    """Largest integer e with amax * 2^e <= 448 (0 where amax == 0)."""
    amax = np.asarray(amax, dtype=np.float64)
    safe = np.where(amax > 0, amax, 1.0)
    e = np.floor(np.log2(E4M3_MAX / safe)).astype(np.int64)
    # settle the floor exactly: scaling by a power of two is exact
    e = np.where(safe * np.exp2(e + 1.0) <= E4M3_MAX, e + 1, e)
    e = np.where(safe * np.exp2(e * 1.0) > E4M3_MAX, e - 1, e)
    return np.where(amax > 0, e, 0)


def hadamard(d):
    """Sylvester Hadamard matrix of order d (a power of two), entries +-1."""
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    if h.shape[0] != d:
        raise ValueError("d must be a power of two")
    return h


def fwht_fp32(x):
    """x @ H along the last axis, radix-2 stages h = 1, 2, 4, ..., all in float32."""
    y = np.array(x, dtype=np.float32, copy=True)
    d = y.shape[-1]
    h = 1
    while h < d:
        z = y.reshape(y.shape[:-1] + (d // (2 * h), 2, h))
        a = z[..., 0, :].copy()
        b = z[..., 1, :].copy()
        z[..., 0, :] = a + b
        z[..., 1, :] = a - b
        y = z.reshape(y.shape)
        h *= 2
    return y


def rotate_fp32(x, signs):
    """Incoherent processing in float32: fp32(FWHT(sigma o x) * fp32(1/sqrt(d)))."""
    x = np.asarray(x, dtype=np.float32)
    d = x.shape[-1]
    s = np.asarray(signs, dtype=np.float32)
    c = np.float32(1.0 / np.sqrt(d))
    return (fwht_fp32(x * s) * c).astype(np.float32)


def rotate_f64(x, signs):
    """The same rotation as a dense float64 product x diag(sigma) H / sqrt(d)."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    return (x * np.asarray(signs, dtype=np.float64)) @ hadamard(d) / np.sqrt(d)


def rope_tables(n, d, base=10000.0):
    """cos/sin tables [n, d/2] float32 of n * base^(-2i/d), computed in float64."""
    i = np.arange(d // 2, dtype=np.float64)
    ang = np.arange(n, dtype=np.float64)[:, None] * base ** (-2.0 * i / d)[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def rope_fp32(x, cos, sin):
    """Rotate-half RoPE along the last axis of x [..., N, d] in float32, every
    product and sum rounded separately; cos/sin [N, d/2] float32."""
    x = np.asarray(x, dtype=np.float32)
    c = np.asarray(cos, dtype=np.float32)
    s = np.asarray(sin, dtype=np.float32)
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    y = np.empty_like(x)
    y[..., :h] = (a * c).astype(np.float32) - (b * s).astype(np.float32)
    y[..., h:] = (b * c).astype(np.float32) + (a * s).astype(np.float32)
    return y.astype(np.float32)


def rope_f64(x, cos, sin):
    """The same rotation in float64 (the definition, for pins)."""
    x = np.asarray(x, dtype=np.float64)
    c = np.asarray(cos, dtype=np.float64)
    s = np.asarray(sin, dtype=np.float64)
    h = x.shape[-1] // 2
    a, b = x[..., :h], x[..., h:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def quantize_blocks(x, signs=None, block=BLOCK, rope=None):
    """[B, H, N, d] -> (codes uint8 [B, H, N, d], factors float32 [B, H, ceil(N/block)]).

    x is taken in float32 (as the GPU sees bf16/fp16 inputs); with ``rope``
    = (cos, sin) RoPE is applied first, then with ``signs`` the rotation. Each
    block of ``block`` rows of one (batch, head) gets its own power-of-two
    factor.
    """
    if hasattr(x, "detach"):
        x = x.detach().float().numpy()
    x = np.asarray(x, dtype=np.float32)
    if rope is not None:
        x = rope_fp32(x, *rope)
    if signs is not None:
        x = rotate_fp32(x, signs)
    b_, h_, n, d = x.shape
    nb = (n + block - 1) // block
    codes = np.empty(x.shape, dtype=np.uint8)
    fac = np.empty((b_, h_, nb), dtype=np.float32)
    for i in range(nb):
        blk = x[:, :, i * block:(i + 1) * block, :].astype(np.float64)
        e = pow2_exponent(np.abs(blk).max(axis=(2, 3)))
        codes[:, :, i * block:(i + 1) * block, :] = e4m3_encode(blk * np.exp2(e * 1.0)[:, :, None, None])
        fac[:, :, i] = np.exp2(-e * 1.0)
    return codes, fac


def quantize_tensor(x, signs=None, block=BLOCK):
    """Per-tensor power-of-two scaling (the baseline): one factor for all of x.

    Returns the factor broadcast to the block-scale shape so that the same
    attention routine consumes either form.
    """
    if hasattr(x, "detach"):
        x = x.detach().float().numpy()
    x = np.asarray(x, dtype=np.float32)
    if signs is not None:
        x = rotate_fp32(x, signs)
    b_, h_, n, d = x.shape
    xd = x.astype(np.float64)
    e = int(pow2_exponent(np.abs(xd).max()))
    codes = e4m3_encode(xd * 2.0 ** e)
    nb = (n + block - 1) // block
    fac = np.full((b_, h_, nb), 2.0 ** -e, dtype=np.float32)
    return codes, fac


def _fp8_rows(qrows, q_fac, kf, vf, sk, sv, tiles, n, scale, causal=False, rows=None, block=BLOCK, p_shift=4,
              tau=0.0, kv_tile=None, round_p=True, bound=False, window=None):
    """Algorithm 1 in its FP8 form for query rows ``qrows`` [R, d] (decoded,
    with per-row factors q_fac) over the key tiles ``tiles`` (indices of tiles
    of kv_tile keys, in order) of one KV head: kf/vf [N, d] decoded, sk/sv the
    factors of the ``block``-key quantisation blocks. A tile may span blocks:
    each key takes its own block's factors, and F is raised to the largest V
    exponent among the tile's keys. Starts from m = -inf, l = 0, O = 0.
    ``round_p=False`` leaves out the E4M3 rounding of P~ (for pins: the rest
    is then exact). Returns (O [R, d], LSE [R]); with ``bound`` also E [R, d],
    the sum over keys of each rounded entry's half_step times |V|, carried
    through the same corrections as O: |O - O_unrounded| <= E elementwise.
    ``window`` (left, right): key j is visible to row i iff i - left <= j <=
    i + right, -1 leaving that side open; causal is (-1, 0). Keys outside it
    get the score -inf, as causal masking does."""
    kv_tile = block if kv_tile is None else kv_tile
    left, right = window if window is not None else ((-1, 0) if causal else (-1, -1))
    d = qrows.shape[1]
    m = np.full(len(qrows), -np.inf)
    l = np.zeros(len(qrows))
    acc = np.zeros((len(qrows), d))
    err = np.zeros((len(qrows), d))
    f_run = -np.inf
    for j in tiles:
        cols = np.arange(j * kv_tile, min(n, (j + 1) * kv_tile))
        blk = cols // block
        s = scale * q_fac[:, None] * sk[blk][None, :] * (qrows @ kf[cols].T)
        if right >= 0:
            s = np.where(cols[None, :] > rows[:, None] + right, -np.inf, s)
        if left >= 0:
            s = np.where(cols[None, :] < rows[:, None] - left, -np.inf, s)
        mx = s.max(axis=1)
        m_new = np.where(mx > m + tau * np.log(2.0), mx, m)   # tau = 0: the running max itself
        m_use = np.where(np.isfinite(m_new), m_new, 0.0)
        corr = np.exp(m - m_use)
        f_c = np.log2(sv[blk])                                # V exponent of each key
        f_new = max(f_run, f_c.max())
        v_corr = np.exp2(f_run - f_new)
        pt = np.exp(s - m_use[:, None])
        l = corr * l + pt.sum(axis=1)
        p8 = pt * np.exp2(p_shift + f_c - f_new)[None, :]
        hs = half_step(p8)
        if round_p:
            p8 = e4m3_decode(e4m3_encode(p8))
        acc = (corr * v_corr)[:, None] * acc + p8 @ vf[cols]
        err = (corr * v_corr)[:, None] * err + hs @ np.abs(vf[cols])
        m, f_run = m_new, f_new
    out = acc * np.exp2(f_run - p_shift) / l[:, None], m + np.log(l)
    if bound:
        return out + (err * np.exp2(f_run - p_shift) / l[:, None],)
    return out


def attention_fp8(q8, k8, v8, sq, sk, sv, scale, causal=False, block=BLOCK, p_shift=4, tau=0.0, heads=None,
                  rows=None, kv_tile=None, round_p=True, bound=False, window=None):
    """FP8 forward following Algorithm 1 tile by tile (Bc = kv_tile keys per
    tile, by default the quantisation block; the stale max and the V exponent
    F move at tile granularity, so the E4M3 rounding of P~ depends on it).

    q8 [B, Hq, N, d], k8/v8 [B, Hkv, N, d] are E4M3 codes; sq/sk/sv are the
    dequantisation factors per 128-row block. Arithmetic is float64 except the
    E4M3 rounding of P~ before the second product. Returns (O, LSE).
    ``heads`` (list of (b, h)) and ``rows`` restrict the work to those query
    heads and rows (rows are independent); other entries are left as NaN.
    ``round_p=False`` leaves out the E4M3 rounding of P~ (for pins).
    ``tau`` = 0 is the running max of Algorithm 1; STALE_MAX_TAU the stale-max
    variant. With ``bound`` a third array E (like O) bounds the effect of the
    E4M3 rounding of P~: |O - O(round_p=False)| <= E elementwise.
    ``window`` (left, right) as in ``_fp8_rows`` (it replaces ``causal``).
    """
    qf, kf, vf = e4m3_decode(q8), e4m3_decode(k8), e4m3_decode(v8)
    sq, sk, sv = (np.asarray(a, dtype=np.float64) for a in (sq, sk, sv))
    b_, hq, n, d = qf.shape
    g = hq // kf.shape[1]
    o = np.full(qf.shape, np.nan)
    e = np.full(qf.shape, np.nan)
    lse = np.full((b_, hq, n), np.nan)
    rows = np.arange(n) if rows is None else np.asarray(rows)
    heads = [(b, h) for b in range(b_) for h in range(hq)] if heads is None else heads
    kvt = block if kv_tile is None else kv_tile
    for b, h in heads:
        kv = h // g
        o[b, h, rows], lse[b, h, rows], e[b, h, rows] = _fp8_rows(
            qf[b, h, rows], sq[b, h, rows // block], kf[b, kv], vf[b, kv], sk[b, kv], sv[b, kv],
            range((n + kvt - 1) // kvt), n, scale, causal, rows, block, p_shift, tau, kvt, round_p, bound=True,
            window=window)
    return (o, lse, e) if bound else (o, lse)


def combine_splits(o_parts, lse_parts):
    """Partial results of disjoint key ranges -> the result over their union:
    LSE = log sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s (float64).
    o_parts [S, ..., d], lse_parts [S, ...]; a part with LSE = -inf adds nothing."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    mx = lse_parts.max(axis=0)
    w = np.exp(lse_parts - mx[None])
    tot = w.sum(axis=0)
    o = (w[..., None] * np.nan_to_num(o_parts)).sum(axis=0) / tot[..., None]
    return o, mx + np.log(tot)


def decode_fp8(q8, sq, k8, v8, sk, sv, lens, scale, tiles_per_split, block=BLOCK, p_shift=4, tau=0.0,
               round_p=True):
    """FP8 decode over a block-quantised KV cache, split by key tiles.

    q8 [B, Hkv, g, d]: E4M3 codes of the g query heads of each KV group at the
    decoded position (query head h = kv * g + i), sq [B, Hkv] their factors;
    k8/v8 [B, Hkv, Nmax, d] and sk/sv [B, Hkv, ceil(Nmax/block)] the cache;
    lens[b] the valid cache length of sequence b. Split s holds key tiles
    [s * tiles_per_split, (s + 1) * tiles_per_split) below ceil(lens[b]/block);
    each split runs the FP8 form of Algorithm 1 on its own and the splits are
    combined with combine_splits. ``round_p=False`` leaves out the E4M3
    rounding of P~ (for pins). Returns (O [B, Hkv, g, d], LSE [B, Hkv, g]).
    """
    qf, kf, vf = e4m3_decode(q8), e4m3_decode(k8), e4m3_decode(v8)
    sq, sk, sv = (np.asarray(a, dtype=np.float64) for a in (sq, sk, sv))
    b_, hkv, g, d = qf.shape
    o = np.empty((b_, hkv, g, d))
    lse = np.empty((b_, hkv, g))
    for b in range(b_):
        n = int(lens[b])
        nt = (n + block - 1) // block
        splits = [range(t, min(t + tiles_per_split, nt)) for t in range(0, nt, tiles_per_split)]
        for kv in range(hkv):
            parts = [_fp8_rows(qf[b, kv], np.full(g, sq[b, kv]), kf[b, kv], vf[b, kv], sk[b, kv], sv[b, kv],
                               tiles, n, scale, block=block, p_shift=p_shift, tau=tau, round_p=round_p)
                     for tiles in splits]
            o[b, kv], lse[b, kv] = combine_splits([p[0] for p in parts], [p[1] for p in parts])
    return o, lse
