"""Mutation check of the oracle's pins (CPU only).

Each case plants one plausible mistake in a copy of an oracle module (a
dropped term, a wrong sign, axis or index, an off-by-one bound, a wrong
logarithm base), reruns every pin test of that module against the copy and
requires that at least one pin fails with an assertion. The copies live only
in this test; the real modules are never modified.
"""
import importlib.util
import inspect
import itertools
import os
import types
import warnings

import pytest

from oracle import attention as A
from oracle import fp8 as F

HERE = os.path.dirname(os.path.abspath(__file__))


def mutant(module, old, new):
    """A fresh module built from ``module``'s source with ``old`` (which must
    occur exactly once) replaced by ``new``."""
    src = inspect.getsource(module)
    assert src.count(old) == 1, (module.__name__, old, src.count(old))
    m = types.ModuleType(module.__name__ + "_mutant")
    exec(compile(src.replace(old, new), f"<mutant of {module.__name__}>", "exec"), m.__dict__)
    return m


def load_pins(filename, attr, module):
    """A private copy of a pin test module whose global ``attr`` is ``module``."""
    spec = importlib.util.spec_from_file_location("pins_" + filename[:-3], os.path.join(HERE, filename))
    pins = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(pins)
    setattr(pins, attr, module)
    return pins


def pin_calls(pins, skip=()):
    """(name, callable) for every test function of ``pins`` and every
    combination of its parametrize values."""
    out = []
    for name, fn in vars(pins).items():
        if not name.startswith("test_") or not callable(fn) or name in skip:
            continue
        marks = [m for m in getattr(fn, "pytestmark", []) if m.name == "parametrize"]
        if any(m.name == "skip" for m in getattr(fn, "pytestmark", [])):
            continue
        axes = []
        for m in marks:
            names = [s.strip() for s in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
            vals = [v if len(names) > 1 else (v,) for v in m.args[1]]
            axes.append([dict(zip(names, v)) for v in vals])
        for combo in itertools.product(*axes):
            kw = {k: v for d in combo for k, v in d.items()}
            out.append((f"{name}{kw or ''}", lambda fn=fn, kw=kw: fn(**kw)))
    return out


def first_failing_pin(calls):
    for name, call in calls:
        try:
            with warnings.catch_warnings():
                warnings.simplefilter("ignore")
                call()
        except AssertionError:
            return name
        except pytest.skip.Exception:
            continue
    return None


# ------------------------------------------------------------ attention oracle

ATTENTION_MUTANTS = {
    "row max over the wrong axis": ("m = s.max(axis=1, keepdims=True)", "m = s.max(axis=0, keepdims=True)"),
    "LSE in base 2": ("return p @ v, (m + np.log(l))[:, 0], p", "return p @ v, (m + np.log2(l))[:, 0], p"),
    "scale dropped from the scores": ("s = scale * (q @ k.T)", "s = q @ k.T"),
    "causal bound off by one": ("vis &= j <= i + right", "vis &= j < i + right"),
    "left window bound off by one": ("vis &= j >= i - left", "vis &= j > i - left"),
    "dS without the D term": ("ds = p * (dp - d_row)", "ds = p * dp"),
    "dS grouped wrongly": ("ds = p * (dp - d_row)", "ds = p * dp - d_row"),
    "scale dropped from dK": ("dk = scale * (ds.T @ q)", "dk = ds.T @ q"),
    "dV from O instead of dO": ("dv = p.T @ do", "dv = p.T @ o"),
    "D from dO alone": ("d_row = (do * o).sum(axis=1, keepdims=True)", "d_row = do.sum(axis=1, keepdims=True)"),
    "GQA head map h % g": ("head_forward(q[b, h], k[b, h // g], v[b, h // g], scale, causal, window)",
                           "head_forward(q[b, h], k[b, h % k.shape[1]], v[b, h % k.shape[1]], scale, causal, window)"),
    "GQA gradients overwritten, not summed": ("dk[b, h // g] += bb", "dk[b, h // g] = bb"),
    "sampled rows: causal bound off by one": ("s[i + right + 1:] = -np.inf", "s[i + right:] = -np.inf"),
    "sampled rows: left bound off by one": ("s[:max(i - left, 0)] = -np.inf", "s[:max(i - left - 1, 0)] = -np.inf"),
    "varlen ignores the causal flag": (
        "o[a:e, h], lse[h, a:e], _ = head_forward(q[a:e, h], k[a:e, h // g], v[a:e, h // g], scale, causal)",
        "o[a:e, h], lse[h, a:e], _ = head_forward(q[a:e, h], k[a:e, h // g], v[a:e, h // g], scale, False)"),
    "varlen GQA dK overwritten, not summed": ("dk[a:e, h // g] += y", "dk[a:e, h // g] = y"),
}


@pytest.mark.parametrize("what", sorted(ATTENTION_MUTANTS))
def test_attention_pins_catch(what):
    old, new = ATTENTION_MUTANTS[what]
    pins = load_pins("test_oracle_attention.py", "A", mutant(A, old, new))
    caught = first_failing_pin(pin_calls(pins, skip=("test_pins_catch_planted_mistakes",)))
    assert caught is not None, f"no pin fails when the oracle has: {what}"


# ------------------------------------------------------------------ FP8 oracle

FP8_MUTANTS = {
    "E4M3 decode with bias 8": ("(1.0 + m / 8.0) * np.exp2(e - 7.0)", "(1.0 + m / 8.0) * np.exp2(e - 8.0)"),
    "E4M3 subnormal step 2^-8": ("mag = np.where(e == 0, m * 2.0 ** -9,", "mag = np.where(e == 0, m * 2.0 ** -8,"),
    "E4M3 encode truncates": ("q_norm = np.rint((2.0 * mant - 1.0) * 8.0)", "q_norm = np.floor((2.0 * mant - 1.0) * 8.0)"),
    "E4M3 encode without saturation clamp": ("a = np.minimum(np.abs(np.where(nan, 0.0, x)), E4M3_MAX)",
                                             "a = np.abs(np.where(nan, 0.0, x))"),
    "largest E4M3 value of the IEEE-style format (240)": ("E4M3_MAX = 448.0", "E4M3_MAX = 240.0"),
    "scale exponent one too low at exact powers": ("e = np.where(safe * np.exp2(e * 1.0) > E4M3_MAX, e - 1, e)",
                                                   "e = np.where(safe * np.exp2(e * 1.0) >= E4M3_MAX, e - 1, e)"),
    "FWHT butterfly sign swapped": ("z[..., 1, :] = a - b", "z[..., 1, :] = b - a"),
    "rotation normalised by 1/d": ("c = np.float32(1.0 / np.sqrt(d))", "c = np.float32(1.0 / d)"),
    "rotation signs dropped": ("return (fwht_fp32(x * s) * c).astype(np.float32)",
                               "return (fwht_fp32(x) * c).astype(np.float32)"),
    "RoPE sign of the sine term": ("y[..., :h] = (a * c).astype(np.float32) - (b * s).astype(np.float32)",
                                   "y[..., :h] = (a * c).astype(np.float32) + (b * s).astype(np.float32)"),
    "RoPE f64 sign of the sine term": ("return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)",
                                       "return np.concatenate([a * c + b * s, b * c - a * s], axis=-1)"),
    "RoPE after the rotation": ("    if rope is not None:\n        x = rope_fp32(x, *rope)\n"
                                "    if signs is not None:\n        x = rotate_fp32(x, signs)\n",
                                "    if signs is not None:\n        x = rotate_fp32(x, signs)\n"
                                "    if rope is not None:\n        x = rope_fp32(x, *rope)\n"),
    "one factor per head, not per block": ("e = pow2_exponent(np.abs(blk).max(axis=(2, 3)))",
                                           "e = pow2_exponent(np.abs(x).max(axis=(2, 3)))"),
    "stored factor inverted": ("fac[:, :, i] = np.exp2(-e * 1.0)", "fac[:, :, i] = np.exp2(e * 1.0)"),
    "K factor dropped from the scores": ("s = scale * q_fac[:, None] * sk[blk][None, :] * (qrows @ kf[cols].T)",
                                         "s = scale * q_fac[:, None] * (qrows @ kf[cols].T)"),
    "Q factor dropped from the scores": ("s = scale * q_fac[:, None] * sk[blk][None, :] * (qrows @ kf[cols].T)",
                                         "s = scale * sk[blk][None, :] * (qrows @ kf[cols].T)"),
    "each tile takes its first key's block": ("blk = cols // block", "blk = np.full(len(cols), cols[0] // block)"),
    "causal mask off by one": ("s = np.where(cols[None, :] > rows[:, None] + right, -np.inf, s)",
                               "s = np.where(cols[None, :] >= rows[:, None] + right, -np.inf, s)"),
    "window's left bound off by one": ("s = np.where(cols[None, :] < rows[:, None] - left, -np.inf, s)",
                                       "s = np.where(cols[None, :] <= rows[:, None] - left, -np.inf, s)"),
    "O not rescaled when F grows": ("v_corr = np.exp2(f_run - f_new)", "v_corr = 1.0"),
    "F correction with the wrong sign": ("v_corr = np.exp2(f_run - f_new)", "v_corr = np.exp2(f_new - f_run)"),
    "row max correction with the wrong sign": ("corr = np.exp(m - m_use)", "corr = np.exp(m_use - m)"),
    "O not rescaled when m grows": ("acc = (corr * v_corr)[:, None] * acc + p8 @ vf[cols]",
                                    "acc = v_corr * acc + p8 @ vf[cols]"),
    "l not rescaled when m grows": ("l = corr * l + pt.sum(axis=1)", "l = l + pt.sum(axis=1)"),
    "P shift not undone": ("out = acc * np.exp2(f_run - p_shift) / l[:, None], m + np.log(l)",
                           "out = acc * np.exp2(f_run) / l[:, None], m + np.log(l)"),
    "stale-max threshold in the wrong units": ("m_new = np.where(mx > m + tau * np.log(2.0), mx, m)",
                                              "m_new = np.where(mx > m + tau, mx, m)"),
    "stale running max as the default": ("p_shift=4, tau=0.0, heads=None,", "p_shift=4, tau=STALE_MAX_TAU, heads=None,"),
    "half step a binade too small": ("return np.where(x >= 2.0 ** -6, np.exp2(ex - 5.0), 2.0 ** -10)",
                                     "return np.where(x >= 2.0 ** -6, np.exp2(ex - 6.0), 2.0 ** -10)"),
    "rounding bound not rescaled with O": ("err = (corr * v_corr)[:, None] * err + hs @ np.abs(vf[cols])",
                                           "err = err + hs @ np.abs(vf[cols])"),
    "V factor taken per tile, not per key": ("p8 = pt * np.exp2(p_shift + f_c - f_new)[None, :]",
                                             "p8 = pt * np.exp2(p_shift + f_c.max() - f_new)"),
    "P~ not rounded to E4M3": ("        if round_p:\n            p8 = e4m3_decode(e4m3_encode(p8))",
                               "        pass"),
    "split combine without normalisation": ("o = (w[..., None] * np.nan_to_num(o_parts)).sum(axis=0) / tot[..., None]",
                                            "o = (w[..., None] * np.nan_to_num(o_parts)).sum(axis=0)"),
    "split combine LSE in base 2": ("return o, mx + np.log(tot)", "return o, mx + np.log2(tot)"),
    "decode ignores the cache lengths": ("n = int(lens[b])", "n = kf.shape[2]"),
    "decode drops the last split": ("splits = [range(t, min(t + tiles_per_split, nt)) for t in range(0, nt, tiles_per_split)]",
                                    "splits = [range(t, min(t + tiles_per_split, nt)) for t in range(0, nt, tiles_per_split)]\n"
                                    "        splits = splits[:-1] if len(splits) > 1 else splits"),
}


@pytest.mark.parametrize("what", sorted(FP8_MUTANTS))
def test_fp8_pins_catch(what):
    old, new = FP8_MUTANTS[what]
    pins = load_pins("test_oracle_fp8.py", "F", mutant(F, old, new))
    caught = first_failing_pin(pin_calls(pins))
    assert caught is not None, f"no pin fails when the oracle has: {what}"


def test_unmutated_oracles_pass_every_pin():
    """The harness itself: with nothing planted, no pin fails."""
    for fname, attr, mod, skip in (("test_oracle_attention.py", "A", A, ("test_pins_catch_planted_mistakes",)),
                                   ("test_oracle_fp8.py", "F", F, ())):
        pins = load_pins(fname, attr, mutant(mod, "import numpy as np\n", "import numpy as np\n"))
        assert first_failing_pin(pin_calls(pins, skip=skip)) is None, fname
