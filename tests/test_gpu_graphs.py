"""The library's calls inside CUDA graphs (GPU only).

After the first call on a device (which probes it and looks up the status
word) and the first launch of each kernel instance (which raises its
shared-memory limit), an entry point only encodes tensor maps on the host
and enqueues kernels on the given stream; the maps travel by value in the
kernel parameters. So a training or decode step can be captured once and
replayed on new contents of the same buffers. These tests capture whole
steps with torch.cuda.CUDAGraph after one direct call, write new inputs into
the captured buffers, replay, and compare with the same calls made directly:
bit-identical for every output with one writer per element and a fixed
summation order (O, LSE, dK, dV, FP8 codes, factors and O, decode O and LSE),
and for dQ, whose FP32 partial sums arrive by reduce-adds in a varying order,
within 1e-3 relative RMS (a reordered FP32 sum moves a BF16 result by at most
one ulp, 2^-8 relative, and only rarely). One head of each replay is also
checked against the oracle with the tolerances of the other parity tests
(the decode against the oracle's split FP8 emulation on its own codes).
The shapes take the split last wave with its dependent launch (fewer units
than SMs), the persistent short-row forward and backward, GQA, causal
masking, d = 64, 128 and 256, packed sequences and split decode.
"""
import numpy as np
import pytest
import torch

from exact_attention_73_gb300 import binding as L
from exact_attention_73_gb300 import inputs
from oracle import attention as A
from oracle import fp8 as F

pytestmark = pytest.mark.gpu


def rel_rms(x, ref):
    x = np.asarray(x, dtype=np.float64)
    assert np.isfinite(x).all()
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-3 * np.sqrt(ref.size)))


def poison(outputs):
    """NaN into floating outputs and zeros into code tensors before each call, so that the
    comparison sees only what that call wrote."""
    for t in outputs.values():
        if t.is_floating_point():
            t.fill_(float("nan"))
        else:
            t.zero_()


def replay_and_compare(step, fill, outputs, loose=()):
    """Capture step() once, then for two new fillings of the inputs compare the
    replayed outputs with a direct call. Returns the last replay's outputs."""
    fill(0)
    step()                                   # first call: device probe, kernel attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    got = None
    for it in (1, 2):
        fill(it)
        poison(outputs)
        g.replay()
        torch.cuda.synchronize()
        assert L.attn_get_device_status() == 0
        got = {k: t.clone() for k, t in outputs.items()}
        poison(outputs)
        step()
        torch.cuda.synchronize()
        for name, t in outputs.items():
            if name in loose:
                assert rel_rms(got[name].double().cpu().numpy(), t.double().cpu().numpy()) <= 1e-3, (name, it)
            else:
                assert torch.equal(got[name], t), (name, it)
    return got


def fill_from(bufs, seed_base, dtype="bf16"):
    def fill(it):
        drawn = inputs.normal(seed_base + it, [tuple(b.shape) for b in bufs], dtype=dtype)
        for b, x in zip(bufs, drawn):
            b.copy_(x)
    return fill


@pytest.mark.parametrize("B,Hq,Hkv,N,d,causal", [
    (2, 4, 2, 1000, 128, False),     # GQA, fewer units than SMs: split last wave, dependent launch
    (2, 4, 2, 1000, 128, True),      # GQA, causal (heavy-first order, no split)
    (8, 16, 16, 512, 64, False),     # persistent forward and backward walks
    (1, 2, 1, 700, 256, False),      # d = 256: two CTAs per key tile, split last wave
])
def test_training_step_replays(B, Hq, Hkv, N, d, causal):
    q = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device="cuda")
    do = torch.empty_like(q)
    k = torch.empty((B, Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    o, lse = torch.empty_like(q), torch.empty((B, Hq, N), device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((L.attn_bwd_workspace_size(B, Hq, Hkv, N, d),), dtype=torch.uint8, device="cuda")

    def step():
        L.attn_fwd(q, k, v, o, lse, causal=causal)
        L.attn_bwd(q, k, v, o, lse, do, dq, dk, dv, ws, causal=causal)

    got = replay_and_compare(step, fill_from([q, k, v, do], 600 + d), {"o": o, "lse": lse, "dq": dq, "dk": dk,
                                                                       "dv": dv}, loose=("dq",))
    b, h = B - 1, Hq - 1
    one = lambda x: x[b:b + 1, h:h + 1].cpu()
    kv = lambda x: x[b:b + 1, h // (Hq // Hkv):h // (Hq // Hkv) + 1].cpu()
    o_ref, lse_ref = A.forward(one(q), kv(k), kv(v), d ** -0.5, causal)
    err = np.abs(one(got["o"]).double().numpy() - o_ref)
    assert err.max() <= 1e-2 and np.sqrt((err ** 2).mean()) <= 2e-3
    assert np.abs(one(got["lse"]).double().numpy() - lse_ref).max() <= 1e-3
    dq_ref, _, _ = A.backward(one(q), kv(k), kv(v), one(do), d ** -0.5, causal)
    assert rel_rms(one(got["dq"]).double().numpy(), dq_ref) <= 1e-2


def test_noalloc_backward_replays():
    # the library-owned workspace: its address is looked up by the first
    # (direct) call, after which the call captures like the others
    B, Hq, Hkv, N, d = 1, 4, 2, 1000, 128
    q = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device="cuda")
    do = torch.empty_like(q)
    k = torch.empty((B, Hkv, N, d), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    o, lse = torch.empty_like(q), torch.empty((B, Hq, N), device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)

    def step():
        L.attn_fwd(q, k, v, o, lse, causal=True)
        L.attn_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, causal=True)

    got = replay_and_compare(step, fill_from([q, k, v, do], 650), {"o": o, "lse": lse, "dq": dq, "dk": dk,
                                                                   "dv": dv}, loose=("dq",))
    # KV head 0 and the query heads 0 and 1 that read it, against the oracle
    full = A.backward(q[:, :2].cpu(), k[:, :1].cpu(), v[:, :1].cpu(), do[:, :2].cpu(), d ** -0.5, True)
    assert rel_rms(got["dk"][:, :1].double().cpu().numpy(), full[1]) <= 1e-2
    assert rel_rms(got["dv"][:, :1].double().cpu().numpy(), full[2]) <= 1e-2
    assert rel_rms(got["dq"][:, 1:2].double().cpu().numpy(), full[0][:, 1:2]) <= 1e-2


def test_fp8_step_replays():
    B, H, N, d = 2, 4, 1000, 128
    x = [torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    signs = inputs.random_signs(4, d).cuda()
    nb = (N + 127) // 128
    codes = [torch.empty((B, H, N, d), dtype=torch.uint8, device="cuda") for _ in range(3)]
    facs = [torch.empty((B, H, nb), device="cuda") for _ in range(3)]
    o, lse = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda"), torch.empty((B, H, N), device="cuda")

    def step():
        for t, c, f, s in zip(x, codes, facs, (signs, signs, None)):
            L.attn_quantize_fp8(t, c, f, s)
        L.attn_fwd_fp8(*codes, *facs, o, lse, causal=True)

    outs = {"o": o, "lse": lse, **{f"c{i}": c for i, c in enumerate(codes)}, **{f"s{i}": f for i, f in enumerate(facs)}}
    replay_and_compare(step, fill_from(x, 700), outs)


def test_varlen_step_replays_with_new_offsets():
    # the same lengths in another order each time: T and the longest length
    # (which size the grid) stay, the offsets read on the device change
    lens = [300, 1000, 5, 129, 640]
    T, Hq, Hkv, d = sum(lens), 4, 2, 128
    q = torch.empty((T, Hq, d), dtype=torch.bfloat16, device="cuda")
    do = torch.empty_like(q)
    k = torch.empty((T, Hkv, d), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    cu = torch.empty((len(lens) + 1,), dtype=torch.int32, device="cuda")
    o, lse = torch.empty_like(q), torch.empty((Hq, T), device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty((L.attn_bwd_varlen_workspace_size(T, Hq, Hkv, d),), dtype=torch.uint8, device="cuda")
    orders = [lens, lens[::-1], lens[2:] + lens[:2]]
    fill_x = fill_from([q, k, v, do], 800)

    def fill(it):
        fill_x(it)
        cu.copy_(inputs.cu_seqlens(orders[it]))

    def step():
        L.attn_fwd_varlen(q, k, v, o, lse, cu, max(lens), causal=True)
        L.attn_bwd_varlen(q, k, v, o, lse, do, dq, dk, dv, ws, cu, max(lens), causal=True)

    got = replay_and_compare(step, fill, {"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, loose=("dq",))
    # the longest sequence of the last order, against the oracle
    c = inputs.cu_seqlens(orders[2]).numpy()
    s = orders[2].index(1000)
    a, e = int(c[s]), int(c[s + 1])
    dense = lambda t: t[a:e].cpu().transpose(0, 1).unsqueeze(0)
    o_ref, lse_ref = A.forward(dense(q), dense(k), dense(v), d ** -0.5, True)
    err = np.abs(dense(got["o"]).double().numpy() - o_ref)
    assert err.max() <= 1e-2 and np.sqrt((err ** 2).mean()) <= 2e-3
    assert np.abs(got["lse"][:, a:e].cpu().double().numpy()[None] - lse_ref).max() <= 1e-3


def test_decode_replays_with_new_lengths():
    B, Hq, Hkv, nmax, d, splits = 4, 16, 4, 2000, 128, 4
    g = Hq // Hkv
    q = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((B, Hkv, nmax, d), dtype=torch.bfloat16, device="cuda")
    v = torch.empty_like(k)
    nb = (nmax + 127) // 128
    q8 = torch.empty((B, Hkv, g, d), dtype=torch.uint8, device="cuda")
    sq3 = torch.empty((B, Hkv, 1), device="cuda")
    sq = torch.empty((B, Hkv), device="cuda")
    k8, v8 = (torch.empty((B, Hkv, nmax, d), dtype=torch.uint8, device="cuda") for _ in range(2))
    sk, sv = (torch.empty((B, Hkv, nb), device="cuda") for _ in range(2))
    seqlens = torch.empty((B,), dtype=torch.int32, device="cuda")
    o, lse = torch.empty((B, Hq, d), dtype=torch.bfloat16, device="cuda"), torch.empty((B, Hq), device="cuda")
    ws = torch.empty((L.attn_decode_fp8_workspace_size(B, Hq, d, splits),), dtype=torch.uint8, device="cuda")
    signs = inputs.random_signs(9, d).cuda()
    fill_x = fill_from([q, k, v], 900)
    lengths = [[1, 2000, 129, 700], [2000, 2000, 2000, 2000], [5, 128, 1999, 1000]]

    def fill(it):
        fill_x(it)
        seqlens.copy_(torch.tensor(lengths[it], dtype=torch.int32))

    def step():
        # the step quantises the new token's query and decodes it
        L.attn_quantize_fp8(q.view(B, Hkv, g, d), q8, sq3, signs)
        sq.copy_(sq3[:, :, 0])
        L.attn_decode_fp8(q8.view(B, Hq, d), sq, k8, v8, sk, sv, o, lse, ws, splits, seqlens=seqlens)

    def fill_and_quantise_cache(it):
        fill(it)
        L.attn_quantize_fp8(k, k8, sk, signs)
        L.attn_quantize_fp8(v, v8, sv)

    got = replay_and_compare(step, fill_and_quantise_cache, {"o": o, "lse": lse})
    # the oracle quantises the last replay's bf16 inputs itself; the GPU's codes must equal its own
    sg = signs.cpu().numpy()
    rq8, rsq = F.quantize_blocks(q.cpu().view(B, Hkv, g, d), sg)
    rk8, rsk = F.quantize_blocks(k.cpu(), sg)
    rv8, rsv = F.quantize_blocks(v.cpu())
    rsq = rsq[:, :, 0]
    for name, gpu, ref in (("q8", q8, rq8), ("sq", sq, rsq), ("k8", k8, rk8), ("sk", sk, rsk), ("v8", v8, rv8),
                           ("sv", sv, rsv)):
        assert np.array_equal(gpu.cpu().numpy(), ref), name
    o_ref, lse_ref = F.decode_fp8(rq8, rsq, rk8, rv8, rsk, rsv, lengths[2], d ** -0.5, -(-nb // splits),
                                  tau=F.STALE_MAX_TAU)
    err = np.abs(got["o"].cpu().double().numpy().reshape(B, Hkv, g, d) - o_ref)
    assert np.sqrt((err ** 2).mean()) <= 2e-3 and np.quantile(err, 0.999) <= 1e-2 and err.max() <= 1e-1
    assert np.abs(got["lse"].cpu().double().numpy().reshape(B, Hkv, g) - lse_ref).max() <= 1e-3
