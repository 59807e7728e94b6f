"""The seeded input recipes (CPU): reproducible, of the stated shape, dtype
and distribution, and disjoint between seeds."""
import numpy as np
import torch

from exact_attention_73_gb300 import inputs


def test_host_normal_is_reproducible_and_standard():
    a, b = inputs.normal(3, [(4, 1000), (7,)])
    a2, _ = inputs.normal(3, [(4, 1000), (7,)])
    assert a.dtype == torch.bfloat16 and a.shape == (4, 1000) and b.shape == (7,)
    assert torch.equal(a, a2) and not torch.equal(a, inputs.normal(4, [(4, 1000)])[0])
    x = a.double().numpy()
    assert abs(x.mean()) < 0.05 and abs(x.std() - 1) < 0.05


def test_device_normal_is_reproducible_and_standard():
    # drawn by torch's seeded generator of the given device (the CPU here)
    a, b = inputs.normal_device(5, [(64, 1024), (3, 5)], dtype="fp16", device="cpu")
    a2, b2 = inputs.normal_device(5, [(64, 1024), (3, 5)], dtype="fp16", device="cpu")
    assert a.dtype == torch.float16 and a.shape == (64, 1024) and b.shape == (3, 5)
    assert torch.equal(a, a2) and torch.equal(b, b2)
    assert not torch.equal(a, inputs.normal_device(6, [(64, 1024)], dtype="fp16", device="cpu")[0])
    x = a.double().numpy()
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02


def test_varlen_recipe_and_signs():
    lens = inputs.varlen_lengths(9, 500, 900, 1250)
    assert min(lens) >= 900 and max(lens) <= 1250 and len(set(lens)) > 100
    cu = inputs.cu_seqlens(lens).numpy()
    assert cu.dtype == np.int32 and cu[0] == 0 and (np.diff(cu) == lens).all()
    s = inputs.random_signs(2, 128).numpy()
    assert s.dtype == np.int8 and set(s.tolist()) == {-1, 1}
