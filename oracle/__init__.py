"""Float64 CPU oracle for exact attention: TEST INFRASTRUCTURE ONLY.

Nothing in the product path may import this package. Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` use it.
It shares no code with the CUDA library and takes its inputs as plain arrays.

Modules
-------
attention : the plain definition of scaled-dot-product attention, its
            log-sum-exp, its analytic backward, GQA and variable-length forms.
fp8       : the E4M3 codec, power-of-two block scales, the random-sign
            Hadamard rotation and an emulation of block-quantised FP8
            attention that follows the tiled algorithm step by step.

Parity status: every function is pinned by ``tests/test_oracle_*.py``. For
``fp8.attention_fp8`` and ``fp8.decode_fp8`` everything but the E4M3 rounding
of P~ is pinned on arbitrary inputs (with ``round_p=False`` they equal float64
attention of the dequantised inputs); which value is rounded is pinned only by
a worked example, the saturation bound and inputs on the E4M3 grid (parity
partly unpinned: on general inputs the rounding's effect is checked through
the stated tolerance and the ordering against the per-tensor emulation).
``tests/test_oracle_mutations.py`` plants mistakes in copies of both modules
and checks that a pin fails for each.
"""
