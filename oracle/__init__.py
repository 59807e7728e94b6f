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
attention of the dequantised inputs). The rounding itself is pinned by worked
examples (one per running-max rule), the saturation bound, inputs on the E4M3
grid, and on arbitrary inputs by its own bound: every rounded entry moves by
at most half an E4M3 step (``fp8.half_step``), so O moves by at most the
returned E. The default running max is the one of Algorithm 1 (tau = 0);
``STALE_MAX_TAU`` selects the stale-max variant, which differs from it only in
which values are rounded, by at most one step per entry in total.
``tests/test_oracle_mutations.py`` plants mistakes in copies of both modules
and checks that a pin fails for each.
"""
