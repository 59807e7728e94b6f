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

Parity status: every function is pinned by ``tests/test_oracle_*.py`` except
``fp8.attention_fp8`` beyond its closed-form special cases (parity unpinned
for general inputs: only the stated tolerance and the ordering against the
per-tensor emulation are checked).
"""
