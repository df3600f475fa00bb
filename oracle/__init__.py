"""CPU oracle for the batch-invariant decoder forward — TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, obviously-correct numpy restatement of what the
GPU path computes.  Only the test-suite, the smoke check and the benchmark's
CPU-baseline leg may import it; the product library never does, and the two
share no code (no kernels, headers, tables or helpers).  The only thing both
sides consume is the seeded input generator in ``synthetic``.

Sources (cited as "<page>, <section>" in every docstring):
  * [Article]  "vLLM Achieves Bitwise-Consistent RL Training: Eliminating
    Numerical Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91%
    Throughput" (todayforai.com copy of the vLLM post).
  * [News]     "vLLM Makes RL Training and Inference Bitwise-Identical on
    DeepSeek-V4-Flash" (ainewsbites.com).
  * [README]   "zero-mismatch-rl" repository README (Inferact).

Numerical contract (the article's "same numerical contract", §2): fp32
accumulation with round-to-nearest-even bf16 rounding at the same layer
boundaries as the GPU path; the vocab-wide logsumexp is taken in fp64.

Pinning: every function is pinned by tests under ``tests/test_oracle_pins.py``
to closed forms, invariants, library routines or brute force.  No function is
left "parity unpinned".
"""
from .bf16 import round_bf16, bf16_bits_to_f32, f32_to_bf16_bits  # noqa: F401
from . import ops, model, moe  # noqa: F401
