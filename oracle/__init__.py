"""CPU oracle of the fused MoE expert FFN with top-k combine (float64, plain numpy).

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import it. The product path (the CUDA library and its binding) never
does, and the oracle imports nothing from it.

Parity status of each function (what pins it, in ``tests/test_oracle_*.py``):
  plan            -- worked count/prefix-sum/scatter example (golden), bijection and count
                     invariants, brute-force counting.
  codecs          -- every e4m3/e2m1/UE8M0 code against the format definitions and torch's
                     own conversions; bf16 rounding against torch's conversion.
  silu/swiglu     -- closed forms (SiLU(0)=0, odd-part identity, limits, known minimum),
                     hand-derived gate/up example (golden).
  quantisers      -- range, symmetry, argmax -> +-127, error <= scale/2, MX exponent rule.
  expert_ffn      -- hand-derived closed-form examples in bf16 and int8 (golden), reduction
                     to a dense SwiGLU FFN computed with library routines, int32 range check.
  forward         -- brute force per token (no plan) equals the pooled path bit for bit;
                     linearity in the gate weights; masked routes.

``ref.c`` states the plan and the A16W16, A8W8-INT and FP8 x FP4 layers a second time in plain C (loops in double
precision, the same readings), compiled by ``__graft_entry__.build_oracle()``; the CPU tests
require the two to agree (the plan exactly, y bit for bit but for ties).
"""
from . import codecs, moe  # noqa: F401
