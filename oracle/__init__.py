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
  expert_ffn      -- hand-derived closed-form examples in bf16, int8, FP8 e4m3, FP8 e5m2 and
                     FP8 x FP4 (golden; non-square weights, two block scales per row, one
                     hand-derived MX exponent per block of A), reduction to a dense SwiGLU FFN
                     computed with library routines, int32 range check; mistakes planted in the
                     oracle (untransposed weights, a per-channel weight scale, swapped nibbles,
                     no re-quantisation of A, swapped gate/up) fail the FP8 goldens.
  forward         -- brute force per token (no plan) equals the pooled path bit for bit;
                     linearity in the gate weights; masked routes.

``ref.c`` states the plan, the shared-expert slots and the layer of every mode a second time in plain C
(loops in double precision, number formats decoded from their bit fields, integer products formed
directly), compiled by ``__graft_entry__.build_oracle()``; the CPU tests require the two to agree: the
plan, the integer accumulators, the re-quantised A of the integer modes and their y exactly; the float
modes' y and FP8 codes but for ties moved by the order of a float64 sum.
"""
from . import codecs, moe  # noqa: F401
