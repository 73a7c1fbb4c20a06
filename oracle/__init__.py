"""Plain CPU oracle for the speculative-decoding verify round (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing in the product (the CUDA library and its
Python binding) imports, links or runs this package; only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference arm
do.  It shares no code with the CUDA path: the only common module is
``synth`` (seeded random inputs, no method arithmetic).

What it computes, and where the pages define it:

* ``ops.linear`` / ``ops.verify_attention`` / ``ops.target_probs`` — the
  target model's single parallel pass over [last token, x_1..x_gamma]
  ("Speculative Decoding Spends Arithmetic You May Not Have", section
  "What one iteration actually does", Algorithm 1, the parallel Mp line;
  "How Speculative Decoding Works (and When It Doesn't)", "Prefill and
  Decode").  These are exact definitions evaluated in fp64.
* ``sampler.reject_sample`` — the acceptance test, prefix truncation,
  residual correction and bonus token, in the order of Algorithm 1 of the
  first page (same section), with the readings of the open points stated in
  that module's header.
* ``ops.rmsnorm`` / ``ops.rope`` / ``ops.silu_mul`` and ``stack`` — the
  layer glue of a Qwen3-8B-shaped stack.  The pages only give the layer and
  head counts; the layer internals are the builder's reading.
* ``formulas`` — the closed forms the pages print (expected tokens per
  round, Theorem 3.11's arithmetic increase, the speedup / break-even model,
  the verify-cost division, vLLM's acceptance metrics).

Parity pins (tests marked ``not gpu``) tie every function here to values the
pages print, closed forms, invariants or brute force; see ``tests/``.
"""
from . import bf16, formulas, ops, sampler, stack  # noqa: F401
