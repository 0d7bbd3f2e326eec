"""CPU oracle for the Flash-Overlap hot path -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, deliberately unoptimised restatement of what the
method computes, written from the method description in "FlashOverlap:
Minimizing Tail Latency in Communication Overlap for Distributed LLM Training"
(technical summary, section 2 "Methodology: Flash-Overlap").  It shares no
code with the CUDA library and never imports it; only the seeded input
generators (``fo_workloads``) are common to both.

Who may use it: the tests under ``tests/``, ``__graft_entry__.smoke()`` (to
check one small GPU result) and ``bench.py`` (its CPU-baseline and
``--impl reference`` legs).  The product path (the C-ABI library and its Python
binding) must never call into this package.

Arithmetic policy: inputs are bf16 bit patterns; all arithmetic is fp64 (every
bf16 product is exact in fp64, and integer-valued workloads stay exact);
results are rounded once, to the output dtype of the operation (bf16
round-to-nearest-even), at the same operation boundaries as the layer
definition.

Modules:
  bf16      -- bf16 <-> fp64 conversion from the IEEE-754 rounding rule.
  ring      -- explicit simulated ring (tagged messages, per-step buffers).
  ops       -- definitions (undecomposed) and ring-decomposed versions of
               AG-GEMM, GEMM-RS, the MLP layer and query-split attention.
  schedule  -- step orders (local-first, kept-slice-last, naive) and a
               unit-time timeline model of exposed communication.

Pinned by ``tests/test_oracle_*.py`` (no GPU needed).  Nothing in this package
is "parity unpinned".
"""
from . import bf16, ring, ops, schedule  # noqa: F401
