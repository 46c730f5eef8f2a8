"""Reference oracle for the fused reduce + residual + RMSNorm step and the
wave-aware token-split planner.

THIS PACKAGE IS TEST INFRASTRUCTURE. It is a plain, slow, obviously correct
CPU restatement of what the GPU path computes, written in NumPy (fp64 for the
floating-point results, Python integers for the planner). Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and its
``--impl reference`` arm) may import or run it. The product path
(``reduce_rmsnorm_gb300`` and ``libtw``) never imports it, and it imports
nothing from the product path: the two share no code, tables or helpers.

Pages cited (by title and section):

  [W] "TokenWeave: Why Hiding Tensor-Parallel Communication Needs Wave
      Arithmetic, Not Finer Tiles" (technical blog summarising the paper)
  [G] "TokenWeave Guide: Compute-Communication Overlap for LLMs"
  [A] "TokenWeave: Efficient Compute-Communication Overlap for Distributed LLM
      Inference" (paper index page, "Abstract (arXiv)")

Functions and what pins each one (tests/test_oracle_*.py, ``-m "not gpu"``):

  bf16.decode / bf16.encode_rne   IEEE-754 bit patterns from the binary32
                                  definition; torch's own fp32->bf16 cast on
                                  random values; tie-to-even cases by hand.
  fused.reduce_residual_rmsnorm   fp64 plain definition of [W] "Fix two" and
                                  the RMSNorm formula of [G] "The Standard
                                  RMSNorm Memory Round-Trip". Pinned by closed
                                  forms (H=2 (3,4); constant rows; one-hot
                                  rows; zero rows), the mean-square invariant,
                                  exact small-integer sums, and shard
                                  invariance.
  fused.residual_fp32_rank_order  fp32 left-to-right sum in rank order, then
                                  one RNE rounding. Pinned by a hand-built
                                  case whose bf16 result depends on the order.
  planner.wave_split              Brute force over every prefix length. Pinned
                                  by the 300-CTA / 132-SM worked example of
                                  [W] "The overlap trap" and "Fix one", the
                                  single-wave and threshold rules of "Fix
                                  one", and hand-computed cases.
  shards.shard_rows               Row-by-row owner rule of the token-boundary
                                  shards ([W] "Fix two"). Pinned by the
                                  partition's invariants (every row owned
                                  once, contiguous and in rank order, sizes
                                  ceil(T/world) but the tail) and by
                                  hand-computed cases (1024 over 8 ranks;
                                  5 over 4 ranks).
  unfused.*                       The two-kernel (reduce, then standalone
                                  RMSNorm) baseline's numerics; pinned by the
                                  same closed forms.

No function here is "parity unpinned".
"""

from . import bf16, fused, planner, shards, unfused  # noqa: F401
