"""Brute-force oracle of the wave-aware token-split planner.

TEST INFRASTRUCTURE (see the package docstring). Integer arithmetic only
(Python ints, no overflow).

The rule, from [W] "The overlap trap" and "Fix one: split at wave boundaries,
unequally":

* A kernel of c CTAs runs in waves of S SMs: waves(c) = ceil(c / S)
  ("The overlap trap": 300 CTAs on 132 SMs run as 132 + 132 + 36, 3 waves).
* The batch is split exactly twice, into a prefix of p tokens and a suffix of
  T - p tokens, and a split is admissible only if the waves of the two pieces
  do not exceed the unsplit wave count ("Fix one").
* The prefix is half + offset and the suffix half - offset, half = T // 2,
  offset drawn from {0, 64, 128, 192, 256, 512} with offset < half ("Fix one",
  the sweep). The page's own worked example puts the SMALLER piece first
  (132 / 168), so an offset is applied with both signs; among candidates the
  smallest |offset| wins and a tie goes to the smaller prefix.
* When the unsplit kernel is a single wave, or the token count is below the
  per-iteration threshold (1K tokens for dense models), every token goes to
  the prefix and splitting is disabled ("Fix one").

The pages state the constraint in CTAs, not tokens. The CTA count of t tokens
is taken as linear in t with ceil rounding, c(t) = ceil(t * C / T), where C is
the unsplit kernel's CTA count for T tokens (a GEMM with 128-token row tiles
has C = ceil(T/128) * tiles_per_row, for which this is exact at every
128-token boundary).

This oracle does not enumerate candidates the way a planner would: it tests
EVERY prefix length p in [1, T-1] for feasibility, then keeps those whose
distance from half is an allowed offset, and picks the first in the order
(|p - half|, p).
"""

DEFAULT_OFFSETS = (0, 64, 128, 192, 256, 512)
DEFAULT_MIN_SPLIT_TOKENS = 1024


def ctas(t, T, C):
    """CTA count of a t-token piece of a T-token, C-CTA kernel: ceil(t*C/T)."""
    if T == 0:
        return 0
    return -((-t * C) // T)


def waves(c, S):
    """Waves of a c-CTA kernel on S SMs: ceil(c/S)."""
    return -((-c) // S)


def feasible(p, T, C, S):
    """True if prefix p / suffix T-p keeps the unsplit wave count."""
    return waves(ctas(p, T, C), S) + waves(ctas(T - p, T, C), S) <= waves(C, S)


def wave_split(T, C, S, offsets=DEFAULT_OFFSETS, min_split_tokens=DEFAULT_MIN_SPLIT_TOKENS):
    """Return (prefix_tokens, suffix_tokens).

    offsets=None means every integer offset 0 .. half-1 (used to check the
    pages' 132/168 example, whose offset of 18 is off the default grid).
    Raises ValueError for S <= 0, C < 0, T < 0 or a negative offset.
    """
    if S <= 0 or C < 0 or T < 0:
        raise ValueError("invalid planner arguments")
    if offsets is not None and any(o < 0 for o in offsets):
        raise ValueError("offsets must be non-negative (both signs are tried)")
    if T == 0:
        return (0, 0)
    if T < min_split_tokens or waves(C, S) <= 1:
        return (T, 0)
    half = T // 2
    allowed = set(range(half)) if offsets is None else {o for o in offsets if 0 <= o < half}
    best = None
    for p in range(1, T):
        if abs(p - half) not in allowed:
            continue
        if not feasible(p, T, C, S):
            continue
        key = (abs(p - half), p)
        if best is None or key < best:
            best = key
    if best is None:
        return (T, 0)
    p = best[1]
    return (p, T - p)
