"""Communication-volume arithmetic behind vocab-parallel cross-entropy.

TEST INFRASTRUCTURE ONLY (see ``vpce_oracle``): used by the tests to pin the
byte counts the pages print; nothing on the product path imports it.

The reason the method exists ("Distributed Training III: Model Parallelism",
CMU 11-868 Lecture 16 notes, §5.5 "Embedding and output layer", and exercise 9
of §9 with its answer): gathering the full logits onto every card moves
``tokens * V`` values, while the fused cross-entropy exchanges three fp32
scalars per token.  Both are counted per card for a ring collective, which
sends (t - 1)/t of the gathered tensor for an all-gather and 2 (t - 1)/t of
the reduced tensor for an all-reduce.  "LLM Internals" §7.3.4 gives the size
of the ``[s, V]`` logits themselves and the per-card column count V / t.
"""
from __future__ import annotations

from fractions import Fraction


def allgather_logits_bytes(tokens: int, V: int, t: int, elem_bytes: int) -> Fraction:
    """Bytes one card sends to all-gather the ``[tokens, V]`` logits (ring)."""
    return Fraction(tokens * V * elem_bytes) * Fraction(t - 1, t)


def fused_ce_bytes(tokens: int, t: int, scalars: int = 3, scalar_bytes: int = 4) -> Fraction:
    """Bytes one card sends for the fused loss: ``scalars`` ring all-reduces
    of one fp32 per token, each costing 2 (t - 1)/t of its payload."""
    return Fraction(tokens * scalars * scalar_bytes) * 2 * Fraction(t - 1, t)


def logits_bytes(s: int, V: int, elem_bytes: int) -> int:
    """Size of the unsharded ``[s, V]`` logits."""
    return s * V * elem_bytes


def columns_per_card(V: int, t: int) -> int:
    """Vocabulary columns each of t cards holds when t divides V."""
    if V % t:
        raise ValueError("V is not divisible by t: the vocabulary needs padding")
    return V // t
