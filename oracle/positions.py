"""Snapshot positions and reusable prefixes (test infrastructure).

"Kimi K3 Tech Intro", sections 2.1-2.2: a recurrent state can only be reused at a
position where it was saved.  With states saved only at the 4096-token physical
block, two requests sharing 4800 and 4900 tokens reuse just 4096 and recompute
704 and 804 tokens; decoupling the prefix-match unit (256 tokens) from the
physical block lets them reuse the state at the last multiple of 256 instead.
"""


def snapshot_positions(start_pos: int, length: int, interval: int):
    """Absolute positions p (0 < p, start_pos < p <= start_pos + length) with
    p % interval == 0: the positions after which a snapshot is taken.  The
    snapshot at p has ordinal p // interval - 1."""
    first = (start_pos // interval + 1) * interval
    return list(range(first, start_pos + length + 1, interval))


def reusable_prefix(shared_tokens: int, interval: int) -> int:
    """Longest prefix of ``shared_tokens`` that ends on a saved state."""
    return (shared_tokens // interval) * interval
