"""Vocabulary slices of a frozen head, as the distillation head lays them out.

The cut rule follows cortiq-engine ``train_head.rs``, ``Head::new``: a slice
holds at most ``max_rows`` vocabulary rows rounded down to a multiple of 128
(by default the most that fit a 2 GiB storage binding of f16 weights with
``hs`` columns); the vocabulary is split into the fewest slices of that size,
and every slice but the last has the same width, the per-slice share rounded
up to a multiple of 128.
"""
from __future__ import annotations


def vocab_cuts(V: int, hs: int = 0, max_rows: int | None = None) -> list[tuple[int, int]]:
    """(offset, width) of each vocabulary slice."""
    if V <= 0:
        raise ValueError("V must be positive")
    if max_rows is None:
        if hs <= 0:
            raise ValueError("give max_rows or the hidden size hs")
        max_rows = ((1 << 31) - 4) // (2 * hs)
    cap = max_rows // 128 * 128
    n = -(-V // max(cap, 128))
    per = -(-(-(-V // n)) // 128) * 128
    cuts, off = [], 0
    while off < V:
        width = min(per, V - off)
        cuts.append((off, width))
        off += width
    return cuts


def cuts_for_slices(V: int, nslices: int) -> list[tuple[int, int]]:
    """The cuts ``Head::new`` yields when the vocabulary needs ``nslices`` slices.

    Uses the smallest 128-multiple cap that gives ``nslices`` slices.
    """
    per = -(-(-(-V // nslices)) // 128) * 128
    cuts = vocab_cuts(V, max_rows=per)
    if len(cuts) != nslices:
        raise ValueError(f"V={V} cannot be cut into {nslices} slices")
    return cuts
