"""Guard bands around device outputs: the stand-in for a memory checker.

A tensor is copied into the middle of one larger allocation whose ends (GUARD
elements on each side) hold a fixed pattern. After a fold writes through the
middle view, every guard element must still hold the pattern: any write past
either end of base_out or xa would change it.
"""
from __future__ import annotations

import torch

GUARD = 4096            # elements on each side (8 KiB of int16: keeps 16-byte alignment)
PATTERN = 0x5AA5        # int16 guard value (not a value the folds are likely to write)


def guarded(t: torch.Tensor):
    """(big, view): `view` holds a copy of t (same shape) between two guard bands of big."""
    n = t.numel()
    big = torch.full((GUARD + n + GUARD,), PATTERN, dtype=t.dtype, device=t.device)
    view = big[GUARD:GUARD + n].view(t.shape)
    view.copy_(t)
    return big, view


def guards_intact(big: torch.Tensor, view: torch.Tensor) -> bool:
    """True when both guard bands of `big` around `view` still hold the pattern."""
    n = view.numel()
    host = big.cpu()
    return bool((host[:GUARD] == PATTERN).all()) and bool((host[GUARD + n:] == PATTERN).all())
