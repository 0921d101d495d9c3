"""The guard-band check used by the -m gpu write-bounds tests, on the host."""
from __future__ import annotations

import torch

from guard_bands import GUARD, PATTERN, guarded, guards_intact


def test_guard_helpers_catch_a_write_past_either_end():
    t = torch.arange(24, dtype=torch.int16).view(4, 6)
    big, view = guarded(t)
    assert torch.equal(view, t) and view.is_contiguous()
    assert view.data_ptr() == big.data_ptr() + 2 * GUARD and view.data_ptr() % 16 == 0
    view.fill_(7)                                   # writes inside the view are fine
    assert guards_intact(big, view)
    big[GUARD + t.numel()] = 1                      # one element past the end
    assert not guards_intact(big, view)
    big[GUARD + t.numel()] = PATTERN
    big[GUARD - 1] = 0                              # one element before the start
    assert not guards_intact(big, view)
