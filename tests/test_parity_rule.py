"""The GPU parity rule (tests/parity.py) itself, on the host.

The oracle's own result, offered as the GPU result, must pass; each kind of
mistake a kernel could make must be rejected: a changed byte outside a folded
segment or in a row without a delta, a folded value far off, a wrong xa, and
too many values that are each within the bound but not bit-exact.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gather_lora_gb300 import workloads as W
from gpu_util import oracle_bgmv, oracle_delta, oracle_gather, oracle_moe
from parity import (compare_bgmv, compare_delta, compare_gather, compare_moe, gather_routes,
                    moe_routes, routed_bgmv_rows)

F = W.bf16_bits_to_f32


@pytest.fixture(scope="module")
def bg():
    oracle.load()
    wl = W.make_bgmv("parity_rule", n=24, k_in=256, n_out=96, max_loras=6, max_rank=16,
                     rank_choices=(8, 16), alpha=32.0, rslora=False, slot_law="uniform",
                     slot_base_frac=0.2, seed=5, x_row_stride=264, out_row_stride=160,
                     out_offset=32, null_slots=(5,))
    out, xa, d = oracle_bgmv(wl)
    return wl, out, xa, d


def _big_element(wl, out, i):
    """A column of row i's folded segment whose value is far from zero."""
    seg = out[i, wl.out_offset:wl.out_offset + wl.n_out]
    return wl.out_offset + int(np.argmax(np.abs(F(seg))))


def test_oracle_result_passes(bg):
    wl, out, xa, d = bg
    st = compare_bgmv(wl, out.copy(), out, xa.copy(), xa, d)
    assert st["rows"] > 5 and st["exact"] == st["total"] > 0


def test_one_ulp_passes_and_a_sign_flip_fails(bg):
    wl, out, xa, d = bg
    i, _ = routed_bgmv_rows(wl)[0]
    j = _big_element(wl, out, i)
    g = out.copy()
    g[i, j] = out[i, j] + 1                      # the next BF16 value: one ulp away
    compare_bgmv(wl, g, out, xa, xa, d)
    g[i, j] = out[i, j] ^ 0x8000                 # same magnitude, other sign
    with pytest.raises(AssertionError, match="fold"):
        compare_bgmv(wl, g, out, xa, xa, d)


def test_bytes_outside_the_segment_and_base_rows_are_exact(bg):
    wl, out, xa, d = bg
    routed = {i for i, _ in routed_bgmv_rows(wl)}
    i = min(routed)
    g = out.copy()
    g[i, wl.out_offset - 1] ^= 1                 # just before the folded segment
    with pytest.raises(AssertionError, match="outside the folded segments"):
        compare_bgmv(wl, g, out, xa, xa, d)
    g = out.copy()
    g[i, wl.out_offset + wl.n_out] ^= 1          # just after it
    with pytest.raises(AssertionError, match="outside the folded segments"):
        compare_bgmv(wl, g, out, xa, xa, d)
    base = min(set(range(wl.n)) - routed)        # a row without a delta
    g = out.copy()
    g[base, wl.out_offset + 5] ^= 1
    with pytest.raises(AssertionError, match="outside the folded segments"):
        compare_bgmv(wl, g, out, xa, xa, d)


def test_wrong_xa_fails(bg):
    wl, out, xa, d = bg
    i, _ = routed_bgmv_rows(wl)[0]
    gx = xa.copy()
    gx[i, 0] ^= 0x4000                           # far from the oracle's value
    with pytest.raises(AssertionError, match="xa"):
        compare_bgmv(wl, out, out, gx, xa, d)


def test_too_many_inexact_values_fail(bg):
    wl, out, xa, d = bg
    g = out.copy()
    seg = slice(wl.out_offset, wl.out_offset + wl.n_out)
    routed = [i for i, _ in routed_bgmv_rows(wl)]
    for i in routed[:3]:                         # every value of three rows one ulp off
        g[i, seg] = out[i, seg] + 1
    with pytest.raises(AssertionError, match="bit-exact"):
        compare_bgmv(wl, g, out, xa, xa, d)
    compare_bgmv(wl, g, out, xa, xa, d, min_exact=0.0)   # each value is within the bound


def test_moe_rule_passes_oracle_and_rejects_mistakes():
    oracle.load()
    wl = W.make_moe("parity_rule_moe", num_tokens=24, top_k=3, num_experts=6, k_in=32, n_out=40,
                    max_loras=3, max_rank=8, rank=8, alpha=16.0, adapter_base_frac=0.25, cap=40,
                    seed=7)
    windows = wl.windows()
    out, xas, d = oracle_moe(wl, windows)
    routes = [rt for lo, hi in windows for rt in moe_routes(wl, lo, hi)]
    compare_moe(wl, windows, out.copy(), out, [x.copy() for x in xas], xas, d, routes)
    routed = {r for r, _ in routes}
    base = min(set(range(wl.te)) - routed)
    g = out.copy()
    g[base, 0] ^= 1
    with pytest.raises(AssertionError, match="without a delta"):
        compare_moe(wl, windows, g, out, xas, xas, d, routes)
    r = min(routed)
    g = out.copy()
    j = int(np.argmax(np.abs(F(out[r]))))
    g[r, j] ^= 0x8000
    with pytest.raises(AssertionError, match="fold"):
        compare_moe(wl, windows, g, out, xas, xas, d, routes)


def test_gather_rule_passes_oracle_and_rejects_mistakes():
    oracle.load()
    wl = W.make_moe_gather("parity_rule_gather", num_tokens=9, top_k=3, num_experts=5, k_in=40,
                           n_out=24, max_loras=3, max_rank=8, rank=8, alpha=16.0,
                           adapter_base_frac=0.25, seed=21, present_frac=0.8)
    out, xa, d = oracle_gather(wl)
    routes = gather_routes(wl)
    compare_gather(wl, out.copy(), out, xa.copy(), xa, d, routes)
    r = routes[0][0]
    gx = xa.copy()
    gx[r, 0] ^= 0x4000
    with pytest.raises(AssertionError, match="xa"):
        compare_gather(wl, out, out, gx, xa, d, routes)


def test_delta_rule_passes_oracle_and_rejects_mistakes():
    oracle.load()
    wl = W.make_delta("parity_rule_delta", m=12, k_in=200, n_out=72, max_rank=16, rank=12,
                      alpha=32.0, rslora=False, seed=9, x_row_stride=208, out_row_stride=96,
                      out_offset=16)
    out, xa, d = oracle_delta(wl)
    compare_delta(wl, out.copy(), out, xa.copy(), xa, d)
    g = out.copy()
    g[3, wl.out_offset + wl.n_out] ^= 1          # a byte after the folded segment
    with pytest.raises(AssertionError, match="outside the folded segments"):
        compare_delta(wl, g, out, xa, xa, d)
