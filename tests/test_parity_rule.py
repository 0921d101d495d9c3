"""The GPU parity rule (tests/parity.py) itself, on the host.

The oracle's own result, offered as the GPU result, must pass; each kind of
mistake a kernel could make must be rejected: a changed byte outside a folded
segment or in a row without a delta, a folded value far off, a wrong xa, a few
values a few ulps off, an xa (and the fold made from it) missing the last k
terms of a row, and too many values that are each one ulp off.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from gather_lora_gb300 import workloads as W
from gpu_util import oracle_bgmv, oracle_delta, oracle_gather, oracle_moe
from parity import (bf16_of_f64, compare_bgmv, compare_delta, compare_gather, compare_moe,
                    expand_oracle_order, fold_bits, gather_routes, moe_routes, routed_bgmv_rows)

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


def _consistent_row(wl, i, s, xa_row):
    """Row i's folded segment as a correct kernel would give it from `xa_row`: the
    expand in the oracle's order, the BF16 delta, one fp32 fma and BF16 rounding."""
    S = expand_oracle_order(xa_row[None], wl.b_pool[s])[0]
    d = bf16_of_f64(S.astype(np.float64))
    seg = wl.out_buf[i, wl.out_offset:wl.out_offset + wl.n_out]
    return fold_bits(wl.scale[s], d, seg)


def test_xa_flip_and_its_fold_pass_and_a_sign_flip_fails(bg):
    """An xa value one ulp off (a summation-order flip), with the fold made from it,
    passes; the same magnitude with the other sign in the output fails."""
    wl, out, xa, d = bg
    i, s = routed_bgmv_rows(wl)[0]
    c = int(np.argmax(np.abs(F(xa[i]))))
    gx = xa.copy()
    gx[i, c] = xa[i, c] + 1
    g = out.copy()
    seg = slice(wl.out_offset, wl.out_offset + wl.n_out)
    g[i, seg] = _consistent_row(wl, i, s, gx[i])
    st = compare_bgmv(wl, g, out, gx, xa, d, min_exact=0.0)
    assert st["xa_max_ulps"] == 1
    j = _big_element(wl, out, i)
    g = out.copy()
    g[i, j] = out[i, j] ^ 0x8000                 # same magnitude, other sign
    with pytest.raises(AssertionError, match="fold"):
        compare_bgmv(wl, g, out, xa, xa, d)


def test_a_one_ulp_fold_change_without_a_flip_fails(bg):
    """With xa equal to the oracle's and the expand sum away from a rounding
    boundary, a folded value one ulp off is not a summation-order effect."""
    wl, out, xa, d = bg
    i, _ = routed_bgmv_rows(wl)[0]
    j = _big_element(wl, out, i)
    g = out.copy()
    g[i, j] = out[i, j] + 1
    with pytest.raises(AssertionError, match="fold"):
        compare_bgmv(wl, g, out, xa, xa, d, min_exact=0.0)


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
    """Three rows whose every xa value is one ulp off (folds made from them): each
    value passes the rules, but the bit-exact floor rejects that many."""
    wl, out, xa, d = bg
    g, gx = out.copy(), xa.copy()
    seg = slice(wl.out_offset, wl.out_offset + wl.n_out)
    for i, s in routed_bgmv_rows(wl)[:3]:
        gx[i] = xa[i] + 1
        g[i, seg] = _consistent_row(wl, i, s, gx[i])
    with pytest.raises(AssertionError, match="bit-exact"):
        compare_bgmv(wl, g, out, gx, xa, d)
    compare_bgmv(wl, g, out, gx, xa, d, min_exact=0.0)   # each value is within the rules


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


def test_few_values_a_few_ulps_off_fail(bg):
    """+3 ulps on 0.5% of the folded values (at least one) is not a summation-order
    effect: the fold is no longer the fold of the row's own xa."""
    wl, out, xa, d = bg
    seg = slice(wl.out_offset, wl.out_offset + wl.n_out)
    routed = [i for i, _ in routed_bgmv_rows(wl)]
    rng = np.random.default_rng(0)
    n_bad = max(1, int(0.005 * len(routed) * wl.n_out))
    g = out.copy()
    for _ in range(n_bad):
        i = int(rng.choice(routed))
        j = wl.out_offset + int(rng.integers(wl.n_out))
        g[i, j] = out[i, j] + 3
    with pytest.raises(AssertionError, match="fold"):
        compare_bgmv(wl, g, out, xa, xa, d, min_exact=0.0)


def test_one_xa_value_three_ulps_off_fails(bg):
    wl, out, xa, d = bg
    i, _ = routed_bgmv_rows(wl)[0]
    c = int(np.argmax(np.abs(F(xa[i]))))        # a large, well-conditioned value
    gx = xa.copy()
    gx[i, c] = xa[i, c] + 3
    with pytest.raises(AssertionError, match="xa"):
        compare_bgmv(wl, out, out, gx, xa, d, min_exact=0.0)


def test_dropped_k_tail_on_one_row_fails(bg):
    """A kernel that drops the last 16 k terms of one row (and folds consistently
    from that wrong xa) is caught by the xa rule."""
    wl, out, xa, d = bg
    i, _ = routed_bgmv_rows(wl)[1]
    bad = W.BgmvWorkload(**{**wl.__dict__})
    bad.x = wl.x.copy()
    bad.x[i, wl.k_in - 16:wl.k_in] = 0
    b_out, b_xa, b_d = oracle_bgmv(bad)
    g, gx = out.copy(), xa.copy()
    g[i], gx[i] = b_out[i], b_xa[i]
    assert not np.array_equal(gx[i], xa[i])
    with pytest.raises(AssertionError, match="xa"):
        compare_bgmv(wl, g, out, gx, xa, d, min_exact=0.0)


def test_reported_ulp_distances(bg):
    wl, out, xa, d = bg
    st = compare_bgmv(wl, out.copy(), out, xa.copy(), xa, d)
    assert st["max_ulps"] == 0 and st["xa_max_ulps"] == 0 and st["beyond_1ulp"] == 0


def test_fold_helpers_against_the_oracle(bg):
    """The rule's own fp32 fma and BF16 rounding reproduce the oracle's folded
    values from the oracle's deltas bit for bit."""
    wl, out, xa, d = bg
    seg = slice(wl.out_offset, wl.out_offset + wl.n_out)
    for i, s in routed_bgmv_rows(wl):
        assert np.array_equal(fold_bits(wl.scale[s], d[i], wl.out_buf[i, seg]), out[i, seg])
        S = expand_oracle_order(xa[i][None], wl.b_pool[s])[0]
        assert np.array_equal(bf16_of_f64(S.astype(np.float64)), d[i])
