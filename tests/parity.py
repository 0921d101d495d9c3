"""GPU-vs-oracle comparison rules for the fold.

Index and routing work is compared bit-exactly: every row the oracle leaves
alone, and every element outside a row's folded segment, must be byte-identical
on the GPU.

Folded values: the GPU sums in a different (fixed) fp32 order, with tensor-core
accumulation, so a BF16 rounding of xa or of the delta may land on the other
neighbour when the exact sum sits next to a rounding boundary. The bound used
follows the arithmetic:
  * if xa_c flips, it moves by one BF16 ulp <= 2^-7 |xa_c|, which moves the
    expand sum by at most 2^-7 * sum_c |xa_c| |B_jc| (= 2^-7 * mag_ij);
  * if the delta d flips, it moves by at most 2^-7 |d|;
  * the fold multiplies the delta change by |scale| and rounds once more, so
      |gpu - oracle| <= max(ulp(gpu), ulp(oracle)) + |scale| * 2^-7 * (mag + |d|).
Without any intermediate flip this is the 1-ulp rule. A sanity floor on the
fraction of bit-exact elements is checked too.
"""
from __future__ import annotations

import numpy as np

from gather_lora_gb300 import workloads as W

F = W.bf16_bits_to_f32


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    e = (np.asarray(bits, dtype=np.uint16).astype(np.int64) >> 7) & 0xFF
    return np.where(e == 0, 2.0 ** -133, np.ldexp(1.0, (e - 127 - 7).astype(np.int64)))


def fold_bound(ora_bits, gpu_bits, d_bits, mag, scale) -> np.ndarray:
    ulp = np.maximum(bf16_ulp(ora_bits), bf16_ulp(gpu_bits))
    return ulp + np.abs(np.float64(scale)) * 2.0 ** -7 * (mag + np.abs(F(d_bits).astype(np.float64)))


def check_row_fold(gpu_row, ora_row, d_row, xa_row, B, scale):
    """Compare one routed row's folded segment; returns (n_exact, n, worst err/bound)."""
    mag = np.abs(B.astype(np.float64)) @ np.abs(F(xa_row).astype(np.float64))
    gf, of = F(gpu_row).astype(np.float64), F(ora_row).astype(np.float64)
    err = np.abs(gf - of)
    bound = fold_bound(ora_row, gpu_row, d_row, mag, scale)
    worst = float(np.max(err / bound)) if err.size else 0.0
    assert np.all(err <= bound), f"fold outside bound: worst err/bound = {worst}"
    return int(np.sum(gpu_row == ora_row)), int(gpu_row.size), worst


def check_xa(gpu_xa_row, ora_xa_row):
    """xa may differ from the oracle by one BF16 ulp (a flipped rounding)."""
    g, o = F(gpu_xa_row).astype(np.float64), F(ora_xa_row).astype(np.float64)
    ulp = np.maximum(bf16_ulp(gpu_xa_row), bf16_ulp(ora_xa_row))
    assert np.all(np.abs(g - o) <= ulp), "xa differs from the oracle by more than one BF16 ulp"
    return int(np.sum(gpu_xa_row == ora_xa_row))


def routed_bgmv_rows(wl: W.BgmvWorkload):
    out = []
    for i, s in enumerate(wl.seq_slot):
        if 0 <= s < wl.max_loras and wl.present[s]:
            out.append((i, int(s)))
    return out


def compare_bgmv(wl: W.BgmvWorkload, gpu_out, ora_out, gpu_xa, ora_xa, ora_d, min_exact=0.99):
    """Full comparison of a bgmv result. gpu_out/ora_out: [n, out_row_stride] uint16."""
    routed = routed_bgmv_rows(wl)
    routed_set = {i for i, _ in routed}
    seg = slice(wl.out_offset, wl.out_offset + wl.n_out)
    # bit-exact: everything outside the folded segments of routed rows
    mask = np.ones(gpu_out.shape, dtype=bool)
    for i in routed_set:
        mask[i, seg] = False
    assert np.array_equal(gpu_out[mask], ora_out[mask]), "bytes outside the folded segments changed"
    assert np.array_equal(ora_out[mask], wl.out_buf[mask])
    n_exact = n_tot = xa_exact = xa_tot = 0
    worst = 0.0
    for i, s in routed:
        xa_exact += check_xa(gpu_xa[i], ora_xa[i])
        xa_tot += wl.max_rank
        e, t, w = check_row_fold(gpu_out[i, seg], ora_out[i, seg], ora_d[i], ora_xa[i],
                                 wl.b_pool[s], wl.scale[s])
        n_exact, n_tot, worst = n_exact + e, n_tot + t, max(worst, w)
    if n_tot:
        assert n_exact / n_tot >= min_exact, f"only {n_exact}/{n_tot} folded values bit-exact"
    return dict(rows=len(routed), exact=n_exact, total=n_tot, xa_exact=xa_exact, xa_total=xa_tot,
                worst=worst)


def moe_routes(wl: W.MoeWorkload, lo: int, hi: int, offsets=None, sorted_ids=None, row_adapter="wl"):
    """(row, table index) of every routed sorted row of window [lo, hi), per the skip rules."""
    offs = wl.expert_offsets if offsets is None else offsets
    sti = wl.sorted_token_ids if sorted_ids is None else sorted_ids
    ra = wl.row_adapter if isinstance(row_adapter, str) else row_adapter
    E = wl.num_experts
    out = []
    for r in range(lo, hi):
        if r < offs[0] or r >= offs[E]:
            continue
        e = int(np.searchsorted(offs, r, side="right") - 1)
        if not (offs[e] <= r < offs[e + 1]):
            continue
        a = 0
        if ra is not None:
            t = int(sti[r])
            if t < 0 or t >= wl.num_tokens:
                continue
            a = int(ra[t])
        if a < 0 or a >= wl.max_loras:
            continue
        idx = a * E + e
        if not wl.present[idx]:
            continue
        out.append((r, idx))
    return out


def compare_moe(wl: W.MoeWorkload, windows, gpu_out, ora_out, gpu_xas, ora_xas, ora_d, routes,
                min_exact=0.99):
    """gpu_xas/ora_xas: per window [rows, max_rank] arrays (window-local rows)."""
    routed = {r for r, _ in routes}
    mask = np.ones(gpu_out.shape[0], dtype=bool)
    mask[list(routed)] = False
    assert np.array_equal(gpu_out[mask], ora_out[mask]), "rows without a delta changed"
    assert np.array_equal(ora_out[mask], wl.out_buf[mask])
    n_exact = n_tot = xa_exact = 0
    worst = 0.0
    for (lo, hi), gx, ox in zip(windows, gpu_xas, ora_xas):
        for r, idx in routes:
            if lo <= r < hi:
                xa_exact += check_xa(gx[r - lo], ox[r - lo])
    for r, idx in routes:
        # the oracle's xa of row r lives in its window's buffer
        w = next(k for k, (lo, hi) in enumerate(windows) if lo <= r < hi)
        xa_row = ora_xas[w][r - windows[w][0]]
        e, t, wst = check_row_fold(gpu_out[r], ora_out[r], ora_d[r], xa_row, wl.b_pool[idx],
                                   wl.scale[idx])
        n_exact, n_tot, worst = n_exact + e, n_tot + t, max(worst, wst)
    if n_tot:
        assert n_exact / n_tot >= min_exact, f"only {n_exact}/{n_tot} folded values bit-exact"
    return dict(rows=len(routes), exact=n_exact, total=n_tot, xa_exact=xa_exact, worst=worst)
