"""GPU-vs-oracle comparison rules for the fold.

Index and routing work is compared bit-exactly: every row the oracle leaves
alone, and every element outside a row's folded segment, must be byte-identical
on the GPU.

Floating point: the GPU sums the same BF16 products in another fixed order
(tensor-core steps of 16, k-slices reduced in rank order), so each fp32 sum may
differ from the oracle's sequential one by the standard summation bound. With
u = 2^-24 and gamma_m = m*u / (1 - m*u), for a sum of m products:
    |S_gpu - S_oracle| <= 2 * gamma_m * sum |terms|        (both orders' errors)
A BF16 rounding after the sum adds at most one ulp of the result. So
  * xa:    |xa_gpu - xa_ora| <= ulp + 2*gamma_{k_in} * sum_k |x_k A_ck|;
  * delta: the expand sum moves by sum_c |xa_gpu_c - xa_ora_c| |B_jc| (the
           observed xa difference, itself checked above) plus
           2*gamma_{max_rank} * sum_c |xa_c| |B_jc|, then one BF16 rounding;
  * fold:  |scale| times the delta change, plus one ulp of the result.
Where no intermediate rounding flips, this is the 1-ulp rule of the method.
A floor on the fraction of bit-exact elements is checked too.
"""
from __future__ import annotations

import numpy as np

from gather_lora_gb300 import workloads as W

F = W.bf16_bits_to_f32


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    e = (np.asarray(bits, dtype=np.uint16).astype(np.int64) >> 7) & 0xFF
    return np.where(e == 0, 2.0 ** -133, np.ldexp(1.0, (e - 127 - 7).astype(np.int64)))


def ulp_of_value(v: np.ndarray) -> np.ndarray:
    """BF16 ulp at magnitude |v| (float64 input)."""
    v = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(v)).astype(np.int64) - 7)


def gamma(m: int, u: float = 2.0 ** -24) -> float:
    return m * u / (1.0 - m * u)


def check_xa(gpu_xa_row, ora_xa_row, x_row, A):
    """xa within one ulp plus both summation errors of the k_in-term sums."""
    g, o = F(gpu_xa_row).astype(np.float64), F(ora_xa_row).astype(np.float64)
    mag = np.abs(F(A).astype(np.float64)) @ np.abs(F(x_row).astype(np.float64))
    bound = np.maximum(bf16_ulp(gpu_xa_row), bf16_ulp(ora_xa_row)) + 2.0 * gamma(A.shape[1]) * mag
    err = np.abs(g - o)
    if not np.all(err <= bound):
        c = int(np.argmax(err / bound))
        raise AssertionError(f"xa[{c}] gpu {g[c]!r} oracle {o[c]!r} err {err[c]:.3g} > bound {bound[c]:.3g}")
    return int(np.sum(gpu_xa_row == ora_xa_row))


def check_row_fold(gpu_row, ora_row, d_row, ora_xa_row, gpu_xa_row, B, scale):
    """Compare one routed row's folded segment; returns (n_exact, n, worst err/bound)."""
    Bf = np.abs(F(B).astype(np.float64))
    xo, xg = F(ora_xa_row).astype(np.float64), F(gpu_xa_row).astype(np.float64)
    dT = Bf @ np.abs(xg - xo) + 2.0 * gamma(B.shape[1]) * (Bf @ np.abs(xo))
    d = np.abs(F(d_row).astype(np.float64))
    d_change = dT + np.maximum(bf16_ulp(d_row), ulp_of_value(d + dT))
    gf, of = F(gpu_row).astype(np.float64), F(ora_row).astype(np.float64)
    err = np.abs(gf - of)
    bound = np.maximum(bf16_ulp(ora_row), bf16_ulp(gpu_row)) + abs(float(scale)) * d_change
    worst = float(np.max(err / bound)) if err.size else 0.0
    if not np.all(err <= bound):
        j = int(np.argmax(err / bound))
        raise AssertionError(f"fold[{j}] gpu {gf[j]!r} oracle {of[j]!r} err {err[j]:.3g} > bound {bound[j]:.3g}")
    return int(np.sum(gpu_row == ora_row)), int(gpu_row.size), worst


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
        xa_exact += check_xa(gpu_xa[i], ora_xa[i], wl.x[i, :wl.k_in], wl.a_pool[s])
        xa_tot += wl.max_rank
        e, t, w = check_row_fold(gpu_out[i, seg], ora_out[i, seg], ora_d[i], ora_xa[i], gpu_xa[i],
                                 wl.b_pool[s], wl.scale[s])
        n_exact, n_tot, worst = n_exact + e, n_tot + t, max(worst, w)
    if n_tot:
        assert n_exact / n_tot >= min_exact, f"only {n_exact}/{n_tot} folded values bit-exact"
    if xa_tot:
        assert xa_exact / xa_tot >= min_exact, f"only {xa_exact}/{xa_tot} xa values bit-exact"
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
        if ra is not None or wl.x_gather:
            t = int(sti[r])
            if t < 0 or t >= wl.num_tokens:
                continue
            if ra is not None:
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
                xrow = wl.x[wl.sorted_token_ids[r]] if wl.x_gather else wl.x[r]
                xa_exact += check_xa(gx[r - lo], ox[r - lo], xrow, wl.a_pool[idx])
    for r, idx in routes:
        # the xa of row r lives in its window's buffer, at the local row
        w = next(k for k, (lo, hi) in enumerate(windows) if lo <= r < hi)
        lr = r - windows[w][0]
        e, t, wst = check_row_fold(gpu_out[r], ora_out[r], ora_d[r], ora_xas[w][lr],
                                   gpu_xas[w][lr], wl.b_pool[idx], wl.scale[idx])
        n_exact, n_tot, worst = n_exact + e, n_tot + t, max(worst, wst)
    if n_tot:
        assert n_exact / n_tot >= min_exact, f"only {n_exact}/{n_tot} folded values bit-exact"
    return dict(rows=len(routes), exact=n_exact, total=n_tot, xa_exact=xa_exact, worst=worst)


def gather_routes(wl: W.MoeGatherWorkload, indices=None, row_adapter="wl"):
    """(row, table index) of every routed row of a decode-path MoE fold."""
    idx = wl.indices if indices is None else indices
    ra = wl.row_adapter if isinstance(row_adapter, str) else row_adapter
    E = wl.num_experts
    out = []
    for r in range(wl.n_rows):
        e = int(idx[r])
        t = r // wl.top_k
        if e < 0 or e >= E or t >= wl.num_tokens:
            continue
        a = 0 if ra is None else int(ra[t])
        if a < 0 or a >= wl.max_loras or not wl.present[a * E + e]:
            continue
        out.append((r, a * E + e))
    return out


def compare_gather(wl: W.MoeGatherWorkload, gpu_out, ora_out, gpu_xa, ora_xa, ora_d, routes,
                   min_exact=0.99):
    """Full comparison of a decode-path MoE fold (rows in flat (token, slot) order)."""
    routed = {r for r, _ in routes}
    mask = np.ones(gpu_out.shape[0], dtype=bool)
    mask[list(routed)] = False
    assert np.array_equal(gpu_out[mask], ora_out[mask]), "rows without a delta changed"
    assert np.array_equal(ora_out[mask], wl.out_buf[mask])
    n_exact = n_tot = xa_exact = xa_tot = 0
    worst = 0.0
    for r, idx in routes:
        xa_exact += check_xa(gpu_xa[r], ora_xa[r], wl.x[r], wl.a_pool[idx])
        xa_tot += wl.max_rank
        e, t, w = check_row_fold(gpu_out[r], ora_out[r], ora_d[r], ora_xa[r], gpu_xa[r],
                                 wl.b_pool[idx], wl.scale[idx])
        n_exact, n_tot, worst = n_exact + e, n_tot + t, max(worst, w)
    if n_tot:
        assert n_exact / n_tot >= min_exact, f"only {n_exact}/{n_tot} folded values bit-exact"
    if xa_tot:
        assert xa_exact / xa_tot >= min_exact, f"only {xa_exact}/{xa_tot} xa values bit-exact"
    return dict(rows=len(routes), exact=n_exact, total=n_tot, worst=worst)


def delta_as_bgmv(wl: W.DeltaWorkload) -> W.BgmvWorkload:
    """The single-adapter delta as a routed fold with every row on slot 0 (its
    definition, lora_delta.rs apply_lora_delta), for the bgmv comparison rules."""
    return W.BgmvWorkload(wl.name, wl.m, wl.k_in, wl.n_out, 1, wl.max_rank, wl.x_row_stride,
                          wl.out_row_stride, wl.out_offset, wl.x, wl.out_buf,
                          np.zeros(wl.m, dtype=np.int32), np.array([wl.rank], np.int32),
                          np.ones(1, dtype=bool), wl.a[None], wl.b[None],
                          np.array([wl.scale], dtype=np.float32))


def compare_delta(wl: W.DeltaWorkload, gpu_out, ora_out, gpu_xa, ora_xa, ora_d, min_exact=0.99):
    return compare_bgmv(delta_as_bgmv(wl), gpu_out, ora_out, gpu_xa, ora_xa, ora_d, min_exact)
