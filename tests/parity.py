"""GPU-vs-oracle comparison rules for the fold.

Index and routing work is compared bit-exactly: every row the oracle leaves
alone, and every element outside a row's folded segment, must be byte-identical
on the GPU.

Floating point. The GPU sums the same BF16 products as the oracle (each product
is exact in fp32) in another fixed order: tensor-core steps of 16, k-slices
reduced in rank order. The rule ("Function apply_lora_bgmv" summary: fp32
accumulate, xa rounded to BF16, the delta rounded to BF16, then one fp32 fold)
is checked in three parts, with u = 2^-24:

  xa     |xa_gpu - xa_ora| <= ulp + 2 * LAMBDA * sqrt(k_in) * u * sum_k |x_k A_ck|.
         The second term is the probabilistic bound on two fp32 summation
         orders of k_in terms (each error at most LAMBDA * sqrt(m) * u * sum|t|,
         failing with probability below 2 exp(-LAMBDA^2 / 2) ~ 3e-8 per value).
         Where it is below one ulp this is the one-ulp rule; more than one ulp
         is only allowed where the sum cancels so far that the two orders can
         straddle several BF16 values.
  fold   every folded value must be the fold of the GPU's own xa up to the
         expand's summation order: with S' the oracle-order fp32 expand sum of
         the GPU's xa and delta = 2 * gamma_{max_rank} * sum_c |xa_c B_jc|
         (the worst case of two orders, gamma_m = m*u / (1 - m*u)), the GPU value
         must lie between bf16(fma(scale, bf16(S' -+ delta), base)). A fold that
         is off by even one ulp for any other reason fails.
  stated the folded value is within one ulp of the oracle's wherever neither
         the row's xa nor the element's delta differs from the oracle's; beyond
         one ulp only where one of them flipped (the relative error is then the
         flip's, at most 2^-7 of the delta term for a delta flip).
A floor on the fraction of bit-exact elements is checked too, and the largest
ulp distance of xa and of the folded values is reported.
"""
from __future__ import annotations

import math
from collections import defaultdict

import numpy as np

from gather_lora_gb300 import workloads as W

F = W.bf16_bits_to_f32
U = 2.0 ** -24
LAMBDA = 6.0


def bf16_ulp(bits: np.ndarray) -> np.ndarray:
    e = (np.asarray(bits, dtype=np.uint16).astype(np.int64) >> 7) & 0xFF
    return np.where(e == 0, 2.0 ** -133, np.ldexp(1.0, (e - 127 - 7).astype(np.int64)))


def ulp_of_value(v: np.ndarray) -> np.ndarray:
    """BF16 ulp at magnitude |v| (float64 input)."""
    v = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(v)).astype(np.int64) - 7)


def gamma(m: int, u: float = U) -> float:
    return m * u / (1.0 - m * u)


def ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in BF16 steps between two arrays of BF16 patterns (sign-aware)."""
    def key(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        return np.where(b & 0x8000, -(b & 0x7FFF), b)
    return np.abs(key(a_bits) - key(b_bits))


def _f64_to_f32_odd(v: np.ndarray) -> np.ndarray:
    """float64 -> float32 rounded to odd (exact values stay; an inexact one takes
    the neighbour with an odd last bit). Rounding that to BF16 (RNE) gives the
    correctly rounded BF16 of v, since 24 >= 8 + 2."""
    v = np.asarray(v, dtype=np.float64)
    r = v.astype(np.float32)
    inexact = r.astype(np.float64) != v
    even = (r.view(np.uint32) & 1) == 0
    toward = np.where(v > r.astype(np.float64), np.float32(np.inf), np.float32(-np.inf))
    return np.where(inexact & even, np.nextafter(r, toward), r)


def bf16_of_f64(v: np.ndarray) -> np.ndarray:
    """Round float64 values to BF16 bit patterns (round to nearest even)."""
    return W.to_bf16_bits(_f64_to_f32_odd(v))


def fmaf32(a: np.ndarray, b: np.ndarray, c: np.ndarray) -> np.ndarray:
    """fp32 fma(a, b, c) with one rounding, for float32 a and c and b holding BF16
    values: a*b is exact in float64; the sum is made exact by TwoSum and rounded
    to odd in float64, then rounded to float32 (53 >= 24 + 2)."""
    p = np.asarray(a, np.float64) * np.asarray(b, np.float64)
    q = np.asarray(c, np.float64)
    s = p + q
    bb = s - p
    err = (p - (s - bb)) + (q - bb)
    even = (s.view(np.int64) & 1) == 0
    s = np.where((err != 0) & even, np.nextafter(s, np.where(err > 0, np.inf, -np.inf)), s)
    return s.astype(np.float32)


def fold_bits(scale: float, d_bits: np.ndarray, base_bits: np.ndarray) -> np.ndarray:
    """The method's fold of BF16 deltas into BF16 base values: bf16(fma(scale, d, base))."""
    r = fmaf32(np.float32(scale), F(d_bits), F(base_bits))
    return W.to_bf16_bits(r)


def check_xa(gpu_xa_row, ora_xa_row, x_row, A):
    """xa within one ulp plus the probabilistic bound of two k_in-term summation
    orders. Returns (bit-exact count, largest ulp distance)."""
    g, o = F(gpu_xa_row).astype(np.float64), F(ora_xa_row).astype(np.float64)
    mag = np.abs(F(A).astype(np.float64)) @ np.abs(F(x_row).astype(np.float64))
    k_in = A.shape[1]
    bound = (np.maximum(bf16_ulp(gpu_xa_row), bf16_ulp(ora_xa_row))
             + 2.0 * LAMBDA * math.sqrt(k_in) * U * mag)
    err = np.abs(g - o)
    if not np.all(err <= bound):
        c = int(np.argmax(err / bound))
        raise AssertionError(f"xa[{c}] gpu {g[c]!r} oracle {o[c]!r} err {err[c]:.3g} > bound {bound[c]:.3g}")
    dist = ulp_distance(gpu_xa_row, ora_xa_row)
    return int(np.sum(gpu_xa_row == ora_xa_row)), int(dist.max()) if dist.size else 0


def expand_oracle_order(xa_bits: np.ndarray, B: np.ndarray) -> np.ndarray:
    """fp32 expand sums of rows xa [R, max_rank] against B [n_out, max_rank], summed
    term by term in rank order as the oracle does (float32 arrays, no fma)."""
    xa = F(xa_bits).astype(np.float32)
    Bf = F(B).astype(np.float32)
    S = np.zeros((xa.shape[0], Bf.shape[0]), dtype=np.float32)
    for c in range(Bf.shape[1]):
        S = S + xa[:, c:c + 1] * Bf[None, :, c]
    return S


def check_fold_group(gpu_rows, ora_rows, base_rows, ora_d, ora_xa, gpu_xa, B, scale):
    """All routed rows of one adapter table entry: [R, n_out] BF16 folded segments of
    the GPU and the oracle, the original base values, the oracle's deltas and both
    xa [R, max_rank]. Returns (bit-exact count, total, largest ulp distance, values
    beyond one ulp)."""
    gpu_rows, ora_rows = np.atleast_2d(gpu_rows), np.atleast_2d(ora_rows)
    R = gpu_rows.shape[0]
    if R == 0:
        return 0, 0, 0, 0
    # fold: the GPU value must be the fold of a delta its own xa allows
    S = expand_oracle_order(gpu_xa, B).astype(np.float64)
    mag = np.abs(F(gpu_xa).astype(np.float64)) @ np.abs(F(B).astype(np.float64)).T
    delta = 2.0 * gamma(B.shape[1]) * mag
    f_lo = fold_bits(scale, bf16_of_f64(S - delta), base_rows)
    f_hi = fold_bits(scale, bf16_of_f64(S + delta), base_rows)
    lo = np.minimum(F(f_lo).astype(np.float64), F(f_hi).astype(np.float64))
    hi = np.maximum(F(f_lo).astype(np.float64), F(f_hi).astype(np.float64))
    g = F(gpu_rows).astype(np.float64)
    bad = ~((g >= lo) & (g <= hi))
    if bad.any():
        r, j = map(int, np.argwhere(bad)[0])
        raise AssertionError(f"fold[{r},{j}] gpu {g[r, j]!r} is not the fold of its own xa: "
                             f"allowed [{lo[r, j]!r}, {hi[r, j]!r}] (oracle {F(ora_rows)[r, j]!r})")
    # stated rule: one ulp, beyond it only where xa or the delta flipped
    dist = ulp_distance(gpu_rows, ora_rows)
    beyond = dist > 1
    if beyond.any():
        xa_flip = np.any(gpu_xa != ora_xa, axis=1)[:, None]
        d_flip = np.zeros_like(beyond)
        for step in (-1, 1):   # the oracle's fold with its delta one BF16 step away
            d_alt = (ora_d.astype(np.int64) + np.where(ora_d & 0x8000, -step, step)).astype(np.uint16)
            d_flip |= fold_bits(scale, d_alt, base_rows) == gpu_rows
        unexplained = beyond & ~(xa_flip | d_flip)
        if unexplained.any():
            r, j = map(int, np.argwhere(unexplained)[0])
            raise AssertionError(f"fold[{r},{j}] gpu {g[r, j]!r} oracle {F(ora_rows)[r, j]!r}: "
                                 f"{int(dist[r, j])} ulps with no xa or delta flip")
    return (int(np.sum(gpu_rows == ora_rows)), int(gpu_rows.size), int(dist.max()),
            int(beyond.sum()))


def _fold_groups(groups, stats):
    """groups: {table: [(gpu_row, ora_row, base_row, ora_d, ora_xa, gpu_xa), ...]} with the
    table's (B, scale) in groups[table].meta. Accumulates into stats."""
    for (B, scale), items in groups.values():
        cols = list(zip(*items))
        e, t, dmax, beyond = check_fold_group(*(np.stack(c) for c in cols), B, scale)
        stats["exact"] += e
        stats["total"] += t
        stats["max_ulps"] = max(stats["max_ulps"], dmax)
        stats["beyond_1ulp"] += beyond


def _finish(stats, xa_exact, xa_tot, xa_max, min_exact):
    n_exact, n_tot = stats["exact"], stats["total"]
    if n_tot:
        assert n_exact / n_tot >= min_exact, f"only {n_exact}/{n_tot} folded values bit-exact"
    if xa_tot:
        assert xa_exact / xa_tot >= min_exact, f"only {xa_exact}/{xa_tot} xa values bit-exact"
    return dict(exact=n_exact, total=n_tot, xa_exact=xa_exact, xa_total=xa_tot,
                max_ulps=stats["max_ulps"], xa_max_ulps=xa_max, beyond_1ulp=stats["beyond_1ulp"])


def _new_stats():
    return dict(exact=0, total=0, max_ulps=0, beyond_1ulp=0)


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
    xa_exact = xa_tot = xa_max = 0
    groups = {}
    for i, s in routed:
        e, m = check_xa(gpu_xa[i], ora_xa[i], wl.x[i, :wl.k_in], wl.a_pool[s])
        xa_exact, xa_tot, xa_max = xa_exact + e, xa_tot + wl.max_rank, max(xa_max, m)
        groups.setdefault(s, ((wl.b_pool[s], wl.scale[s]), []))[1].append(
            (gpu_out[i, seg], ora_out[i, seg], wl.out_buf[i, seg], ora_d[i], ora_xa[i], gpu_xa[i]))
    stats = _new_stats()
    _fold_groups(groups, stats)
    res = _finish(stats, xa_exact, xa_tot, xa_max, min_exact)
    res["rows"] = len(routed)
    return res


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
    xa_exact = xa_tot = xa_max = 0
    groups = {}
    for r, idx in routes:
        # the xa of row r lives in its window's buffer, at the local row
        w = next(k for k, (lo, hi) in enumerate(windows) if lo <= r < hi)
        lr = r - windows[w][0]
        gx, ox = gpu_xas[w][lr], ora_xas[w][lr]
        xrow = wl.x[wl.sorted_token_ids[r]] if wl.x_gather else wl.x[r]
        e, m = check_xa(gx, ox, xrow, wl.a_pool[idx])
        xa_exact, xa_tot, xa_max = xa_exact + e, xa_tot + wl.max_rank, max(xa_max, m)
        groups.setdefault(idx, ((wl.b_pool[idx], wl.scale[idx]), []))[1].append(
            (gpu_out[r], ora_out[r], wl.out_buf[r], ora_d[r], ox, gx))
    stats = _new_stats()
    _fold_groups(groups, stats)
    res = _finish(stats, xa_exact, xa_tot, xa_max, min_exact)
    res["rows"] = len(routes)
    return res


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
    xa_exact = xa_tot = xa_max = 0
    groups = {}
    for r, idx in routes:
        e, m = check_xa(gpu_xa[r], ora_xa[r], wl.x[r], wl.a_pool[idx])
        xa_exact, xa_tot, xa_max = xa_exact + e, xa_tot + wl.max_rank, max(xa_max, m)
        groups.setdefault(idx, ((wl.b_pool[idx], wl.scale[idx]), []))[1].append(
            (gpu_out[r], ora_out[r], wl.out_buf[r], ora_d[r], ora_xa[r], gpu_xa[r]))
    stats = _new_stats()
    _fold_groups(groups, stats)
    res = _finish(stats, xa_exact, xa_tot, xa_max, min_exact)
    res["rows"] = len(routes)
    return res


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
