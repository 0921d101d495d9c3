"""A CPU model of the MoE fold kernel's planner (`lora_moe_fold_kernel`).

The planner is index arithmetic over the routing arrays of a window
("Module moe_lora_grouped", moe_lora_grouped_down: rows sorted by expert, the
expert of a row from the offsets, the adapter from the token's row_adapter
entry, tables adapter-major). Each CTA b of a grid of G plans its own units
(one expert of the window and a chunk of `ac` adapters; units b, b + G, ...),
scans its units' rows in planning rounds of a bounded number of rows, numbers
each routed row within its (expert, adapter) group, makes the groups with rows
the round's runs and their rows positions, and folds the positions in passes of
kMaxRows, split into groups of at most gmax rows of one run.

This file restates that arithmetic step by step, with the kernel's constants
read from its sources, and checks for the routings of the MoE GPU tests and of
the benchmarked workloads, on the launcher's grid and on other grid sizes (the
kernel reads its grid size, so any G must work):

- every routed row (the skip rules of the fold: inside the window and the
  expert spans, a token in range where one is read, an adapter in range, a
  non-NULL table entry) is folded exactly once, in a group of its own expert
  and adapter, and nothing else is folded;
- every table the planner writes stays inside its shared-memory reservation:
  units per round, group counters, runs, positions, rows per thread and group
  starts per pass;
- every row, token and xa index the fold uses lies inside its buffer.

It is a restatement, not the kernel: the GPU tests compare the kernel's folds
with the oracle on the same routings.
"""
from __future__ import annotations

import math
import os
import re

import numpy as np
import pytest

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "gather_lora_gb300", "csrc")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    """The launcher's geometry comes from the library's host code (no GPU needed)."""
    if not os.path.exists(L.LIB_PATH):
        from gather_lora_gb300 import build
        build.build()
    L.load()


def _source(name):
    with open(os.path.join(CSRC, name)) as f:
        return f.read()


def _const(text, pattern):
    m = re.search(pattern, text)
    assert m, f"constant not found: {pattern}"
    return int(m.group(1))


_FT, _KC, _ABI = _source("fold_types.h"), _source("kernels.cu"), _source("abi.cpp")
MAX_DESC = _const(_FT, r"constexpr int kMoeMaxDesc = (\d+);")
ROUND_ROWS = _const(_FT, r"#define GLORA_MOE_ROUND_ROWS (\d+)")
MAX_ROWS = _const(_FT, r"constexpr int kMaxRows = (\d+);")
MAX_GROUP_ROWS = _const(_FT, r"constexpr int kMaxGroupRows = (\d+);")
MAX_BINS = _const(_FT, r"constexpr int kMoeMaxBins = (\d+);")
UNITS_PER_CTA = _const(_KC, r"#define GLORA_MOE_UNITS_PER_CTA (\d+)")
MAX_MY_UNITS = _const(_KC, r"constexpr int kMoeMaxMyUnits = (\d+);")
GMAX = min(_const(_ABI, r"#define GLORA_MOE_GROUP_ROWS (\d+)"), MAX_GROUP_ROWS)
THREADS = {cfg: 32 * (_const(_FT, rf"struct MoeShape<{cfg}> {{ static constexpr int cw = (\d+)")
                      + _const(_FT, rf"struct MoeShape<{cfg}> {{ static constexpr int cw = \d+, pw = (\d+)"))
           for cfg in (0, 1)}


def test_constants_were_read():
    assert MAX_DESC > 0 and ROUND_ROWS >= MAX_DESC and MAX_ROWS == 64 and GMAX >= 1
    assert UNITS_PER_CTA >= 1 and MAX_MY_UNITS >= 1 and min(THREADS.values()) >= MAX_DESC
    # a group counter is packed with its run as (run << 16) | 1, a run index held in a short
    assert MAX_DESC < (1 << 15)


def _expert_of(offs, E, r):
    """Vector form of the kernel's binary search over [0, E) (the same halving, so
    the same answer on offsets out of order): the e with offs[e] <= r < offs[e+1]
    it lands on, -1 outside [offs[0], offs[E]) or when it lands outside a span."""
    r = np.asarray(r, dtype=np.int64)
    lo = np.zeros(r.shape, dtype=np.int64)
    hi = np.full(r.shape, E, dtype=np.int64)
    while True:
        open_ = hi - lo > 1
        if not open_.any():
            break
        mid = (lo + hi) >> 1
        go = open_ & (offs[np.minimum(mid, E)] <= r)
        lo = np.where(go, mid, lo)
        hi = np.where(open_ & ~go, mid, hi)
    ok = (r >= offs[0]) & (r < offs[E]) & (offs[lo] <= r) & (r < offs[lo + 1])
    return np.where(ok, lo, -1)


def plan_window(wl, lo, hi, G, use_row_adapter=True, cfg=0, mutant=None):
    """All CTAs' plans of window [lo, hi) on a grid of G CTAs.

    Returns {row: (cta, expert, adapter)} of the folded rows and checks every
    table bound on the way. `mutant` plants a mistake (tests of the checks)."""
    E = wl.num_experts
    ra = wl.row_adapter if use_row_adapter else None
    A = wl.max_loras if ra is not None else 1
    need_token = ra is not None or wl.x_gather
    offs = np.asarray(wl.expert_offsets, dtype=np.int64)
    sti = np.asarray(wl.sorted_token_ids, dtype=np.int64)
    present = np.asarray(wl.present)
    rows_per_thread = -(-ROUND_ROWS // THREADS[cfg])
    folded = {}
    lo_w, hi_w = max(lo, int(offs[0])), min(hi, int(offs[E]))
    if hi_w <= lo_w:
        return folded
    e_first, e_last = int(_expert_of(offs, E, lo_w)), int(_expert_of(offs, E, hi_w - 1))
    if e_first < 0 or e_last < e_first:
        e_first, e_last = 0, E - 1
    E_w = e_last - e_first + 1
    n_chunks0 = min(A, max(1, (UNITS_PER_CTA * G) // E_w))
    ac = -(-A // n_chunks0)
    n_chunks = -(-A // ac)
    n_units = E_w * n_chunks
    assert n_units <= E * A <= MAX_BINS
    round_rows = MAX_DESC if ac > MAX_DESC else ROUND_ROWS
    assert round_rows <= rows_per_thread * THREADS[cfg]
    for b in range(G):
        my_units = -(-(n_units - b) // G) if n_units > b else 0
        if mutant == "units_floor":
            my_units = (n_units - b) // G if n_units > b else 0
        v0 = row_cur = 0
        while v0 < my_units:
            v1 = min(my_units, v0 + min(MAX_MY_UNITS, max(1, MAX_DESC // ac)))
            nu = v1 - v0
            assert 1 <= nu <= MAX_MY_UNITS and nu <= THREADS[cfg]
            # group counters: reserved for max(kMoeMaxDesc, adapters) groups
            assert nu * ac <= max(MAX_DESC, A)
            u = b + (v0 + np.arange(nu)) * G
            ue = e_first + u // n_chunks
            assert ue.min() >= 0 and ue.max() < E
            ua0 = (u % n_chunks) * ac
            ulo = np.maximum(offs[ue], lo_w)
            cnt = np.maximum(0, np.minimum(offs[ue + 1], hi_w) - ulo)
            row0 = np.concatenate([[0], np.cumsum(cnt)])
            rows_all = int(row0[nu])
            row_end = min(rows_all, row_cur + round_rows)
            q = np.arange(row_cur, row_end)
            v = np.searchsorted(row0, q, side="right") - 1
            r = ulo[v] + (q - row0[v])
            assert len(r) == 0 or (r.min() >= lo_w and r.max() < hi_w)
            if need_token:
                t = sti[r]
                tok_ok = (t >= 0) & (t < wl.num_tokens)
            else:
                t = np.zeros_like(r)
                tok_ok = np.ones(len(r), dtype=bool)
            a = np.zeros_like(r)
            if ra is not None:
                a[tok_ok] = np.asarray(ra, dtype=np.int64)[t[tok_ok]]
            mine = tok_ok & (_expert_of(offs, E, r) == ue[v]) & (a >= ua0[v]) & (a < np.minimum(A, ua0[v] + ac))
            grp = v[mine] * ac + (a[mine] - ua0[v[mine]])
            bcnt = np.bincount(grp, minlength=nu * ac)
            has = np.nonzero(bcnt)[0]
            nd, npos = len(has), int(bcnt.sum())
            assert nd <= MAX_DESC and npos <= ROUND_ROWS, (nd, npos)
            # runs in group order; a run's positions follow the groups before it
            pos0 = np.concatenate([[0], np.cumsum(bcnt)])[has]
            run_of_group = np.full(nu * ac, -1)
            run_of_group[has] = np.arange(nd)
            desc_e = ue[has // ac]
            desc_a = ua0[has // ac] + has % ac
            order = np.argsort(grp, kind="stable")        # any order inside a group is valid
            pos_row = r[mine][order]
            pos_tok = (t if wl.x_gather else r)[mine][order]
            pos_desc = run_of_group[grp[order]]
            assert np.all(pos_tok >= 0) and np.all(pos_tok < (wl.num_tokens if wl.x_gather else wl.te))
            # passes of kMaxRows positions, groups of at most gmax rows of one run
            for P0 in range(0, npos, MAX_ROWS):
                P = min(MAX_ROWS, npos - P0)
                qs = np.arange(P0, P0 + P)
                k = pos_desc[qs]
                first = pos0[k] if mutant == "group_start" else np.maximum(P0, pos0[k])
                start = ((qs - first) % GMAX) == 0
                assert start[0]
                starts = np.nonzero(start)[0]
                assert len(starts) <= MAX_ROWS
                bounds = np.append(starts, P)
                for g0, g1 in zip(bounds[:-1], bounds[1:]):
                    d = int(k[g0])
                    assert g1 - g0 <= GMAX and np.all(k[g0:g1] == d)
                    e, ad = int(desc_e[d]), int(desc_a[d])
                    if not present[ad * E + e]:
                        continue                           # a NULL entry: the group is dropped
                    for row in pos_row[qs[g0:g1]]:
                        row = int(row)
                        assert row not in folded, f"row {row} folded twice"
                        assert 0 <= row - lo < hi - lo    # its xa row
                        folded[row] = (b, e, ad)
            if row_end >= rows_all:
                v0, row_cur = v1, 0
            else:
                row_cur = row_end + (mutant == "round_skip")
    return folded


def routed_rows(wl, lo, hi, use_row_adapter=True):
    """{row: (expert, adapter)} of the rows the fold must fold, by the skip rules."""
    E = wl.num_experts
    ra = wl.row_adapter if use_row_adapter else None
    A = wl.max_loras if ra is not None else 1
    out = {}
    for r in range(lo, hi):
        e = int(_expert_of(np.asarray(wl.expert_offsets, dtype=np.int64), E, r))
        if e < 0:
            continue
        a = 0
        if ra is not None or wl.x_gather:
            t = int(wl.sorted_token_ids[r])
            if not 0 <= t < wl.num_tokens:
                continue
            if ra is not None:
                a = int(ra[t])
        if 0 <= a < A and wl.present[a * E + e]:
            out[r] = (e, a)
    return out


def launcher_grid(wl, lo, hi, use_row_adapter=True):
    """The launcher's grid for this window (one CTA set per SM of a 152-SM GPU)."""
    A = wl.max_loras if (use_row_adapter and wl.row_adapter is not None) else 1
    g = L.lora_launch_geometry(1, hi - lo, A, wl.max_rank, wl.k_in, wl.n_out)
    return int(g["clusters"]), int(g["direct"])


def check_routing(wl, windows, use_row_adapter=True, grids=(1, 5, 152, 304), mutant=None, exact=True):
    total = 0
    for lo, hi in windows:
        want = routed_rows(wl, lo, hi, use_row_adapter)
        G0, cfg = launcher_grid(wl, lo, hi, use_row_adapter) if hi > lo else (1, 0)
        assert 1 <= G0 <= 152 * 2 and G0 <= max(1, math.ceil((hi - lo) / 16))
        for G in sorted({G0, *grids}):
            got = {r: ea[1:] for r, ea in plan_window(wl, lo, hi, G, use_row_adapter, cfg, mutant).items()}
            if exact:
                assert got == want, (lo, hi, G)
            else:   # bad data: whatever is folded is folded once, as a routed row of its own pair
                assert all(want.get(r) == ea for r, ea in got.items()), (lo, hi, G)
        total += len(want)
    return total


SMALL = [   # the random MoE cases of the GPU tests
    (24, 3, 6, 32, 40, 3, 8, 40, True, 1.0),
    (300, 4, 16, 136, 264, 5, 16, 500, True, 0.7),
    (512, 8, 64, 768, 2048, 4, 16, 1000, False, 1.0),
    (200, 2, 8, 520, 1032, 2, 24, 130, True, 1.0),
    (64, 8, 128, 1024, 512, 3, 64, 4096, True, 0.9),
    (128, 1, 4, 2048, 1024, 2, 128, 256, True, 1.0),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_plan_of_the_random_cases(case):
    tok, k, E, k_in, n_out, Lr, R, cap, use_ra, pf = SMALL[case]
    wl = W.make_moe(f"moe{case}", num_tokens=tok, top_k=k, num_experts=E, k_in=k_in, n_out=n_out,
                    max_loras=Lr, max_rank=R, rank=R, alpha=16.0, adapter_base_frac=0.25,
                    cap=cap, seed=200 + case, use_row_adapter=use_ra, present_frac=pf)
    assert check_routing(wl, wl.windows(), use_ra) > 0


@pytest.mark.parametrize("name", ["moe_down_fold", "moe_gateup_fold"])
def test_plan_of_the_benchmarked_workloads(name):
    """The four windows of 4096 sorted rows, one call over all rows, and windows of 1000 and 300."""
    wl = W.by_name(name)
    n = check_routing(wl, wl.windows(), grids=(152,))
    assert n > 10000
    assert check_routing(wl, [(0, wl.te)], grids=(152, 304)) == n
    for cap in (1000, 300):
        ws = [(lo, min(lo + cap, wl.te)) for lo in range(0, wl.te, cap)]
        assert check_routing(wl, ws, grids=()) == n


def test_plan_of_skewed_groups():
    """One adapter takes 90% of the tokens: groups far larger than gmax, spanning passes."""
    wl = W.make_moe("moe_skew", num_tokens=1024, top_k=4, num_experts=8, k_in=256, n_out=512,
                    max_loras=16, max_rank=16, rank=16, alpha=16.0, adapter_base_frac=0.0,
                    cap=4096, seed=321)
    rng = np.random.default_rng(321)
    wl.row_adapter = np.where(rng.random(wl.num_tokens) < 0.9, 0,
                              rng.integers(1, 16, wl.num_tokens)).astype(np.int32)
    for cap in (4096, 1000, 300):
        check_routing(wl, [(lo, min(lo + cap, wl.te)) for lo in range(0, wl.te, cap)])


def test_plan_over_several_rounds():
    """200000 sorted rows in one window: each CTA takes several planning rounds."""
    wl = W.make_moe("moe_rounds", num_tokens=25000, top_k=8, num_experts=16, k_in=16, n_out=24,
                    max_loras=4, max_rank=8, rank=8, alpha=16.0, adapter_base_frac=0.1,
                    cap=200000, seed=333)
    n = check_routing(wl, wl.windows(), grids=(152,))
    assert n > 152 * ROUND_ROWS


def test_plan_with_rows_outside_spans_bad_tokens_and_an_empty_window():
    wl = W.make_moe("moe_bad", num_tokens=40, top_k=4, num_experts=8, k_in=64, n_out=64,
                    max_loras=2, max_rank=16, rank=16, alpha=16.0, adapter_base_frac=0.0,
                    cap=1000, seed=300)
    wl.expert_offsets = wl.expert_offsets.copy()
    wl.expert_offsets[0] = min(9, int(wl.expert_offsets[1]))
    wl.sorted_token_ids = wl.sorted_token_ids.copy()
    wl.sorted_token_ids[20] = wl.num_tokens + 5
    wl.sorted_token_ids[21] = -3
    ra = wl.row_adapter.copy()
    ra[wl.sorted_token_ids[30]] = 7
    wl.row_adapter = ra
    check_routing(wl, [(0, 50), (50, 50), (50, wl.te)])


@pytest.mark.parametrize("use_ra", [True, False])
def test_plan_of_the_gateup_form(use_ra):
    wl = W.make_moe("gateup_small", num_tokens=150, top_k=4, num_experts=12, k_in=264,
                    n_out=136, max_loras=3, max_rank=16, rank=16, alpha=16.0,
                    adapter_base_frac=0.25, cap=230, seed=410 + int(use_ra),
                    use_row_adapter=use_ra, present_frac=0.8, x_gather=True)
    wl.sorted_token_ids = wl.sorted_token_ids.copy()
    wl.sorted_token_ids[5] = wl.num_tokens + 1
    wl.sorted_token_ids[9] = -2
    check_routing(wl, wl.windows(), use_ra)


def test_plan_with_more_adapters_than_a_round_holds_runs():
    """One expert, 4096 adapters: a unit's chunk alone has more groups than a
    round holds runs, so a round scans at most kMoeMaxDesc rows."""
    wl = W.make_moe("wide", num_tokens=3000, top_k=1, num_experts=1, k_in=768, n_out=256,
                    max_loras=4096, max_rank=8, rank=8, alpha=16.0, adapter_base_frac=0.0,
                    cap=3000, seed=5)
    check_routing(wl, wl.windows(), grids=(1, 152))


def test_plan_with_many_experts():
    wl = W.make_moe("limits_moe", num_tokens=512, top_k=4, num_experts=1024, k_in=128, n_out=256,
                    max_loras=4, max_rank=16, rank=16, alpha=32.0, adapter_base_frac=0.2,
                    cap=1024, seed=902)
    check_routing(wl, wl.windows())


def test_plan_with_expert_offsets_out_of_order():
    """Bad device data: offsets that decrease make spans overlap or vanish. Each
    row is folded at most once (by the unit of the expert the binary search
    finds), and every index stays in bounds."""
    wl = W.make_moe("moe_disorder", num_tokens=300, top_k=4, num_experts=16, k_in=136, n_out=264,
                    max_loras=5, max_rank=16, rank=16, alpha=16.0, adapter_base_frac=0.25,
                    cap=500, seed=203)
    rng = np.random.default_rng(17)
    for _ in range(4):
        offs = wl.expert_offsets.copy()
        offs[1:-1] = rng.integers(0, wl.te, size=len(offs) - 2)     # inner offsets scrambled
        wl.expert_offsets = offs.astype(np.int32)
        check_routing(wl, wl.windows(), grids=(1, 7, 152), exact=False)


@pytest.mark.parametrize("mutant", ["units_floor", "round_skip", "group_start"])
def test_planted_planner_mistakes_are_caught(mutant):
    """The checks are not vacuous: a CTA's unit count rounded down, a row skipped
    between planning rounds, or fold groups counted from the run's start instead
    of the pass's each fail them."""
    wl = W.make_moe("moe_skew", num_tokens=1024, top_k=4, num_experts=8, k_in=256, n_out=512,
                    max_loras=16, max_rank=16, rank=16, alpha=16.0, adapter_base_frac=0.0,
                    cap=4096, seed=321)
    rng = np.random.default_rng(321)
    wl.row_adapter = np.where(rng.random(wl.num_tokens) < 0.9, 0,
                              rng.integers(1, 16, wl.num_tokens)).astype(np.int32)
    check_routing(wl, wl.windows(), grids=(1, 7))
    with pytest.raises(AssertionError):
        check_routing(wl, wl.windows(), grids=(1, 7), mutant=mutant)
