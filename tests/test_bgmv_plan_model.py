"""A CPU model of the routed fold kernel's planner (`lora_bgmv_fold_kernel`).

The launcher sizes a static grid from host integers alone, so that a call
captured once replays with new routing ("Function apply_lora_bgmv", GRAPH-SAFE
paragraph): rows / rt + min(rows, max_loras) clusters, each owning one unit, a
tile of at most rt rows of one slot. Units are numbered either directly (unit s < max_loras is tile 0
of slot s, the units after them the further tiles of the slots in slot order)
or slot by slot (the tiles of the slots with rows, in slot order). A unit takes
the rows of its slot in ascending order, ranks [tile * rt, tile * rt + rt).

This file restates that numbering with the launcher's own geometry (rt, the
numbering and the grid, from `lora_launch_geometry`) and checks, for the
benchmarked routings and adversarial ones (all rows on one slot, every slot
one row past a tile, more slots than rows, slots out of range, the largest
batch), that every routed row is folded exactly once, by a unit of its own
slot, and that no unit is left without a (slot, tile) that a routing can need:
the grid bound covers the tiles of every routing of that many rows.

It is a restatement, not the kernel: the GPU tests compare the kernel's folds
with the oracle on routings of these kinds.
"""
from __future__ import annotations

import os

import numpy as np
import pytest

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W

MAX_ROWS = 8192      # LORA_MAX_ROWS
MAX_LORAS = 4096     # LORA_MAX_LORAS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    """The launcher's geometry comes from the library's host code (no GPU needed)."""
    if not os.path.exists(L.LIB_PATH):
        from gather_lora_gb300 import build
        build.build()
    L.load()


def plan(slots, max_loras, rt, direct, clusters, mutant=None):
    """{row: (unit, slot)} of the rows the grid's units fold."""
    slots = np.asarray(slots, dtype=np.int64)
    valid = (slots >= 0) & (slots < max_loras)
    cnt = np.bincount(slots[valid], minlength=max_loras)
    rows_of = {s: np.nonzero(slots == s)[0] for s in np.nonzero(cnt)[0]}
    t0 = 1 if direct else 0
    tiles = np.maximum(0, -(-cnt // rt) - t0)
    if mutant == "tiles_floor":
        tiles = np.maximum(0, cnt // rt - t0)
    start = np.concatenate([[0], np.cumsum(tiles)])          # first unit (after the direct ones) of each slot
    folded = {}
    for unit in range(clusters):
        if direct and unit < max_loras:
            slot, tile = unit, 0
        else:
            v = unit - max_loras if direct else unit
            s = int(np.searchsorted(start, v, side="right") - 1)
            if s >= max_loras or not (start[s] <= v < start[s] + tiles[s]):
                continue                                     # no (slot, tile): the unit leaves
            slot, tile = s, t0 + v - int(start[s])
        rows = rows_of.get(slot)
        if rows is None:
            continue
        mine = rows[tile * rt: tile * rt + rt]
        assert len(mine) <= rt
        for r in mine:
            r = int(r)
            assert r not in folded, f"row {r} folded by units {folded[r][0]} and {unit}"
            folded[r] = (unit, slot)
    return folded


def check(slots, max_loras, rt, direct, clusters, mutant=None):
    slots = np.asarray(slots)
    got = plan(slots, max_loras, rt, direct, clusters, mutant)
    want = {i: int(s) for i, s in enumerate(slots) if 0 <= s < max_loras}
    assert {r: s for r, (_, s) in got.items()} == want
    return len(want)


def geometry(kind, rows, max_loras, max_rank, k_in, n_out, maps=False):
    g = L.lora_launch_geometry(kind | (16 if maps else 0), rows, max_loras, max_rank, k_in, n_out)
    assert g["clusters"] == (rows // g["rows_per_tile"] + min(rows, max_loras) if rows > 0 else 0)
    return g["rows_per_tile"], g["direct"], g["clusters"]


@pytest.mark.parametrize("name,maps", [("decode_qproj_bgmv", False), ("qkv_kfold_bgmv", True),
                                       ("ffn_down_bgmv", True), ("ffn_down_bgmv", False)])
def test_benchmarked_routings(name, maps):
    wl = W.by_name(name)
    rt, direct, clusters = geometry(0, wl.n, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, maps)
    assert check(wl.seq_slot, wl.max_loras, rt, direct, clusters) > 0


def _gather_slots(wl):
    """Derived slot a * E + e of each flat row of the decode gather fold (-1: skipped)."""
    E = wl.num_experts
    tok = np.arange(wl.n_rows) // wl.top_k
    a = np.zeros(wl.n_rows, dtype=np.int64) if wl.row_adapter is None else np.asarray(wl.row_adapter)[tok]
    e = np.asarray(wl.indices, dtype=np.int64)
    ok = (e >= 0) & (e < E) & (a >= 0) & (a < wl.max_loras) & (tok < wl.num_tokens)
    return np.where(ok, a * E + e, -1)


@pytest.mark.parametrize("maps", [False, True])
def test_decode_gather_routing(maps):
    wl = W.by_name("moe_decode_gather")
    tables = wl.max_loras * wl.num_experts
    rt, direct, clusters = geometry(2, wl.n_rows, tables, wl.max_rank, wl.k_in, wl.n_out, maps)
    assert check(_gather_slots(wl), tables, rt, direct, clusters) > 0


def _adversarial(rng, n, max_loras, rt):
    """Routings that stress the grid bound and the numbering."""
    yield np.zeros(n, dtype=np.int64)                                   # every row on one slot
    yield np.full(n, max_loras - 1, dtype=np.int64)                     # on the last slot
    k = max(1, min(max_loras, n // (rt + 1)))                           # slots one row past a tile
    s = np.repeat(np.arange(k), rt + 1)[:n]
    yield np.concatenate([s, rng.integers(0, max_loras, n - len(s))]) if len(s) < n else s
    yield rng.permutation(np.arange(n) % max_loras)                     # as many slots as rows allow
    yield rng.integers(-1, max_loras + 2, n)                            # out-of-range slots skipped
    yield np.full(n, -1, dtype=np.int64)                                # nothing routed
    z = rng.zipf(1.1, n) - 1                                            # heavy head
    yield np.where(z < max_loras, z, -1)


SHAPES = [   # rows, max_loras, max_rank, k_in, n_out: direct and slot-by-slot numbering, tiny and largest
    (64, 32, 16, 4096, 4096),
    (256, 128, 64, 4096, 1024),
    (512, 64, 128, 12288, 4096),
    (17, 3, 8, 256, 256),
    (5, 40, 16, 128, 96),
    (1, 1, 16, 64, 64),
    (MAX_ROWS, MAX_LORAS, 16, 128, 96),
    (MAX_ROWS, 16, 32, 1024, 1024),
    (3000, 2999, 16, 512, 512),
]


@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_adversarial_routings_fold_every_row_once(shape):
    n, max_loras, max_rank, k_in, n_out = SHAPES[shape]
    rng = np.random.default_rng(700 + shape)
    for maps in ((False, True) if max_rank >= 32 else (False,)):
        rt, direct, clusters = geometry(0, n, max_loras, max_rank, k_in, n_out, maps)
        for slots in _adversarial(rng, n, max_loras, rt):
            check(slots, max_loras, rt, direct, clusters)
            # the other numbering over the same grid folds the same rows
            check(slots, max_loras, rt, 1 - direct if max_loras <= n else 0, clusters)


def test_grid_bound_is_tight_for_some_routing():
    """A routing that needs every unit of the grid exists (the bound is not loose
    by more than the empty direct units): max_loras slots, each with one row
    more than a multiple of the tile."""
    n, max_loras = 17 * 16, 16
    rt, direct, clusters = geometry(0, n, max_loras, 16, 256, 256)
    slots = np.repeat(np.arange(max_loras), n // max_loras)
    got = plan(slots, max_loras, rt, 0, clusters)
    used = {u for u, _ in got.values()}
    assert len(got) == n and len(used) == -(-(n // max_loras) // rt) * max_loras <= clusters


@pytest.mark.parametrize("mutant", ["tiles_floor"])
def test_a_planted_numbering_mistake_is_caught(mutant):
    rng = np.random.default_rng(5)
    rt, direct, clusters = geometry(0, 256, 128, 64, 4096, 1024, True)
    slots = next(x for i, x in enumerate(_adversarial(rng, 256, 128, rt)) if i == 2)
    check(slots, 128, rt, direct, clusters)
    with pytest.raises(AssertionError):
        check(slots, 128, rt, direct, clusters, mutant=mutant)


def test_single_adapter_rows_on_the_routed_engine():
    """lora_delta below the tensor-core size runs the routed engine with every row on slot 0."""
    for m in (1, 7, 16, 17, 255):
        rt, direct, clusters = geometry(0, m, 1, 16, 4096, 4096)
        assert check(np.zeros(m, dtype=np.int64), 1, rt, direct, clusters) == m
