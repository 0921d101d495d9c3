"""CUDA lora_moe_grouped_fold against the CPU oracle (-m gpu), through the C ABI.

Covers the MoE down-projection workload and its gate/up form (token-major x
gathered per sorted row) at full size over their four windows of 4096 sorted
rows (every element compared), window invariance (one full-window call == the
windowed calls, bit for bit), small random routings with ragged windows, NULL
row_adapter, absent (adapter, expert) entries, rows outside the expert spans,
bad tokens, an empty window, and graph replay with new routing.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W
from gpu_util import gpu_moe, oracle_moe, require_gpu, to_u16
from parity import compare_moe, moe_routes

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    L.lora_read_device_status(clear=True)


def _routes_all(wl, windows, **kw):
    r = []
    for lo, hi in windows:
        r += moe_routes(wl, lo, hi, **kw)
    return r


def test_moe_down_workload_parity():
    wl = W.moe_down_fold()
    windows = wl.windows()
    assert windows == [(0, 4096), (4096, 8192), (8192, 12288), (12288, 16384)]
    g_out, g_xas = gpu_moe(wl, windows)
    o_out, o_xas, o_d = oracle_moe(wl, windows)
    st = compare_moe(wl, windows, g_out, o_out, g_xas, o_xas, o_d, _routes_all(wl, windows))
    assert st["rows"] > 10000
    assert L.lora_read_device_status(clear=True) == 0


def test_moe_full_window_equals_windowed():
    wl = W.moe_down_fold()
    windows = wl.windows()
    g_out, g_xas = gpu_moe(wl, windows)
    f_out, (f_xa,) = gpu_moe(wl, [(0, wl.te)])
    assert np.array_equal(g_out, f_out)
    assert np.array_equal(np.concatenate(g_xas), f_xa)


SMALL = [
    # tokens, top_k, experts, k_in, n_out, loras, rank, cap, row_adapter, present_frac
    (24, 3, 6, 32, 40, 3, 8, 40, True, 1.0),
    (300, 4, 16, 136, 264, 5, 16, 500, True, 0.7),
    (512, 8, 64, 768, 2048, 4, 16, 1000, False, 1.0),
    (200, 2, 8, 520, 1032, 2, 24, 130, True, 1.0),       # ragged tails, few experts -> large groups
    (64, 8, 128, 1024, 512, 3, 64, 4096, True, 0.9),
    (128, 1, 4, 2048, 1024, 2, 128, 256, True, 1.0),     # groups of > 32 rows at rank 128
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_moe_random(case):
    tok, k, E, k_in, n_out, Lr, R, cap, use_ra, pf = SMALL[case]
    wl = W.make_moe(f"moe{case}", num_tokens=tok, top_k=k, num_experts=E, k_in=k_in, n_out=n_out,
                    max_loras=Lr, max_rank=R, rank=R, alpha=16.0, adapter_base_frac=0.25,
                    cap=cap, seed=200 + case, use_row_adapter=use_ra, present_frac=pf)
    windows = wl.windows()
    g_out, g_xas = gpu_moe(wl, windows, use_row_adapter=use_ra)
    o_out, o_xas, o_d = oracle_moe(wl, windows, use_row_adapter=use_ra)
    routes = _routes_all(wl, windows, row_adapter=wl.row_adapter if use_ra else None)
    compare_moe(wl, windows, g_out, o_out, g_xas, o_xas, o_d, routes, min_exact=0.97)


def _skewed(seed):
    """One adapter takes 90% of the tokens: its (expert, adapter) groups are far
    larger than the 16 rows of one fold group, and a CTA's share of them spans
    several passes of 64 rows."""
    wl = W.make_moe("moe_skew", num_tokens=1024, top_k=4, num_experts=8, k_in=256, n_out=512,
                    max_loras=16, max_rank=16, rank=16, alpha=16.0, adapter_base_frac=0.0,
                    cap=4096, seed=seed)
    rng = np.random.default_rng(seed)
    wl.row_adapter = np.where(rng.random(wl.num_tokens) < 0.9, 0,
                              rng.integers(1, 16, wl.num_tokens)).astype(np.int32)
    return wl


def test_moe_large_groups_and_other_windows():
    wl = _skewed(321)
    assert wl.te == 4096
    windows = [(0, 4096)]
    g_out, g_xas = gpu_moe(wl, windows)
    o_out, o_xas, o_d = oracle_moe(wl, windows)
    compare_moe(wl, windows, g_out, o_out, g_xas, o_xas, o_d, _routes_all(wl, windows))
    # windows of 1000 and 300 rows (other grids, other CTA shares) give the same bits
    for cap in (1000, 300):
        ws = [(lo, min(lo + cap, wl.te)) for lo in range(0, wl.te, cap)]
        w_out, w_xas = gpu_moe(wl, ws)
        assert np.array_equal(w_out, g_out)
        assert np.array_equal(np.concatenate(w_xas), g_xas[0])


@pytest.mark.parametrize("name", ["moe_down_fold", "moe_gateup_fold"])
def test_moe_workload_windows_of_any_size_give_the_same_bits(name):
    """The benchmarked MoE workloads: windows of 4096 (as configured), 1000 and 300
    sorted rows and one call over all rows fold every row to the same bits (the
    grid and each CTA's share of the rows change with the window; a row's
    arithmetic does not)."""
    wl = W.by_name(name)
    ref_out, ref_xa = gpu_moe(wl, [(0, wl.te)])
    for cap in (4096, 1000, 300):
        ws = [(lo, min(lo + cap, wl.te)) for lo in range(0, wl.te, cap)]
        w_out, w_xas = gpu_moe(wl, ws)
        assert np.array_equal(w_out, ref_out), cap
        assert np.array_equal(np.concatenate(w_xas), ref_xa[0]), cap


def test_moe_window_with_more_rows_than_one_planning_round():
    """200000 sorted rows in one window: each of the 152 CTAs gets more rows than
    one planning round holds (1024), and the window has more rows than the group
    keys kept in shared memory (the rest are recomputed from the routing data)."""
    wl = W.make_moe("moe_rounds", num_tokens=25000, top_k=8, num_experts=16, k_in=16, n_out=24,
                    max_loras=4, max_rank=8, rank=8, alpha=16.0, adapter_base_frac=0.1,
                    cap=200000, seed=333)
    assert wl.te == 200000
    windows = wl.windows()
    g_out, g_xas = gpu_moe(wl, windows)
    o_out, o_xas, o_d = oracle_moe(wl, windows)
    st = compare_moe(wl, windows, g_out, o_out, g_xas, o_xas, o_d, _routes_all(wl, windows))
    assert st["rows"] > 152 * 1024
    assert L.lora_read_device_status(clear=True) == 0


def test_moe_rows_outside_spans_bad_tokens_and_empty_window():
    wl = W.make_moe("moe_bad", num_tokens=40, top_k=4, num_experts=8, k_in=64, n_out=64,
                    max_loras=2, max_rank=16, rank=16, alpha=16.0, adapter_base_frac=0.0,
                    cap=1000, seed=300)
    wl.expert_offsets = wl.expert_offsets.copy()
    wl.expert_offsets[0] = min(9, int(wl.expert_offsets[1]))   # rows before expert 0's span
    wl.sorted_token_ids = wl.sorted_token_ids.copy()
    wl.sorted_token_ids[20] = wl.num_tokens + 5   # token out of range
    wl.sorted_token_ids[21] = -3
    ra = wl.row_adapter.copy()
    ra[wl.sorted_token_ids[30]] = 7               # adapter >= max_loras
    wl.row_adapter = ra
    windows = [(0, 50), (50, 50), (50, wl.te)]
    g_out, g_xas = gpu_moe(wl, windows)
    o_out, o_xas, o_d = oracle_moe(wl, windows)
    routes = _routes_all(wl, windows)
    compare_moe(wl, windows, g_out, o_out, g_xas, o_xas, o_d, routes)
    for r in list(range(int(wl.expert_offsets[0]))) + [20, 21]:
        assert np.array_equal(g_out[r], wl.out_buf[r])


def test_moe_graph_replay_with_new_row_adapter():
    wl = W.make_moe("moe_graph", num_tokens=512, top_k=8, num_experts=32, k_in=768, n_out=2048,
                    max_loras=8, max_rank=16, rank=16, alpha=32.0, adapter_base_frac=0.2,
                    cap=1024, seed=301)
    windows = wl.windows()
    d = W.moe_to_device(wl, xa_rows=wl.cap)
    xa_w = torch.zeros((len(windows), wl.cap, wl.max_rank), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()

    def run():
        for w, (lo, hi) in enumerate(windows):
            L.lora_moe_grouped_fold(d.x, wl.k_in, d.out_buf, wl.n_out, d.expert_offsets,
                                    wl.num_experts, d.sorted_token_ids, wl.te, d.row_adapter,
                                    wl.num_tokens, lo, hi, d.a_table, d.b_table, d.scale,
                                    wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=xa_w[w],
                                    stream=s)

    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        run()
    rng = np.random.default_rng(9)
    for _ in range(2):
        ra = rng.integers(0, wl.max_loras, size=wl.num_tokens).astype(np.int32)
        ra[rng.random(wl.num_tokens) < 0.3] = -1
        wl.row_adapter = ra
        wl.out_buf = W.to_bf16_bits(rng.standard_normal(wl.out_buf.shape).astype(np.float32))
        d.row_adapter.copy_(torch.from_numpy(ra))
        d.out_buf.copy_(torch.from_numpy(wl.out_buf.view(np.int16)))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        o_out, o_xas, o_d = oracle_moe(wl, windows)
        routes = _routes_all(wl, windows)
        g_xas = [to_u16(xa_w[w])[: hi - lo] for w, (lo, hi) in enumerate(windows)]
        compare_moe(wl, windows, to_u16(d.out_buf), o_out, g_xas, o_xas, o_d, routes)


# ---------------------------------------------------------- gate/up (x_gather)
def test_moe_gateup_workload_parity():
    wl = W.moe_gateup_fold()
    assert wl.x_gather and wl.x.shape == (wl.num_tokens, wl.k_in)
    windows = wl.windows()
    g_out, g_xas = gpu_moe(wl, windows)
    o_out, o_xas, o_d = oracle_moe(wl, windows)
    st = compare_moe(wl, windows, g_out, o_out, g_xas, o_xas, o_d, _routes_all(wl, windows))
    assert st["rows"] > 10000
    assert L.lora_read_device_status(clear=True) == 0


def test_moe_gateup_full_window_equals_windowed():
    wl = W.moe_gateup_fold()
    windows = wl.windows()
    g_out, g_xas = gpu_moe(wl, windows)
    f_out, (f_xa,) = gpu_moe(wl, [(0, wl.te)])
    assert np.array_equal(g_out, f_out)
    assert np.array_equal(np.concatenate(g_xas), f_xa)


@pytest.mark.parametrize("use_ra", [True, False])
def test_moe_gateup_random_and_bad_tokens(use_ra):
    wl = W.make_moe("gateup_small", num_tokens=150, top_k=4, num_experts=12, k_in=264,
                    n_out=136, max_loras=3, max_rank=16, rank=16, alpha=16.0,
                    adapter_base_frac=0.25, cap=230, seed=410 + int(use_ra),
                    use_row_adapter=use_ra, present_frac=0.8, x_gather=True)
    wl.sorted_token_ids = wl.sorted_token_ids.copy()
    wl.sorted_token_ids[5] = wl.num_tokens + 1    # token out of range: row skipped
    wl.sorted_token_ids[9] = -2
    windows = wl.windows()
    g_out, g_xas = gpu_moe(wl, windows, use_row_adapter=use_ra)
    o_out, o_xas, o_d = oracle_moe(wl, windows, use_row_adapter=use_ra)
    routes = _routes_all(wl, windows, row_adapter=wl.row_adapter if use_ra else None)
    compare_moe(wl, windows, g_out, o_out, g_xas, o_xas, o_d, routes, min_exact=0.97)
    for r in (5, 9):
        assert np.array_equal(g_out[r], wl.out_buf[r])
