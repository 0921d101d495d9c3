"""CUDA lora_bgmv against the CPU oracle (-m gpu), through the C ABI.

Covers the four bgmv workloads at full size (every output element compared),
random small shapes with ragged k / n_out / rank tails, strided outputs, slots
holding more rows than one work unit, skip rules, batch invariance (one row per
call is bit-identical), CUDA-graph replay with new routing, and the
misaligned-table status bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W
from gpu_util import device_a_tmaps, gpu_bgmv, oracle_bgmv, require_gpu, to_u16
from parity import compare_bgmv

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    L.lora_read_device_status(clear=True)


@pytest.mark.parametrize("name", ["tiny_bgmv", "decode_qproj_bgmv", "qkv_kfold_bgmv", "ffn_down_bgmv"])
def test_bgmv_workload_parity(name):
    wl = W.by_name(name)
    g_out, g_xa = gpu_bgmv(wl)
    o_out, o_xa, o_d = oracle_bgmv(wl)
    st = compare_bgmv(wl, g_out, o_out, g_xa, o_xa, o_d)
    assert st["rows"] > 0
    assert L.lora_read_device_status(clear=True) == 0


SMALL = [
    # n, k_in, n_out, max_loras, max_rank, ranks, slot_law, x_stride, out_stride, out_offset
    (1, 8, 8, 1, 8, (8,), "uniform", None, None, 0),
    (5, 24, 40, 3, 8, (8, 4), "uniform_all", 40, 64, 16),
    (33, 136, 72, 4, 24, (24, 8, 16), "uniform", 144, 96, 8),
    (70, 520, 264, 2, 16, (16,), "uniform", None, None, 0),      # > one work unit per slot
    (100, 1040, 392, 9, 40, (8, 40), "zipf:1.1", 1048, 400, 8),
    (64, 4104, 1032, 5, 128, (128, 72), "uniform", None, None, 0),
    (17, 2056, 4096, 3, 256, (256, 200), "uniform_all", None, None, 0),
    (40, 12296, 512, 6, 64, (64, 32), "uniform", None, None, 0),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_bgmv_random_shapes(case):
    n, k_in, n_out, L_, R, ranks, law, xs, os_, off = SMALL[case]
    wl = W.make_bgmv(f"small{case}", n=n, k_in=k_in, n_out=n_out, max_loras=L_, max_rank=R,
                     rank_choices=ranks, alpha=16.0, rslora=bool(case % 2), slot_law=law,
                     slot_base_frac=0.15, seed=100 + case, x_row_stride=xs,
                     out_row_stride=(os_ or n_out) if off == 0 else os_, out_offset=off,
                     x_law="silu_gate" if case % 3 == 0 else "normal")
    g_out, g_xa = gpu_bgmv(wl)
    o_out, o_xa, o_d = oracle_bgmv(wl)
    compare_bgmv(wl, g_out, o_out, g_xa, o_xa, o_d, min_exact=0.97)


def test_bgmv_skip_rules_and_null_tables():
    wl = W.tiny_bgmv()
    wl.seq_slot = np.array([-5, 3, 4, 1], np.int32)   # base, NULL slot, >= max_loras, routed
    g_out, _ = gpu_bgmv(wl)
    assert np.array_equal(g_out[:3], wl.out_buf[:3])
    o_out, o_xa, o_d = oracle_bgmv(wl)
    assert not np.array_equal(g_out[3], wl.out_buf[3])
    assert np.array_equal(g_out[:3], o_out[:3])


def test_bgmv_all_rows_base_and_empty():
    wl = W.decode_qproj_bgmv()
    wl.seq_slot = np.full(wl.n, -1, np.int32)
    g_out, _ = gpu_bgmv(wl)
    assert np.array_equal(g_out, wl.out_buf)
    d = W.bgmv_to_device(wl)
    L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, 0, d.a_table,
                d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa)
    torch.cuda.synchronize()
    assert np.array_equal(to_u16(d.out_buf), wl.out_buf)


def test_bgmv_one_hot_slot_heavy():
    """Every row on one slot: many work units of the same adapter."""
    wl = W.make_bgmv("heavy", n=300, k_in=2048, n_out=1024, max_loras=4, max_rank=16,
                     rank_choices=(16,), alpha=32.0, rslora=False,
                     slot_law="list:" + ",".join(["2"] * 300), slot_base_frac=0.0, seed=7)
    g_out, g_xa = gpu_bgmv(wl)
    o_out, o_xa, o_d = oracle_bgmv(wl)
    compare_bgmv(wl, g_out, o_out, g_xa, o_xa, o_d)


def test_bgmv_units_numbered_slot_by_slot():
    """max_loras > n: units are numbered over the slots that have rows (not one
    per slot), including a slot with more than one tile of rows and slots at
    both ends of the table."""
    seq = np.random.default_rng(3).permutation([150] * 40 + [3] * 30 + [199] * 5 + [0] * 5)
    wl = W.make_bgmv("many_slots", n=80, k_in=1032, n_out=520, max_loras=200, max_rank=16,
                     rank_choices=(16, 8), alpha=32.0, rslora=False,
                     slot_law="list:" + ",".join(str(int(v)) for v in seq), slot_base_frac=0.0, seed=11)
    g_out, g_xa = gpu_bgmv(wl)
    o_out, o_xa, o_d = oracle_bgmv(wl)
    compare_bgmv(wl, g_out, o_out, g_xa, o_xa, o_d)


def _one_row_calls(wl, d, rows, maps):
    """Fold each of `rows` alone (n = 1 per call) on device copy d."""
    for i in rows:
        L.lora_bgmv(d.x[i], wl.x_row_stride, d.out_buf[i].data_ptr() + 2 * wl.out_offset,
                    wl.out_row_stride, d.seq_slot[i:i + 1], 1, d.a_table, d.b_table, d.scale,
                    wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa[i], a_tmaps=maps)
    torch.cuda.synchronize()
    return to_u16(d.out_buf), to_u16(d.xa)


def _batch_invariant(wl, rows, maps: bool):
    """The batched call and one call per row give the same bits (out and xa);
    both with A tensor maps when `maps` (the launch geometry then follows them)."""
    d = W.bgmv_to_device(wl)
    m = device_a_tmaps(d.a_table, wl.max_rank, wl.k_in) if maps else None
    L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, wl.n, d.a_table,
                d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa, a_tmaps=m)
    torch.cuda.synchronize()
    g_out, g_xa = to_u16(d.out_buf), to_u16(d.xa)
    d1 = W.bgmv_to_device(wl)
    m1 = device_a_tmaps(d1.a_table, wl.max_rank, wl.k_in) if maps else None
    s_out, s_xa = _one_row_calls(wl, d1, rows, m1)
    rows = list(rows)
    assert np.array_equal(s_out[rows], g_out[rows])
    routed = [i for i in rows if 0 <= wl.seq_slot[i] < wl.max_loras and wl.present[wl.seq_slot[i]]]
    assert np.array_equal(s_xa[routed], g_xa[routed])
    return g_out, g_xa


@pytest.mark.parametrize("name,maps", [("decode_qproj_bgmv", False), ("qkv_kfold_bgmv", False),
                                       ("qkv_kfold_bgmv", True), ("ffn_down_bgmv", False),
                                       ("ffn_down_bgmv", True)])
def test_bgmv_batch_invariance(name, maps):
    """Each row folded alone (n = 1 per call) is bit-identical to the batched call
    ("Function apply_lora_bgmv", BYTE-IDENTICAL paragraph), on every shrink path a
    routed call can take: mma.sync with A rows or A boxes, and the tcgen05 shrink
    (ffn_down_bgmv with maps)."""
    wl = W.by_name(name)
    g = L.lora_launch_geometry(16 if maps else 0, wl.n, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out)
    if name == "ffn_down_bgmv":
        assert g["tc"] == int(maps)
    rows = range(wl.n) if wl.n <= 64 else list(range(0, wl.n, 3))
    _batch_invariant(wl, rows, maps)


def test_bgmv_tc_shrink_small_units_batch_invariant():
    """tcgen05 shrink with units of fewer than 16 rows (the N = 16 atom then holds
    x columns past the unit's rows): parity with the oracle and bit-identity with
    one row per call."""
    wl = W.make_bgmv("tc_small", n=45, k_in=2056, n_out=520, max_loras=7, max_rank=128,
                     rank_choices=(128, 96), alpha=16.0, rslora=True, slot_law="uniform",
                     slot_base_frac=0.1, seed=77)
    assert L.lora_launch_geometry(16, wl.n, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out)["tc"] == 1
    counts = np.bincount(wl.seq_slot[wl.seq_slot >= 0], minlength=wl.max_loras)
    assert counts.max() < 16
    g_out, g_xa = _batch_invariant(wl, range(wl.n), maps=True)
    o_out, o_xa, o_d = oracle_bgmv(wl)
    compare_bgmv(wl, g_out, o_out, g_xa, o_xa, o_d, min_exact=0.97)


def test_bgmv_graph_replay_with_new_routing():
    """Capture once; replay with new seq_slot and base_out contents."""
    wl = W.decode_qproj_bgmv()
    d = W.bgmv_to_device(wl)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, wl.n,
                    d.a_table, d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out,
                    xa=d.xa, stream=s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, wl.n,
                    d.a_table, d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out,
                    xa=d.xa, stream=s)
    rng = np.random.default_rng(5)
    for step in range(3):
        wl.seq_slot = W.zipf_slots(rng, wl.n, wl.max_loras, 1.1)
        wl.seq_slot[rng.random(wl.n) < 0.2] = -1
        wl.out_buf = W.to_bf16_bits(rng.standard_normal(wl.out_buf.shape).astype(np.float32))
        d.seq_slot.copy_(torch.from_numpy(wl.seq_slot))
        d.out_buf.copy_(torch.from_numpy(wl.out_buf.view(np.int16)))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        o_out, o_xa, o_d = oracle_bgmv(wl)
        compare_bgmv(wl, to_u16(d.out_buf), o_out, to_u16(d.xa), o_xa, o_d)


def test_bgmv_misaligned_table_entry_is_skipped_and_reported():
    wl = W.tiny_bgmv()
    wl.seq_slot = np.array([0, 1, 2, 1], np.int32)
    d = W.bgmv_to_device(wl)
    tab = d.a_table.clone()
    tab[1] += 2                                   # not 16-byte aligned (inside the pool)
    L.lora_read_device_status(clear=True)
    L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, wl.n, tab,
                d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa)
    torch.cuda.synchronize()
    out = to_u16(d.out_buf)
    assert np.array_equal(out[[1, 3]], wl.out_buf[[1, 3]])
    assert not np.array_equal(out[0], wl.out_buf[0])
    assert L.lora_read_device_status(clear=True) & L.LORA_DEV_MISALIGNED
