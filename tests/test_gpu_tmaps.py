"""A loaded as 2-D TMA boxes (lora_encode_a_tmaps + a_tmaps) on the GPU (-m gpu).

The maps change how A reaches shared memory (64-column boxes with the 128-byte
swizzle instead of one copy per row). Where the shrink stays on mma.sync the
arithmetic is unchanged and the fold must give the same bits with and without
them; at max_rank 128 with units of at most 16 rows the shrink moves to the
tcgen05 tensor cores (another fp32 summation order), and every result must
match the CPU oracle.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W
from gpu_util import device_a_tmaps, gpu_bgmv, oracle_bgmv, oracle_gather, require_gpu, to_u16
from parity import compare_bgmv, compare_gather, gather_routes

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    L.lora_read_device_status(clear=True)


def _bgmv_run(wl, maps=None):
    d = W.bgmv_to_device(wl)
    m = device_a_tmaps(d.a_table, wl.max_rank, wl.k_in) if maps else None
    L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, wl.n, d.a_table,
                d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa, a_tmaps=m)
    torch.cuda.synchronize()
    return to_u16(d.out_buf), to_u16(d.xa)


@pytest.mark.parametrize("name", ["tiny_bgmv", "decode_qproj_bgmv", "qkv_kfold_bgmv", "ffn_down_bgmv"])
def test_bgmv_maps_give_the_same_bits(name):
    wl = W.by_name(name)
    g = L.lora_launch_geometry(16, wl.n, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out)
    if wl.max_rank >= L.TMAP_MIN_RANK:
        assert g["k_chunk"] % 64 == 0
    else:   # maps ignored below the threshold
        assert g == L.lora_launch_geometry(0, wl.n, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out)
    o1, x1 = _bgmv_run(wl)
    o2, x2 = _bgmv_run(wl, maps=True)
    if not g["tc"]:     # same arithmetic, other loads: the same bits
        assert np.array_equal(o1, o2)
        routed = [i for i in range(wl.n) if 0 <= wl.seq_slot[i] < wl.max_loras and wl.present[wl.seq_slot[i]]]
        assert np.array_equal(x1[routed], x2[routed])
    o_out, o_xa, o_d = oracle_bgmv(wl)
    compare_bgmv(wl, o2, o_out, x2, o_xa, o_d)
    assert L.lora_read_device_status(clear=True) == 0


SMALL = [
    # n, k_in, n_out, max_loras, max_rank, ranks, slot law
    (9, 72, 40, 3, 32, (32, 8), "uniform"),               # k-slice shorter than one box
    (70, 520, 264, 2, 40, (40, 16), "uniform"),           # chunks reach past the k-slice
    (33, 4104, 1032, 5, 128, (128, 72), "zipf:1.1"),
    (17, 2056, 512, 3, 256, (256, 200), "uniform_all"),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_bgmv_maps_random_shapes(case):
    n, k_in, n_out, Lr, R, ranks, law = SMALL[case]
    wl = W.make_bgmv(f"tm{case}", n=n, k_in=k_in, n_out=n_out, max_loras=Lr, max_rank=R,
                     rank_choices=ranks, alpha=16.0, rslora=False, slot_law=law,
                     slot_base_frac=0.15, seed=600 + case)
    assert R >= L.TMAP_MIN_RANK
    g_out, g_xa = _bgmv_run(wl, maps=True)
    o_out, o_xa, o_d = oracle_bgmv(wl)
    compare_bgmv(wl, g_out, o_out, g_xa, o_xa, o_d, min_exact=0.97)


@pytest.mark.parametrize("max_rank", [16, 64, 128])
def test_gather_maps_give_the_same_bits(max_rank):
    wl = W.make_moe_gather("tmg", num_tokens=64, top_k=8, num_experts=128, k_in=768, n_out=2048,
                           max_loras=16, max_rank=max_rank, rank=max_rank, alpha=32.0,
                           adapter_base_frac=0.20, seed=630 + max_rank)
    res = []
    for maps in (False, True):
        d = W.gather_to_device(wl)
        m = device_a_tmaps(d.a_table, wl.max_rank, wl.k_in) if maps else None
        L.lora_moe_gather_bgmv(d.x, wl.k_in, d.out_buf, wl.n_out, d.indices, wl.n_rows, wl.top_k,
                               d.row_adapter, wl.num_tokens, wl.num_experts, d.a_table, d.b_table,
                               d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                               a_tmaps=m)
        torch.cuda.synchronize()
        res.append((to_u16(d.out_buf), to_u16(d.xa)[: wl.n_rows]))
    g = L.lora_launch_geometry(18, wl.n_rows, wl.max_loras * wl.num_experts, wl.max_rank, wl.k_in, wl.n_out)
    if not g["tc"]:
        assert np.array_equal(res[0][0], res[1][0])
    o_out, o_xa, o_d = oracle_gather(wl)
    compare_gather(wl, res[1][0], o_out, res[1][1], o_xa, o_d, gather_routes(wl))
