"""CUDA lora_moe_gather_bgmv (decode-path MoE fold over flat (token, slot)
rows) against the CPU oracle (-m gpu), through the C ABI.

Covers the decode workload at full size (every element compared), small random
routings, NULL row_adapter, absent (adapter, expert) entries, experts and
tokens out of range, per-token calls equal to the batched call (bit for bit),
and graph replay with new routing.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W
from gpu_util import device_a_tmaps, gpu_gather, oracle_gather, require_gpu, to_u16
from parity import compare_gather, gather_routes

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    L.lora_read_device_status(clear=True)


def test_gather_decode_workload_parity():
    wl = W.moe_decode_gather()
    g_out, g_xa = gpu_gather(wl)
    o_out, o_xa, o_d = oracle_gather(wl)
    st = compare_gather(wl, g_out, o_out, g_xa, o_xa, o_d, gather_routes(wl))
    assert st["rows"] > 300
    assert L.lora_read_device_status(clear=True) == 0


SMALL = [
    # tokens, top_k, experts, k_in, n_out, loras, rank, present_frac, row_adapter
    (3, 2, 4, 40, 24, 2, 8, 1.0, True),
    (37, 4, 16, 264, 520, 3, 16, 0.7, True),
    (20, 8, 64, 768, 2048, 4, 16, 1.0, False),
    (50, 2, 3, 1040, 392, 2, 64, 1.0, True),   # few entries: many rows per work unit
    (9, 6, 32, 2056, 1032, 5, 24, 0.9, True),
]


@pytest.mark.parametrize("case", range(len(SMALL)))
def test_gather_random(case):
    tok, k, E, k_in, n_out, Lr, R, pf, use_ra = SMALL[case]
    wl = W.make_moe_gather(f"g{case}", num_tokens=tok, top_k=k, num_experts=E, k_in=k_in,
                           n_out=n_out, max_loras=Lr, max_rank=R, rank=R, alpha=16.0,
                           adapter_base_frac=0.25, seed=500 + case, use_row_adapter=use_ra,
                           present_frac=pf)
    g_out, g_xa = gpu_gather(wl, use_row_adapter=use_ra)
    o_out, o_xa, o_d = oracle_gather(wl, use_row_adapter=use_ra)
    routes = gather_routes(wl, row_adapter=wl.row_adapter if use_ra else None)
    compare_gather(wl, g_out, o_out, g_xa, o_xa, o_d, routes, min_exact=0.97)


def test_gather_experts_out_of_range_are_skipped():
    wl = W.make_moe_gather("g_bad", num_tokens=16, top_k=4, num_experts=8, k_in=136, n_out=72,
                           max_loras=2, max_rank=16, rank=16, alpha=16.0, adapter_base_frac=0.2,
                           seed=520)
    idx = wl.indices.copy()
    idx[[1, 7, 30]] = [-1, wl.num_experts, 1 << 20]
    g_out, g_xa = gpu_gather(wl, indices=idx)
    o_out, o_xa, o_d = oracle_gather(wl, indices=idx)
    compare_gather(wl, g_out, o_out, g_xa, o_xa, o_d, gather_routes(wl, indices=idx))
    for r in (1, 7, 30):
        assert np.array_equal(g_out[r], wl.out_buf[r])


def test_gather_per_token_calls_equal_batched():
    """Rows are independent: folding one token's top_k rows per call gives the
    same bits as the batched call."""
    wl = W.make_moe_gather("g_inv", num_tokens=12, top_k=4, num_experts=16, k_in=768,
                           n_out=1024, max_loras=4, max_rank=16, rank=16, alpha=32.0,
                           adapter_base_frac=0.2, seed=530)
    g_out, g_xa = gpu_gather(wl)
    d = W.gather_to_device(wl)
    k = wl.top_k
    for t in range(wl.num_tokens):
        rows = slice(t * k, (t + 1) * k)
        L.lora_moe_gather_bgmv(d.x[rows], wl.k_in, d.out_buf[rows], wl.n_out, d.indices[rows], k, k,
                               d.row_adapter[t:t + 1], 1, wl.num_experts, d.a_table, d.b_table,
                               d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out,
                               xa=d.xa[rows])
    torch.cuda.synchronize()
    assert np.array_equal(to_u16(d.out_buf), g_out)
    routed = [r for r, _ in gather_routes(wl)]
    assert np.array_equal(to_u16(d.xa)[routed], g_xa[routed])


@pytest.mark.parametrize("max_rank,maps", [(16, False), (64, True), (128, True)])
def test_gather_decode_shape_per_token_calls_equal_batched(max_rank, maps):
    """The decode workload (64 tokens x top-8 of 128 experts, k_in 768, n_out 2048;
    at ranks 64 and 128 the same rows over 32 experts x 8 adapters, to keep the
    adapter pool small): one token's rows per call give the same bits as the batched
    call, with A row copies (rank 16) and with A tensor maps (ranks 64, 128)."""
    wl = (W.moe_decode_gather() if max_rank == 16 else
          W.make_moe_gather("g_inv_full", num_tokens=64, top_k=8, num_experts=32, k_in=768,
                            n_out=2048, max_loras=8, max_rank=max_rank, rank=max_rank, alpha=32.0,
                            adapter_base_frac=0.2, seed=560 + max_rank))
    res = []
    for per_token in (False, True):
        d = W.gather_to_device(wl)
        m = device_a_tmaps(d.a_table, wl.max_rank, wl.k_in) if maps else None
        k = wl.top_k
        calls = ([(slice(t * k, (t + 1) * k), t) for t in range(wl.num_tokens)] if per_token
                 else [(slice(0, wl.n_rows), None)])
        for rows, t in calls:
            n = rows.stop - rows.start
            ra = d.row_adapter if t is None else d.row_adapter[t:t + 1]
            L.lora_moe_gather_bgmv(d.x[rows], wl.k_in, d.out_buf[rows], wl.n_out, d.indices[rows], n, k,
                                   ra, wl.num_tokens if t is None else 1, wl.num_experts, d.a_table,
                                   d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out,
                                   xa=d.xa[rows], a_tmaps=m)
        torch.cuda.synchronize()
        res.append((to_u16(d.out_buf), to_u16(d.xa)[: wl.n_rows]))
    assert np.array_equal(res[0][0], res[1][0])
    routed = [r for r, _ in gather_routes(wl)]
    assert np.array_equal(res[0][1][routed], res[1][1][routed])
    o_out, o_xa, o_d = oracle_gather(wl)
    compare_gather(wl, res[0][0], o_out, res[0][1], o_xa, o_d, gather_routes(wl))


def test_gather_graph_replay_with_new_routing():
    wl = W.make_moe_gather("g_graph", num_tokens=32, top_k=8, num_experts=64, k_in=768,
                           n_out=2048, max_loras=8, max_rank=16, rank=16, alpha=32.0,
                           adapter_base_frac=0.2, seed=540)
    d = W.gather_to_device(wl)
    s = torch.cuda.Stream()

    def run():
        L.lora_moe_gather_bgmv(d.x, wl.k_in, d.out_buf, wl.n_out, d.indices, wl.n_rows, wl.top_k,
                               d.row_adapter, wl.num_tokens, wl.num_experts, d.a_table, d.b_table,
                               d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                               stream=s)

    with torch.cuda.stream(s):
        run()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        run()
    rng = np.random.default_rng(41)
    for _ in range(2):
        wl.indices = rng.integers(0, wl.num_experts, size=wl.n_rows).astype(np.int32)
        ra = rng.integers(0, wl.max_loras, size=wl.num_tokens).astype(np.int32)
        ra[rng.random(wl.num_tokens) < 0.3] = -1
        wl.row_adapter = ra
        wl.out_buf = W.to_bf16_bits(rng.standard_normal(wl.out_buf.shape).astype(np.float32))
        d.indices.copy_(torch.from_numpy(wl.indices))
        d.row_adapter.copy_(torch.from_numpy(ra))
        d.out_buf.copy_(torch.from_numpy(wl.out_buf.view(np.int16)))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        o_out, o_xa, o_d = oracle_gather(wl)
        compare_gather(wl, to_u16(d.out_buf), o_out, to_u16(d.xa)[: wl.n_rows], o_xa, o_d,
                       gather_routes(wl))
