"""LORA_INPUTS_READY (-m gpu): calls that plan and shrink while the previous
kernel on the stream finishes give the same bits as calls that wait for it.

Every input other than base_out and xa is written (and the device synchronized)
before the flagged calls, as the flag's promise requires. The chained cases
make each flagged call read base_out rows the kernel just before it writes, and
the MoE windows share one xa buffer, so a fold that touched base_out or xa
before its wait would give different bits.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W
from gpu_util import device_a_tmaps, require_gpu, to_u16

pytestmark = pytest.mark.gpu

READY = L.INPUTS_READY


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    L.lora_read_device_status(clear=True)


def _bgmv_chain(wl, d, flags, calls, maps=None, graph=False):
    """`calls` back-to-back folds of the same rows into the same out buffer
    (each reads what the one before wrote); returns (out, xa) after the last."""
    out0 = d.out_buf.clone()
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def run():
        for _ in range(calls):
            L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, wl.n,
                        d.a_table, d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in,
                        wl.n_out, xa=d.xa, stream=stream, a_tmaps=maps, flags=flags)

    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run()
        d.out_buf.copy_(out0)
        torch.cuda.synchronize()
        g.replay()
    else:
        with torch.cuda.stream(stream):
            run()
    torch.cuda.synchronize()
    res = to_u16(d.out_buf), to_u16(d.xa)
    d.out_buf.copy_(out0)
    d.xa.zero_()
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("name,maps", [("decode_qproj_bgmv", False), ("qkv_kfold_bgmv", True),
                                       ("ffn_down_bgmv", True), ("ffn_down_bgmv", False)])
def test_bgmv_ready_chain_matches_the_waiting_chain(name, maps):
    wl = W.by_name(name)
    d = W.bgmv_to_device(wl)
    m = device_a_tmaps(d.a_table, wl.max_rank, wl.k_in) if maps else None
    ref = _bgmv_chain(wl, d, 0, 3, maps=m)
    got = _bgmv_chain(wl, d, READY, 3, maps=m)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    one = _bgmv_chain(wl, d, 0, 1, maps=m)
    assert not np.array_equal(one[0], ref[0])     # the chain really folds three times
    assert L.lora_read_device_status(clear=True) == 0


def test_bgmv_ready_chain_in_a_graph():
    wl = W.by_name("decode_qproj_bgmv")
    d = W.bgmv_to_device(wl)
    ref = _bgmv_chain(wl, d, 0, 8)
    got = _bgmv_chain(wl, d, READY, 8, graph=True)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])


def test_bgmv_ready_call_without_routed_rows():
    """Every CTA finds no rows: the grid still waits for the kernel before it, so
    a waiting call after it sees that kernel's output."""
    wl = W.by_name("decode_qproj_bgmv")
    d = W.bgmv_to_device(wl)
    none = torch.full_like(d.seq_slot, -1)
    out0 = d.out_buf.clone()
    torch.cuda.synchronize()
    for flags in (0, READY):
        for i, f in enumerate((0, flags, 0)):
            seq = none if i == 1 else d.seq_slot
            L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, seq, wl.n, d.a_table,
                        d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                        flags=f)
        torch.cuda.synchronize()
        if flags == 0:
            ref = to_u16(d.out_buf)
        else:
            assert np.array_equal(to_u16(d.out_buf), ref)
        d.out_buf.copy_(out0)
        torch.cuda.synchronize()


def _moe_windows(wl, d, flags, rounds=1):
    out0 = d.out_buf.clone()
    torch.cuda.synchronize()
    for _ in range(rounds):
        for lo, hi in wl.windows():
            L.lora_moe_grouped_fold(d.x, wl.k_in, d.out_buf, wl.n_out, d.expert_offsets,
                                    wl.num_experts, d.sorted_token_ids, wl.te, d.row_adapter,
                                    wl.num_tokens, lo, hi, d.a_table, d.b_table, d.scale,
                                    wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                                    x_gather=wl.x_gather, flags=flags)
    torch.cuda.synchronize()
    res = to_u16(d.out_buf), to_u16(d.xa)
    d.out_buf.copy_(out0)
    d.xa.zero_()
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("name", ["moe_down_fold", "moe_gateup_fold"])
def test_moe_ready_windows_share_xa_and_match(name):
    """Four windows of one layer, flagged, one shared xa buffer, folded twice in
    a row (the second pass reads the first pass's base_out)."""
    wl = W.by_name(name)
    d = W.moe_to_device(wl, xa_rows=wl.cap)
    ref = _moe_windows(wl, d, 0, rounds=2)
    got = _moe_windows(wl, d, READY, rounds=2)
    assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1])
    assert L.lora_read_device_status(clear=True) == 0


def test_gather_ready_chain_matches():
    wl = W.by_name("moe_decode_gather")
    d = W.gather_to_device(wl)
    out0 = d.out_buf.clone()
    res = []
    for flags in (0, READY):
        torch.cuda.synchronize()
        for _ in range(3):
            L.lora_moe_gather_bgmv(d.x, wl.k_in, d.out_buf, wl.n_out, d.indices, wl.n_rows,
                                   wl.top_k, d.row_adapter, wl.num_tokens, wl.num_experts,
                                   d.a_table, d.b_table, d.scale, wl.max_loras, wl.max_rank,
                                   wl.k_in, wl.n_out, xa=d.xa, flags=flags)
        torch.cuda.synchronize()
        res.append((to_u16(d.out_buf), to_u16(d.xa)))
        d.out_buf.copy_(out0)
        d.xa.zero_()
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])
