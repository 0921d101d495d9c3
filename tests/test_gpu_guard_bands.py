"""No fold writes outside its outputs (-m gpu): guard bands around base_out and xa.

Each fold runs twice on the same inputs: once on plain device buffers and once
with base_out and xa copied into the middle of larger allocations whose ends
hold a fixed pattern (tests/guard_bands.py). The guarded run must leave every
guard element unchanged and give the same bits as the plain run. This covers
the routed bgmv (rows, A tensor maps, the tcgen05 shrink), the MoE grouped
fold (four windows, and one call over all sorted rows), the decode gather fold
and both paths of the single-adapter delta at full workload sizes.
"""
from __future__ import annotations

from dataclasses import replace

import numpy as np
import pytest
import torch

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W
from guard_bands import guarded, guards_intact
from gpu_util import delta_rows, device_a_tmaps, require_gpu, to_u16

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    L.lora_read_device_status(clear=True)


def _guard(d, guard, *fields):
    """Replace the named output tensors of a device workload by guarded copies."""
    if not guard:
        return d, []
    bands, new = [], {}
    for f in fields:
        big, view = guarded(getattr(d, f))
        bands.append((big, view))
        new[f] = view
    return replace(d, **new), bands


def _check(bands):
    torch.cuda.synchronize()
    for big, view in bands:
        assert guards_intact(big, view)
    assert L.lora_read_device_status(clear=True) == 0


@pytest.mark.parametrize("name,maps", [("tiny_bgmv", False), ("decode_qproj_bgmv", False),
                                       ("qkv_kfold_bgmv", False), ("qkv_kfold_bgmv", True),
                                       ("ffn_down_bgmv", False), ("ffn_down_bgmv", True)])
def test_bgmv_writes_stay_inside(name, maps):
    wl = W.by_name(name)
    res = []
    for guard in (False, True):
        d, bands = _guard(W.bgmv_to_device(wl), guard, "out_buf", "xa")
        out_ptr = d.out_buf.data_ptr() + 2 * wl.out_offset
        m = device_a_tmaps(d.a_table, wl.max_rank, wl.k_in) if maps else None
        L.lora_bgmv(d.x, wl.x_row_stride, out_ptr, wl.out_row_stride, d.seq_slot, wl.n, d.a_table,
                    d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                    a_tmaps=m)
        _check(bands)
        res.append((to_u16(d.out_buf), to_u16(d.xa)))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])


@pytest.mark.parametrize("name,one_call", [("moe_down_fold", False), ("moe_gateup_fold", True)])
def test_moe_writes_stay_inside(name, one_call):
    wl = W.by_name(name)
    windows = [(0, wl.te)] if one_call else wl.windows()
    res = []
    for guard in (False, True):
        d = W.moe_to_device(wl, xa_rows=max(hi - lo for lo, hi in windows))
        # xa holds exactly the largest window's rows: its band starts at row xa_rows
        assert d.xa.shape[0] == max(hi - lo for lo, hi in windows)
        d, bands = _guard(d, guard, "out_buf", "xa")
        for lo, hi in windows:
            L.lora_moe_grouped_fold(d.x, wl.k_in, d.out_buf, wl.n_out, d.expert_offsets,
                                    wl.num_experts, d.sorted_token_ids, wl.te, d.row_adapter,
                                    wl.num_tokens, lo, hi, d.a_table, d.b_table, d.scale,
                                    wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                                    x_gather=wl.x_gather)
        _check(bands)
        res.append((to_u16(d.out_buf), to_u16(d.xa)))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])


@pytest.mark.parametrize("maps", [False, True])
def test_gather_writes_stay_inside(maps):
    wl = W.moe_decode_gather()
    res = []
    for guard in (False, True):
        d, bands = _guard(W.gather_to_device(wl), guard, "out_buf", "xa")
        m = device_a_tmaps(d.a_table, wl.max_rank, wl.k_in) if maps else None
        L.lora_moe_gather_bgmv(d.x, wl.k_in, d.out_buf, wl.n_out, d.indices, wl.n_rows, wl.top_k,
                               d.row_adapter, wl.num_tokens, wl.num_experts, d.a_table, d.b_table,
                               d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                               a_tmaps=m)
        _check(bands)
        res.append((to_u16(d.out_buf), to_u16(d.xa)))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])


@pytest.mark.parametrize("name,rows", [("prefill_down_delta", None), ("prefill_qproj_delta", None),
                                       ("prefill_qproj_delta", 100)])
def test_delta_writes_stay_inside(name, rows):
    wl = W.by_name(name)
    if rows is not None:            # below the tensor-core threshold: the routed engine
        wl = delta_rows(wl, range(rows))
    assert (wl.m >= L.DELTA_DENSE_MIN_ROWS) == (rows is None)
    res = []
    for guard in (False, True):
        d, bands = _guard(W.delta_to_device(wl), guard, "out_buf", "xa")
        out_ptr = d.out_buf.data_ptr() + 2 * wl.out_offset
        L.lora_delta(d.x, wl.x_row_stride, out_ptr, wl.out_row_stride, wl.m, d.a, d.b, wl.scale,
                     wl.max_rank, wl.k_in, wl.n_out, xa=d.xa)
        _check(bands)
        res.append((to_u16(d.out_buf), to_u16(d.xa)))
    assert np.array_equal(res[0][0], res[1][0]) and np.array_equal(res[0][1], res[1][1])



def test_moe_undersized_xa_is_rejected_before_launch():
    """An xa of fewer rows than the window is refused on the host; nothing runs."""
    wl = W.moe_down_fold()
    lo, hi = wl.windows()[0]
    d = W.moe_to_device(wl, xa_rows=hi - lo)
    with pytest.raises(L.LoraError, match="LORA_ERR_SIZE"):
        L.lora_moe_grouped_fold(d.x, wl.k_in, d.out_buf, wl.n_out, d.expert_offsets, wl.num_experts,
                                d.sorted_token_ids, wl.te, d.row_adapter, wl.num_tokens, lo, hi,
                                d.a_table, d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in,
                                wl.n_out, xa=d.xa, xa_rows=hi - lo - 1)
    torch.cuda.synchronize()
    assert np.array_equal(to_u16(d.out_buf), wl.out_buf)
