"""Helpers for the -m gpu tests: run the CUDA path and the oracle on one workload."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import oracle
from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if not os.path.exists(L.LIB_PATH):
        from gather_lora_gb300 import build
        build.build()
    L.load()


def to_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def gpu_bgmv(wl: W.BgmvWorkload, d: W.DeviceBgmv = None, seq=None, stream=None):
    """Run lora_bgmv on the device copy of wl. Returns (out_buf, xa) as uint16 numpy."""
    d = d or W.bgmv_to_device(wl)
    n = wl.n if seq is None else int(seq.numel())
    L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride,
                d.seq_slot if seq is None else seq, n, d.a_table, d.b_table, d.scale,
                wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa, stream=stream)
    torch.cuda.synchronize()
    return to_u16(d.out_buf), to_u16(d.xa)


def oracle_bgmv(wl: W.BgmvWorkload):
    out = wl.out_buf.copy()
    seg = out.reshape(-1)[wl.out_offset:]
    xa, dd = oracle.lora_bgmv(wl.x.reshape(-1), wl.x_row_stride, seg, wl.out_row_stride,
                              wl.seq_slot, wl.a_list(), wl.b_list(), wl.scale, wl.max_rank,
                              wl.k_in, wl.n_out)
    return out, xa, dd


def gpu_moe(wl: W.MoeWorkload, windows, d: W.DeviceMoe = None, use_row_adapter=True):
    d = d or W.moe_to_device(wl, xa_rows=max(hi - lo for lo, hi in windows) or 1)
    xas = []
    for lo, hi in windows:
        d.xa.zero_()
        L.lora_moe_grouped_fold(d.x, wl.k_in, d.out_buf, wl.n_out, d.expert_offsets,
                                wl.num_experts, d.sorted_token_ids, wl.te,
                                d.row_adapter if use_row_adapter else None, wl.num_tokens, lo, hi,
                                d.a_table, d.b_table, d.scale, wl.max_loras, wl.max_rank,
                                wl.k_in, wl.n_out, xa=d.xa, x_gather=wl.x_gather)
        torch.cuda.synchronize()
        xas.append(to_u16(d.xa)[: hi - lo].copy())
    return to_u16(d.out_buf), xas


def oracle_moe(wl: W.MoeWorkload, windows, use_row_adapter=True):
    out = wl.out_buf.copy()
    xas = []
    d_all = np.zeros((max(wl.te, 1), wl.n_out), dtype=np.uint16)
    for lo, hi in windows:
        xa, dd = oracle.lora_moe_grouped_fold(
            wl.x, wl.k_in, out, wl.n_out, wl.expert_offsets, wl.sorted_token_ids,
            wl.row_adapter if use_row_adapter else None, wl.num_tokens, lo, hi, wl.a_list(),
            wl.b_list(), wl.scale, wl.max_rank, wl.k_in, wl.n_out, x_gather=wl.x_gather)
        xas.append(xa)
        d_all[lo:hi] = dd[lo:hi]
    return out, xas, d_all


def gpu_gather(wl: W.MoeGatherWorkload, d: W.DeviceMoeGather = None, use_row_adapter=True,
               indices=None):
    d = d or W.gather_to_device(wl)
    if indices is not None:
        d.indices.copy_(torch.from_numpy(np.ascontiguousarray(indices, dtype=np.int32)))
    d.xa.zero_()
    L.lora_moe_gather_bgmv(d.x, wl.k_in, d.out_buf, wl.n_out, d.indices, wl.n_rows, wl.top_k,
                           d.row_adapter if use_row_adapter else None, wl.num_tokens,
                           wl.num_experts, d.a_table, d.b_table, d.scale, wl.max_loras,
                           wl.max_rank, wl.k_in, wl.n_out, xa=d.xa)
    torch.cuda.synchronize()
    return to_u16(d.out_buf), to_u16(d.xa)[: wl.n_rows]


def oracle_gather(wl: W.MoeGatherWorkload, use_row_adapter=True, indices=None):
    out = wl.out_buf.copy()
    xa, dd = oracle.lora_moe_gather_bgmv(
        wl.x, wl.k_in, out, wl.n_out, wl.indices if indices is None else indices, wl.top_k,
        wl.row_adapter if use_row_adapter else None, wl.num_tokens, wl.num_experts, wl.a_list(),
        wl.b_list(), wl.scale, wl.max_rank, wl.k_in, wl.n_out)
    return out, xa, dd


def device_a_tmaps(a_table: torch.Tensor, max_rank: int, k_in: int) -> torch.Tensor:
    """Encode the A tensor maps of a device table (read back once, as at adapter
    load) and place them in device memory."""
    ptrs = a_table.cpu().numpy().astype(np.uint64)
    maps = L.lora_encode_a_tmaps(ptrs, max_rank, k_in)
    t = torch.from_numpy(maps).to(a_table.device)
    assert t.data_ptr() % 64 == 0
    return t


def gpu_delta(wl: W.DeltaWorkload, d: W.DeviceDelta = None, with_xa=True, stream=None):
    """Run lora_delta on the device copy of wl. Returns (out_buf, xa [m, max_rank]) as uint16."""
    d = d or W.delta_to_device(wl)
    L.lora_delta(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, wl.m, d.a, d.b, wl.scale,
                 wl.max_rank, wl.k_in, wl.n_out, xa=d.xa if with_xa else None, stream=stream)
    torch.cuda.synchronize()
    return to_u16(d.out_buf), to_u16(d.xa)[: wl.m]


def oracle_delta(wl: W.DeltaWorkload):
    out = wl.out_buf.copy()
    seg = out.reshape(-1)[wl.out_offset:]
    xa, dd = oracle.lora_delta(wl.x.reshape(-1), wl.x_row_stride, seg, wl.out_row_stride, wl.m,
                               wl.a, wl.b, wl.scale, wl.max_rank, wl.k_in, wl.n_out)
    return out, xa, dd


def delta_rows(wl: W.DeltaWorkload, rows) -> W.DeltaWorkload:
    """The same problem restricted to the given rows (for oracle samples of a full-size run)."""
    rows = np.asarray(rows)
    return W.DeltaWorkload(wl.name, len(rows), wl.k_in, wl.n_out, wl.max_rank, wl.rank,
                           wl.x_row_stride, wl.out_row_stride, wl.out_offset,
                           np.ascontiguousarray(wl.x[rows]), np.ascontiguousarray(wl.out_buf[rows]),
                           wl.a, wl.b, wl.scale, wl.meta)
