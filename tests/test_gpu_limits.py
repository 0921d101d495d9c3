"""The folds at the limits the header states (-m gpu).

n = LORA_MAX_ROWS routed rows over LORA_MAX_LORAS table slots (most of them
NULL); the MoE fold over LORA_MAX_EXPERTS experts; the single-adapter delta at
LORA_MAX_DELTA_ROWS rows on the tensor-core path, and past LORA_MAX_ROWS on the
routed engine (one launch per 8192 rows). Each result is compared with the
oracle (whole output, or rows sampled across the launch boundaries).
"""
from __future__ import annotations

import numpy as np
import pytest

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W
from gpu_util import (delta_rows, gpu_bgmv, gpu_delta, gpu_moe, oracle_bgmv, oracle_delta, oracle_moe,
                      require_gpu)
from parity import compare_bgmv, compare_delta, compare_moe, moe_routes

pytestmark = pytest.mark.gpu

MAX_ROWS, MAX_LORAS, MAX_EXPERTS, MAX_DELTA_ROWS = 8192, 4096, 1024, 1 << 20


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    L.lora_read_device_status(clear=True)


def test_bgmv_max_rows_and_slots():
    rng = np.random.default_rng(900)
    present = np.sort(rng.choice(MAX_LORAS, size=96, replace=False))
    wl = W.make_bgmv("limits", n=MAX_ROWS, k_in=128, n_out=96, max_loras=MAX_LORAS, max_rank=16,
                     rank_choices=(8, 16), alpha=16.0, rslora=False, slot_law="uniform_all",
                     slot_base_frac=0.05, seed=901, present_slots=present.tolist())
    assert L.lora_launch_geometry(0, wl.n, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out)["clusters"] > 0
    g_out, g_xa = gpu_bgmv(wl)
    o_out, o_xa, o_d = oracle_bgmv(wl)
    st = compare_bgmv(wl, g_out, o_out, g_xa, o_xa, o_d)
    assert st["rows"] > 100          # rows on present slots; the rest (NULL or base) stay byte-identical
    assert L.lora_read_device_status(clear=True) == 0


def test_moe_max_experts():
    wl = W.make_moe("limits_moe", num_tokens=512, top_k=4, num_experts=MAX_EXPERTS, k_in=128, n_out=256,
                    max_loras=4, max_rank=16, rank=16, alpha=32.0, adapter_base_frac=0.2, cap=1024, seed=902)
    windows = wl.windows()
    g_out, g_xas = gpu_moe(wl, windows)
    o_out, o_xas, o_d = oracle_moe(wl, windows)
    routes = [r for lo, hi in windows for r in moe_routes(wl, lo, hi)]
    compare_moe(wl, windows, g_out, o_out, g_xas, o_xas, o_d, routes)
    assert L.lora_read_device_status(clear=True) == 0


def _sampled(wl, g_out, g_xa, boundaries):
    rows = sorted({r for b in boundaries for r in (b - 2, b - 1, b, b + 1) if 0 <= r < wl.m} |
                  set(np.random.default_rng(7).integers(0, wl.m, size=24).tolist()))
    sub = delta_rows(wl, rows)
    o_out, o_xa, o_d = oracle_delta(sub)
    compare_delta(sub, g_out[rows], o_out, g_xa[rows], o_xa, o_d)


def test_delta_engine_path_past_max_rows():
    """A rank the tensor-core path does not take, over 2.5 x LORA_MAX_ROWS rows: three launches."""
    m = 2 * MAX_ROWS + MAX_ROWS // 2
    wl = W.make_delta("limits_eng", m=m, k_in=64, n_out=72, max_rank=24, rank=24, alpha=16.0,
                      rslora=False, seed=903)
    assert L.lora_delta_geometry(m, 24, 64, 72)["dense"] == 0
    g_out, g_xa = gpu_delta(wl)
    _sampled(wl, g_out, g_xa, [MAX_ROWS, 2 * MAX_ROWS, m])
    assert L.lora_read_device_status(clear=True) == 0


def test_delta_max_rows_tensor_cores():
    wl = W.make_delta("limits_tc", m=MAX_DELTA_ROWS, k_in=64, n_out=64, max_rank=16, rank=16, alpha=16.0,
                      rslora=False, seed=904)
    assert L.lora_delta_geometry(wl.m, 16, 64, 64)["dense"] == 1
    g_out, g_xa = gpu_delta(wl)
    _sampled(wl, g_out, g_xa, [128, wl.m // 2, wl.m])
    assert L.lora_read_device_status(clear=True) == 0
