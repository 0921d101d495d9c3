"""Failure path of the bounded waits, on the GPU without a fault (-m gpu).

Every mbarrier wait in the fold kernels gives up after a limit of SM clocks,
records LORA_DEV_TIMEOUT in the device status word and lets the kernel finish.
Here a wait that nothing completes runs out on purpose (a short limit): the
host reads the status bit, clears it, and the context still runs folds that
match the oracle.
"""
from __future__ import annotations

import time

import pytest
import torch

from gather_lora_gb300 import lib as L
from gather_lora_gb300 import workloads as W
from gpu_util import gpu_bgmv, oracle_bgmv, require_gpu
from parity import compare_bgmv

pytestmark = pytest.mark.gpu

LORA_DEV_TIMEOUT = 0x2


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    require_gpu()
    L.lora_read_device_status(clear=True)


def test_wait_that_runs_out_sets_the_timeout_bit_and_returns():
    assert L.lora_read_device_status(clear=True) == 0
    t0 = time.perf_counter()
    L.lora_selftest_wait_timeout(4_000_000)          # ~2 ms at 2 GHz
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    assert elapsed < 5.0                              # it gave up; it did not hang
    assert L.lora_read_device_status(clear=True) & LORA_DEV_TIMEOUT
    assert L.lora_read_device_status(clear=True) == 0


def test_context_still_folds_after_a_timeout():
    L.lora_selftest_wait_timeout(1_000_000)
    torch.cuda.synchronize()
    assert L.lora_read_device_status(clear=True) & LORA_DEV_TIMEOUT
    wl = W.tiny_bgmv()
    g_out, g_xa = gpu_bgmv(wl)
    o_out, o_xa, o_d = oracle_bgmv(wl)
    compare_bgmv(wl, g_out, o_out, g_xa, o_xa, o_d)
    assert L.lora_read_device_status(clear=True) == 0


def test_limit_is_checked_on_the_host():
    with pytest.raises(L.LoraError):
        L.lora_selftest_wait_timeout(0)
