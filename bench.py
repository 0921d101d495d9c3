#!/usr/bin/env python3
"""Benchmark of the routed LoRA fold on GB300 (one JSON line on stdout).

Headline workload: the MoE grouped down fold (2048 tokens x top-8 of 128
experts = 16384 expert-sorted rows, k_in 768, n_out 2048, 16 adapters x 128
experts at max_rank 16, 20% of tokens without an adapter), folded in its four
windows of 4096 sorted rows: a step is the four lora_moe_grouped_fold calls over
one batch. The other fold workloads (decode q_proj, strided K fold into an
interleaved QKV row, dense FFN down_proj, the MoE gate/up form, both MoE folds
as one call over all rows, the decode-path MoE gather fold, single-adapter
prefill deltas) are measured the same way and reported under "workloads".

Calls pass LORA_INPUTS_READY (routing, x and adapters of a step are written
before its calls are issued, as in a model layer): each call plans and runs its
shrink while the kernel before it finishes. Every figure is also taken with
calls that wait for the previous kernel first (--wait-previous makes those the
main figures).

Timing: inputs are resident in HBM; consecutive steps rotate through enough
independent copies of every input (adapter pools included) to exceed 2x the L2
size, so no step finds its data in L2. The K steps are replayed from CUDA graphs
and timed with CUDA events on the launching stream, bracketed by a barrier and
a device synchronize; with several ranks the time is the max over ranks.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (the reference arm of this comparison),
unchanged, on all host cores (disjoint rows per thread) for the same workload,
metric, unit and config.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "routed LoRA fold rows/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
HEADLINE = "moe_down_fold"
SIDE_WORKLOADS = ("decode_qproj_bgmv", "qkv_kfold_bgmv", "ffn_down_bgmv", "moe_gateup_fold",
                  "moe_down_fold_one_launch", "moe_gateup_fold_one_launch",
                  "moe_decode_gather", "prefill_qproj_delta", "prefill_down_delta")
FALLBACK_HBM_GBS = 6800.0
KERNEL_NAMES = {"bgmv": "lora_bgmv_fold_kernel", "moe": "lora_moe_fold_kernel",
                "gather": "lora_bgmv_fold_kernel", "delta": "lora_dense_fold_kernel"}


# ----------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments, trailing blanks and blank lines."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def kernel_source_digest() -> str:
    """Digest of the kernel and launcher code (comments excluded: they do not
    change what runs), which keys the recorded ncu counters."""
    h = hashlib.sha256()
    for rel in ("gather_lora_gb300/csrc/kernels.cu", "gather_lora_gb300/csrc/common.cuh",
                "gather_lora_gb300/csrc/fold_types.h", "gather_lora_gb300/csrc/abi.cpp",
                "gather_lora_gb300/csrc/dense.cu", "gather_lora_gb300/csrc/dense_types.h",
                "gather_lora_gb300/csrc/tc05.cuh"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernels are unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_digest") != kernel_source_digest():
        return None
    v = d.get("workloads", {}).get(workload, {}).get("dram_bytes_per_launch")
    return float(v) if v is not None else None


def bgmv_algorithmic_bytes(wl) -> dict:
    """Bytes one launch must move: each routed row's x row, out row read+write and
    xa row write+read, plus each distinct routed adapter's padded A and B once,
    plus the routing vector and the three table entries of each distinct slot."""
    import numpy as np
    routed = [(i, int(s)) for i, s in enumerate(wl.seq_slot) if 0 <= s < wl.max_loras and wl.present[s]]
    slots = sorted({s for _, s in routed})
    per_row = wl.k_in * 2 + wl.n_out * 2 * 2 + wl.max_rank * 2 * 2
    per_adapter = wl.max_rank * wl.k_in * 2 + wl.n_out * wl.max_rank * 2
    total = len(routed) * per_row + len(slots) * (per_adapter + 20) + wl.n * 4
    return dict(bytes=int(total), routed_rows=len(routed), rows=int(wl.n), adapters=len(slots),
                per_row=per_row, per_adapter=per_adapter,
                flops=int(2 * len(routed) * wl.max_rank * (wl.k_in + wl.n_out)))


def delta_algorithmic_bytes(wl) -> dict:
    """Bytes of one single-adapter delta: every row's x row, out row read+write and
    xa row write+read (as for the routed fold), plus the pair's A and B once."""
    per_row = wl.k_in * 2 + wl.n_out * 2 * 2 + wl.max_rank * 2 * 2
    per_adapter = wl.max_rank * wl.k_in * 2 + wl.n_out * wl.max_rank * 2
    total = wl.m * per_row + per_adapter
    return dict(bytes=int(total), routed_rows=int(wl.m), rows=int(wl.m), adapters=1,
                per_row=per_row, per_adapter=per_adapter,
                flops=int(2 * wl.m * wl.max_rank * (wl.k_in + wl.n_out)))


def moe_algorithmic_bytes(wl) -> dict:
    E = wl.num_experts
    routed, pairs = 0, set()
    for lo, hi in wl.windows():
        for r in range(lo, hi):
            e = int((wl.expert_offsets[1:] <= r).sum())
            a = 0 if wl.row_adapter is None else int(wl.row_adapter[wl.sorted_token_ids[r]])
            if a < 0 or a >= wl.max_loras or not wl.present[a * E + e]:
                continue
            routed += 1
            pairs.add((a * E + e, lo))          # an adapter is read once per window it serves
    per_row = wl.k_in * 2 + wl.n_out * 2 * 2 + wl.max_rank * 2 * 2 + 4 + 4
    per_adapter = wl.max_rank * wl.k_in * 2 + wl.n_out * wl.max_rank * 2
    total = routed * per_row + len(pairs) * (per_adapter + 20) + len(wl.windows()) * (E + 1) * 4
    return dict(bytes=int(total), routed_rows=routed, rows=int(wl.te), adapters=len(pairs),
                per_row=per_row, per_adapter=per_adapter,
                flops=int(2 * routed * wl.max_rank * (wl.k_in + wl.n_out)))


def gather_algorithmic_bytes(wl) -> dict:
    """Decode-path MoE fold: like the bgmv, with the (adapter, expert) table entry of
    each row as its slot, plus the expert index per row and the adapter per token."""
    E = wl.num_experts
    routed, tables = 0, set()
    for r in range(wl.n_rows):
        e, t = int(wl.indices[r]), r // wl.top_k
        a = 0 if wl.row_adapter is None else int(wl.row_adapter[t])
        if not 0 <= e < E or a < 0 or a >= wl.max_loras or not wl.present[a * E + e]:
            continue
        routed += 1
        tables.add(a * E + e)
    per_row = wl.k_in * 2 + wl.n_out * 2 * 2 + wl.max_rank * 2 * 2 + 4
    per_adapter = wl.max_rank * wl.k_in * 2 + wl.n_out * wl.max_rank * 2
    total = routed * per_row + len(tables) * (per_adapter + 20) + wl.num_tokens * 4
    return dict(bytes=int(total), routed_rows=routed, rows=int(wl.n_rows), adapters=len(tables),
                per_row=per_row, per_adapter=per_adapter,
                flops=int(2 * routed * wl.max_rank * (wl.k_in + wl.n_out)))


USE_TMAPS = True     # load A as 2-D TMA boxes through host-encoded tensor maps (--no-tmaps: rows)
READY = 1            # calls pass LORA_INPUTS_READY (--wait-previous: 0)
E2E_SPLIT_INPUTS = True   # e2e: base_out's host copy on its own stream beside the other inputs


def a_load(wl) -> str:
    """How the fold loads A for this workload (the library's own choice: the
    bgmv and gather folds take the maps from LORA_TMAP_MIN_RANK up; the grouped
    MoE fold loads rows)."""
    from gather_lora_gb300 import lib as L
    kind = workload_kind(wl)
    if kind == "delta":
        dense = L.lora_delta_geometry(wl.m, wl.max_rank, wl.k_in, wl.n_out)["dense"]
        return ("2-D TMA boxes into tcgen05 tensor cores (tensor maps encoded per call)" if dense
                else "one TMA copy per row")
    tiled = 0
    if USE_TMAPS and kind == "bgmv":
        tiled = L.lora_launch_geometry(16, wl.n, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out)["a_tiled"]
    elif USE_TMAPS and kind == "gather":
        tiled = L.lora_launch_geometry(18, wl.n_rows, wl.max_loras * wl.num_experts, wl.max_rank,
                                       wl.k_in, wl.n_out)["a_tiled"]
    return "2-D TMA boxes via tensor maps" if tiled else "one TMA copy per row"


def a_maps_for(a_table, max_rank: int, k_in: int):
    """Device A tensor maps for a device table (encoded once, as at adapter load), or None."""
    if not USE_TMAPS:
        return None
    import torch
    from gather_lora_gb300 import lib as L
    maps = L.lora_encode_a_tmaps(a_table.cpu().numpy().astype("uint64"), max_rank, k_in)
    return torch.from_numpy(maps).to(a_table.device)


def workload_kind(wl) -> str:
    from gather_lora_gb300 import workloads as W
    if isinstance(wl, W.MoeGatherWorkload):
        return "gather"
    if isinstance(wl, W.DeltaWorkload):
        return "delta"
    return "moe" if isinstance(wl, W.MoeWorkload) else "bgmv"


def algorithmic_bytes(wl) -> dict:
    k = workload_kind(wl)
    return {"bgmv": bgmv_algorithmic_bytes, "moe": moe_algorithmic_bytes,
            "gather": gather_algorithmic_bytes, "delta": delta_algorithmic_bytes}[k](wl)


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_selector: str):
        self.sel = device_selector
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", self.sel], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
            time.sleep(0.3)          # let the first sample land before the timed region
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def smi_selector(torch, dev) -> str:
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        return str(getattr(dev, "index", 0) or 0)


# ------------------------------------------------------------- device runs
class BgmvRunner:
    def __init__(self, wl, copies, device):
        import torch
        from gather_lora_gb300 import workloads as W
        self.wl = wl
        base = W.bgmv_to_device(wl, device)
        self.copies = [base] + [self._clone(base, wl) for _ in range(copies - 1)]
        self.maps = [a_maps_for(d.a_table, wl.max_rank, wl.k_in) for d in self.copies]
        self.launches_per_step = 1
        self.flags = READY

    @staticmethod
    def _clone(d, wl):
        import torch
        from gather_lora_gb300 import workloads as W
        a_pool, b_pool = d.a_pool.clone(), d.b_pool.clone()
        out = d.out_buf.clone()
        return W.DeviceBgmv(
            x=d.x.clone(), out_buf=out, out_ptr=out.data_ptr() + 2 * wl.out_offset,
            seq_slot=d.seq_slot.clone(), a_pool=a_pool, b_pool=b_pool,
            a_table=W._table_of(a_pool, wl.present, a_pool.device),
            b_table=W._table_of(b_pool, wl.present, b_pool.device), scale=d.scale.clone(),
            xa=d.xa.clone())

    def bytes_per_copy(self):
        d = self.copies[0]
        return sum(t.numel() * t.element_size() for t in (d.x, d.out_buf, d.a_pool, d.b_pool))

    def step(self, c, stream):
        from gather_lora_gb300 import lib as L
        wl, d = self.wl, self.copies[c]
        L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, wl.n,
                    d.a_table, d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out,
                    xa=d.xa, stream=stream, a_tmaps=self.maps[c], flags=self.flags)


class MoeRunner:
    def __init__(self, wl, copies, device):
        from gather_lora_gb300 import workloads as W
        self.wl = wl
        self.windows = wl.windows()
        self.copies = [W.moe_to_device(wl, device, xa_rows=wl.cap) for _ in range(copies)]
        self.launches_per_step = len(self.windows)
        self.flags = READY

    def bytes_per_copy(self):
        d = self.copies[0]
        return sum(t.numel() * t.element_size() for t in (d.x, d.out_buf, d.a_pool, d.b_pool))

    def step(self, c, stream):
        from gather_lora_gb300 import lib as L
        wl, d = self.wl, self.copies[c]
        for lo, hi in self.windows:
            L.lora_moe_grouped_fold(d.x, wl.k_in, d.out_buf, wl.n_out, d.expert_offsets,
                                    wl.num_experts, d.sorted_token_ids, wl.te, d.row_adapter,
                                    wl.num_tokens, lo, hi, d.a_table, d.b_table, d.scale,
                                    wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                                    stream=stream, x_gather=wl.x_gather, flags=self.flags)


class GatherRunner:
    def __init__(self, wl, copies, device):
        from gather_lora_gb300 import workloads as W
        self.wl = wl
        self.copies = [W.gather_to_device(wl, device) for _ in range(copies)]
        self.maps = [a_maps_for(d.a_table, wl.max_rank, wl.k_in) for d in self.copies]
        self.launches_per_step = 1
        self.flags = READY

    def bytes_per_copy(self):
        d = self.copies[0]
        return sum(t.numel() * t.element_size() for t in (d.x, d.out_buf, d.a_pool, d.b_pool))

    def step(self, c, stream):
        from gather_lora_gb300 import lib as L
        wl, d = self.wl, self.copies[c]
        L.lora_moe_gather_bgmv(d.x, wl.k_in, d.out_buf, wl.n_out, d.indices, wl.n_rows, wl.top_k,
                               d.row_adapter, wl.num_tokens, wl.num_experts, d.a_table, d.b_table,
                               d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                               stream=stream, a_tmaps=self.maps[c], flags=self.flags)


class DeltaRunner:
    def __init__(self, wl, copies, device):
        from gather_lora_gb300 import workloads as W
        self.wl = wl
        self.copies = [W.delta_to_device(wl, device) for _ in range(copies)]
        self.launches_per_step = 1
        self.flags = 0      # lora_delta takes no flags

    def bytes_per_copy(self):
        d = self.copies[0]
        return sum(t.numel() * t.element_size() for t in (d.x, d.out_buf, d.a, d.b))

    def step(self, c, stream):
        from gather_lora_gb300 import lib as L
        wl, d = self.wl, self.copies[c]
        L.lora_delta(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, wl.m, d.a, d.b, wl.scale,
                     wl.max_rank, wl.k_in, wl.n_out, xa=d.xa, stream=stream)


RUNNERS = {"bgmv": BgmvRunner, "moe": MoeRunner, "gather": GatherRunner, "delta": DeltaRunner}


def copies_needed(bytes_per_copy, l2_bytes, touched_per_step=None):
    """Input copies to rotate through so that a step never finds its data in L2:
    the bytes the steps of one rotation touch (the algorithmic bytes of a step,
    not the whole buffers: an adapter pool is mostly untouched by one batch)
    exceed 2x L2."""
    per = max(1, min(bytes_per_copy, touched_per_step or bytes_per_copy))
    return max(1, min(64, math.ceil(2 * l2_bytes / per)))


def time_steps(runner, steps, warmup, device, dist_ctx, sampler=None):
    """Warm up, capture CUDA graphs over the rotating copies, time exactly `steps` steps."""
    import torch
    C = len(runner.copies)
    stream = torch.cuda.Stream(device=device)
    with torch.cuda.stream(stream):
        for w in range(max(warmup, 1)):
            runner.step(w % C, stream)
    torch.cuda.synchronize(device)

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                runner.step(i % C, stream)
        return g

    per_graph = C * max(1, 64 // C) if C < 64 else C     # >= 64 launches per replay when cheap
    full, tail = divmod(steps, per_graph)
    g_full = capture(per_graph) if full else None
    g_tail = capture(tail) if tail else None
    for _ in range(2):                                   # graph warm-up (untimed)
        if g_full:
            g_full.replay()
        if g_tail:
            g_tail.replay()
    torch.cuda.synchronize(device)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    dist_ctx.barrier()
    torch.cuda.synchronize(device)
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(full):
                g_full.replay()
            if g_tail:
                g_tail.replay()
            end.record(stream)
        torch.cuda.synchronize(device)
    dist_ctx.barrier()
    ms = start.elapsed_time(end)
    return dist_ctx.max(ms), ms


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


class DistCtx:
    """Barrier and max-over-ranks; a no-op with one process."""

    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend)
            self.dist = dist
            self.backend = backend

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, v: float) -> float:
        return self._reduce(v, "max")

    def sum(self, v: float) -> float:
        return self._reduce(v, "sum")

    def _reduce(self, v, op):
        if self.dist is None:
            return v
        import torch
        dev = f"cuda:{self.local_rank}" if self.backend == "nccl" else "cpu"
        t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX if op == "max" else self.dist.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


def aggregate(rows_per_rank: float, ms_max: float, steps: int, n_ranks: int):
    """Whole-job throughput: all ranks' rows over the slowest rank's time."""
    total_rows = rows_per_rank * steps * n_ranks
    return total_rows / (ms_max / 1e3), ms_max / steps


# --------------------------------------------------------------- e2e
def _pinned(a):
    import numpy as np
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).pin_memory()


def e2e_run(wl, device, steps, warmup, copies):
    """The headline metric through the C ABI with host buffers. Every step copies
    the step's inputs from pinned host memory (bgmv: x, seq_slot, base_out; MoE:
    x, expert_offsets, sorted_token_ids, row_adapter, base_out), makes the fold's
    calls (MoE: one per window), and reads base_out back into pinned host memory,
    all inside the timed region. Steps are pipelined the way a serving loop would
    run them: the copies in, the calls and the copy out go on three streams, over
    at least two device copies of the inputs, so step i's inputs travel while step
    i - 1 folds and step i - 2's result comes back (events order each copy's uses).
    Returns rows/s, the H2D and D2H bytes per step, and the time and rows/s of one
    step's copies alone (in and out at once, no fold): the bound of the pipeline."""
    import torch
    from gather_lora_gb300 import lib as L
    from gather_lora_gb300 import workloads as W
    kind = workload_kind(wl)
    copies = max(2, copies)
    s_in, s_run, s_out = (torch.cuda.Stream(device=device) for _ in range(3))
    # the largest input (base_out) travels on a stream of its own, beside the others
    s_big = torch.cuda.Stream(device=device) if E2E_SPLIT_INPUTS else s_in
    if kind == "bgmv":
        devs = [W.bgmv_to_device(wl, device) for _ in range(copies)]
        maps = [a_maps_for(d.a_table, wl.max_rank, wl.k_in) for d in devs]
        pairs = lambda d: [(d.x, _pinned(wl.x)), (d.seq_slot, _pinned(wl.seq_slot)),
                           (d.out_buf, _pinned(wl.out_buf))]

        def call(c, d):
            L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, wl.n,
                        d.a_table, d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out,
                        xa=d.xa, stream=s_run, a_tmaps=maps[c])
        rows = wl.n
    elif kind == "moe":
        devs = [W.moe_to_device(wl, device, xa_rows=wl.cap) for _ in range(copies)]
        pairs = lambda d: [(d.x, _pinned(wl.x)), (d.expert_offsets, _pinned(wl.expert_offsets)),
                           (d.sorted_token_ids, _pinned(wl.sorted_token_ids)),
                           (d.row_adapter, _pinned(wl.row_adapter)), (d.out_buf, _pinned(wl.out_buf))]

        def call(c, d):
            # the first window follows this step's input copies (another stream): it
            # waits for everything; the later windows follow only the window before
            for j, (lo, hi) in enumerate(wl.windows()):
                L.lora_moe_grouped_fold(d.x, wl.k_in, d.out_buf, wl.n_out, d.expert_offsets,
                                        wl.num_experts, d.sorted_token_ids, wl.te, d.row_adapter,
                                        wl.num_tokens, lo, hi, d.a_table, d.b_table, d.scale,
                                        wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                                        stream=s_run, x_gather=wl.x_gather,
                                        flags=READY if j > 0 else 0)
        rows = wl.te
    else:
        raise ValueError(f"no end-to-end run for {kind}")
    host = [pairs(d) for d in devs]
    hres = [_pinned(wl.out_buf).clone().pin_memory() for _ in range(copies)]
    ev_in = [torch.cuda.Event() for _ in range(copies)]
    ev_run = [torch.cuda.Event() for _ in range(copies)]
    ev_out = [torch.cuda.Event() for _ in range(copies)]
    ev_big = [torch.cuda.Event() for _ in range(copies)]

    def one(i):
        c = i % copies
        d = devs[c]
        if i >= copies:                      # copy c's last result has left the device
            s_in.wait_event(ev_out[c])
            if s_big is not s_in:
                s_big.wait_event(ev_out[c])
        big = max(host[c], key=lambda ds: ds[1].numel() * ds[1].element_size())
        for pair in host[c]:
            with torch.cuda.stream(s_big if pair is big else s_in):
                pair[0].copy_(pair[1], non_blocking=True)
        ev_in[c].record(s_in)
        ev_big[c].record(s_big)
        s_run.wait_event(ev_in[c])
        s_run.wait_event(ev_big[c])
        call(c, d)
        ev_run[c].record(s_run)
        s_out.wait_event(ev_run[c])
        with torch.cuda.stream(s_out):
            hres[c].copy_(d.out_buf, non_blocking=True)
        ev_out[c].record(s_out)

    for i in range(warmup):
        one(i)
    torch.cuda.synchronize(device)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(s_in)
    for i in range(steps):
        one(warmup + i)
    for st in (s_in, s_big, s_run):
        s_out.wait_stream(st)
    end.record(s_out)
    torch.cuda.synchronize(device)
    ms = start.elapsed_time(end)
    # every step folds the same host inputs: each copy's last result must equal
    # one step run alone with nothing overlapping it
    last = [hres[c].clone() for c in range(copies)]
    with torch.cuda.stream(s_run):
        for dst, src in host[0]:
            dst.copy_(src, non_blocking=True)
        call(0, devs[0])
        hres[0].copy_(devs[0].out_buf, non_blocking=True)
    torch.cuda.synchronize(device)
    if not all(torch.equal(x, hres[0]) for x in last):
        raise RuntimeError("end-to-end steps gave different results from a step run alone")
    h2d = sum(src.numel() * src.element_size() for _, src in host[0])
    d2h = hres[0].numel() * hres[0].element_size()
    # The bound the pipeline can reach: one step's copies alone, its inputs in and
    # a result out at once on the same streams, with no fold (steps serialized).
    big0 = max(host[0], key=lambda ds: ds[1].numel() * ds[1].element_size())
    cur = torch.cuda.current_stream(device)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 20
    for r in range(reps + 3):
        if r == 3:
            t0.record(cur)
        for st in (s_in, s_big, s_out):
            st.wait_stream(cur)
        for pair in host[0]:
            with torch.cuda.stream(s_big if pair is big0 else s_in):
                pair[0].copy_(pair[1], non_blocking=True)
        with torch.cuda.stream(s_out):
            hres[1].copy_(devs[1].out_buf, non_blocking=True)
        for st in (s_in, s_big, s_out):
            cur.wait_stream(st)
    t1.record(cur)
    torch.cuda.synchronize(device)
    copy_ms = t0.elapsed_time(t1) / reps
    return rows * steps / (ms / 1e3), h2d, d2h, copy_ms, rows / (copy_ms / 1e3)


# ------------------------------------------------------------ CPU oracle
def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the baseline line."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_fold(wl, idx) -> None:
    """Fold the batch rows `idx` with the oracle, into a copy of their out rows."""
    import oracle
    out = wl.out_buf[idx].copy()
    seg = out.reshape(-1)[wl.out_offset:]
    oracle.lora_bgmv(wl.x[idx].reshape(-1), wl.x_row_stride, seg, wl.out_row_stride,
                     wl.seq_slot[idx], wl.a_list(), wl.b_list(), wl.scale, wl.max_rank,
                     wl.k_in, wl.n_out)


def oracle_fold_moe(wl, lo: int, hi: int) -> None:
    """Fold sorted rows [lo, hi) of an MoE workload with the oracle, into a copy of
    their out rows. The rows are handed over as the same problem on fewer rows:
    their x (or, for gate/up, the token-major x itself) and out rows, their token
    ids, and the expert offsets shifted by lo and clipped to [0, hi - lo], so every
    row keeps its expert, token and adapter."""
    import numpy as np
    import oracle
    offs = np.clip(wl.expert_offsets.astype(np.int64) - lo, 0, hi - lo).astype(np.int32)
    out = wl.out_buf[lo:hi].copy()
    x = wl.x if wl.x_gather else wl.x[lo:hi]
    oracle.lora_moe_grouped_fold(x, wl.k_in, out, wl.n_out, offs, wl.sorted_token_ids[lo:hi],
                                 wl.row_adapter, wl.num_tokens, 0, hi - lo, wl.a_list(), wl.b_list(),
                                 wl.scale, wl.max_rank, wl.k_in, wl.n_out, x_gather=wl.x_gather)


def oracle_total_rows(wl) -> int:
    return int(wl.te) if workload_kind(wl) == "moe" else int(wl.n)


def oracle_fold_rows(wl, start: int, count: int) -> None:
    """Fold `count` consecutive rows of the workload from `start` (wrapping)."""
    import numpy as np
    total = oracle_total_rows(wl)
    if workload_kind(wl) == "moe":
        lo = start % total
        hi = min(total, lo + count)
        oracle_fold_moe(wl, lo, hi)
        if lo + count > total:
            oracle_fold_moe(wl, 0, lo + count - total)
    else:
        oracle_fold(wl, np.arange(start, start + count) % total)


def oracle_rows_per_s(wl, budget_s: float, rows_per_call=None, threads: int = 1):
    """Time the oracle on the host over a bounded sample of the workload's rows.

    One thread folds rotating rows, rows_per_call at a time, until budget_s has
    passed. With several threads the rows go in rounds, as the reference arm's
    steps do: each round hands every thread its own rows_per_call rows (the
    oracle is a C call that releases the interpreter lock, so they run in
    parallel; the oracle itself is unchanged) and ends when all are done.
    Returns (rows/s over all threads, rows timed, seconds)."""
    from concurrent.futures import ThreadPoolExecutor
    total = oracle_total_rows(wl)
    # MoE: 1/16 of the sorted rows per call (1024 of 16384), the chunk the
    # reference arm gives each of 16 host threads
    default = max(1, -(-total // 16)) if workload_kind(wl) == "moe" else max(1, total // threads)
    rows_per_call = rows_per_call or default
    done = 0
    i0 = 0
    t0 = time.perf_counter()
    if threads == 1:
        while True:
            oracle_fold_rows(wl, i0, rows_per_call)
            done += rows_per_call
            i0 = (i0 + rows_per_call) % total
            if time.perf_counter() - t0 >= budget_s:
                break
    else:
        with ThreadPoolExecutor(threads) as ex:
            while True:
                starts = [(i0 + t * rows_per_call) % total for t in range(threads)]
                # a failed call re-raises here: it must not shorten the count silently
                list(ex.map(lambda st: oracle_fold_rows(wl, st, rows_per_call), starts))
                done += threads * rows_per_call
                i0 = (i0 + threads * rows_per_call) % total
                if time.perf_counter() - t0 >= budget_s:
                    break
    el = time.perf_counter() - t0
    return done / el, done, el


def _rows_word(wl) -> str:
    return "expert-sorted rows" if workload_kind(wl) == "moe" else "decode rows"


def cpu_baseline(wl, seconds: float) -> dict:
    """The oracle on all host cores (rows partitioned over threads), with its
    one-thread figure beside it; `seconds` of wall time in all."""
    threads = host_threads()
    v1, n1, s1 = oracle_rows_per_s(wl, seconds / 2)
    vt, nt, st = oracle_rows_per_s(wl, seconds / 2, threads=threads)
    return {"value": vt, "unit": "rows/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{nt} {_rows_word(wl)} of the {wl.name} batch in rounds of one call per host "
                      f"thread ({threads} threads, disjoint rows; {st:.1f} s)",
            "single_thread": {"value": v1, "cores": 1,
                              "sample": f"{n1} {_rows_word(wl)}, 1 host thread ({s1:.1f} s)"}}


def workload_config(wl, alg, world: int = 1) -> dict:
    """The `config` object of the JSON line: the workload and its shapes, the same
    in both arms (the reference arm is launched the same way, on the same N)."""
    kind = workload_kind(wl)
    cfg = {"workload": wl.name, "rows": alg["rows"], "routed_rows": alg["routed_rows"],
           "k_in": wl.k_in, "n_out": wl.n_out, "max_loras": getattr(wl, "max_loras", 1),
           "max_rank": wl.max_rank, "distinct_adapters": alg["adapters"]}
    if kind == "moe":
        cfg.update(num_experts=wl.num_experts, num_tokens=wl.num_tokens, te=wl.te,
                   windows=len(wl.windows()), window_rows=wl.cap, x_gather=bool(wl.x_gather))
    cfg["l2"] = "inputs rotate through device copies totalling more than 2x L2 between steps"
    cfg["inputs_ready"] = bool(READY)
    cfg["parallelism"] = f"replicas{world}"
    return cfg


def run_reference(args):
    """CPU oracle arm: same workload, metric, unit and config, on the host cores
    (each step's rows partitioned over all host threads)."""
    from concurrent.futures import ThreadPoolExecutor
    import numpy as np
    dctx = DistCtx()
    if dctx.rank != 0:
        dctx.close()
        return 0
    from gather_lora_gb300 import workloads as W
    import oracle
    wl = W.by_name(HEADLINE)
    oracle.load()
    threads = host_threads()
    total = oracle_total_rows(wl)
    state = {"i0": 0}

    def split(rows):
        per = max(1, -(-rows // threads))
        return [(o, min(per, rows - o)) for o in range(0, rows, per)]

    def step(ex, chunks, rows):
        i0 = state["i0"]
        list(ex.map(lambda c: oracle_fold_rows(wl, i0 + c[0], c[1]), chunks))
        state["i0"] = (i0 + rows) % total

    with ThreadPoolExecutor(threads) as ex:
        # calibrate on parallel steps of a part of the batch: seconds per row as the
        # threads actually share it (the second of two steps; the first starts them)
        cal_rows = min(total, 64 * threads)
        cal = split(cal_rows)
        for _ in range(2):
            t0 = time.perf_counter()
            step(ex, cal, cal_rows)
            t_row = (time.perf_counter() - t0) / cal_rows
        # rows per step: all warm-up and timed steps within about `budget` seconds,
        # at least one row per thread
        budget = 150.0
        rows_per_step = int(max(min(threads, total),
                                min(total, budget / max(args.steps + args.warmup, 1) / t_row)))
        chunks = split(rows_per_step)
        for _ in range(args.warmup):
            step(ex, chunks, rows_per_step)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            step(ex, chunks, rows_per_step)
        el = time.perf_counter() - t0
    value = rows_per_step * args.steps / el
    sample = (f"{rows_per_step} of the {total} {_rows_word(wl)} per step (rotating), split over "
              f"{len(chunks)} host threads")
    alg = algorithmic_bytes(wl)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el * 1e3 / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl, alg, dctx.world),
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": len(chunks), "kind": "oracle",
                         "sample": sample, "cpu_model": cpu_model()},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    dctx.close()
    return 0


# ------------------------------------------------------------------- main
def geometry_of(L, wl):
    kind = workload_kind(wl)
    if kind == "moe":
        return L.lora_launch_geometry(1, wl.cap, wl.max_loras if wl.row_adapter is not None else 1,
                                      wl.max_rank, wl.k_in, wl.n_out)
    if kind == "delta":
        return L.lora_delta_geometry(wl.m, wl.max_rank, wl.k_in, wl.n_out)
    if kind == "gather":
        return L.lora_launch_geometry(18 if USE_TMAPS else 2, wl.n_rows, wl.max_loras * wl.num_experts,
                                      wl.max_rank, wl.k_in, wl.n_out)
    return L.lora_launch_geometry(16 if USE_TMAPS else 0, wl.n, wl.max_loras, wl.max_rank,
                                  wl.k_in, wl.n_out)


def run_ours(args):
    import torch
    from gather_lora_gb300 import lib as L
    from gather_lora_gb300 import workloads as W
    dctx = DistCtx()
    device = torch.device("cuda", dctx.local_rank)
    torch.cuda.set_device(device)
    L.load()
    props = torch.cuda.get_device_properties(device)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2 ** 20)
    peak, peak_kind = measured_peaks()

    # headline
    head = args.only or HEADLINE
    wl = W.by_name(head)
    head_kind = workload_kind(wl)
    alg = algorithmic_bytes(wl)
    mk = RUNNERS[head_kind]
    probe = mk(wl, 1, device)
    C = copies_needed(probe.bytes_per_copy(), l2, alg["bytes"])
    runner = probe if C == 1 else mk(wl, C, device)
    del probe
    sampler = ClockSampler(smi_selector(torch, device)) if dctx.rank == 0 else None
    ms_max, ms_local = time_steps(runner, args.steps, args.warmup, device, dctx, sampler)
    value, ms_per_step = aggregate(alg["rows"], ms_max, args.steps, dctx.world)
    kernel_ms = ms_max / args.steps / runner.launches_per_step
    bytes_per_launch = alg["bytes"] / runner.launches_per_step
    achieved = bytes_per_launch / (kernel_ms / 1e3) / 1e9
    clocks = sampler.summary() if sampler else None
    launches = args.steps * runner.launches_per_step
    geometry = geometry_of(L, wl)

    def other_mode(r, steps_alt):
        """The same steps with the other call mode (calls that wait for the
        previous kernel first, or inputs-ready calls under --wait-previous)."""
        if workload_kind(r.wl) == "delta":
            return None
        r.flags = 0 if READY else L.INPUTS_READY
        m_alt, _ = time_steps(r, steps_alt, 5, device, dctx)
        r.flags = READY
        return m_alt / steps_alt

    alt_steps = int(max(50, min(args.steps, 2000.0 / max(ms_max / args.steps, 1e-3))))
    alt_ms = other_mode(runner, alt_steps)
    other = None
    if alt_ms is not None:
        alt_gbs = bytes_per_launch / (alt_ms / runner.launches_per_step / 1e3) / 1e9
        other = {"calls": "wait for the previous kernel" if READY else "LORA_INPUTS_READY",
                 "ms_per_step": alt_ms, "steps": alt_steps, "rows_per_s": alg["rows"] / (alt_ms / 1e3),
                 "achieved_gbs": alt_gbs, "frac_of_peak": alt_gbs / peak}

    # the other fold workloads (per-GPU numbers, same timing rules)
    side = {}
    for name in ([] if args.only else SIDE_WORKLOADS):
        w2 = W.by_name(name)
        a2 = algorithmic_bytes(w2)
        mk = RUNNERS[workload_kind(w2)]
        pr = mk(w2, 1, device)
        c2 = copies_needed(pr.bytes_per_copy(), l2, a2["bytes"])
        r2 = pr if c2 == 1 else mk(w2, c2, device)
        del pr
        # about 0.3 s of timed work, at least 20 steps
        est_ms = a2["bytes"] / (0.8 * peak * 1e9) * 1e3 + 0.004 * r2.launches_per_step
        k2 = int(max(20, min(20000, 300.0 / est_ms)))
        m2, _ = time_steps(r2, k2, 5, device, dctx)
        ms2 = m2 / k2
        gbs2 = a2["bytes"] / (ms2 / 1e3) / 1e9
        side[name] = {
            "rows_per_s": a2["rows"] / (ms2 / 1e3), "routed_rows_per_s": a2["routed_rows"] / (ms2 / 1e3),
            "ms_per_step": ms2, "launches_per_step": r2.launches_per_step, "steps": k2,
            "algorithmic_bytes": a2["bytes"], "achieved_gbs": gbs2, "frac_of_peak": gbs2 / peak,
            "frac_of_8tbs": gbs2 / 8000.0, "input_copies": len(r2.copies), "a_load": a_load(w2),
            "traffic": recorded_traffic(name), "inputs_ready": bool(r2.flags)}
        ms_o = other_mode(r2, k2)
        if ms_o is not None:
            gbs_o = a2["bytes"] / (ms_o / 1e3) / 1e9
            side[name]["other_calls"] = {"inputs_ready": not bool(r2.flags), "ms_per_step": ms_o,
                                         "achieved_gbs": gbs_o, "frac_of_peak": gbs_o / peak}
        if dctx.rank == 0 and not args.no_cpu_baseline and workload_kind(w2) in ("bgmv", "moe") \
                and not name.endswith("_one_launch"):
            vt, nt, st = oracle_rows_per_s(w2, 1.0, threads=host_threads())
            side[name]["cpu_oracle_rows_per_s"] = vt
            side[name]["cpu_oracle_sample"] = f"{nt} rows, {host_threads()} host threads ({st:.1f} s)"
        del r2
        torch.cuda.empty_cache()

    # e2e through the C ABI with host buffers
    e2e = None
    if head_kind in ("bgmv", "moe"):
        e2e_steps = max(50, min(args.steps, 2000 if head_kind == "bgmv" else 400))
        e2e_val, h2d, d2h, copy_ms, copy_rows = e2e_run(wl, device, e2e_steps, 10, C)
        e2e = {"value": dctx.sum(e2e_val), "unit": "rows/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps,
               "copy_bound": {"value": dctx.sum(copy_rows), "unit": "rows/s", "ms_per_step": copy_ms,
                              "what": "one step's host copies alone, inputs in and base_out out at once, "
                                      "no fold"},
               "frac_of_copy_bound": e2e_val / copy_rows}

    cpu = None
    if dctx.rank == 0 and not args.no_cpu_baseline and head_kind in ("bgmv", "moe"):
        cpu = cpu_baseline(wl, args.cpu_seconds)

    if dctx.rank == 0:
        config = workload_config(wl, alg, dctx.world)
        line = {
            "metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": dctx.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": config,
            "timing": {"input_copies": C,
                       "copies_mib": round(C * runner.bytes_per_copy() / 2 ** 20),
                       "l2_mib": round(l2 / 2 ** 20),
                       "graph": "CUDA graph replay, programmatic dependent launch",
                       "launches_per_step": runner.launches_per_step, "a_load": a_load(wl),
                       "calls": "LORA_INPUTS_READY" if READY else "wait for the previous kernel",
                       "other_calls": other},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": recorded_traffic(head),
                         "peak_kind": peak_kind, "kernel": KERNEL_NAMES[head_kind],
                         "algorithmic_bytes_per_launch": bytes_per_launch,
                         "kernel_ms": kernel_ms, "frac_of_8tbs": achieved / 8000.0},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "geometry": geometry,
            "workloads": side,
        }
        print(json.dumps(line), flush=True)
    dctx.close()
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100000)
    p.add_argument("--warmup", type=int, default=200)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-tmaps", action="store_true", help="load A row by row (no tensor maps)")
    p.add_argument("--only", default=None, help="time one named workload alone (profiling runs)")
    p.add_argument("--wait-previous", action="store_true",
                   help="calls wait for the previous kernel before reading anything (no LORA_INPUTS_READY)")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    global USE_TMAPS, READY
    USE_TMAPS = not args.no_tmaps
    READY = 0 if args.wait_previous else 1
    return run_reference(args) if args.impl == "reference" else run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
