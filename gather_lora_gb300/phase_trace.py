"""Phase breakdown of one fold launch per CTA (a diagnostic, GPU only).

Builds a variant of the library with -DGLORA_TRACE=1 (SM-clock stamps at the
phase boundaries of every CTA, one thread each; see kernels.cu) into
_build/trace, runs a workload's calls a few times the way bench.py does, and
prints, over the CTAs that folded rows in the last launch, the median / p90 /
max time from CTA entry to each phase boundary, the spread of entries and exits
on the global timer, and the rows per CTA.

    python -m gather_lora_gb300.phase_trace decode_qproj_bgmv [--ready] [--sm-mhz 2070]

The stamps themselves cost a few clocks each; the product library is built
without them.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
TRACE_LIB = os.path.join(HERE, "_build", "trace", "libgather_lora_trace.so")
SLOTS = 12
PHASES = [(1, "entry wait passed"), (2, "planned (engine entry)"), (3, "producer: first item issued"),
          (4, "shrink done"), (5, "exchange done"), (6, "first expand data"), (7, "expand done"),
          (8, "exit")]


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("workload")
    ap.add_argument("--ready", action="store_true", help="calls pass LORA_INPUTS_READY")
    ap.add_argument("--sm-mhz", type=float, default=2070.0, help="SM clock of the stamps")
    ap.add_argument("--calls", type=int, default=20)
    args = ap.parse_args(argv)

    import numpy as np
    import torch
    sys.path.insert(0, ROOT)
    from gather_lora_gb300 import build as B
    from gather_lora_gb300 import lib as L
    from gather_lora_gb300 import workloads as W

    B.build(defines=("GLORA_TRACE=1",), lib=TRACE_LIB, build_dir=os.path.join(HERE, "_build", "trace"))
    L.LIB_PATH = TRACE_LIB
    lib = L.load()
    lib.lora_trace_copy.argtypes = [ctypes.c_void_p, ctypes.c_int]
    flags = L.INPUTS_READY if args.ready else 0

    wl = W.by_name(args.workload)
    if hasattr(wl, "seq_slot"):
        d = W.bgmv_to_device(wl)
        maps = None
        if wl.max_rank >= L.TMAP_MIN_RANK:
            maps = torch.from_numpy(L.lora_encode_a_tmaps(d.a_table.cpu().numpy(), wl.max_rank, wl.k_in)).cuda()

        def call():
            L.lora_bgmv(d.x, wl.x_row_stride, d.out_ptr, wl.out_row_stride, d.seq_slot, wl.n, d.a_table,
                        d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in, wl.n_out, xa=d.xa,
                        a_tmaps=maps, flags=flags)
        windows = 1
    elif hasattr(wl, "expert_offsets"):
        d = W.moe_to_device(wl, xa_rows=wl.cap)

        def call():
            for lo, hi in wl.windows():
                L.lora_moe_grouped_fold(d.x, wl.k_in, d.out_buf, wl.n_out, d.expert_offsets, wl.num_experts,
                                        d.sorted_token_ids, wl.te, d.row_adapter, wl.num_tokens, lo, hi,
                                        d.a_table, d.b_table, d.scale, wl.max_loras, wl.max_rank, wl.k_in,
                                        wl.n_out, xa=d.xa, x_gather=wl.x_gather, flags=flags)
        windows = len(wl.windows())
    else:
        raise SystemExit(f"{args.workload}: bgmv and MoE workloads only")

    lib.lora_trace_clear()
    for _ in range(args.calls):
        call()
    torch.cuda.synchronize()
    buf = np.zeros((4096, SLOTS), dtype=np.uint64)
    rc = lib.lora_trace_copy(buf.ctypes.data, buf.nbytes)
    if rc != 0:
        raise SystemExit(f"trace copy failed ({rc})")
    t = buf.astype(np.int64)
    folded = (t[:, 2] > 0) & (t[:, 7] > 0)
    t = t[folded]
    us = lambda cyc: cyc / args.sm_mhz
    print(f"{args.workload}: {len(t)} CTAs folded rows in the last launch "
          f"({'inputs-ready' if args.ready else 'waiting'} calls, {windows} launch(es) per call)")
    print(f"{'phase (from CTA entry)':>30}   median      p90      max  (us)")
    for k, name in PHASES:
        v = us(t[:, k] - t[:, 0])
        print(f"{name:>30} {np.median(v):8.2f} {np.percentile(v, 90):8.2f} {v.max():8.2f}")
    g0, g1 = t[:, 9], t[:, 10]
    print(f"global timer: entries spread {(g0.max() - g0.min()) / 1e3:.2f} us, exits spread "
          f"{(g1.max() - g1.min()) / 1e3:.2f} us, first entry to last exit {(g1.max() - g0.min()) / 1e3:.2f} us")
    rows = t[:, 11]
    print(f"rows per CTA (last pass): min {rows.min()} median {int(np.median(rows))} max {rows.max()}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
