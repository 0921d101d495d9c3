"""ctypes binding of libgather_lora.so (the C ABI in include/gather_lora.h).

Argument marshalling only: every step of the fold runs in the library's CUDA
kernels. Device buffers may be passed as torch tensors (their data_ptr() is
used) or as raw integer addresses; ``stream`` may be a torch.cuda.Stream, a raw
cudaStream_t integer, or None for torch's current stream. The functions carry
the C names. A missing library raises at first use: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgather_lora.so")

LORA_OK = 0
STATUS_NAMES = {-1: "LORA_ERR_NULL", -2: "LORA_ERR_SIZE", -3: "LORA_ERR_STRIDE",
                -4: "LORA_ERR_ALIGN", -5: "LORA_ERR_WINDOW", -6: "LORA_ERR_CUDA",
                -7: "LORA_ERR_UNSUPPORTED", -8: "LORA_ERR_FLAGS"}
LORA_DEV_MISALIGNED = 0x1
INPUTS_READY = 0x1         # LORA_INPUTS_READY (call flag)
MOE_M_TILE = 64
TMAP_MIN_RANK = 32         # LORA_TMAP_MIN_RANK: a_tmaps are used from this max_rank up
DELTA_DENSE_MIN_ROWS = 256  # LORA_DELTA_DENSE_MIN_ROWS: lora_delta's tensor-core path from this m up


class LoraError(RuntimeError):
    def __init__(self, code: int, text: str):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {text}")
        self.code = code


_lib = None


def load():
    """Load libgather_lora.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with gather_lora_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    lib.lora_bgmv.restype = ctypes.c_int
    U32 = ctypes.c_uint32
    lib.lora_bgmv.argtypes = [P, I64, P, I64, P, I32, P, P, P, I32, I32, I32, I32, P, P, U32, P]
    lib.lora_moe_grouped_fold.restype = ctypes.c_int
    lib.lora_moe_grouped_fold.argtypes = [P, I64, I32, P, I64, P, I32, P, I32, P, I32, I32, I32,
                                          P, P, P, I32, I32, I32, I32, P, I32, U32, P]
    lib.lora_moe_gather_bgmv.restype = ctypes.c_int
    lib.lora_moe_gather_bgmv.argtypes = [P, I64, P, I64, P, I32, I32, P, I32, I32,
                                         P, P, P, I32, I32, I32, I32, P, P, U32, P]
    lib.lora_delta.restype = ctypes.c_int
    lib.lora_delta.argtypes = [P, I64, P, I64, I32, P, P, ctypes.c_float, I32, I32, I32, P, P]
    lib.lora_delta_geometry.restype = ctypes.c_int
    lib.lora_delta_geometry.argtypes = [I32, I32, I32, I32, I32, ctypes.POINTER(I64)]
    lib.lora_encode_a_tmaps.restype = ctypes.c_int
    lib.lora_encode_a_tmaps.argtypes = [P, I32, I32, I32, P]
    lib.lora_selftest_wait_timeout.restype = ctypes.c_int
    lib.lora_selftest_wait_timeout.argtypes = [I64, P]
    lib.lora_last_error.restype = ctypes.c_char_p
    lib.lora_last_error.argtypes = []
    lib.lora_read_device_status.restype = ctypes.c_int
    lib.lora_read_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
    lib.lora_launch_geometry.restype = ctypes.c_int
    lib.lora_launch_geometry.argtypes = [ctypes.c_int, I32, I32, I32, I32, I32, ctypes.POINTER(I64)]
    lib.lora_grouped_down_wc.restype = I32
    lib.lora_grouped_down_wc.argtypes = [I32, I32]
    lib.lora_gather_row_token.restype = I32
    lib.lora_gather_row_token.argtypes = [I32, I32]
    lib.lora_gather_bgmv_grids.restype = ctypes.c_int
    lib.lora_gather_bgmv_grids.argtypes = [I32, I32, I32, ctypes.POINTER(I32), ctypes.POINTER(I32)]
    lib.lora_grouped_down_windows.restype = I32
    lib.lora_grouped_down_windows.argtypes = [I32, I32, ctypes.POINTER(I32), ctypes.POINTER(I32), I32]
    lib.lora_pack_expert_tables.restype = ctypes.c_int
    lib.lora_pack_expert_tables.argtypes = [ctypes.POINTER(I32), ctypes.POINTER(ctypes.c_uint64),
                                            ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_float),
                                            I32, ctypes.POINTER(ctypes.c_uint64),
                                            ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_float),
                                            I32, ctypes.POINTER(I32)]
    _lib = lib
    return lib


def _addr(v):
    if v is None:
        return None
    if isinstance(v, int):
        return v or None
    return v.data_ptr() or None       # torch tensor


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None      # torch.cuda.Stream


def _check(rc: int) -> int:
    if rc != LORA_OK:
        raise LoraError(rc, load().lora_last_error().decode())
    return rc


def lora_bgmv(x, x_row_stride, base_out, out_row_stride, seq_slot, n, a_table, b_table,
              scale_table, max_loras, max_rank, k_in, n_out, xa=None, stream=None, a_tmaps=None,
              flags=0):
    """Routed bgmv fold (see lora_bgmv in include/gather_lora.h). flags: 0 or
    INPUTS_READY."""
    return _check(load().lora_bgmv(_addr(x), x_row_stride, _addr(base_out), out_row_stride,
                                   _addr(seq_slot), n, _addr(a_table), _addr(b_table),
                                   _addr(scale_table), max_loras, max_rank, k_in, n_out,
                                   _addr(xa), _addr(a_tmaps), int(flags), _stream(stream)))


def lora_delta(x, x_row_stride, base_out, out_row_stride, m, a, b, scale, max_rank, k_in, n_out,
               xa=None, stream=None):
    """One adapter pair folded into all m rows (see lora_delta in include/gather_lora.h)."""
    return _check(load().lora_delta(_addr(x), x_row_stride, _addr(base_out), out_row_stride, m,
                                    _addr(a), _addr(b), float(scale), max_rank, k_in, n_out,
                                    _addr(xa), _stream(stream)))


DELTA_GEOMETRY_KEYS = ("dense", "cluster", "ring_stages", "stage_bytes", "smem_bytes", "ctas")


def lora_delta_geometry(m, max_rank, k_in, n_out, sm_count=0) -> dict:
    out = (ctypes.c_int64 * 6)()
    _check(load().lora_delta_geometry(m, max_rank, k_in, n_out, sm_count, out))
    return dict(zip(DELTA_GEOMETRY_KEYS, list(out)))


def lora_moe_grouped_fold(x, x_row_stride, base_out, out_row_stride, expert_offsets, num_experts,
                          sorted_token_ids, te, row_adapter, num_tokens, row_offset, row_end,
                          a_table, b_table, scale_table, max_loras, max_rank, k_in, n_out,
                          xa=None, stream=None, x_gather=False, xa_rows=None, flags=0):
    """MoE grouped fold of one window (see lora_moe_grouped_fold in include/gather_lora.h).
    x_gather: x is token-major and sorted row r reads row sorted_token_ids[r] (gate/up).
    xa_rows: rows allocated for xa; taken from the tensor's size (numel // max_rank) when
    xa is a tensor and xa_rows is not given. flags: 0 or INPUTS_READY."""
    if xa is None:
        xa_rows = 0
    elif xa_rows is None:
        if isinstance(xa, int):
            raise ValueError("xa given as a raw address needs xa_rows")
        xa_rows = xa.numel() // max_rank
    return _check(load().lora_moe_grouped_fold(
        _addr(x), x_row_stride, 1 if x_gather else 0, _addr(base_out), out_row_stride, _addr(expert_offsets),
        num_experts, _addr(sorted_token_ids), te, _addr(row_adapter), num_tokens, row_offset,
        row_end, _addr(a_table), _addr(b_table), _addr(scale_table), max_loras, max_rank, k_in,
        n_out, _addr(xa), int(xa_rows), int(flags), _stream(stream)))


def lora_moe_gather_bgmv(x, x_row_stride, base_out, out_row_stride, indices, n_rows, top_k,
                         row_adapter, num_tokens, num_experts, a_table, b_table, scale_table,
                         max_loras, max_rank, k_in, n_out, xa=None, stream=None, a_tmaps=None,
                         flags=0):
    """Decode-path MoE fold over flat (token, slot) rows (see lora_moe_gather_bgmv in
    include/gather_lora.h). flags: 0 or INPUTS_READY."""
    return _check(load().lora_moe_gather_bgmv(
        _addr(x), x_row_stride, _addr(base_out), out_row_stride, _addr(indices), n_rows, top_k,
        _addr(row_adapter), num_tokens, num_experts, _addr(a_table), _addr(b_table),
        _addr(scale_table), max_loras, max_rank, k_in, n_out, _addr(xa), _addr(a_tmaps),
        int(flags), _stream(stream)))


def lora_encode_a_tmaps(a_ptrs, max_rank: int, k_in: int):
    """Host-encoded A tensor maps (see lora_encode_a_tmaps): returns a uint8 numpy
    array of len(a_ptrs) * 128 bytes to copy to (64-byte aligned) device memory."""
    import numpy as np
    ptrs = np.ascontiguousarray(np.asarray(a_ptrs, dtype=np.uint64))
    n = int(ptrs.shape[0])
    buf = np.zeros(n * 128 + 64, dtype=np.uint8)
    off = (-buf.ctypes.data) % 64
    maps = buf[off:off + n * 128]
    _check(load().lora_encode_a_tmaps(ptrs.ctypes.data if n else None, n, max_rank, k_in,
                                      maps.ctypes.data if n else None))
    return maps.copy()


def lora_last_error() -> str:
    return load().lora_last_error().decode()


def lora_selftest_wait_timeout(limit_cycles, stream=None):
    """Diagnostic: one bounded wait that runs out (see include/gather_lora.h)."""
    return _check(load().lora_selftest_wait_timeout(int(limit_cycles), _stream(stream)))


def lora_read_device_status(stream=None, clear=True) -> int:
    v = ctypes.c_uint32(0)
    _check(load().lora_read_device_status(_stream(stream), ctypes.byref(v), int(clear)))
    return int(v.value)


GEOMETRY_KEYS = ("cluster", "rows_per_tile", "k_slice", "j_slice", "k_chunk", "j_chunk",
                 "ring_stages", "clusters", "smem_bytes", "a_tiled", "tc", "direct")


def lora_launch_geometry(moe, rows, max_loras, max_rank, k_in, n_out) -> dict:
    out = (ctypes.c_int64 * 12)()
    _check(load().lora_launch_geometry(int(moe), rows, max_loras, max_rank, k_in, n_out, out))
    return dict(zip(GEOMETRY_KEYS, list(out)))


def lora_grouped_down_wc(row_offset: int, row_end: int) -> int:
    return int(load().lora_grouped_down_wc(row_offset, row_end))


def lora_gather_row_token(row: int, top_k: int) -> int:
    return int(load().lora_gather_row_token(row, top_k))


def lora_gather_bgmv_grids(max_rank: int, n_out: int, n_slots: int):
    """((shrink grid), (expand grid)) of the pages' decode gather fold, or ValueError."""
    sh, ex = (ctypes.c_int32 * 3)(), (ctypes.c_int32 * 3)()
    if load().lora_gather_bgmv_grids(max_rank, n_out, n_slots, sh, ex) != 0:
        raise ValueError("bad gather grid arguments")
    return tuple(sh), tuple(ex)


def lora_grouped_down_windows(total_rows: int, cap: int):
    """Returns the list of (start, end) windows, or raises ValueError."""
    n_max = max(1, (max(total_rows, 0) + max(cap, 1) - 1) // max(cap, 1))
    starts = (ctypes.c_int32 * n_max)()
    ends = (ctypes.c_int32 * n_max)()
    n = int(load().lora_grouped_down_windows(total_rows, cap, starts, ends, n_max))
    if n < 0:
        raise ValueError(f"lora_grouped_down_windows({total_rows}, {cap}) -> {n}")
    return [(starts[i], ends[i]) for i in range(n)]


def lora_pack_expert_tables(entries, table_len=None):
    """entries: list of (expert_id, a_addr, b_addr, scale). Returns None for an
    empty list, else (a_table, b_table, scale_table) lists of n_experts entries."""
    n = len(entries)
    ids = (ctypes.c_int32 * max(n, 1))(*[e[0] for e in entries])
    aa = (ctypes.c_uint64 * max(n, 1))(*[e[1] for e in entries])
    bb = (ctypes.c_uint64 * max(n, 1))(*[e[2] for e in entries])
    ss = (ctypes.c_float * max(n, 1))(*[e[3] for e in entries])
    tl = table_len if table_len is not None else max([e[0] for e in entries] + [0]) + 1
    at = (ctypes.c_uint64 * max(tl, 1))()
    bt = (ctypes.c_uint64 * max(tl, 1))()
    st = (ctypes.c_float * max(tl, 1))()
    ne = ctypes.c_int32(0)
    rc = load().lora_pack_expert_tables(ids, aa, bb, ss, n, at, bt, st, tl, ctypes.byref(ne))
    if rc == 1:
        return None
    if rc != 0:
        raise ValueError(f"lora_pack_expert_tables -> {rc}")
    k = ne.value
    return list(at[:k]), list(bt[:k]), list(st[:k])
