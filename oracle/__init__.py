"""CPU oracle for the routed multi-LoRA fold: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (``gather_lora_gb300``)
never imports it, and the two share no code: the oracle is plain single-threaded
C (``oracle.c``) built with gcc, loaded here through ctypes.

What each function computes, and the page passages it follows, is written at the
top of ``oracle.c``. Parity of every function is pinned by the ``-m "not gpu"``
tests in ``tests/test_oracle_pins.py`` (exact-integer closed forms, exact
rational brute force, invariants of the pages).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lib = None


def build(out_path: str | None = None, defines: tuple[str, ...] = ()) -> str:
    """Compile oracle.c with gcc into a shared library and return its path."""
    out = out_path or _LIB_PATH
    cmd = ["gcc", *_CFLAGS, *[f"-D{d}" for d in defines], "-o", out, _SRC, "-lm"]
    subprocess.run(cmd, check=True, cwd=_HERE)
    return out


def _stale() -> bool:
    if not os.path.exists(_LIB_PATH):
        return True
    t = os.path.getmtime(_LIB_PATH)
    return any(os.path.getmtime(os.path.join(_HERE, f)) > t for f in ("oracle.c", "oracle.h"))


def _bind(lib):
    u16p = ctypes.c_void_p
    lib.ora_f32_of_bf16.restype = ctypes.c_float
    lib.ora_f32_of_bf16.argtypes = [ctypes.c_uint16]
    lib.ora_bf16_of_f32.restype = ctypes.c_uint16
    lib.ora_bf16_of_f32.argtypes = [ctypes.c_float]
    lib.ora_bf16_of_f64.restype = ctypes.c_uint16
    lib.ora_bf16_of_f64.argtypes = [ctypes.c_double]
    lib.ora_lora_bgmv.restype = ctypes.c_int
    lib.ora_lora_bgmv.argtypes = [
        u16p, ctypes.c_int64, u16p, ctypes.c_int64, u16p, ctypes.c_int32,
        u16p, u16p, u16p, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        u16p, u16p, ctypes.c_int32]
    lib.ora_lora_delta.restype = ctypes.c_int
    lib.ora_lora_delta.argtypes = [
        u16p, ctypes.c_int64, u16p, ctypes.c_int64, ctypes.c_int32,
        u16p, u16p, ctypes.c_float,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        u16p, u16p, ctypes.c_int32]
    lib.ora_lora_moe_grouped_fold.restype = ctypes.c_int
    lib.ora_lora_moe_grouped_fold.argtypes = [
        u16p, ctypes.c_int64, ctypes.c_int32, u16p, ctypes.c_int64,
        u16p, ctypes.c_int32, u16p, ctypes.c_int32, u16p, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32,
        u16p, u16p, u16p, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        u16p, u16p, ctypes.c_int32]
    lib.ora_lora_moe_gather_bgmv.restype = ctypes.c_int
    lib.ora_lora_moe_gather_bgmv.argtypes = [
        u16p, ctypes.c_int64, u16p, ctypes.c_int64,
        u16p, ctypes.c_int32, ctypes.c_int32, u16p, ctypes.c_int32, ctypes.c_int32,
        u16p, u16p, u16p, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
        u16p, u16p, ctypes.c_int32]
    return lib


def load(path: str | None = None):
    """Load (building first if missing or stale) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    override = os.environ.get("GATHER_LORA_ORACLE_LIB")   # mutation tests load a planted copy
    if _lib is None and override:
        _lib = _bind(ctypes.CDLL(override))
    if _lib is None:
        if _stale():
            build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    return None if a is None else a.ctypes.data


def _table(arrays) -> tuple[np.ndarray, list]:
    """Host pointer table from a list of uint16 arrays (None = NULL entry)."""
    keep = [None if a is None else np.ascontiguousarray(a, dtype=np.uint16) for a in arrays]
    tab = np.array([0 if a is None else a.ctypes.data for a in keep], dtype=np.uint64)
    return tab, keep


def bf16_of_f32(v: float) -> int:
    return int(load().ora_bf16_of_f32(float(v)))


def bf16_of_f64(v: float) -> int:
    return int(load().ora_bf16_of_f64(float(v)))


def f32_of_bf16(h: int) -> float:
    return float(load().ora_f32_of_bf16(int(h)))


def lora_bgmv(x, x_row_stride, base_out, out_row_stride, seq_slot, a_list, b_list,
              scale_table, max_rank, k_in, n_out, mode=0, lib=None):
    """Apply the routed bgmv fold in place on the host.

    x: uint16 array holding n rows at ``x_row_stride`` elements; base_out: uint16
    array (modified in place) holding n rows at ``out_row_stride`` elements,
    the folded segment being the first n_out elements of each row; seq_slot:
    int32 [n]; a_list / b_list: per-slot uint16 arrays [max_rank, k_in] /
    [n_out, max_rank] or None (NULL entry); scale_table: float32 [max_loras].
    Returns (xa [n, max_rank] uint16, d [n, n_out] uint16); rows that are not
    routed keep zeros there.
    """
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    assert base_out.dtype == np.uint16 and base_out.flags.c_contiguous
    seq_slot = np.ascontiguousarray(seq_slot, dtype=np.int32)
    n = int(seq_slot.shape[0])
    a_tab, a_keep = _table(a_list)
    b_tab, b_keep = _table(b_list)
    scale = np.ascontiguousarray(scale_table, dtype=np.float32)
    max_loras = len(a_list)
    assert len(b_list) == max_loras and scale.shape[0] >= max_loras
    xa = np.zeros((max(n, 1), max_rank), dtype=np.uint16)
    d = np.zeros((max(n, 1), n_out), dtype=np.uint16)
    rc = lib.ora_lora_bgmv(_ptr(x), x_row_stride, _ptr(base_out), out_row_stride,
                           _ptr(seq_slot), n, _ptr(a_tab), _ptr(b_tab), _ptr(scale), max_loras,
                           max_rank, k_in, n_out, _ptr(xa), _ptr(d), mode)
    if rc != 0:
        raise ValueError(f"oracle lora_bgmv rejected its arguments (rc={rc})")
    return xa[:n], d[:n]


def lora_delta(x, x_row_stride, base_out, out_row_stride, m, a, b, scale, max_rank, k_in,
               n_out, mode=0, lib=None):
    """Fold one adapter pair into all m rows of base_out in place ("lora_delta.rs",
    apply_lora_delta).

    x: uint16 array holding m rows at ``x_row_stride`` elements; base_out: uint16
    array (modified in place) of m rows at ``out_row_stride`` elements, the first
    n_out of each folded; a: uint16 [max_rank, k_in]; b: uint16 [n_out, max_rank];
    scale: the f32 scale. Returns (xa [m, max_rank], d [m, n_out]) as uint16.
    """
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    assert base_out.dtype == np.uint16 and base_out.flags.c_contiguous
    a = np.ascontiguousarray(a, dtype=np.uint16)
    b = np.ascontiguousarray(b, dtype=np.uint16)
    xa = np.zeros((max(m, 1), max_rank), dtype=np.uint16)
    d = np.zeros((max(m, 1), n_out), dtype=np.uint16)
    rc = lib.ora_lora_delta(_ptr(x), x_row_stride, _ptr(base_out), out_row_stride, m, _ptr(a), _ptr(b),
                            float(np.float32(scale)), max_rank, k_in, n_out, _ptr(xa), _ptr(d), mode)
    if rc != 0:
        raise ValueError(f"oracle lora_delta rejected its arguments (rc={rc})")
    return xa[:m], d[:m]


def lora_moe_grouped_fold(x, x_row_stride, base_out, out_row_stride, expert_offsets,
                          sorted_token_ids, row_adapter, num_tokens, row_offset, row_end,
                          a_list, b_list, scale_table, max_rank, k_in, n_out, mode=0,
                          lib=None, x_gather=False):
    """Apply the MoE grouped fold to one window [row_offset, row_end) in place.

    Tables are lists of length max_loras * num_experts, adapter-major
    (index a * num_experts + e). row_adapter may be None (every row adapter 0).
    x_gather: x is token-major and sorted row r reads row sorted_token_ids[r]
    (gate/up); otherwise x is the sorted [te, k_in] activation (down).
    Returns (xa [row_end-row_offset, max_rank], d [te, n_out]).
    """
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    assert base_out.dtype == np.uint16 and base_out.flags.c_contiguous
    offs = np.ascontiguousarray(expert_offsets, dtype=np.int32)
    num_experts = int(offs.shape[0]) - 1
    sti = None if sorted_token_ids is None else np.ascontiguousarray(sorted_token_ids, dtype=np.int32)
    te = int(sti.shape[0]) if sti is not None else int(offs[-1])
    ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, dtype=np.int32)
    a_tab, a_keep = _table(a_list)
    b_tab, b_keep = _table(b_list)
    assert len(a_list) % num_experts == 0
    max_loras = len(a_list) // num_experts
    scale = np.ascontiguousarray(scale_table, dtype=np.float32)
    xa = np.zeros((max(row_end - row_offset, 1), max_rank), dtype=np.uint16)
    d = np.zeros((max(te, 1), n_out), dtype=np.uint16)
    rc = lib.ora_lora_moe_grouped_fold(
        _ptr(x), x_row_stride, 1 if x_gather else 0, _ptr(base_out), out_row_stride,
        _ptr(offs), num_experts, _ptr(sti), te, _ptr(ra), num_tokens,
        row_offset, row_end, _ptr(a_tab), _ptr(b_tab), _ptr(scale), max_loras,
        max_rank, k_in, n_out, _ptr(xa), _ptr(d), mode)
    if rc != 0:
        raise ValueError(f"oracle lora_moe_grouped_fold rejected its arguments (rc={rc})")
    return xa[: row_end - row_offset], d[:te]


def lora_moe_gather_bgmv(x, x_row_stride, base_out, out_row_stride, indices, top_k,
                         row_adapter, num_tokens, num_experts, a_list, b_list, scale_table,
                         max_rank, k_in, n_out, mode=0, lib=None):
    """Apply the decode-path MoE fold over flat (token, slot) rows in place.

    Row r: expert indices[r], adapter row_adapter[r // top_k] (None: adapter 0),
    table index a * num_experts + e. Returns (xa [n_rows, max_rank], d [n_rows, n_out]).
    """
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    assert base_out.dtype == np.uint16 and base_out.flags.c_contiguous
    idx = np.ascontiguousarray(indices, dtype=np.int32)
    n_rows = int(idx.shape[0])
    ra = None if row_adapter is None else np.ascontiguousarray(row_adapter, dtype=np.int32)
    a_tab, a_keep = _table(a_list)
    b_tab, b_keep = _table(b_list)
    assert len(a_list) % num_experts == 0
    max_loras = len(a_list) // num_experts
    scale = np.ascontiguousarray(scale_table, dtype=np.float32)
    xa = np.zeros((max(n_rows, 1), max_rank), dtype=np.uint16)
    d = np.zeros((max(n_rows, 1), n_out), dtype=np.uint16)
    rc = lib.ora_lora_moe_gather_bgmv(
        _ptr(x), x_row_stride, _ptr(base_out), out_row_stride, _ptr(idx), n_rows, top_k,
        _ptr(ra), num_tokens, num_experts, _ptr(a_tab), _ptr(b_tab), _ptr(scale), max_loras,
        max_rank, k_in, n_out, _ptr(xa), _ptr(d), mode)
    if rc != 0:
        raise ValueError(f"oracle lora_moe_gather_bgmv rejected its arguments (rc={rc})")
    return xa[:n_rows], d[:n_rows]
