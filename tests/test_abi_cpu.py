"""The C-ABI library on the CPU: it loads, exports every declared entry point,
rejects bad arguments on the host before any CUDA call, and its pure helpers
follow the MoE window / table rules. No kernel is launched here."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from gather_lora_gb300 import lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gather_lora.h")
FAKE = 0x100000            # a non-NULL, 16-byte aligned address that is never dereferenced


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not os.path.exists(L.LIB_PATH):
        from gather_lora_gb300 import build
        build.build()
    L.load()


def declared_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int32_t|int)\s+(lora_\w+)\s*\(", src, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("lora_bgmv", "lora_moe_grouped_fold", "lora_moe_gather_bgmv", "lora_last_error",
              "lora_read_device_status",
              "lora_launch_geometry", "lora_grouped_down_wc", "lora_grouped_down_windows",
              "lora_pack_expert_tables", "lora_gather_row_token", "lora_gather_bgmv_grids"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(L.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    nm = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = set(re.findall(r" T (lora_\w+)$", nm.stdout, re.M))
        assert set(declared_functions()) <= exported


def _bgmv(**kw):
    a = dict(x=FAKE, xs=4096, out=FAKE, os=4096, seq=FAKE, n=4, at=FAKE, bt=FAKE, sc=FAKE, L=8,
             R=16, k=4096, no=4096, xa=FAKE, maps=None, flags=0)
    a.update(kw)
    return L.load().lora_bgmv(a["x"], a["xs"], a["out"], a["os"], a["seq"], a["n"], a["at"],
                              a["bt"], a["sc"], a["L"], a["R"], a["k"], a["no"], a["xa"], a["maps"],
                              a["flags"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), -2), (dict(n=8193), -2), (dict(L=0), -2), (dict(L=5000), -2),
    (dict(R=0), -2), (dict(R=264), -2), (dict(R=12), -4), (dict(k=4), -2), (dict(k=4100, xs=4104), -4),
    (dict(no=4097, os=8192), -4), (dict(xs=4088), -3), (dict(os=100, no=128), -3),
    (dict(xs=4100), -4), (dict(x=None), -1), (dict(out=None), -1), (dict(seq=None), -1),
    (dict(at=None), -1), (dict(bt=None), -1), (dict(sc=None), -1), (dict(x=FAKE + 2), -4),
    (dict(out=FAKE + 8), -4), (dict(xa=FAKE + 4), -4), (dict(maps=FAKE + 32), -4),
    (dict(flags=2), -8), (dict(flags=0x80000001), -8), (dict(flags=1, x=FAKE + 2), -4),
])
def test_bgmv_rejects_bad_arguments_before_launch(kw, code):
    assert _bgmv(**kw) == code
    assert L.lora_last_error()


def test_bgmv_zero_rows_is_a_no_op():
    assert _bgmv(n=0, x=None, out=None) == 0
    assert L.lora_last_error() == ""


def _moe(**kw):
    a = dict(x=FAKE, xs=768, xg=0, out=FAKE, os=2048, off=FAKE, E=128, sti=FAKE, te=16384, ra=FAKE,
             nt=2048, lo=0, hi=4096, at=FAKE, bt=FAKE, sc=FAKE, L=16, R=16, k=768, no=2048, xa=FAKE,
             xa_rows=4096, flags=0)
    a.update(kw)
    return L.load().lora_moe_grouped_fold(a["x"], a["xs"], a["xg"], a["out"], a["os"], a["off"], a["E"],
                                          a["sti"], a["te"], a["ra"], a["nt"], a["lo"], a["hi"],
                                          a["at"], a["bt"], a["sc"], a["L"], a["R"], a["k"], a["no"],
                                          a["xa"], a["xa_rows"], a["flags"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(E=0), -2), (dict(E=1025), -2), (dict(L=0), -2), (dict(te=-1), -2),
    (dict(lo=-1), -5), (dict(lo=10, hi=5), -5), (dict(hi=16385), -5), (dict(R=4), -2),
    (dict(k=770, xs=776), -4), (dict(xs=700), -3), (dict(x=None), -1), (dict(off=None), -1),
    (dict(sti=None), -1), (dict(at=None), -1), (dict(x=FAKE + 2), -4),
    (dict(sti=None, ra=None, xg=1), -1),
    (dict(xa_rows=4095), -2), (dict(xa_rows=-1), -2), (dict(lo=100, hi=5000, xa_rows=4899), -2),
    (dict(flags=4), -8), (dict(flags=1, x=FAKE + 2), -4),
])
def test_moe_rejects_bad_arguments_before_launch(kw, code):
    assert _moe(**kw) == code


def test_moe_xa_rows_cover_the_window():
    """xa needs the window's rows (written at the local row r - row_offset), not te's;
    with xa NULL the count is not looked at. The check runs before any launch."""
    assert _moe(lo=100, hi=5000, xa_rows=4899) == -2
    assert "xa holds 4899 rows" in L.lora_last_error()
    assert _moe(lo=0, hi=0, xa_rows=0, x=FAKE + 2) == -4      # reaches the alignment check
    assert _moe(xa=None, xa_rows=-5, x=FAKE + 2) == -4         # xa_rows ignored without xa


def test_moe_table_count_and_persistent_grid():
    """The MoE tables hold at most LORA_MAX_LORAS (adapter, expert) entries; the
    grid is persistent (one CTA per SM, fewer for small windows: at least 16 rows
    each), so even the largest window launches a fixed grid."""
    assert _moe(L=33, E=128) == -2            # 33 x 128 > 4096 table entries
    assert "table entries" in L.lora_last_error()
    big = 2 ** 31 - 1
    assert L.lora_launch_geometry(1, big, 16, 16, 768, 2048)["clusters"] == 152
    assert L.lora_launch_geometry(1, 40, 16, 16, 768, 2048)["clusters"] == 3
    assert L.lora_launch_geometry(1, 0, 16, 16, 768, 2048)["clusters"] == 1
    assert _moe(te=big, lo=0, hi=big, xa=None, x=FAKE + 2) == -4   # passes the size checks


def test_strided_k_fold_geometry_takes_256_column_chunks():
    """With A as tensor-map boxes at rank 64, a 256-column k chunk of the strided K
    fold needs a 40.4 KB stage: the 42 KB target takes it (two stages) rather than
    128-column chunks in three."""
    g = L.lora_launch_geometry(16, 256, 128, 64, 4096, 1024)
    assert g["a_tiled"] == 1 and g["cluster"] == 4 and g["k_slice"] == 1024
    assert g["k_chunk"] == 256 and g["ring_stages"] == 2 and g["smem_bytes"] <= 113 * 1024


def test_moe_cta_shape_follows_the_larger_half():
    """The MoE fold runs two CTAs of 8 + 2 warps per SM when its shrink is the larger
    half (k_in > n_out: the gate/up form) and one CTA of 12 + 4 warps otherwise (the
    down form); the grid is then up to two CTAs per SM."""
    up = L.lora_launch_geometry(1, 1 << 20, 16, 16, 2048, 768)
    down = L.lora_launch_geometry(1, 1 << 20, 16, 16, 768, 2048)
    assert up["direct"] == 1 and up["clusters"] == 2 * 152 and up["smem_bytes"] <= 113 * 1024
    assert down["direct"] == 0 and down["clusters"] == 152
    assert L.lora_launch_geometry(1, 4096, 16, 16, 2048, 768)["clusters"] == 256


def _gather(**kw):
    a = dict(x=FAKE, xs=768, out=FAKE, os=2048, idx=FAKE, n=512, k=8, ra=FAKE, nt=64, E=128,
             at=FAKE, bt=FAKE, sc=FAKE, L=16, R=16, kin=768, no=2048, xa=FAKE, maps=None, flags=0)
    a.update(kw)
    return L.load().lora_moe_gather_bgmv(a["x"], a["xs"], a["out"], a["os"], a["idx"], a["n"],
                                         a["k"], a["ra"], a["nt"], a["E"], a["at"], a["bt"],
                                         a["sc"], a["L"], a["R"], a["kin"], a["no"], a["xa"],
                                         a["maps"], a["flags"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(n=-1), -2), (dict(n=8193), -2), (dict(k=0), -2), (dict(nt=-1), -2), (dict(E=0), -2),
    (dict(E=1025), -2), (dict(L=0), -2), (dict(L=33), -2), (dict(R=4), -2), (dict(xs=700), -3),
    (dict(x=None), -1), (dict(idx=None), -1), (dict(at=None), -1), (dict(x=FAKE + 2), -4),
    (dict(flags=8), -8),
])
def test_gather_bgmv_rejects_bad_arguments_before_launch(kw, code):
    assert _gather(**kw) == code
    assert L.lora_last_error()


def test_gather_bgmv_zero_rows_is_a_no_op():
    assert _gather(n=0, x=None, idx=None) == 0


def test_grouped_down_wc():
    assert L.lora_grouped_down_wc(0, 16384) == 256          # full window: ceil(te / 64)
    assert L.lora_grouped_down_wc(0, 4096) == 64
    assert L.lora_grouped_down_wc(4096, 4097) == 1
    assert L.lora_grouped_down_wc(100, 100) == 1              # at least one tile
    assert L.lora_grouped_down_wc(0, 65) == 2
    assert L.lora_grouped_down_wc(5, 4) == -1
    for lo, hi in [(0, 1), (3, 131), (64, 128), (7, 7000)]:
        assert L.lora_grouped_down_wc(lo, hi) == max(1, -(-(hi - lo) // 64))


def test_encode_a_tmaps_checks_arguments():
    enc = L.load().lora_encode_a_tmaps
    assert enc(None, 0, 16, 4096, None) == 0                   # nothing to encode
    assert enc(None, -1, 16, 4096, None) == -2
    assert enc(None, 2, 4, 4096, None) == -2                   # max_rank out of range
    assert enc(None, 2, 16, 4100, None) == -4                  # k_in not a multiple of 8
    assert enc(None, 2, 16, 4096, None) == -1                  # pointers required
    ptrs = (ctypes.c_uint64 * 2)(0x10000, 0x20000)
    buf = ctypes.create_string_buffer(2 * 128 + 64)
    base = ctypes.addressof(buf)
    aligned = base + (-base) % 64
    assert enc(ptrs, 2, 16, 4096, aligned + 16) == -4          # maps_out not 64-byte aligned
    bad = (ctypes.c_uint64 * 2)(0x10000, 0x20008)
    rc = enc(bad, 2, 16, 4096, aligned)
    assert rc in (-4, -6)     # misaligned A pointer; or no CUDA driver on this machine


def test_gather_row_token():
    assert L.lora_gather_row_token(0, 8) == 0
    assert L.lora_gather_row_token(7, 8) == 0
    assert L.lora_gather_row_token(8, 8) == 1
    assert L.lora_gather_row_token(511, 8) == 63
    assert L.lora_gather_row_token(5, 1) == 5
    assert L.lora_gather_row_token(-1, 8) == -1 and L.lora_gather_row_token(3, 0) == -1


def test_gather_bgmv_grids():
    assert L.lora_gather_bgmv_grids(16, 2048, 512) == ((4, 512, 1), (512, 512, 1))
    assert L.lora_gather_bgmv_grids(24, 1030, 3) == ((6, 3, 1), (258, 3, 1))   # ceil(./4)
    assert L.lora_gather_bgmv_grids(8, 8, 0) == ((2, 0, 1), (2, 0, 1))
    with pytest.raises(ValueError):
        L.lora_gather_bgmv_grids(0, 8, 1)
    with pytest.raises(ValueError):
        L.lora_gather_bgmv_grids(8, 8, -1)


def test_grouped_down_windows():
    assert L.lora_grouped_down_windows(16384, 4096) == [(0, 4096), (4096, 8192), (8192, 12288), (12288, 16384)]
    assert L.lora_grouped_down_windows(10, 4) == [(0, 4), (4, 8), (8, 10)]
    assert L.lora_grouped_down_windows(0, 4) == []
    assert L.lora_grouped_down_windows(3, 4096) == [(0, 3)]
    with pytest.raises(ValueError):
        L.lora_grouped_down_windows(10, 0)
    rng = np.random.default_rng(0)
    for _ in range(50):
        total, cap = int(rng.integers(0, 5000)), int(rng.integers(1, 700))
        w = L.lora_grouped_down_windows(total, cap)
        covered = [r for lo, hi in w for r in range(lo, hi)]
        assert covered == list(range(total))
        assert all(0 < hi - lo <= cap for lo, hi in w)


def test_pack_expert_tables():
    assert L.lora_pack_expert_tables([]) is None
    a, b, s = L.lora_pack_expert_tables([(2, 0x1000, 0x2000, 0.5), (0, 0x3000, 0x4000, 2.0)])
    assert a == [0x3000, 0, 0x1000] and b == [0x4000, 0, 0x2000] and s == [2.0, 0.0, 0.5]
    a, b, s = L.lora_pack_expert_tables([(1, 0x10, 0x20, 1.0), (1, 0x30, 0x40, 3.0)])
    assert a == [0, 0x30] and b == [0, 0x40] and s == [0.0, 3.0]   # the last entry wins
    with pytest.raises(ValueError):
        L.lora_pack_expert_tables([(-1, 1, 2, 1.0)])
    with pytest.raises(ValueError):
        L.lora_pack_expert_tables([(5, 1, 2, 1.0)], table_len=3)


def test_geometry_depends_on_shapes_only():
    """The per-row arithmetic (cluster split, k chunks) must not depend on n."""
    for (L_, R, k, no) in [(32, 16, 4096, 4096), (128, 64, 4096, 1024), (64, 128, 12288, 4096),
                           (4, 8, 256, 256), (3, 256, 2056, 4096)]:
        g1 = L.lora_launch_geometry(0, 1, L_, R, k, no)
        g2 = L.lora_launch_geometry(0, 512, L_, R, k, no)
        for key in ("cluster", "k_slice", "k_chunk", "j_slice", "j_chunk"):
            assert g1[key] == g2[key]
        assert g1["smem_bytes"] <= 227 * 1024
        assert g1["k_chunk"] % 16 == 0 and g1["j_chunk"] % 16 == 0
        assert g1["k_slice"] * g1["cluster"] >= k and g1["j_slice"] * g1["cluster"] >= no


def test_every_supported_shape_has_a_launch_geometry():
    """Every max_rank of the supported range (multiples of 8 up to 256), k_in and
    n_out from 8 to 2^20, for each fold kind (bgmv with and without A maps, the
    decode gather fold, the MoE fold): a geometry exists, fits the 227 KB of
    shared memory a CTA may take, has at least two ring stages, and its cluster
    slices cover k_in and n_out."""
    dims = (8, 64, 136, 768, 2048, 4096, 12288, 65536, 1 << 20)
    for R in range(8, 256 + 1, 8):      # LORA_MAX_RANK
        for k in dims:
            for no in dims:
                for kind in (0, 16, 2, 18, 1):
                    g = L.lora_launch_geometry(kind, 512, 16 if kind == 1 else 64, R, k, no)
                    assert g["smem_bytes"] <= 227 * 1024 and g["ring_stages"] >= 2, (kind, R, k, no)
                    assert g["cluster"] in (1, 2, 4, 8)
                    assert g["k_slice"] * g["cluster"] >= k and g["j_slice"] * g["cluster"] >= no
                    assert g["k_chunk"] % 8 == 0 and g["j_chunk"] % 8 == 0
                # the largest batch and slot count (the planner's scratch is the largest)
                for kind in (0, 16, 2):
                    g = L.lora_launch_geometry(kind, 8192, 4096, R, k, 2048)
                    assert g["smem_bytes"] <= 227 * 1024 and g["ring_stages"] >= 2, (kind, R, k)


def test_bgmv_grid_bounds_every_routing():
    """clusters = n/rt + min(n, max_loras) covers sum_s ceil(count_s / rt) for any routing."""
    rng = np.random.default_rng(1)
    for _ in range(200):
        n, L_ = int(rng.integers(1, 600)), int(rng.integers(1, 300))
        g = L.lora_launch_geometry(0, n, L_, 16, 1024, 1024)
        rt = g["rows_per_tile"]
        slots = rng.integers(-1, L_, size=n) if rng.random() < 0.5 else np.zeros(n, int)
        counts = np.bincount(slots[slots >= 0], minlength=L_)
        need = int(np.sum((counts + rt - 1) // rt))
        assert need <= g["clusters"]


def test_gather_geometry_has_no_cluster_split():
    g = L.lora_launch_geometry(2, 512, 2048, 16, 768, 2048)
    assert g["cluster"] == 1 and g["clusters"] == 512 // 8 + 512 and g["rows_per_tile"] == 8
    assert L.lora_launch_geometry(0, 512, 2048, 16, 768, 2048)["cluster"] == 4


def test_moe_geometry_persistent():
    """The MoE grid: one CTA per SM (152 without a device), fewer for windows of
    under 16 rows per CTA; passes of 64 rows; the arithmetic (k chunk, j chunk)
    from the shapes alone, whatever the window."""
    g = L.lora_launch_geometry(1, 4096, 16, 16, 768, 2048)
    assert g["rows_per_tile"] == 64 and g["cluster"] == 1 and g["clusters"] == 152
    assert g["ring_stages"] >= 2 and g["smem_bytes"] <= 227 * 1024
    assert L.lora_launch_geometry(1, 100, 1, 16, 768, 2048)["clusters"] == 7
    for rows in (0, 100, 4096, 16384, 10 ** 6):
        h = L.lora_launch_geometry(1, rows, 16, 16, 768, 2048)
        assert (h["k_chunk"], h["j_chunk"], h["k_slice"], h["j_slice"]) == \
            (g["k_chunk"], g["j_chunk"], g["k_slice"], g["j_slice"])


def test_tensor_maps_only_from_the_minimum_rank():
    m = re.search(r"#define LORA_TMAP_MIN_RANK (\d+)", open(HEADER).read())
    assert m and int(m.group(1)) == L.TMAP_MIN_RANK
    for mode, rows, tables in ((0, 64, 32), (2, 512, 2048)):
        for rank in (8, 16, L.TMAP_MIN_RANK - 8):
            args = (rows, tables, rank, 4096, 4096)
            assert L.lora_launch_geometry(mode + 16, *args) == L.lora_launch_geometry(mode, *args)
            assert L.lora_launch_geometry(mode + 16, *args)["a_tiled"] == 0
        for rank in (L.TMAP_MIN_RANK, 64, 128):
            g = L.lora_launch_geometry(mode + 16, rows, tables, rank, 4104, 4096)
            assert g["a_tiled"] == 1 and g["k_chunk"] % 64 == 0
            assert L.lora_launch_geometry(mode, rows, tables, rank, 4104, 4096)["a_tiled"] == 0
    # the grouped MoE fold loads A rows whatever it is given
    assert L.lora_launch_geometry(17, 4096, 16, 64, 768, 2048) == L.lora_launch_geometry(1, 4096, 16, 64, 768, 2048)


def _delta(**kw):
    a = dict(x=FAKE, xs=4096, out=FAKE, os=4096, m=512, a=FAKE, b=FAKE, sc=1.0, R=64, k=4096, no=4096,
             xa=None)
    a.update(kw)
    return L.load().lora_delta(a["x"], a["xs"], a["out"], a["os"], a["m"], a["a"], a["b"], a["sc"],
                               a["R"], a["k"], a["no"], a["xa"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(m=-1), -2), (dict(m=(1 << 20) + 1), -2), (dict(R=0), -2), (dict(R=264), -2), (dict(R=12), -4),
    (dict(k=4100, xs=4104), -4), (dict(xs=4088), -3), (dict(os=100, no=128), -3), (dict(x=None), -1),
    (dict(out=None), -1), (dict(a=None), -1), (dict(b=None), -1), (dict(a=FAKE + 8), -4),
    (dict(b=FAKE + 2), -4), (dict(xa=FAKE + 4), -4), (dict(out=FAKE + 8), -4),
])
def test_delta_rejects_bad_arguments_before_launch(kw, code):
    assert _delta(**kw) == code
    assert L.lora_last_error()


def test_delta_zero_rows_is_a_no_op():
    assert _delta(m=0, x=None, out=None) == 0


def test_delta_geometry():
    g = L.lora_delta_geometry(4096, 16, 4096, 4096, 152)
    assert g["dense"] == 1 and g["cluster"] == 4 and g["ctas"] == 128 and g["ring_stages"] == 8
    g = L.lora_delta_geometry(4096, 128, 12288, 4096, 152)
    assert g["dense"] == 1 and g["cluster"] == 4 and g["ring_stages"] == 4
    assert L.lora_delta_geometry(16384, 64, 4096, 4096, 152)["cluster"] == 1    # 128 tiles fill the SMs
    assert L.lora_delta_geometry(1024, 64, 4096, 4096, 152)["cluster"] == 8
    assert L.lora_delta_geometry(4096, 64, 64, 4096, 152)["cluster"] == 1       # one k-chunk
    for r, ns in ((16, 8), (32, 7), (64, 6), (128, 4)):
        g = L.lora_delta_geometry(L.DELTA_DENSE_MIN_ROWS, r, 4096, 4096, 152)
        assert g["dense"] == 1 and g["ring_stages"] == ns and 116 * 1024 < g["smem_bytes"] <= 227 * 1024
        assert g["stage_bytes"] % 1024 == 0
    # small m or a rank the tensor-core path does not take: the routed engine
    assert L.lora_delta_geometry(L.DELTA_DENSE_MIN_ROWS - 1, 64, 4096, 4096, 152)["dense"] == 0
    for r in (8, 24, 48, 256):
        assert L.lora_delta_geometry(4096, r, 4096, 4096, 152)["dense"] == 0
    m = re.search(r"#define LORA_DELTA_DENSE_MIN_ROWS (\d+)", open(HEADER).read())
    assert m and int(m.group(1)) == L.DELTA_DENSE_MIN_ROWS


def test_tcgen05_shrink_geometry():
    """The bgmv shrink moves to tcgen05 only with A tensor maps at max_rank 128 (units of 16 rows)."""
    assert L.lora_launch_geometry(16, 512, 64, 128, 12288, 4096)["tc"] == 1
    assert L.lora_launch_geometry(0, 512, 64, 128, 12288, 4096)["tc"] == 0     # no maps
    assert L.lora_launch_geometry(16, 256, 128, 64, 4096, 1024)["tc"] == 0     # rank 64
    assert L.lora_launch_geometry(17, 4096, 16, 128, 768, 2048)["tc"] == 0     # grouped MoE
    assert L.lora_launch_geometry(18, 512, 2048, 128, 768, 2048)["tc"] == 0    # gather units: 8 rows


def test_unit_numbering_rule():
    """Direct numbering unless the grid is more than one wave of CTAs and the slots
    are many for the rows (152 SMs without a device)."""
    assert L.lora_launch_geometry(0, 64, 32, 16, 4096, 4096)["direct"] == 1      # one wave
    assert L.lora_launch_geometry(16, 512, 64, 128, 12288, 4096)["direct"] == 1  # few slots per row
    assert L.lora_launch_geometry(16, 256, 128, 64, 4096, 1024)["direct"] == 0   # many sparse slots
    assert L.lora_launch_geometry(0, 16, 128, 16, 4096, 4096)["direct"] == 0     # more slots than rows
    for args in [(0, 64, 32, 16, 4096, 4096), (16, 256, 128, 64, 4096, 1024)]:
        g = L.lora_launch_geometry(*args)
        assert g["clusters"] == args[1] // g["rows_per_tile"] + min(args[1], args[2])
