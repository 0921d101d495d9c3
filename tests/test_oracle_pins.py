"""Pins of the CPU oracle against things other than itself (CPU only).

Each pin targets a different plausible mistake:
  * BF16 rounding  -> torch's fp32->bf16 conversion and exact rational RNE;
  * routing, strides, layouts, transposes, padded rank, skip rules
                   -> the exact-integer special case, where every rounding is
                      exact and the result is an integer matrix product;
  * summation / rounding order of each stage
                   -> exact rational evaluation of the definition, within the
                      standard fp32 (fp64) summation error bound;
  * the pages' invariants: batched == one row per call, padded rank == true
    rank, skipped rows byte-identical, B = 0 leaves out unchanged, a one-hot x
    row gives that column of A, the MoE full window == its sub-windows, the MoE
    fold of one (adapter, expert) group == the bgmv of the same rows.
``test_oracle_mutants.py`` shows that planted mistakes fail these pins.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from gather_lora_gb300 import workloads as W
from oracle_refs import (bf16_bits_to_frac, exact_row, f32_to_frac, rne_bf16,
                         sum_is_unambiguous)

U32 = Fraction(1, 2 ** 24)
U64 = Fraction(1, 2 ** 53)


# ---------------------------------------------------------------- BF16 rounding
def test_bf16_of_f32_matches_torch():
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(100.0),
        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-30),
        # exact ties: low 16 bits == 0x8000, both parities of bit 16
        (np.arange(0x3F800000, 0x3F800000 + 0x40000, 0x8000, dtype=np.uint32)
         | np.uint32(0x8000)).view(np.float32),
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 1e-40], dtype=np.float32),
    ])
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    lib = oracle.load()
    got = np.array([lib.ora_bf16_of_f32(float(a)) for a in v], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_of_f64_exact_rne():
    rng = np.random.default_rng(12)
    vals = list(rng.standard_normal(3000) * 37.0) + list(rng.standard_normal(300) * 1e-39)
    # doubles just around BF16 midpoints (where rounding through fp32 would be wrong)
    for m in (1.0, 1.5, 3.0, 0.1):
        b = float(np.float32(m))
        vals += [b + 2.0 ** -9 * b, b + 2.0 ** -9 * b + 2.0 ** -40, b + 2.0 ** -9 * b - 2.0 ** -40]
    for v in vals:
        want = rne_bf16(Fraction(v))
        got = bf16_bits_to_frac(oracle.bf16_of_f64(v))
        assert got == want, v


def test_f32_of_bf16_roundtrip():
    for h in (0, 0x8000, 0x3F80, 0xBF80, 0x0001, 0x7F7F, 0x4049):
        f = oracle.f32_of_bf16(h)
        assert oracle.bf16_of_f32(f) == h


# ------------------------------------------------------------ bgmv helpers
def _int_bits(a):
    return W.to_bf16_bits(np.asarray(a, dtype=np.float32))


def _run_bgmv(wl: W.BgmvWorkload, mode=0):
    out = wl.out_buf.copy()
    seg = out.reshape(-1)[wl.out_offset:]
    xa, d = oracle.lora_bgmv(wl.x.reshape(-1), wl.x_row_stride, seg, wl.out_row_stride,
                             wl.seq_slot, wl.a_list(), wl.b_list(), wl.scale,
                             wl.max_rank, wl.k_in, wl.n_out, mode=mode)
    return out, xa, d


def _int_workload(seed, n=7, k_in=16, n_out=24, max_loras=5, max_rank=8, xs_pad=8,
                  out_pad=16, out_offset=8):
    """Small-integer bgmv where every fp32 and BF16 step is exact."""
    rng = np.random.default_rng(seed)
    ranks = [3, 8, 5, 0, 8]          # slot 3: NULL entry
    present = np.array([r > 0 for r in ranks])
    xs, os_ = k_in + xs_pad, out_offset + n_out + out_pad
    x = rng.integers(-1, 2, size=(n, xs))
    base = rng.integers(-6, 7, size=(n, os_))
    a_pool = np.zeros((max_loras, max_rank, k_in), dtype=np.uint16)
    b_pool = np.zeros((max_loras, n_out, max_rank), dtype=np.uint16)
    a_int = np.zeros((max_loras, max_rank, k_in), dtype=np.int64)
    b_int = np.zeros((max_loras, n_out, max_rank), dtype=np.int64)
    for s, r in enumerate(ranks):
        if r:
            a_int[s, :r] = rng.integers(-1, 2, size=(r, k_in))
            b_int[s, :, :r] = rng.integers(-1, 2, size=(n_out, r))
            a_pool[s] = _int_bits(a_int[s])
            b_pool[s] = _int_bits(b_int[s])
    scale = np.array([1.0, 2.0, 0.5, 0.0, 1.0], dtype=np.float32)
    seq = np.array([0, 1, -1, 2, 3, 7, 4][:n], dtype=np.int32)   # -1, NULL slot 3, slot 7 >= max_loras
    wl = W.BgmvWorkload("int", n, k_in, n_out, max_loras, max_rank, xs, os_, out_offset,
                        _int_bits(x), _int_bits(base), seq, np.array(ranks, np.int32), present,
                        a_pool, b_pool, scale)
    return wl, x, base, a_int, b_int


@pytest.mark.parametrize("seed", [1, 2, 3, 4])
def test_bgmv_exact_integer_case(seed):
    """All values small integers (or halves): the fold equals the integer
    matrix product out + scale * (x @ A^T) @ B^T exactly, untouched bytes stay."""
    wl, x, base, a_int, b_int = _int_workload(seed)
    out, xa, d = _run_bgmv(wl)
    want = base.astype(np.float64).copy()
    for i, s in enumerate(wl.seq_slot):
        if s < 0 or s >= wl.max_loras or not wl.present[s]:
            continue
        xa_i = a_int[s] @ x[i, :wl.k_in]                    # int64 matmul (library)
        d_i = b_int[s] @ xa_i
        assert np.abs(xa_i).max() <= 256 and np.abs(d_i).max() <= 256
        seg = slice(wl.out_offset, wl.out_offset + wl.n_out)
        want[i, seg] = base[i, seg] + float(wl.scale[s]) * d_i
        assert np.array_equal(W.bf16_bits_to_f32(xa[i]), xa_i.astype(np.float32))
        assert np.array_equal(W.bf16_bits_to_f32(d[i]), d_i.astype(np.float32))
    assert np.abs(want).max() <= 256
    assert np.array_equal(out, _int_bits(want))


# ------------------------------------------------ exact rational brute force
def _rand_tiny(seed, n=3, k_in=40, n_out=12, max_rank=8, ranks=(8, 5)):
    return W.make_bgmv("tiny_rand", n=n, k_in=k_in, n_out=n_out, max_loras=len(ranks),
                       max_rank=max_rank, rank_choices=dict(enumerate(ranks)), alpha=16.0,
                       rslora=False, slot_law="uniform", slot_base_frac=0.0, seed=seed,
                       x_row_stride=k_in + 8, out_row_stride=n_out + 8, out_offset=8,
                       a_bound=0.5, b_std=0.3)


@pytest.mark.parametrize("seed,mode", [(21, 0), (22, 0), (23, 1), (24, 1)])
def test_bgmv_stagewise_exact_rational(seed, mode):
    """Each stage of the oracle equals the exact-rational definition, except where
    the summation error bound straddles a BF16 rounding boundary (rare)."""
    wl = _rand_tiny(seed)
    out, xa, d = _run_bgmv(wl, mode)
    unit = U32 if mode == 0 else U64
    ambiguous = 0
    total = 0
    for i, s in enumerate(wl.seq_slot):
        A, B = wl.a_pool[s], wl.b_pool[s]
        xrow = wl.x[i, :wl.k_in]
        base_row = wl.out_buf[i, wl.out_offset:wl.out_offset + wl.n_out]
        xa_e, sx, d_e, sd, out_e = exact_row(xrow, A, B, wl.scale[s], base_row,
                                             wl.max_rank, wl.k_in, wl.n_out,
                                             xa_given=xa[i], d_given=d[i])
        for c in range(wl.max_rank):
            absx = sum(abs(bf16_bits_to_frac(xrow[k]) * bf16_bits_to_frac(A[c][k]))
                       for k in range(wl.k_in))
            total += 1
            if sum_is_unambiguous(sx[c], absx, wl.k_in, unit):
                assert xa[i][c] == xa_e[c], (i, c)
            else:
                ambiguous += 1
        for j in range(wl.n_out):
            absd = sum(abs(bf16_bits_to_frac(xa[i][c]) * bf16_bits_to_frac(B[j][c]))
                       for c in range(wl.max_rank))
            total += 1
            if sum_is_unambiguous(sd[j], absd, wl.max_rank, unit):
                assert d[i][j] == d_e[j], (i, j)
            else:
                ambiguous += 1
        # the fold is a single fp32 fma of the oracle's own d, then BF16: exact
        assert list(out[i, wl.out_offset:wl.out_offset + wl.n_out]) == out_e
    assert ambiguous <= total // 50


def test_bgmv_fp32_vs_fp64_within_bound():
    """fp32 and fp64 summation agree except where an intermediate BF16 rounding
    flips; then the fold differs by at most the flip's propagated size."""
    wl = W.decode_qproj_bgmv()
    wl.n = 16
    wl.x, wl.out_buf, wl.seq_slot = wl.x[:16], wl.out_buf[:16], wl.seq_slot[:16]
    o32, xa32, d32 = _run_bgmv(wl, 0)
    o64, xa64, d64 = _run_bgmv(wl, 1)
    routed = [i for i, s in enumerate(wl.seq_slot) if s >= 0]
    f = W.bf16_bits_to_f32
    for i in routed:
        rel = np.abs(f(xa32[i]) - f(xa64[i])) / np.maximum(np.abs(f(xa64[i])), 1e-30)
        assert rel.max() <= 2.0 ** -7
    same = np.mean([np.array_equal(o32[i], o64[i]) for i in routed])
    assert same >= 0.5
    diff = np.abs(f(o32).astype(np.float64) - f(o64).astype(np.float64))
    assert diff.max() <= 2.0 ** -6 * max(1.0, np.abs(f(o64)).max())


# -------------------------------------------------------------- invariants
def test_bgmv_batched_equals_one_row_per_call():
    wl = W.qkv_kfold_bgmv()
    keep = 24
    wl.n, wl.x, wl.out_buf, wl.seq_slot = keep, wl.x[:keep], wl.out_buf[:keep], wl.seq_slot[:keep]
    out_b, xa_b, d_b = _run_bgmv(wl)
    out_s = wl.out_buf.copy()
    for i in range(keep):
        seg = out_s[i].reshape(-1)[wl.out_offset:]
        xa, d = oracle.lora_bgmv(wl.x[i], wl.x_row_stride, seg, wl.out_row_stride,
                                 wl.seq_slot[i:i + 1], wl.a_list(), wl.b_list(), wl.scale,
                                 wl.max_rank, wl.k_in, wl.n_out)
    assert np.array_equal(out_b, out_s)


def test_bgmv_padded_rank_equals_true_rank():
    """An adapter packed at max_rank 16 (zero pad) folds bit-identically to the
    same adapter packed at max_rank = its true rank 5."""
    rng = np.random.default_rng(5)
    k_in, n_out, r, R, n = 64, 48, 5, 16, 6
    A = W.to_bf16_bits(rng.uniform(-0.2, 0.2, (r, k_in)).astype(np.float32))
    B = W.to_bf16_bits(rng.normal(0, 0.1, (n_out, r)).astype(np.float32))
    Ap = np.zeros((R, k_in), np.uint16); Ap[:r] = A
    Bp = np.zeros((n_out, R), np.uint16); Bp[:, :r] = B
    x = W.to_bf16_bits(rng.standard_normal((n, k_in)).astype(np.float32))
    base = W.to_bf16_bits(rng.standard_normal((n, n_out)).astype(np.float32))
    seq = np.zeros(n, np.int32)
    sc = np.array([3.2], np.float32)
    o1 = base.copy(); xa1, d1 = oracle.lora_bgmv(x, k_in, o1, n_out, seq, [A], [B], sc, r, k_in, n_out)
    o2 = base.copy(); xa2, d2 = oracle.lora_bgmv(x, k_in, o2, n_out, seq, [Ap], [Bp], sc, R, k_in, n_out)
    assert np.array_equal(o1, o2) and np.array_equal(d1, d2)
    assert np.array_equal(xa2[:, :r], xa1) and not xa2[:, r:].any()


def test_bgmv_skip_rules_leave_rows_byte_identical():
    wl = W.tiny_bgmv()
    wl.seq_slot = np.array([-1, 3, 9, 1], np.int32)    # base, NULL slot, out of range, routed
    out, xa, d = _run_bgmv(wl)
    assert np.array_equal(out[:3], wl.out_buf[:3])
    assert not np.array_equal(out[3], wl.out_buf[3])
    # NULL B alone also skips
    b_list = wl.b_list(); b_list[1] = None
    o2 = wl.out_buf.copy()
    oracle.lora_bgmv(wl.x, wl.x_row_stride, o2, wl.out_row_stride, wl.seq_slot, wl.a_list(),
                     b_list, wl.scale, wl.max_rank, wl.k_in, wl.n_out)
    assert np.array_equal(o2, wl.out_buf)


def test_bgmv_strided_fold_touches_only_its_segment():
    wl = W.qkv_kfold_bgmv()
    keep = 16
    wl.n, wl.x, wl.out_buf, wl.seq_slot = keep, wl.x[:keep], wl.out_buf[:keep], wl.seq_slot[:keep]
    out, _, _ = _run_bgmv(wl)
    seg = slice(wl.out_offset, wl.out_offset + wl.n_out)
    mask = np.ones_like(out, dtype=bool); mask[:, seg] = False
    assert np.array_equal(out[mask], wl.out_buf[mask])
    routed = wl.seq_slot >= 0
    assert not np.array_equal(out[routed][:, seg], wl.out_buf[routed][:, seg])


def test_bgmv_zero_b_leaves_output_unchanged():
    wl = W.tiny_bgmv()
    wl.b_pool[:] = 0
    out, xa, d = _run_bgmv(wl)
    assert not d.any()
    assert np.array_equal(out, wl.out_buf)


def test_bgmv_one_hot_row_gives_column_of_a():
    wl = W.tiny_bgmv()
    wl.x[:] = 0
    ks = [5, 77, 200, 255]
    for i, k in enumerate(ks):
        wl.x[i, k] = 0x3F80                        # 1.0
    wl.seq_slot = np.array([0, 1, 2, 0], np.int32)
    out, xa, d = _run_bgmv(wl)
    for i, k in enumerate(ks):
        s = wl.seq_slot[i]
        assert np.array_equal(xa[i], wl.a_pool[s][:, k])


def test_bgmv_scale_rules():
    """scale = alpha / r, or alpha / sqrt(r) under rsLoRA (LoraPair doc comment)."""
    assert W.lora_scale(32.0, 16, False) == np.float32(2.0)
    assert W.lora_scale(64.0, 16, True) == np.float32(16.0)
    assert W.lora_scale(64.0, 64, True) == np.float32(8.0)


# ---------------------------------------------------------------------- MoE
def _small_moe(seed=7, use_row_adapter=True, present_frac=1.0, cap=40):
    return W.make_moe("moe_small", num_tokens=24, top_k=3, num_experts=6, k_in=32, n_out=40,
                      max_loras=3, max_rank=8, rank=8, alpha=16.0, adapter_base_frac=0.25,
                      cap=cap, seed=seed, use_row_adapter=use_row_adapter,
                      present_frac=present_frac)


def _run_moe(wl: W.MoeWorkload, windows, mode=0, row_adapter="wl", out=None):
    out = wl.out_buf.copy() if out is None else out
    ra = wl.row_adapter if isinstance(row_adapter, str) else row_adapter
    xas = []
    for lo, hi in windows:
        xa, d = oracle.lora_moe_grouped_fold(
            wl.x, wl.k_in, out, wl.n_out, wl.expert_offsets, wl.sorted_token_ids, ra,
            wl.num_tokens, lo, hi, wl.a_list(), wl.b_list(), wl.scale, wl.max_rank,
            wl.k_in, wl.n_out, mode=mode)
        xas.append(xa)
    return out, xas


def test_moe_full_window_equals_sub_windows():
    wl = _small_moe()
    full, (xa_full,) = _run_moe(wl, [(0, wl.te)])
    parts, xas = _run_moe(wl, [(0, 17), (17, 40), (40, wl.te)])
    assert np.array_equal(full, parts)
    assert np.array_equal(np.concatenate(xas), xa_full)


def test_moe_delta_rows_are_sorted_rows_in_every_window():
    """The d output of a window sits at the sorted row index r (as base_out
    does), so each window's d equals the full call's d on its rows and is zero
    elsewhere; xa alone is window-local."""
    wl = _small_moe()

    def run_d(lo, hi):
        out = wl.out_buf.copy()
        _, d = oracle.lora_moe_grouped_fold(
            wl.x, wl.k_in, out, wl.n_out, wl.expert_offsets, wl.sorted_token_ids, wl.row_adapter,
            wl.num_tokens, lo, hi, wl.a_list(), wl.b_list(), wl.scale, wl.max_rank, wl.k_in,
            wl.n_out)
        return d

    d_full = run_d(0, wl.te)
    assert d_full.any()
    for lo, hi in [(0, 17), (17, 40), (40, wl.te)]:
        d = run_d(lo, hi)
        assert np.array_equal(d[lo:hi], d_full[lo:hi])
        assert not d[:lo].any() and not d[hi:].any()


def test_moe_group_equals_bgmv_on_same_rows():
    """The fold of the rows of one (adapter, expert) group equals the bgmv of the
    same rows with that adapter in slot 0."""
    wl = _small_moe(seed=8)
    out, _ = _run_moe(wl, [(0, wl.te)])
    E = wl.num_experts
    for e in range(E):
        rows = np.arange(wl.expert_offsets[e], wl.expert_offsets[e + 1])
        for a in range(wl.max_loras):
            sel = [r for r in rows if wl.row_adapter[wl.sorted_token_ids[r]] == a]
            if not sel:
                continue
            ob = wl.out_buf[sel].copy()
            i = a * E + e
            oracle.lora_bgmv(wl.x[sel], wl.k_in, ob, wl.n_out, np.zeros(len(sel), np.int32),
                             [wl.a_pool[i]], [wl.b_pool[i]], wl.scale[i:i + 1], wl.max_rank,
                             wl.k_in, wl.n_out)
            assert np.array_equal(out[sel], ob)


def test_moe_skip_rules():
    wl = _small_moe(seed=9, present_frac=0.6)
    out, _ = _run_moe(wl, [(0, wl.te)])
    E = wl.num_experts
    for r in range(wl.te):
        e = int(np.searchsorted(wl.expert_offsets, r, side="right") - 1)
        a = wl.row_adapter[wl.sorted_token_ids[r]]
        routed = a >= 0 and wl.present[a * E + e]
        assert np.array_equal(out[r], wl.out_buf[r]) != routed, r


def test_moe_rows_outside_offsets_and_bad_tokens_skipped():
    wl = _small_moe(seed=10)
    offs = wl.expert_offsets.copy()
    offs[0] = 5                                  # rows 0..4 lie before expert 0's span
    sti = wl.sorted_token_ids.copy()
    sti[7] = wl.num_tokens + 3                   # token out of range
    out = wl.out_buf.copy()
    oracle.lora_moe_grouped_fold(wl.x, wl.k_in, out, wl.n_out, offs, sti, wl.row_adapter,
                                 wl.num_tokens, 0, wl.te, wl.a_list(), wl.b_list(), wl.scale,
                                 wl.max_rank, wl.k_in, wl.n_out)
    assert np.array_equal(out[:5], wl.out_buf[:5])
    assert np.array_equal(out[7], wl.out_buf[7])


def test_moe_null_row_adapter_is_adapter_zero():
    wl = _small_moe(seed=11)
    zeros = np.zeros(wl.num_tokens, np.int32)
    o1, _ = _run_moe(wl, [(0, wl.te)], row_adapter=None)
    o2, _ = _run_moe(wl, [(0, wl.te)], row_adapter=zeros)
    assert np.array_equal(o1, o2)


def test_moe_exact_rational_rows():
    wl = _small_moe(seed=12)
    out, (xa,) = _run_moe(wl, [(0, wl.te)])
    E = wl.num_experts
    checked = 0
    for r in range(0, wl.te, 5):
        e = int(np.searchsorted(wl.expert_offsets, r, side="right") - 1)
        a = wl.row_adapter[wl.sorted_token_ids[r]]
        if a < 0:
            continue
        i = a * E + e
        _, _, _, _, out_e = exact_row(wl.x[r], wl.a_pool[i], wl.b_pool[i], wl.scale[i],
                                      wl.out_buf[r], wl.max_rank, wl.k_in, wl.n_out,
                                      xa_given=xa[r])
        # d differs from the exact one only where a rounding is ambiguous; the
        # fold of exact-rational d must then agree in at least 90% of elements
        agree = np.mean(np.array(out_e, np.uint16) == out[r])
        assert agree >= 0.9
        checked += 1
    assert checked > 5


# ------------------------------------------------ MoE gate/up (x_gather) and decode gather
def test_moe_gate_up_reads_token_rows():
    """x_gather: sorted row r reads row sorted_token_ids[r] of the token-major
    input, so the fold equals the down fold of the pre-gathered rows; without
    a row_adapter, rows whose token is out of range are skipped."""
    wl = _small_moe(seed=13)
    rng = np.random.default_rng(13)
    x_tok = W.to_bf16_bits(rng.standard_normal((wl.num_tokens, wl.k_in), dtype=np.float32))
    for ra in (wl.row_adapter, None):
        o1, o2 = wl.out_buf.copy(), wl.out_buf.copy()
        xa1, d1 = oracle.lora_moe_grouped_fold(
            x_tok, wl.k_in, o1, wl.n_out, wl.expert_offsets, wl.sorted_token_ids, ra,
            wl.num_tokens, 0, wl.te, wl.a_list(), wl.b_list(), wl.scale, wl.max_rank,
            wl.k_in, wl.n_out, x_gather=True)
        xa2, d2 = oracle.lora_moe_grouped_fold(
            x_tok[wl.sorted_token_ids], wl.k_in, o2, wl.n_out, wl.expert_offsets,
            wl.sorted_token_ids, ra, wl.num_tokens, 0, wl.te, wl.a_list(), wl.b_list(),
            wl.scale, wl.max_rank, wl.k_in, wl.n_out)
        assert np.array_equal(o1, o2) and np.array_equal(xa1, xa2) and np.array_equal(d1, d2)
        assert not np.array_equal(o1, wl.out_buf)
    sti = wl.sorted_token_ids.copy()
    sti[3] = -1
    o3 = wl.out_buf.copy()
    oracle.lora_moe_grouped_fold(x_tok, wl.k_in, o3, wl.n_out, wl.expert_offsets, sti, None,
                                 wl.num_tokens, 0, wl.te, wl.a_list(), wl.b_list(), wl.scale,
                                 wl.max_rank, wl.k_in, wl.n_out, x_gather=True)
    assert np.array_equal(o3[3], wl.out_buf[3])


def _small_gather(seed=21, use_row_adapter=True, present_frac=0.8):
    return W.make_moe_gather("gather_small", num_tokens=9, top_k=3, num_experts=5, k_in=40,
                             n_out=24, max_loras=3, max_rank=8, rank=8, alpha=16.0,
                             adapter_base_frac=0.25, seed=seed, use_row_adapter=use_row_adapter,
                             present_frac=present_frac)


def _run_gather(wl, indices=None, row_adapter="wl"):
    out = wl.out_buf.copy()
    ra = wl.row_adapter if isinstance(row_adapter, str) else row_adapter
    xa, d = oracle.lora_moe_gather_bgmv(wl.x, wl.k_in, out, wl.n_out,
                                        wl.indices if indices is None else indices, wl.top_k,
                                        ra, wl.num_tokens, wl.num_experts, wl.a_list(),
                                        wl.b_list(), wl.scale, wl.max_rank, wl.k_in, wl.n_out)
    return out, xa, d


def test_gather_bgmv_equals_bgmv_with_derived_slots():
    """Row r of the decode gather fold is the bgmv row with slot
    row_adapter[r // top_k] * E + indices[r] over the adapter-major tables."""
    wl = _small_gather()
    idx = wl.indices.copy()
    idx[2] = wl.num_experts          # expert out of range
    idx[5] = -1
    out, xa, d = _run_gather(wl, indices=idx)
    E = wl.num_experts
    ra = wl.row_adapter[np.arange(wl.n_rows) // wl.top_k]
    slot = np.where((ra >= 0) & (idx >= 0) & (idx < E), ra * E + idx, -1).astype(np.int32)
    ob = wl.out_buf.copy()
    xb, db = oracle.lora_bgmv(wl.x, wl.k_in, ob, wl.n_out, slot, wl.a_list(), wl.b_list(),
                              wl.scale, wl.max_rank, wl.k_in, wl.n_out)
    assert np.array_equal(out, ob) and np.array_equal(d, db)
    routed = [r for r in range(wl.n_rows) if slot[r] >= 0 and wl.present[slot[r]]]
    assert len(routed) > 5
    assert np.array_equal(xa[routed], xb[routed])
    for r in range(wl.n_rows):
        if r not in routed:
            assert np.array_equal(out[r], wl.out_buf[r])


def test_gather_bgmv_equals_grouped_fold_after_sorting():
    """Sorting the flat rows by (expert, token) and folding them with the grouped
    fold gives the same rows."""
    wl = _small_gather(seed=22, present_frac=1.0)
    out, xa, d = _run_gather(wl)
    tok = np.arange(wl.n_rows) // wl.top_k
    order = np.lexsort((tok, wl.indices))
    counts = np.bincount(wl.indices, minlength=wl.num_experts)
    offs = np.zeros(wl.num_experts + 1, np.int32)
    offs[1:] = np.cumsum(counts)
    os_ = wl.out_buf[order].copy()
    xs, _ = oracle.lora_moe_grouped_fold(wl.x[order], wl.k_in, os_, wl.n_out, offs,
                                         tok[order].astype(np.int32), wl.row_adapter,
                                         wl.num_tokens, 0, wl.n_rows, wl.a_list(), wl.b_list(),
                                         wl.scale, wl.max_rank, wl.k_in, wl.n_out)
    assert np.array_equal(out[order], os_)


def test_gather_bgmv_null_row_adapter_is_adapter_zero():
    wl = _small_gather(seed=23)
    o1, _, _ = _run_gather(wl, row_adapter=None)
    o2, _, _ = _run_gather(wl, row_adapter=np.zeros(wl.num_tokens, np.int32))
    assert np.array_equal(o1, o2)


# ------------------------------------------------ single-adapter delta
def _int_delta(seed, m=6, k_in=24, n_out=20, max_rank=16, rank=11, xs_pad=8, out_offset=8, out_pad=8):
    """Small-integer single-adapter delta where every fp32 and BF16 step is exact."""
    rng = np.random.default_rng(seed)
    xs, os_ = k_in + xs_pad, out_offset + n_out + out_pad
    x = rng.integers(-1, 2, size=(m, xs))
    base = rng.integers(-6, 7, size=(m, os_))
    a_int = np.zeros((max_rank, k_in), dtype=np.int64)
    b_int = np.zeros((n_out, max_rank), dtype=np.int64)
    a_int[:rank] = rng.integers(-1, 2, size=(rank, k_in))
    b_int[:, :rank] = rng.integers(-1, 2, size=(n_out, rank))
    wl = W.DeltaWorkload("int_delta", m, k_in, n_out, max_rank, rank, xs, os_, out_offset,
                         _int_bits(x), _int_bits(base), _int_bits(a_int), _int_bits(b_int),
                         np.float32(2.0))
    return wl, x, base, a_int, b_int


def _run_delta(wl: W.DeltaWorkload, mode=0):
    out = wl.out_buf.copy()
    seg = out.reshape(-1)[wl.out_offset:]
    xa, d = oracle.lora_delta(wl.x.reshape(-1), wl.x_row_stride, seg, wl.out_row_stride, wl.m,
                              wl.a, wl.b, wl.scale, wl.max_rank, wl.k_in, wl.n_out, mode=mode)
    return out, xa, d


@pytest.mark.parametrize("seed", [31, 32, 33])
def test_delta_exact_integer_case(seed):
    """lora_delta.rs, apply_lora_delta on small integers: every row equals the
    integer product out + scale * (x @ A^T) @ B^T exactly; bytes outside each
    row's [out_offset, out_offset + n_out) stay."""
    wl, x, base, a_int, b_int = _int_delta(seed)
    out, xa, d = _run_delta(wl)
    want = base.astype(np.float64).copy()
    seg = slice(wl.out_offset, wl.out_offset + wl.n_out)
    for i in range(wl.m):
        xa_i = a_int @ x[i, :wl.k_in]                      # int64 matmul (library)
        d_i = b_int @ xa_i
        assert np.abs(xa_i).max() <= 256 and np.abs(d_i).max() <= 256
        want[i, seg] = base[i, seg] + float(wl.scale) * d_i
        assert np.array_equal(W.bf16_bits_to_f32(xa[i]), xa_i.astype(np.float32))
    assert np.abs(want).max() <= 256
    assert np.array_equal(out, _int_bits(want))


@pytest.mark.parametrize("mode", [0, 1])
def test_delta_equals_bgmv_with_one_slot(mode):
    """apply_lora_delta over m rows == apply_lora_bgmv with every row on one slot
    holding the same pair (the routed fold's definition, pinned above)."""
    wl = W.make_delta("d", m=9, k_in=72, n_out=40, max_rank=16, rank=12, alpha=16.0, rslora=False,
                      seed=41, x_row_stride=80, out_row_stride=56, out_offset=8)
    out_d, xa_d, d_d = _run_delta(wl, mode)
    bg = W.BgmvWorkload("b", wl.m, wl.k_in, wl.n_out, 1, wl.max_rank, wl.x_row_stride,
                        wl.out_row_stride, wl.out_offset, wl.x, wl.out_buf.copy(),
                        np.zeros(wl.m, dtype=np.int32), np.array([wl.rank], np.int32),
                        np.ones(1, dtype=bool), wl.a[None], wl.b[None],
                        np.array([wl.scale], dtype=np.float32))
    out_b, xa_b, d_b = _run_bgmv(bg, mode)
    assert np.array_equal(out_d, out_b) and np.array_equal(xa_d, xa_b) and np.array_equal(d_d, d_b)
    assert not np.array_equal(out_d, wl.out_buf)


def test_delta_zero_rows_is_a_no_op():
    wl = W.make_delta("z", m=0, k_in=16, n_out=16, max_rank=8, rank=8, alpha=8.0, rslora=False, seed=1)
    out, xa, d = _run_delta(wl)
    assert out.shape == (0, 16) and xa.shape == (0, 8)
