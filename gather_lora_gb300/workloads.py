"""Seeded synthetic inputs for the routed LoRA fold (bgmv and MoE grouped fold).

This module only draws inputs: activations, adapter pools, routing tables and
scales. It holds none of the fold's arithmetic (no shrink, expand, rounding
order or fold), so the CUDA path and the CPU oracle can both be fed from it.

Layouts follow the pages:
  * lora_delta.rs page (metrale source listing), ``LoraPair`` doc comment: A is
    ``[max_rank, k_in]`` row-major BF16 and B is ``[n_out, max_rank]`` row-major
    BF16, the adapter's true rank in the first rows of A / first columns of B
    and zeros after (the pool is zeroed before packing).
  * the same comment: ``scale = lora_alpha / r``, or ``lora_alpha / sqrt(r)``
    under rsLoRA. The scale is computed here in double and stored as f32 once;
    every consumer reads that same f32.
  * Function apply_lora_bgmv page: ``seq_slot[n]`` i32, ``< 0`` = no delta;
    NULL table entry = slot that does not adapt this module.
  * Module moe_lora_grouped page, ``moe_lora_grouped_down``: rows sorted by
    expert, ``expert_offsets`` ``[E+1]`` i32 prefix sum, ``sorted_token_ids``
    ``[te]`` sorted-row -> token, ``moe_row_adapter`` ``[num_tokens]`` i32
    (< 0 = base), windows of ``cap`` rows.

BF16 values are carried as raw uint16 bit patterns (round-to-nearest-even of
fp32 samples, done by torch's CPU conversion).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """fp32 samples -> BF16 bit patterns (uint16), round-to-nearest-even."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """BF16 bit patterns -> fp32 values (exact)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def lora_scale(alpha: float, rank: int, rslora: bool) -> np.float32:
    """Per-adapter scale as stored in the scale table (f32 of a double)."""
    return np.float32(alpha / math.sqrt(rank) if rslora else alpha / rank)


def zipf_slots(rng: np.random.Generator, n: int, num: int, s: float) -> np.ndarray:
    """n draws of a bounded Zipf law over slots 0..num-1: P(slot k-1) ∝ k^-s."""
    p = np.arange(1, num + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    return rng.choice(num, size=n, p=p).astype(np.int32)


@dataclass
class BgmvWorkload:
    """One routed-bgmv problem on the host.

    ``out_buf`` is the whole output buffer ``[n, out_buf_cols]``; the folded
    segment of row i starts at element ``out_offset`` of that row and is
    ``n_out`` wide, rows ``out_row_stride`` (= out_buf_cols) apart.
    ``present[s]`` False means a NULL table entry for slot s.
    """
    name: str
    n: int
    k_in: int
    n_out: int
    max_loras: int
    max_rank: int
    x_row_stride: int
    out_row_stride: int
    out_offset: int
    x: np.ndarray            # uint16 [n, x_row_stride]
    out_buf: np.ndarray      # uint16 [n, out_row_stride]
    seq_slot: np.ndarray     # int32 [n]
    ranks: np.ndarray        # int32 [max_loras], 0 where not present
    present: np.ndarray      # bool [max_loras]
    a_pool: np.ndarray       # uint16 [max_loras, max_rank, k_in]
    b_pool: np.ndarray       # uint16 [max_loras, n_out, max_rank]
    scale: np.ndarray        # float32 [max_loras]
    meta: dict = field(default_factory=dict)

    def a_list(self):
        return [self.a_pool[s] if self.present[s] else None for s in range(self.max_loras)]

    def b_list(self):
        return [self.b_pool[s] if self.present[s] else None for s in range(self.max_loras)]


@dataclass
class MoeWorkload:
    """One MoE grouped-fold problem (all windows) on the host.

    Tables are adapter-major: entry ``a * num_experts + e``.
    """
    name: str
    num_tokens: int
    top_k: int
    num_experts: int
    te: int
    k_in: int
    n_out: int
    max_loras: int
    max_rank: int
    cap: int
    x: np.ndarray                # uint16 [te, k_in] (down), or [num_tokens, k_in] token-major (x_gather)
    out_buf: np.ndarray          # uint16 [te, n_out]
    expert_offsets: np.ndarray   # int32 [E+1]
    sorted_token_ids: np.ndarray  # int32 [te]
    row_adapter: np.ndarray | None  # int32 [num_tokens] or None
    present: np.ndarray          # bool [max_loras * E]
    a_pool: np.ndarray           # uint16 [max_loras * E, max_rank, k_in]
    b_pool: np.ndarray           # uint16 [max_loras * E, n_out, max_rank]
    scale: np.ndarray            # float32 [max_loras * E]
    meta: dict = field(default_factory=dict)
    x_gather: bool = False       # gate/up: sorted row r reads token row sorted_token_ids[r] of x

    def windows(self):
        return [(s, min(s + self.cap, self.te)) for s in range(0, self.te, self.cap)] or [(0, 0)]

    def a_list(self):
        return [self.a_pool[i] if self.present[i] else None for i in range(len(self.present))]

    def b_list(self):
        return [self.b_pool[i] if self.present[i] else None for i in range(len(self.present))]


@dataclass
class DeltaWorkload:
    """One single-adapter delta problem (lora_delta.rs page, apply_lora_delta):
    every one of the m rows is adapted by the same pair. Layout of ``out_buf`` as
    for BgmvWorkload (the folded segment of row i starts at ``out_offset``)."""
    name: str
    m: int
    k_in: int
    n_out: int
    max_rank: int
    rank: int
    x_row_stride: int
    out_row_stride: int
    out_offset: int
    x: np.ndarray            # uint16 [m, x_row_stride]
    out_buf: np.ndarray      # uint16 [m, out_row_stride]
    a: np.ndarray            # uint16 [max_rank, k_in], rows >= rank zero
    b: np.ndarray            # uint16 [n_out, max_rank], columns >= rank zero
    scale: np.float32
    meta: dict = field(default_factory=dict)


def _pack_pool(rng, count, present, ranks, max_rank, k_in, n_out, a_bound, b_std):
    """Zeroed pool, then each present adapter's true-rank A rows / B columns."""
    a_pool = np.zeros((count, max_rank, k_in), dtype=np.uint16)
    b_pool = np.zeros((count, n_out, max_rank), dtype=np.uint16)
    for s in range(count):
        if not present[s]:
            continue
        r = int(ranks[s])
        a = rng.uniform(-a_bound, a_bound, size=(r, k_in)).astype(np.float32)
        b = rng.normal(0.0, b_std, size=(n_out, r)).astype(np.float32)
        a_pool[s, :r, :] = to_bf16_bits(a)
        b_pool[s, :, :r] = to_bf16_bits(b)
    return a_pool, b_pool


def make_bgmv(name, *, n, k_in, n_out, max_loras, max_rank, rank_choices, alpha, rslora,
              slot_law, slot_base_frac, seed, x_row_stride=None, out_row_stride=None,
              out_offset=0, null_slots=(), x_law="normal", present_slots=None,
              a_bound=None, b_std=0.02) -> BgmvWorkload:
    """Draw one bgmv workload.

    slot_law: "uniform" over present slots, "zipf:<s>" over all max_loras slots,
    or "list:<i,j,...>" (explicit per-row slots). slot_base_frac: fraction of rows
    given slot -1. x_law: "normal" (N(0,1)) or "silu_gate" (SiLU(N(0,1))*N(0,1)).
    A ~ U(+-a_bound) with a_bound = 1/sqrt(k_in) unless given; B ~ N(0, b_std).
    """
    rng = np.random.default_rng(seed)
    xs = x_row_stride or k_in
    os_ = out_row_stride or n_out
    present = np.ones(max_loras, dtype=bool)
    if present_slots is not None:
        present[:] = False
        present[list(present_slots)] = True
    for s in null_slots:
        present[s] = False
    ranks = np.zeros(max_loras, dtype=np.int32)
    if isinstance(rank_choices, dict):
        for s, r in rank_choices.items():
            ranks[s] = r
    else:
        ranks[present] = rng.choice(np.asarray(rank_choices), size=int(present.sum()))
    ranks[~present] = 0
    scale = np.zeros(max_loras, dtype=np.float32)
    for s in range(max_loras):
        if present[s]:
            scale[s] = lora_scale(alpha, int(ranks[s]), rslora)
    # routing
    if slot_law.startswith("list:"):
        seq = np.array([int(v) for v in slot_law[5:].split(",")], dtype=np.int32)
        assert seq.shape[0] == n
    else:
        if slot_law == "uniform":
            seq = rng.choice(np.flatnonzero(present), size=n).astype(np.int32)
        elif slot_law == "uniform_all":
            seq = rng.integers(-1, max_loras, size=n).astype(np.int32)
        elif slot_law.startswith("zipf:"):
            seq = zipf_slots(rng, n, max_loras, float(slot_law[5:]))
        else:
            raise ValueError(slot_law)
        base = rng.random(n) < slot_base_frac
        seq[base] = -1
    # activations and output buffer
    if x_law == "normal":
        xf = rng.standard_normal((n, xs), dtype=np.float32)
    elif x_law == "silu_gate":
        g = rng.standard_normal((n, xs), dtype=np.float32)
        u = rng.standard_normal((n, xs), dtype=np.float32)
        xf = (g / (1.0 + np.exp(-g))) * u
    else:
        raise ValueError(x_law)
    x = to_bf16_bits(xf)
    out_buf = to_bf16_bits(rng.standard_normal((n, os_), dtype=np.float32))
    a_pool, b_pool = _pack_pool(rng, max_loras, present, ranks, max_rank, k_in, n_out,
                                a_bound if a_bound is not None else 1.0 / math.sqrt(k_in), b_std)
    return BgmvWorkload(name, n, k_in, n_out, max_loras, max_rank, xs, os_, out_offset,
                        x, out_buf, seq, ranks, present, a_pool, b_pool, scale,
                        meta=dict(seed=seed, slot_law=slot_law, alpha=alpha, rslora=rslora))


def make_delta(name, *, m, k_in, n_out, max_rank, rank, alpha, rslora, seed, x_law="normal",
               x_row_stride=None, out_row_stride=None, out_offset=0, a_bound=None,
               b_std=0.02) -> DeltaWorkload:
    """Draw one single-adapter delta problem: x ~ N(0,1) (or SiLU(N)*N), base_out ~
    N(0,1), A ~ U(+-1/sqrt(k_in)) in its first ``rank`` rows, B ~ N(0, b_std) in
    its first ``rank`` columns, zeros elsewhere; scale as for the pool."""
    rng = np.random.default_rng(seed)
    xs = x_row_stride or k_in
    os_ = out_row_stride or (out_offset + n_out)
    if x_law == "normal":
        xf = rng.standard_normal((m, xs), dtype=np.float32)
    elif x_law == "silu_gate":
        g = rng.standard_normal((m, xs), dtype=np.float32)
        u = rng.standard_normal((m, xs), dtype=np.float32)
        xf = (g / (1.0 + np.exp(-g))) * u
    else:
        raise ValueError(x_law)
    x = to_bf16_bits(xf)
    out_buf = to_bf16_bits(rng.standard_normal((m, os_), dtype=np.float32))
    a_pool, b_pool = _pack_pool(rng, 1, np.ones(1, dtype=bool), np.array([rank]), max_rank, k_in,
                                n_out, a_bound if a_bound is not None else 1.0 / math.sqrt(k_in), b_std)
    return DeltaWorkload(name, m, k_in, n_out, max_rank, rank, xs, os_, out_offset, x, out_buf,
                         a_pool[0], b_pool[0], lora_scale(alpha, rank, rslora),
                         meta=dict(seed=seed, alpha=alpha, rslora=rslora, x_law=x_law))


def make_moe(name, *, num_tokens, top_k, num_experts, k_in, n_out, max_loras, max_rank,
             rank, alpha, adapter_base_frac, cap, seed, use_row_adapter=True,
             present_frac=1.0, b_std=0.02, x_gather=False) -> MoeWorkload:
    """Draw one MoE grouped-fold workload.

    Routing: each token takes the top_k experts of N(0,1) logits (softmax is
    monotone, so top-k by logit; ties go to the lower expert id). Rows are the
    (token, expert) pairs sorted by (expert, token); expert_offsets is their
    prefix sum over experts. x = SiLU(N)*N per sorted row (post-SiLU down_proj
    input), base_out ~ N(0,1). Every (adapter, expert) pair is an adapter of
    the given rank unless present_frac < 1. row_adapter per token: -1 with
    probability adapter_base_frac, else uniform over 0..max_loras-1.
    """
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((num_tokens, num_experts), dtype=np.float32)
    topk = np.argsort(-logits, axis=1, kind="stable")[:, :top_k]
    tok = np.repeat(np.arange(num_tokens, dtype=np.int32), top_k)
    exp_ = topk.reshape(-1).astype(np.int32)
    order = np.lexsort((tok, exp_))                     # by expert, then token
    sorted_token_ids = tok[order].astype(np.int32)
    counts = np.bincount(exp_, minlength=num_experts)
    expert_offsets = np.zeros(num_experts + 1, dtype=np.int32)
    expert_offsets[1:] = np.cumsum(counts)
    te = int(expert_offsets[-1])
    if x_gather:   # gate/up input: token-major hidden states ~ N(0, 1)
        x = to_bf16_bits(rng.standard_normal((num_tokens, k_in), dtype=np.float32))
    else:          # down input: post-SiLU sorted activations
        g = rng.standard_normal((te, k_in), dtype=np.float32)
        u = rng.standard_normal((te, k_in), dtype=np.float32)
        x = to_bf16_bits((g / (1.0 + np.exp(-g))) * u)
    out_buf = to_bf16_bits(rng.standard_normal((te, n_out), dtype=np.float32))
    if use_row_adapter:
        ra = rng.integers(0, max_loras, size=num_tokens).astype(np.int32)
        ra[rng.random(num_tokens) < adapter_base_frac] = -1
    else:
        ra = None
    count = max_loras * num_experts
    present = np.ones(count, dtype=bool)
    if present_frac < 1.0:
        present = rng.random(count) < present_frac
    ranks = np.where(present, rank, 0).astype(np.int32)
    a_pool, b_pool = _pack_pool(rng, count, present, ranks, max_rank, k_in, n_out,
                                1.0 / math.sqrt(k_in), b_std)
    scale = np.where(present, lora_scale(alpha, rank, False), 0.0).astype(np.float32)
    return MoeWorkload(name, num_tokens, top_k, num_experts, te, k_in, n_out, max_loras,
                       max_rank, cap, x, out_buf, expert_offsets, sorted_token_ids, ra,
                       present, a_pool, b_pool, scale, meta=dict(seed=seed), x_gather=x_gather)


@dataclass
class MoeGatherWorkload:
    """One decode-path MoE fold over flat, unsorted (token, slot) rows on the host:
    row r = token * top_k + j takes expert indices[r] and adapter
    row_adapter[r // top_k]; tables are adapter-major (a * E + e)."""
    name: str
    num_tokens: int
    top_k: int
    num_experts: int
    k_in: int
    n_out: int
    max_loras: int
    max_rank: int
    x: np.ndarray                # uint16 [n_rows, k_in]
    out_buf: np.ndarray          # uint16 [n_rows, n_out]
    indices: np.ndarray          # int32 [n_rows]
    row_adapter: np.ndarray | None  # int32 [num_tokens] or None
    present: np.ndarray          # bool [max_loras * E]
    a_pool: np.ndarray
    b_pool: np.ndarray
    scale: np.ndarray            # float32 [max_loras * E]
    meta: dict = field(default_factory=dict)

    @property
    def n_rows(self):
        return self.num_tokens * self.top_k

    def a_list(self):
        return [self.a_pool[i] if self.present[i] else None for i in range(len(self.present))]

    def b_list(self):
        return [self.b_pool[i] if self.present[i] else None for i in range(len(self.present))]


def make_moe_gather(name, *, num_tokens, top_k, num_experts, k_in, n_out, max_loras, max_rank,
                    rank, alpha, adapter_base_frac, seed, use_row_adapter=True,
                    present_frac=1.0, b_std=0.02) -> MoeGatherWorkload:
    """Draw one decode-path MoE workload: routing as in make_moe (top_k experts of
    N(0,1) logits per token), rows left in (token, slot) order; x = SiLU(N)*N per
    row (post-SiLU down_proj input), base_out ~ N(0,1)."""
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((num_tokens, num_experts), dtype=np.float32)
    indices = np.argsort(-logits, axis=1, kind="stable")[:, :top_k].reshape(-1).astype(np.int32)
    n_rows = num_tokens * top_k
    g = rng.standard_normal((n_rows, k_in), dtype=np.float32)
    u = rng.standard_normal((n_rows, k_in), dtype=np.float32)
    x = to_bf16_bits((g / (1.0 + np.exp(-g))) * u)
    out_buf = to_bf16_bits(rng.standard_normal((n_rows, n_out), dtype=np.float32))
    if use_row_adapter:
        ra = rng.integers(0, max_loras, size=num_tokens).astype(np.int32)
        ra[rng.random(num_tokens) < adapter_base_frac] = -1
    else:
        ra = None
    count = max_loras * num_experts
    present = np.ones(count, dtype=bool)
    if present_frac < 1.0:
        present = rng.random(count) < present_frac
    ranks = np.where(present, rank, 0).astype(np.int32)
    a_pool, b_pool = _pack_pool(rng, count, present, ranks, max_rank, k_in, n_out,
                                1.0 / math.sqrt(k_in), b_std)
    scale = np.where(present, lora_scale(alpha, rank, False), 0.0).astype(np.float32)
    return MoeGatherWorkload(name, num_tokens, top_k, num_experts, k_in, n_out, max_loras,
                             max_rank, x, out_buf, indices, ra, present, a_pool, b_pool, scale,
                             meta=dict(seed=seed))


# --- the five named workloads --------------------------------------------------
#
# Shapes and laws of the decode, strided-QKV, dense-FFN and MoE workloads that the
# fold serves. Where a law is not given for a workload (base_out, the A/B laws of
# the larger ones, alpha of the strided K fold and of the MoE fold) the choice of
# the tiny / q_proj workloads is reused: base_out ~ N(0,1), A ~ U(+-1/sqrt(k_in)),
# B ~ N(0, 0.02), alpha = 32.

WORKLOADS = ("tiny_bgmv", "decode_qproj_bgmv", "qkv_kfold_bgmv", "ffn_down_bgmv", "moe_down_fold")


def tiny_bgmv(seed=0):
    """n=4 decode rows, k_in=n_out=256, 4 slots at max_rank 8, ranks {4,8,8}, slot 3 NULL."""
    return make_bgmv("tiny_bgmv", n=4, k_in=256, n_out=256, max_loras=4, max_rank=8,
                     rank_choices={0: 4, 1: 8, 2: 8}, alpha=16.0, rslora=False,
                     slot_law="uniform_all", slot_base_frac=0.0, seed=seed, null_slots=(3,))


def decode_qproj_bgmv(seed=1):
    """n=64, k_in=n_out=4096, 32 adapters, max_rank 16, ranks {8,16}, Zipf(1.1), 10% base."""
    return make_bgmv("decode_qproj_bgmv", n=64, k_in=4096, n_out=4096, max_loras=32,
                     max_rank=16, rank_choices=(8, 16), alpha=32.0, rslora=False,
                     slot_law="zipf:1.1", slot_base_frac=0.10, seed=seed)


def qkv_kfold_bgmv(seed=2):
    """n=256, k_in=4096, fold n_out=1024 into the K segment of an interleaved
    Q4096|K1024|V1024 row (offset 4096, row stride 6144); 128 adapters, max_rank 64."""
    return make_bgmv("qkv_kfold_bgmv", n=256, k_in=4096, n_out=1024, max_loras=128,
                     max_rank=64, rank_choices=(8, 16, 32, 64), alpha=32.0, rslora=False,
                     slot_law="zipf:1.1", slot_base_frac=0.10, seed=seed,
                     out_row_stride=6144, out_offset=4096)


def ffn_down_bgmv(seed=3):
    """n=512, k_in=12288, n_out=4096, post-SiLU x, 64 adapters at max_rank 128,
    ranks {16,64,128}, rsLoRA alpha=64, uniform slots with 5% base."""
    return make_bgmv("ffn_down_bgmv", n=512, k_in=12288, n_out=4096, max_loras=64,
                     max_rank=128, rank_choices=(16, 64, 128), alpha=64.0, rslora=True,
                     slot_law="uniform", slot_base_frac=0.05, seed=seed, x_law="silu_gate")


def moe_down_fold(seed=4):
    """2048 tokens, top-8 of 128 experts, te=16384 sorted rows, k_in=768, n_out=2048,
    16 adapters over every expert at rank 16 (alpha 32), 20% base tokens, windows of 4096."""
    return make_moe("moe_down_fold", num_tokens=2048, top_k=8, num_experts=128, k_in=768,
                    n_out=2048, max_loras=16, max_rank=16, rank=16, alpha=32.0,
                    adapter_base_frac=0.20, cap=4096, seed=seed)


def moe_gateup_fold(seed=5):
    """Gate/up form of the MoE fold on the same model: 2048 tokens, top-8 of 128
    experts, te=16384, token-major x [2048, 2048] ~ N(0,1) gathered per sorted row,
    n_out=768 (the expert width), 16 adapters at rank 16 (alpha 32), 20% base
    tokens, windows of 4096."""
    return make_moe("moe_gateup_fold", num_tokens=2048, top_k=8, num_experts=128, k_in=2048,
                    n_out=768, max_loras=16, max_rank=16, rank=16, alpha=32.0,
                    adapter_base_frac=0.20, cap=4096, seed=seed, x_gather=True)


def moe_decode_gather(seed=6):
    """Decode-path MoE down fold: 64 tokens x top-8 of 128 experts = 512 flat rows,
    x [512, 768] post-SiLU, base_out [512, 2048], 16 adapters at rank 16 (alpha
    32), 20% base tokens."""
    return make_moe_gather("moe_decode_gather", num_tokens=64, top_k=8, num_experts=128,
                           k_in=768, n_out=2048, max_loras=16, max_rank=16, rank=16, alpha=32.0,
                           adapter_base_frac=0.20, seed=seed)


def prefill_qproj_delta(seed=7):
    """Prefill with one active adapter on the decode q_proj's model: m=4096 rows,
    k_in=n_out=4096, x ~ N(0,1), the adapter at rank 16 (alpha 32)."""
    return make_delta("prefill_qproj_delta", m=4096, k_in=4096, n_out=4096, max_rank=16, rank=16,
                      alpha=32.0, rslora=False, seed=seed)


def prefill_down_delta(seed=8):
    """Prefill with one active adapter on the FFN down_proj's model: m=4096 rows,
    k_in=12288, n_out=4096, post-SiLU x, the adapter at rank 128 (rsLoRA, alpha 64)."""
    return make_delta("prefill_down_delta", m=4096, k_in=12288, n_out=4096, max_rank=128, rank=128,
                      alpha=64.0, rslora=True, seed=seed, x_law="silu_gate")


def one_launch(wl: MoeWorkload) -> MoeWorkload:
    """The same MoE problem folded by one call over all te sorted rows: one
    window of cap = te, so the xa output holds every row."""
    return replace(wl, name=wl.name + "_one_launch", cap=wl.te)


def by_name(name: str, seed=None):
    if name.endswith("_one_launch"):
        return one_launch(by_name(name[: -len("_one_launch")], seed))
    fn = {"tiny_bgmv": tiny_bgmv, "decode_qproj_bgmv": decode_qproj_bgmv,
          "qkv_kfold_bgmv": qkv_kfold_bgmv, "ffn_down_bgmv": ffn_down_bgmv,
          "moe_down_fold": moe_down_fold, "moe_gateup_fold": moe_gateup_fold,
          "moe_decode_gather": moe_decode_gather, "prefill_qproj_delta": prefill_qproj_delta,
          "prefill_down_delta": prefill_down_delta}[name]
    return fn() if seed is None else fn(seed)


# --- device placement (data movement only) -------------------------------------

@dataclass
class DeviceBgmv:
    x: "torch.Tensor"         # int16 [n, x_row_stride] (BF16 bits)
    out_buf: "torch.Tensor"   # int16 [n, out_row_stride]
    out_ptr: int              # address of out_buf[0, out_offset]
    seq_slot: "torch.Tensor"  # int32 [n]
    a_pool: "torch.Tensor"
    b_pool: "torch.Tensor"
    a_table: "torch.Tensor"   # int64 [max_loras] device addresses (0 = NULL)
    b_table: "torch.Tensor"
    scale: "torch.Tensor"     # float32 [max_loras]
    xa: "torch.Tensor"        # int16 [n, max_rank]


def _dev(a: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(a))
    if t.dtype == torch.uint16:
        t = t.view(torch.int16)
    return t.to(device)


def _table_of(pool: torch.Tensor, present: np.ndarray, device) -> torch.Tensor:
    stride = pool[0].numel() * pool.element_size() if pool.shape[0] else 0
    base = pool.data_ptr()
    addrs = [base + i * stride if present[i] else 0 for i in range(len(present))]
    return torch.tensor(addrs, dtype=torch.int64, device=device)


def bgmv_to_device(wl: BgmvWorkload, device="cuda") -> DeviceBgmv:
    x = _dev(wl.x.view(np.int16), device)
    out = _dev(wl.out_buf.view(np.int16), device)
    a_pool = _dev(wl.a_pool.view(np.int16), device)
    b_pool = _dev(wl.b_pool.view(np.int16), device)
    return DeviceBgmv(
        x=x, out_buf=out, out_ptr=out.data_ptr() + 2 * wl.out_offset,
        seq_slot=_dev(wl.seq_slot, device), a_pool=a_pool, b_pool=b_pool,
        a_table=_table_of(a_pool, wl.present, device), b_table=_table_of(b_pool, wl.present, device),
        scale=_dev(wl.scale, device),
        xa=torch.zeros((max(wl.n, 1), wl.max_rank), dtype=torch.int16, device=device))


@dataclass
class DeviceDelta:
    x: "torch.Tensor"         # int16 [m, x_row_stride]
    out_buf: "torch.Tensor"   # int16 [m, out_row_stride]
    out_ptr: int              # address of out_buf[0, out_offset]
    a: "torch.Tensor"         # int16 [max_rank, k_in]
    b: "torch.Tensor"         # int16 [n_out, max_rank]
    xa: "torch.Tensor"        # int16 [m, max_rank]


def delta_to_device(wl: DeltaWorkload, device="cuda") -> DeviceDelta:
    out = _dev(wl.out_buf.view(np.int16), device)
    return DeviceDelta(x=_dev(wl.x.view(np.int16), device), out_buf=out,
                       out_ptr=out.data_ptr() + 2 * wl.out_offset,
                       a=_dev(wl.a.view(np.int16), device), b=_dev(wl.b.view(np.int16), device),
                       xa=torch.zeros((max(wl.m, 1), wl.max_rank), dtype=torch.int16, device=device))


@dataclass
class DeviceMoe:
    x: "torch.Tensor"
    out_buf: "torch.Tensor"
    expert_offsets: "torch.Tensor"
    sorted_token_ids: "torch.Tensor"
    row_adapter: "torch.Tensor | None"
    a_pool: "torch.Tensor"
    b_pool: "torch.Tensor"
    a_table: "torch.Tensor"
    b_table: "torch.Tensor"
    scale: "torch.Tensor"
    xa: "torch.Tensor"        # int16 [cap, max_rank] (window-local rows)


def moe_to_device(wl: MoeWorkload, device="cuda", xa_rows=None) -> DeviceMoe:
    a_pool = _dev(wl.a_pool.view(np.int16), device)
    b_pool = _dev(wl.b_pool.view(np.int16), device)
    rows = xa_rows if xa_rows is not None else max(wl.cap, 1)
    return DeviceMoe(
        x=_dev(wl.x.view(np.int16), device), out_buf=_dev(wl.out_buf.view(np.int16), device),
        expert_offsets=_dev(wl.expert_offsets, device),
        sorted_token_ids=_dev(wl.sorted_token_ids, device),
        row_adapter=None if wl.row_adapter is None else _dev(wl.row_adapter, device),
        a_pool=a_pool, b_pool=b_pool,
        a_table=_table_of(a_pool, wl.present, device), b_table=_table_of(b_pool, wl.present, device),
        scale=_dev(wl.scale, device),
        xa=torch.zeros((rows, wl.max_rank), dtype=torch.int16, device=device))


@dataclass
class DeviceMoeGather:
    x: "torch.Tensor"
    out_buf: "torch.Tensor"
    indices: "torch.Tensor"
    row_adapter: "torch.Tensor | None"
    a_pool: "torch.Tensor"
    b_pool: "torch.Tensor"
    a_table: "torch.Tensor"
    b_table: "torch.Tensor"
    scale: "torch.Tensor"
    xa: "torch.Tensor"        # int16 [n_rows, max_rank]


def gather_to_device(wl: MoeGatherWorkload, device="cuda") -> DeviceMoeGather:
    a_pool = _dev(wl.a_pool.view(np.int16), device)
    b_pool = _dev(wl.b_pool.view(np.int16), device)
    return DeviceMoeGather(
        x=_dev(wl.x.view(np.int16), device), out_buf=_dev(wl.out_buf.view(np.int16), device),
        indices=_dev(wl.indices, device),
        row_adapter=None if wl.row_adapter is None else _dev(wl.row_adapter, device),
        a_pool=a_pool, b_pool=b_pool,
        a_table=_table_of(a_pool, wl.present, device), b_table=_table_of(b_pool, wl.present, device),
        scale=_dev(wl.scale, device),
        xa=torch.zeros((max(wl.n_rows, 1), wl.max_rank), dtype=torch.int16, device=device))
