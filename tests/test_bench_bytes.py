"""The roofline numerator: algorithmic bytes of each fold kind on hand-built cases.

The expected totals are worked out by hand from the stated count (per routed
row: its x row, its out segment read and written, its xa row written and read;
per distinct adapter table entry: its padded A and B once plus 20 bytes of
table entries; plus the routing data), so a mistake such as counting skipped
rows, counting an adapter once per row, or dropping a term changes the total.
With k_in = 16, n_out = 8 and max_rank = 8: a routed row moves 16*2 + 8*2*2 +
8*2*2 = 96 bytes and an adapter 8*16*2 + 8*8*2 + 20 = 404 bytes.
"""
from __future__ import annotations

import numpy as np

import bench
from gather_lora_gb300 import workloads as W

K, N, R = 16, 8, 8


def _pools(entries):
    return (np.zeros((entries, R, K), np.uint16), np.zeros((entries, N, R), np.uint16),
            np.ones(entries, np.float32))


def test_bgmv_bytes():
    # rows: slot 0, base (-1), slot 0, slot 1, slot 2 (NULL entry) -> 3 routed rows, 2 adapters
    seq = np.array([0, -1, 0, 1, 2], np.int32)
    a, b, s = _pools(3)
    wl = W.BgmvWorkload("bytes", 5, K, N, 3, R, K, N, 0, np.zeros((5, K), np.uint16),
                        np.zeros((5, N), np.uint16), seq, np.array([8, 8, 0], np.int32),
                        np.array([True, True, False]), a, b, s)
    got = bench.algorithmic_bytes(wl)
    assert got["routed_rows"] == 3 and got["adapters"] == 2 and got["rows"] == 5
    assert got["bytes"] == 3 * 96 + 2 * 404 + 5 * 4 == 1116
    assert got["flops"] == 2 * 3 * R * (K + N)


def _moe(cap, present):
    # 5 sorted rows: experts [0, 0, 0, 1, 1]; tokens [0, 1, 2, 0, 1]; token adapters [0, -1, 1]
    a, b, s = _pools(4)
    return W.MoeWorkload("bytes", num_tokens=3, top_k=2, num_experts=2, te=5, k_in=K, n_out=N,
                         max_loras=2, max_rank=R, cap=cap, x=np.zeros((5, K), np.uint16),
                         out_buf=np.zeros((5, N), np.uint16),
                         expert_offsets=np.array([0, 3, 5], np.int32),
                         sorted_token_ids=np.array([0, 1, 2, 0, 1], np.int32),
                         row_adapter=np.array([0, -1, 1], np.int32), present=np.array(present),
                         a_pool=a, b_pool=b, scale=s)


def test_moe_bytes():
    # routed rows 0 (a0,e0), 2 (a1,e0), 3 (a0,e1): 3 rows of 96 + 8 routing bytes, 3 pairs
    one = bench.algorithmic_bytes(_moe(5, [True] * 4))
    assert one["routed_rows"] == 3 and one["adapters"] == 3
    assert one["bytes"] == 3 * 104 + 3 * 404 + 1 * 3 * 4 == 1536
    # two windows [0, 3) and [3, 5): the same pairs, the offsets read once per window
    two = bench.algorithmic_bytes(_moe(3, [True] * 4))
    assert two["bytes"] == 3 * 104 + 3 * 404 + 2 * 3 * 4 == 1548
    # the (a1, e0) entry NULL: row 2 is skipped and its pair not read
    null = bench.algorithmic_bytes(_moe(5, [True, True, False, True]))   # entry a*E+e = 1*2+0
    assert null["routed_rows"] == 2 and null["bytes"] == 2 * 104 + 2 * 404 + 12 == 1028


def test_gather_bytes():
    # 2 tokens x top-2: rows (t0: e0, e2), (t1: e5 out of range, e1); adapters [1, 0]
    a, b, s = _pools(6)
    wl = W.MoeGatherWorkload("bytes", num_tokens=2, top_k=2, num_experts=3, k_in=K, n_out=N,
                             max_loras=2, max_rank=R, x=np.zeros((4, K), np.uint16),
                             out_buf=np.zeros((4, N), np.uint16),
                             indices=np.array([0, 2, 5, 1], np.int32),
                             row_adapter=np.array([1, 0], np.int32), present=np.ones(6, bool),
                             a_pool=a, b_pool=b, scale=s)
    got = bench.algorithmic_bytes(wl)
    assert got["routed_rows"] == 3 and got["adapters"] == 3
    assert got["bytes"] == 3 * (96 + 4) + 3 * 404 + 2 * 4 == 1520


def test_delta_bytes():
    wl = W.DeltaWorkload("bytes", 3, K, N, R, R, K, N, 0, np.zeros((3, K), np.uint16),
                         np.zeros((3, N), np.uint16), np.zeros((R, K), np.uint16),
                         np.zeros((N, R), np.uint16), np.float32(1.0))
    got = bench.algorithmic_bytes(wl)
    assert got["bytes"] == 3 * 96 + (R * K * 2 + N * R * 2) == 672


def test_counter_digest_follows_code_not_comments():
    src = 'int f(int a) {  // add one\n  /* block\n     comment */ return a + 1;\n}\n'
    assert bench.code_only(src) == bench.code_only(src.replace("add one", "increment"))
    assert bench.code_only(src) == bench.code_only(src.replace("block", "other text"))
    assert bench.code_only(src) != bench.code_only(src.replace("a + 1", "a + 2"))
    assert "//" not in bench.code_only(src) and "/*" not in bench.code_only(src)
    assert len(bench.kernel_source_digest()) == 16


def test_input_rotation_counts_the_bytes_a_step_touches():
    """The rotation covers more than 2x L2 with the bytes the steps touch, not with the
    whole buffers: an adapter pool mostly untouched by one batch must not count."""
    import bench
    l2 = 126 * 2 ** 20
    # one step touching 34 MB of a 190 MB copy (the decode gather fold's shape)
    assert bench.copies_needed(190 * 10 ** 6, l2, 34 * 10 ** 6) == 8
    # whole buffers smaller than the touched estimate: the buffers bound it
    assert bench.copies_needed(9 * 10 ** 6, l2, 10 ** 9) == 30
    # a step that streams more than 2x L2 needs no second copy
    assert bench.copies_needed(300 * 10 ** 6, l2, 315 * 10 ** 6) == 1
    # at most 64 copies
    assert bench.copies_needed(10 ** 3, l2, 10 ** 3) == 64
