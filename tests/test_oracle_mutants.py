"""Planted mistakes in the oracle must fail its pins (CPU only).

Each mutant is a copy of oracle.c with one plausible mistake (a transposed
operand, a wrong stride, a dropped or sign-flipped term, a wrong rounding, a
shifted index). It is compiled to a temporary library and the pin suite
(test_oracle_pins.py) is run against it in a subprocess; the suite must fail.
Mutants are chosen so that none reads or writes out of bounds.
"""
from __future__ import annotations

import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "b_transposed": ("acc = acc + ora_f32_of_bf16(xa_row[c]) * ora_f32_of_bf16(brow[c]);",
                     "acc = acc + ora_f32_of_bf16(xa_row[c]) * ora_f32_of_bf16(B[(int64_t)c * n_out + j]);"),
    "a_wrong_stride": ("const uint16_t* arow = A + (int64_t)c * k_in;",
                       "const uint16_t* arow = A + (int64_t)c;"),
    "scale_dropped": ("float folded = fmaf(scale, ", "float folded = fmaf(1.0f, "),
    "scale_sign": ("float folded = fmaf(scale, ", "float folded = fmaf(-scale, "),
    "scale_before_rounding": ("            d = ora_bf16_of_f32(acc);",
                              "            d = ora_bf16_of_f32(acc * scale); scale = 1.0f;"),
    "truncating_bf16": ("        upper += 1u;                               /* carries into the exponent */",
                        "        upper += 0u;"),
    "out_stride": ("base_out + (int64_t)i * out_row_stride", "base_out + (int64_t)i * n_out"),
    "x_stride": ("x + (int64_t)i * x_row_stride", "x + (int64_t)i * k_in"),
    "slot_zero_skipped": ("if (s < 0 || s >= max_loras) continue;", "if (s < 1 || s >= max_loras) continue;"),
    "expert_span_shifted": ("if (expert_offsets[k] <= r && r < expert_offsets[k + 1])",
                            "if (expert_offsets[k] < r && r <= expert_offsets[k + 1])"),
    "moe_table_expert_major": ("int64_t ti = (int64_t)a * num_experts + e;",
                               "int64_t ti = (int64_t)e * max_loras + a;"),
    "gate_up_reads_sorted_row": ("const int64_t xr = x_gather ? t : r;", "const int64_t xr = r;"),
    "gather_token_of_row": ("const int32_t t = r / top_k;", "const int32_t t = r % top_k;"),
    "gather_table_expert_major": ("const int64_t entry = (int64_t)a * num_experts + e;",
                                  "const int64_t entry = (int64_t)e * max_loras + a;"),
    "delta_out_stride": ("uint16_t* out_row = base_out + (int64_t)row * out_row_stride;",
                         "uint16_t* out_row = base_out + (int64_t)row * n_out;"),
    "delta_x_stride": ("const uint16_t* x_row = x + (int64_t)row * x_row_stride;",
                       "const uint16_t* x_row = x + (int64_t)row * k_in;"),
    "xa_truncated": ("            xa_row[c] = ora_bf16_of_f32(acc);",
                     "            { uint32_t u; memcpy(&u, &acc, sizeof u); xa_row[c] = (uint16_t)(u >> 16); }"),
    "delta_truncated": ("            d = ora_bf16_of_f32(acc);",
                        "            { uint32_t u; memcpy(&u, &acc, sizeof u); d = (uint16_t)(u >> 16); }"),
    "fold_rounds_twice": ("float folded = fmaf(scale, ora_f32_of_bf16(d), ora_f32_of_bf16(orow[j]));",
                          "float folded = ora_f32_of_bf16(ora_bf16_of_f32(scale * ora_f32_of_bf16(d)))"
                          " + ora_f32_of_bf16(orow[j]);"),
    "last_rank_dropped": ("for (int32_t c = 0; c < max_rank; ++c)\n                acc = acc + ora_f32_of_bf16(xa_row[c])",
                          "for (int32_t c = 0; c < max_rank - 1; ++c)\n                acc = acc + ora_f32_of_bf16(xa_row[c])"),
    "window_first_row_skipped": ("for (int32_t r = row_offset; r < row_end; ++r) {",
                                 "for (int32_t r = row_offset + 1; r < row_end; ++r) {"),
    "moe_adapter_gate_ignored": ("int32_t a = row_adapter ? row_adapter[t] : 0;\n        if (a < 0 || a >= max_loras) continue;\n        int64_t ti",
                                 "int32_t a = 0;\n        if (a < 0 || a >= max_loras) continue;\n        int64_t ti"),
    "moe_d_at_window_row": ("uint16_t* d_row = d_out ? d_out + (int64_t)r * n_out : NULL;\n        const int64_t xr",
                            "uint16_t* d_row = d_out ? d_out + local * n_out : NULL;\n        const int64_t xr"),
    "gather_expert_zero_skipped": ("if (e < 0 || e >= num_experts) continue;",
                                   "if (e < 1 || e >= num_experts) continue;"),
    "gather_last_token_skipped": ("if (t >= num_tokens) continue;", "if (t >= num_tokens - 1) continue;"),
    "last_k_dropped": ("for (int32_t k = 0; k < k_in; ++k)\n                acc = acc + ora_f32_of_bf16(xrow[k])",
                       "for (int32_t k = 0; k < k_in - 1; ++k)\n                acc = acc + ora_f32_of_bf16(xrow[k])"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_fails_pins(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site for {name} not unique"
    mutated = src.replace(old, new, 1)
    mpath = tmp_path / "oracle.c"
    mpath.write_text(mutated)
    # the mutant includes oracle.h from the oracle directory
    lib = tmp_path / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    "-I", os.path.join(ROOT, "oracle"), "-o", str(lib), str(mpath), "-lm"],
                   check=True)
    env = dict(os.environ, GATHER_LORA_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_pins.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
