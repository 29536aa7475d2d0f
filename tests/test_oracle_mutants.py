"""The pins catch planted mistakes: each case compiles a copy of oracle.c with
one plausible bug (a wrong rank offset, slab stride, dropped term, sign,
operand index, rounding rule, block placement or shard lookup) and checks that
at least one pin of tests/test_oracle_pins.py fails on it.  The mistakes are
planted in the oracle, on the CPU; the shipped oracle is untouched."""
import os
import subprocess

import numpy as np
import pytest

import oracle

from . import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

# (name, exact text in oracle.c, replacement, pins expected to fail)
MUTANTS = [
    ("tgather_rank_offset", "(slab * dst_rows3 + (int64_t)r * H + i) * W + j",
     "(slab * dst_rows3 + (int64_t)(nranks - 1 - r) * H + i) * W + j", ["tg_scheme", "tg_cat"]),
    ("tgather_slab_stride", "(slab * dst_rows3 + (int64_t)r * H + i) * W + j",
     "(slab * (int64_t)nranks * H * 0 + slab * H + (int64_t)r * H + i) * W + j", ["tg_cat"]),
    ("tgather_skips_last_col", "for (int64_t j = 0; j < W; ++j) {", "for (int64_t j = 0; j + 1 < W; ++j) {",
     ["tg_scheme", "tg_cat"]),
    ("bf16_round_half_up", "u += 0x7FFFu + lsb;", "u += 0x8000u + 0u * lsb;", ["bf16"]),
    ("bf16_truncate", "u += 0x7FFFu + lsb;", "u += 0u * lsb;", ["bf16"]),
    ("gemm_dropped_term", "for (int64_t k = 0; k < K; ++k)\n        acc +=",
     "for (int64_t k = 0; k + 1 < K; ++k)\n        acc +=", ["int_exact", "f64"]),
    ("gemm_wrong_sign", "acc += oracle_bf16_to_f32(arow[k]) * oracle_bf16_to_f32(brow[k]);",
     "acc -= oracle_bf16_to_f32(arow[k]) * oracle_bf16_to_f32(brow[k]);", ["int_exact", "f64"]),
    ("gemm_permuted_k", "acc += oracle_bf16_to_f32(arow[k]) * oracle_bf16_to_f32(brow[k]);",
     "acc += oracle_bf16_to_f32(arow[k]) * oracle_bf16_to_f32(brow[(k * 7 + 1) % K]);", ["int_exact", "f64"]),
    ("chunked_wrong_block_row", "int64_t row0 = src_rank * H + split_id * cb;",
     "int64_t row0 = src_rank * H + (S - 1 - split_id) * cb;", ["chunked"]),
    ("strided_row_index", "int64_t row = (int64_t)r * H + i;", "int64_t row = (int64_t)r * H + (H - 1 - i);",
     ["tg_strided"]),
    ("e4m3_truncate", "        k += 1.0;\n    if (k == 8.0) {", "        k += 0.0;\n    if (k == 8.0) {", ["e4m3"]),
    ("e4m3_no_saturation", "if (a >= 448.0)\n        return (uint8_t)(sign | 0x7Eu);",
     "if (a >= 480.0)\n        return (uint8_t)(sign | 0x7Fu);", ["e4m3"]),
    ("rows_wrong_shard", "const uint16_t *arow = a_shards[m / H] + (m % H) * K;",
     "const uint16_t *arow = a_shards[(m / H + 1) % R] + (m % H) * K;", ["rows"]),
]


def _compile(tmp_path, name, old, new):
    text = open(SRC, encoding="utf-8").read()
    assert text.count(old) >= 1, f"mutation anchor for {name} not found"
    mutated = text.replace(old, new, 1)
    c = tmp_path / f"{name}.c"
    c.write_text(mutated, encoding="utf-8")
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-shared", "-fPIC", "-std=c11",
                    "-o", str(so), str(c)], check=True)
    return oracle.load_from(str(so))


def _run_pin(kind, o):
    if kind == "tg_scheme":
        for case in pins._golden_cases():
            if case[2] > 0:
                for n in (2, 4):
                    pins.test_tgather_page_value_scheme(o, case, n)
    elif kind == "tg_cat":
        import torch
        for shape in [(2, 3, 2, 5, 7), (1, 2, 1, 13, 33)]:
            pins.test_tgather_equals_torch_cat_dim3(o, shape, torch.int32, 3)
    elif kind == "bf16":
        pins.test_bf16_rne_matches_torch_on_random_bit_patterns(o)
        pins.test_bf16_rne_edge_cases(o)
    elif kind == "int_exact":
        for args in [(4, 16, 64, 40), (2, 24, 64, 96)]:
            pins.test_ag_matmul_integer_exact(o, *args)
    elif kind == "f64":
        pins.test_ag_matmul_vs_float64(o, 4, 16, 64, 64, 1.0)
    elif kind == "chunked":
        pins.test_chunked_equals_gather_then_matmul(o, 0)
    elif kind == "rows":
        pins.test_rows_variant_matches_full(o)
    elif kind == "e4m3":
        pins.test_e4m3_rne_matches_torch_inside_range(o)
        pins.test_e4m3_grid_points_ties_and_saturation(o)
    elif kind == "tg_strided":
        for case in ("slices", "transposed_w", "padded_dst"):
            pins.test_tgather_strided_views_equal_torch_cat(o, case)
    else:
        raise ValueError(kind)


def test_unmutated_copy_passes_every_pin_used_here(tmp_path):
    o = _compile(tmp_path, "identity", "int oracle_tgather(", "int oracle_tgather(")
    for kind in ("tg_scheme", "tg_cat", "bf16", "int_exact", "f64", "chunked", "rows", "tg_strided", "e4m3"):
        _run_pin(kind, o)


@pytest.mark.parametrize("name,old,new,kinds", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new, kinds):
    o = _compile(tmp_path, name, old, new)
    for kind in kinds:
        with pytest.raises(AssertionError):
            _run_pin(kind, o)
