"""tgc_ag_matmul_noalloc: the fused AllGather-MatMul for callers that cannot
allocate device memory (a memory manager that owns the device and forbids raw
cudaMalloc, or a path where no allocation may happen after start-up).  Its
scratch is a fixed array inside the library, so these tests check that two
calls in a row -- the second one finding the first one's flags and counters in
that array -- give the CPU oracle's result, within the tolerance of every GEMM
parity test here (|C - C_ref| <= 0.02 + 0.01 |C_ref|), and the same result as the
allocating entry point.

This file is named to be collected last, so that a run stopping at its first
failure has already run every other test."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import tile_gather_comm_gb300 as tgc
from tile_gather_comm_gb300 import _lib
from tile_gather_comm_gb300.workloads import AG_CONFIGS, AGConfig, make_ag_inputs

from .helpers import assert_within_tol, bits16, requires_gpu

DEV = "cuda"


def _problem(cfg, seed):
    shards, B = make_ag_inputs(cfg, seed=seed)
    return [s.to(DEV) for s in shards], B.to(DEV)


@pytest.mark.gpu
def test_noalloc_matches_allocating_entry_point_on_consecutive_calls():
    requires_gpu()
    cases = [AGConfig("mid", R=4, H=256, K=512, N=768, cb=64, b_sigma=0.02), AG_CONFIGS["tiny"]]
    for cfg in cases:
        shards, B = _problem(cfg, seed=cfg.H)
        C_ref = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=DEV)
        tgc.tgc_ag_matmul(shards, B, C_ref, cfg.cb)  # existing (allocating) entry point
        ref_bits = bits16(C_ref)
        oracle.build()
        oracle_C, oracle_a = oracle.ag_matmul([bits16(s) for s in shards], bits16(B))
        assert_within_tol(C_ref, oracle_C, f"{cfg.name} allocating entry point")
        for call in range(2):  # two calls in a row share the library's scratch
            C = torch.full((cfg.M, cfg.N), float("nan"), dtype=torch.bfloat16, device=DEV)
            a_out = torch.full((cfg.M, cfg.K), float("nan"), dtype=torch.bfloat16, device=DEV)
            tgc.tgc_ag_matmul_noalloc(shards, B, C, a_out, cfg.cb)
            assert_within_tol(C, oracle_C, f"{cfg.name} call {call} vs oracle")
            assert_within_tol(C, ref_bits, f"{cfg.name} call {call} vs tgc_ag_matmul")
            assert np.array_equal(bits16(a_out), oracle_a), f"{cfg.name} call {call}: gathered A"


def test_noalloc_rejects_too_many_blocks_before_any_device_work():
    fake = 1 << 20
    arr = (ctypes.c_void_p * 4)(*([fake] * 4))
    L = _lib.lib()
    M = 4 * (_lib.NOALLOC_MAX_BLOCKS // 4 + 1) * 8  # one 8-row block more than the limit, per-rank rows % 8 == 0
    rc = L.tgc_ag_matmul_noalloc(arr, 4, fake, fake, fake, M, 64, 64, 8, None)
    assert rc == _lib.TGC_ERR_TOO_LARGE
    assert "noalloc" in tgc.tgc_status_string(rc)
    # within the limit, argument errors are reported as for the other entry points
    assert L.tgc_ag_matmul_noalloc(arr, 4, fake, fake, fake, 66, 64, 64, 8, None) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_ag_matmul_noalloc(arr, 4, fake, fake, fake, 0, 64, 64, 8, None) == _lib.TGC_OK


def test_noalloc_rejects_scratch_overflow_from_tile_rows():
    """Within the block limit, the per-tile-row counters and ready ring can still overflow the
    fixed scratch: 2048 blocks of 512 rows (M = 1,048,576, 4096 tile rows) do."""
    fake = 1 << 20
    arr = (ctypes.c_void_p * 1)(fake)
    L = _lib.lib()
    M = _lib.NOALLOC_MAX_BLOCKS * 512
    assert L.tgc_ag_matmul_noalloc(arr, 1, fake, fake, fake, M, 64, 64, 512, None) == _lib.TGC_ERR_TOO_LARGE


def test_noalloc_python_limits_match_header():
    text = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "tgc.h"),
                encoding="utf-8").read()
    assert int(re.search(r"#define TGC_NOALLOC_MAX_BLOCKS (\d+)", text).group(1)) == _lib.NOALLOC_MAX_BLOCKS
    assert int(re.search(r"#define TGC_NOALLOC_SCRATCH_BYTES (\d+)", text).group(1)) == _lib.NOALLOC_SCRATCH_BYTES
