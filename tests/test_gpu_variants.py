"""The library's non-default compile-time paths, built once into a separate
library under the package's build folder and checked like the default build:

- TGC_COPY_LSU=0: the fused kernel's producer is one warp of bulk async copies
  (global -> shared -> global through four slots) instead of register copies;
- TGC_TG_CHUNK=0: the flat TGATHER kernel gives each CTA one contiguous share
  instead of dealing 32 KiB chunks round-robin;
- TGC_TG_VW32=0: the flat TGATHER kernel moves 16-byte vectors where 32-byte
  ones would do;
- TGC_TMA_STORE_C=0: the GEMM epilogue stores C with per-thread 16-byte stores
  instead of TMA stores of shared-memory boxes (the bulk-copy kernel always
  does).

A second build keeps the default register-copy producer and turns only the
per-thread C stores on, together with the TGATHER release kernel's earliest
form (no publisher block at any chunk count: the block whose count completes
a chunk publishes it, each count a gpu-scope fence then an acq_rel add; no
programmatic dependent launch), so that each of those paths is run on its own.

Results must be identical to the oracle (TGATHER bit for bit, GEMM within the
tolerance, bit for bit on integer-exact inputs) and to the default build's
unfused path.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import tile_gather_comm_gb300 as tgc
from tile_gather_comm_gb300 import _build, _lib
from tile_gather_comm_gb300.workloads import TG_CONFIGS, make_tg_inputs, sample_rows

from .helpers import assert_within_tol, bits16, requires_gpu, trace_buffer
from .test_gpu_ag_matmul import Run, _custom, _expected_pieces, _inputs, _oracle_full

pytestmark = pytest.mark.gpu
DEV = "cuda"
VARIANT = {"TGC_COPY_LSU": 0, "TGC_TG_CHUNK": 0, "TGC_TG_VW32": 0, "TGC_TMA_STORE_C": 0}
VARIANT_CSTORE = {"TGC_TMA_STORE_C": 0, "TGC_TG_REL_ATOM": 0, "TGC_TG_REL_PDL": 0, "TGC_TG_REL_POLL": 0}


@pytest.fixture(scope="module")
def variant_lib():
    requires_gpu()
    path = _build.build_variant(os.path.join(_build.PKG, "_build", "variant_bulk_copy"), VARIANT)
    return _lib.load_library(path)


@pytest.fixture
def use_variant(variant_lib):
    """Route the binding's calls to the variant build for the duration of a test."""
    default = _lib.lib()
    _lib._lib = variant_lib
    try:
        yield variant_lib
    finally:
        _lib._lib = default


@pytest.mark.parametrize("pivot", ["page", "ready_queue"])
def test_bulk_producer_tiny_all_ranks(use_variant, pivot):
    cfg, shards, B = _inputs("tiny")
    C_ref, a_ref = _oracle_full(shards, B)
    run = Run(cfg, shards, B)
    for rank in range(cfg.R):
        run.C.fill_(float("nan"))
        run.a.view(torch.int16).fill_(-1)  # a stale read of `a` shows up as NaN in C
        run(pivot=pivot, rank=rank)
        assert_within_tol(run.C, C_ref, f"bulk producer {pivot} rank {rank}")
        assert np.array_equal(bits16(run.a), a_ref)


def test_bulk_producer_integer_exact_and_trace(use_variant):
    # integer values in {-2..2}, K = 64: every partial sum is exact, so C is exact
    cfg, _, _ = _custom(4, 256, 64, 512, 64, seed=31)
    g = torch.Generator().manual_seed(31)
    shards = [torch.randint(-2, 3, (cfg.H, cfg.K), generator=g).to(torch.bfloat16) for _ in range(cfg.R)]
    B = torch.randint(-2, 3, (cfg.N, cfg.K), generator=g).to(torch.bfloat16)
    run = Run(cfg, shards, B)
    trace = trace_buffer(_lib.TRACE_WORDS)
    run(trace=trace)
    exact = (torch.cat(shards).double() @ B.double().T).to(torch.bfloat16)
    assert torch.equal(run.C.cpu(), exact)
    t = trace.view(-1, _lib.TRACE_WORDS).cpu()
    used = t[t[:, _lib.TRACE["start"]] > 0]
    assert set(used[:, _lib.TRACE["copy_warps"]].tolist()) == {1}
    assert int(used[:, _lib.TRACE["pieces"]].sum()) == _expected_pieces(cfg, used)


def test_bulk_producer_matches_unfused_bitwise(use_variant):
    # ragged: M not a multiple of the 256-row tile, N not a multiple of 256
    cfg, shards, B = _custom(3, 200, 256, 328, 40, seed=32)
    run = Run(cfg, shards, B)
    run(mode="unfused")
    ref = run.C.clone()
    for pivot in ("page", "shard", "ready_queue"):
        for tile_n in (256, 512):
            run.C.zero_()
            run(pivot=pivot, tile_n=tile_n)
            assert torch.equal(run.C, ref), (pivot, tile_n)
    assert torch.equal(run.a, torch.cat(run.shards))


@pytest.mark.parametrize("name", ["bw_f16", "ragged_i32"])
def test_one_share_tgather_bit_exact(use_variant, name):
    cfg = TG_CONFIGS[name]
    srcs = make_tg_inputs(cfg, seed=0)
    D0, D1, D2, H, W = cfg.shape
    dst = torch.empty((D0, D1, D2, cfg.nranks * H, W), dtype=cfg.dtype, device=DEV)
    dst.view(torch.uint8).fill_(0xA5)
    tgc.tgc_tgather(dst, [s.to(DEV) for s in srcs])
    torch.cuda.synchronize()
    ref = oracle.tgather([s.numpy() for s in srcs])
    assert dst.cpu().numpy().tobytes() == ref.tobytes()


# ----------------------------------------------------------------------------- per-thread C stores


@pytest.fixture(scope="module")
def cstore_lib():
    requires_gpu()
    path = _build.build_variant(os.path.join(_build.PKG, "_build", "variant_cstore"), VARIANT_CSTORE)
    return _lib.load_library(path)


@pytest.fixture
def use_cstore(cstore_lib):
    default = _lib.lib()
    _lib._lib = cstore_lib
    try:
        yield cstore_lib
    finally:
        _lib._lib = default


@pytest.mark.parametrize("R,H,K,N,cb", [(3, 100, 200, 264, 20), (4, 256, 136, 256, 64), (2, 160, 72, 40, 32)])
def test_cstore_register_copy_ragged_against_oracle(use_cstore, R, H, K, N, cb):
    """The default producer with per-thread C stores: ragged M and N (stores clipped by hand),
    every tile order, first and last rank, against the oracle and bit for bit with unfused."""
    cfg, shards, B = _custom(R, H, K, N, cb, seed=7 * R + H)
    C_ref, a_ref = _oracle_full(shards, B)
    run = Run(cfg, shards, B)
    run(mode="unfused")
    ref = run.C.clone()
    assert_within_tol(ref, C_ref, "cstore unfused")
    for pivot in ("page", "shard", "ready_queue"):
        for rank in sorted({0, R - 1}):
            for tile_n in (256, 512):
                run.C.fill_(float("nan"))
                run.a.view(torch.int16).fill_(-1)
                run(pivot=pivot, rank=rank, tile_n=tile_n)
                assert torch.equal(run.C, ref), (pivot, rank, tile_n)
                assert np.array_equal(bits16(run.a), a_ref)


def test_cstore_square_workload_sampled_rows(use_cstore):
    cfg, shards, B = _inputs("square")
    run = Run(cfg, shards, B)
    run(pivot="ready_queue")
    rows = sample_rows(cfg, seed=0, per_block_random=1)
    ref = oracle.ag_matmul_rows([bits16(s) for s in shards], bits16(B), rows)
    assert_within_tol(run.C[rows], ref, "cstore square")


@pytest.mark.parametrize("H,W,chunk_rows,D0", [(1024, 1024, 128, 2), (1000, 777, 96, 1)])
def test_cstore_build_release_kernel_bit_exact(use_cstore, H, W, chunk_rows, D0):
    """The TGATHER release kernel's earliest form (the completing block publishes; fence, then an
    acq_rel count per item)."""
    nranks = 8
    shape = (D0, 1, 1, H, W)
    g = torch.Generator().manual_seed(H * W)
    srcs = [torch.randint(-2**31, 2**31, shape, generator=g, dtype=torch.int64).to(torch.int32)
            for _ in range(nranks)]
    S = -(-H // chunk_rows)
    progress = torch.full((nranks * S,), 2, dtype=torch.int32, device=DEV)
    counters = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    dst = torch.zeros((D0, 1, 1, nranks * H, W), dtype=torch.int32, device=DEV)
    tgc.tgc_tgather_ex(dst, [s.to(DEV) for s in srcs], progress=progress, counters=counters,
                       chunk_rows=chunk_rows, epoch=3)
    torch.cuda.synchronize()
    assert dst.cpu().numpy().tobytes() == oracle.tgather([s.numpy() for s in srcs]).tobytes()
    assert torch.all(progress == 3) and torch.all(counters == 0)
