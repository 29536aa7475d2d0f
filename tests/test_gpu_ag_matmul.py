"""Fused AllGather-MatMul on the GPU against the CPU oracle.

Small problems are compared element by element in full; the pages' large
workloads are compared on sampled rows the oracle computes one by one (the
first and last row of every comm block plus seeded random rows, all N
columns), and in full against the library's unfused path, which must match the
fused path bit for bit (same per-tile MMA order).  Tolerance: |C - C_ref| <=
0.02 + 0.01 |C_ref| elementwise -- both sides sum the same bf16 products in fp32,
in different orders, and round once to bf16.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
import tile_gather_comm_gb300 as tgc
from tile_gather_comm_gb300 import _lib
from tile_gather_comm_gb300.workloads import (AG_CONFIGS, AGConfig, make_ag_inputs, make_release_schedule,
                                              sample_rows)

from .helpers import assert_within_tol, bits16, requires_gpu, trace_buffer

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _gpu():
    requires_gpu()


@functools.lru_cache(maxsize=2)
def _inputs(name):
    cfg = AG_CONFIGS[name]
    shards, B = make_ag_inputs(cfg, seed=0)
    return cfg, shards, B


class Run:
    """Device buffers for one problem, reused across calls."""

    def __init__(self, cfg: AGConfig, shards, B):
        self.cfg = cfg
        self.shards = [s.to(DEV) for s in shards]
        self.B = B.to(DEV)
        self.C = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=DEV)
        self.a = torch.empty(cfg.M, cfg.K, dtype=torch.bfloat16, device=DEV)
        self.progress = torch.zeros(cfg.nblocks, dtype=torch.int32, device=DEV)
        nbytes = tgc.tgc_ag_matmul_workspace_bytes(cfg.R, cfg.M, cfg.K, cfg.N, cfg.cb)
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
        self.epoch = 0

    def __call__(self, mode="fused", check=True, **kw):
        self.epoch += 1
        rc = tgc.tgc_ag_matmul_ex(self.shards, self.B, self.C, self.a, self.cfg.cb, mode=mode,
                                  progress=self.progress, epoch=self.epoch, workspace=self.ws, sync=True,
                                  check=check, **kw)
        return rc


def _oracle_full(shards, B):
    return oracle.ag_matmul([bits16(s) for s in shards], bits16(B))


def _expected_pieces(cfg, used):
    """Copy pieces of one call, from the piece size its trace records (one size per call,
    a power of two from 16 to 64 KiB)."""
    sizes = set(int(x) for x in used[:, _lib.TRACE["piece_bytes"]].tolist())
    assert len(sizes) == 1, sizes
    pb = sizes.pop()
    assert pb in (16384, 32768, 65536), pb
    return cfg.nblocks * -(-cfg.cb * cfg.K * 2 // pb)


def _custom(R, H, K, N, cb, seed=0, sigma=1.0):
    cfg = AGConfig("custom", R=R, H=H, K=K, N=N, cb=cb, b_sigma=sigma)
    return (cfg,) + tuple(make_ag_inputs(cfg, seed=seed))


# ----------------------------------------------------------------------------- small, full compare


@pytest.mark.parametrize("mode", ["fused", "unfused", "fused_ce"])
@pytest.mark.parametrize("pivot", ["page", "shard", "none", "ready_queue", "auto"])
def test_tiny_all_ranks(mode, pivot):
    cfg, shards, B = _inputs("tiny")
    C_ref, a_ref = _oracle_full(shards, B)
    run = Run(cfg, shards, B)
    for rank in range(cfg.R):
        run.C.fill_(float("nan"))
        run.a.view(torch.int16).fill_(-1)   # NaN sentinel: a stale read of `a` shows up in C
        run(mode=mode, pivot=pivot, rank=rank)
        assert_within_tol(run.C, C_ref, f"tiny {mode} {pivot} rank {rank}")
        assert np.array_equal(bits16(run.a), a_ref)
        if mode in ("fused", "fused_ce"):
            assert torch.all(run.progress == run.epoch)


@pytest.mark.parametrize("R,H,K,N,cb", [(3, 100, 200, 264, 20), (2, 160, 72, 40, 32), (1, 130, 64, 520, 130),
                                        (4, 256, 136, 256, 64), (8, 128, 64, 8, 128)])
def test_ragged_shapes_full(R, H, K, N, cb):
    """M, N, K that are not multiples of the 128 x 256 x 64 tile; tiles straddling ranks and blocks."""
    cfg, shards, B = _custom(R, H, K, N, cb, seed=R * H)
    C_ref, a_ref = _oracle_full(shards, B)
    run = Run(cfg, shards, B)
    for mode, pivot in (("fused", "page"), ("unfused", "page"), ("fused", "ready_queue"), ("fused_ce", "page")):
        for rank in sorted({0, R - 1}):
            for band_n in (0, -1, 1):  # default (bands for the fused modes), group raster, one-column bands
                for tile_n in ((256,) if mode == "fused_ce" else (256, 512)):
                    run.C.zero_()
                    run(mode=mode, rank=rank, pivot=pivot, band_n=band_n, tile_n=tile_n)
                    assert_within_tol(run.C, C_ref, f"{mode} {pivot} rank {rank} band {band_n} tile {tile_n}")
                    assert np.array_equal(bits16(run.a), a_ref)


@pytest.mark.parametrize("R,H,K,N", [(4, 16, 64, 64), (2, 128, 64, 512), (4, 96, 128, 248)])
def test_integer_exact_bitwise(R, H, K, N):
    """Small-integer inputs: every sum is exact, so C must equal the int64 product bit for bit."""
    g = torch.Generator().manual_seed(R + N)
    lim = 2 if K <= 64 else 1
    si = [torch.randint(-lim, lim + 1, (H, K), generator=g) for _ in range(R)]
    Bi = torch.randint(-lim, lim + 1, (N, K), generator=g)
    ref = torch.cat(si) @ Bi.T
    assert int(ref.abs().max()) <= 256
    cfg = AGConfig("int", R=R, H=H, K=K, N=N, cb=H // 2 if H % 2 == 0 else H, b_sigma=1.0)
    run = Run(cfg, [s.to(torch.bfloat16) for s in si], Bi.to(torch.bfloat16))
    for mode in ("fused", "unfused"):
        for tile_n in (256, 512):
            run.C.zero_()
            run(mode=mode, tile_n=tile_n)
            assert torch.equal(run.C.double().cpu(), ref.double()), (mode, tile_n)


def test_plain_entry_point_tiny_and_ragged():
    for cfg, shards, B in (_inputs("tiny"), _custom(3, 100, 200, 264, 20)):
        C = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=DEV)
        tgc.tgc_ag_matmul([s.to(DEV) for s in shards], B.to(DEV), C, cfg.cb)
        C_ref, _ = _oracle_full(shards, B)
        assert_within_tol(C, C_ref, "plain entry point")


# ----------------------------------------------------------------------------- flags and epochs


def test_stale_epoch_flags_are_not_taken_as_ready():
    """Progress entries hold the previous epoch (a previous round's 1) on entry."""
    cfg, shards, B = _custom(4, 256, 512, 512, 64, seed=3)
    C_ref, _ = _oracle_full(shards, B)
    run = Run(cfg, shards, B)
    run.epoch = 41
    run.progress.fill_(41)
    run.a.view(torch.int16).fill_(-1)
    run(rank=1)
    assert_within_tol(run.C, C_ref, "stale epoch")


def test_repeated_calls_reuse_workspace_and_flags():
    cfg, shards, B = _custom(4, 256, 256, 512, 32, seed=4)
    C_ref, a_ref = _oracle_full(shards, B)
    run = Run(cfg, shards, B)
    for i in range(20):
        run.C.zero_()
        run.a.view(torch.int16).fill_(-1)
        run(rank=i % 4, pivot=["page", "shard", "none", "ready_queue"][i % 4])
        assert_within_tol(run.C, C_ref, f"call {i}")
        assert torch.all(run.ws == 0), "workspace must be left zeroed"


def test_release_order_permutations_and_delays_bit_identical():
    cfg, shards, B = _custom(4, 512, 256, 1024, 64, seed=5)
    run = Run(cfg, shards, B)
    run(mode="unfused")
    C_unf = run.C.clone()
    g = torch.Generator().manual_seed(9)
    for i in range(6):
        order = torch.randperm(cfg.nblocks, generator=g).tolist()
        delay = torch.randint(0, 20000, (cfg.nblocks,), generator=g).tolist() if i % 2 else None
        run.C.zero_()
        run(order=order, delay_ns=delay, rank=i % 4, pivot="ready_queue" if i % 3 == 0 else "page")
        assert torch.equal(run.C, C_unf), f"order {i}"


def test_withheld_block_times_out_and_context_survives():
    """A block left out of the release order is never published: the bounded waits
    expire, the call reports TGC_ERR_TIMEOUT, and the next call works."""
    cfg, shards, B = _custom(4, 256, 128, 256, 64, seed=6)
    run = Run(cfg, shards, B)
    order = [c for c in range(cfg.nblocks) if c != 13]
    rc = run(order=order, spin_timeout_ns=2_000_000, check=False)
    assert rc == _lib.TGC_ERR_TIMEOUT
    run.ws.zero_()
    run.progress.zero_()
    rc = run(order=order, spin_timeout_ns=2_000_000, check=False, pivot="ready_queue")
    assert rc == _lib.TGC_ERR_TIMEOUT
    run.ws.zero_()
    run.progress.zero_()
    rc = run(order=order, spin_timeout_ns=2_000_000, check=False, mode="fused_ce")
    assert rc == _lib.TGC_ERR_TIMEOUT
    torch.cuda.synchronize()
    run.ws.zero_()
    run.progress.zero_()
    run.epoch = 0
    run()
    C_ref, _ = _oracle_full(shards, B)
    assert_within_tol(run.C, C_ref, "after timeout")


# ----------------------------------------------------------------------------- the pages' workloads


@pytest.mark.parametrize("name", ["square", "mlp_up", "large_skewed"])
def test_workload_sampled_rows_and_fused_equals_unfused(name):
    cfg, shards, B = _inputs(name)
    run = Run(cfg, shards, B)
    kw = {}
    if cfg.skewed:
        order, delay = make_release_schedule(cfg, rank=0, seed=0)
        kw = dict(order=order.tolist(), delay_ns=delay.tolist())
    run.a.view(torch.int16).fill_(-1)
    run(mode="fused", **kw)
    C_fused = run.C.clone()
    assert torch.equal(run.a, torch.cat(run.shards))
    # the first and last row of every comm block plus two seeded interior rows of each, so
    # that interior TMEM lanes of both CTAs of a pair are compared with the oracle too
    rows = sample_rows(cfg, seed=0, per_block_random=2)
    ref = oracle.ag_matmul_rows([bits16(s) for s in shards], bits16(B), rows)
    assert_within_tol(C_fused[rows], ref, name)
    run.C.zero_()
    run(mode="unfused")
    assert torch.equal(run.C, C_fused), "fused and unfused differ"
    run.C.zero_()
    run(mode="mm_only")
    assert torch.equal(run.C, C_fused), "mm_only differs"
    run.C.zero_()
    run(mode="fused", pivot="ready_queue", **kw)
    assert torch.equal(run.C, C_fused), "ready-queue order differs"
    run.C.zero_()
    run.a.view(torch.int16).fill_(-1)
    run(mode="fused_ce", **{k: v for k, v in kw.items() if k == "order"})
    assert torch.equal(run.C, C_fused), "copy-engine producer differs"
    assert torch.equal(run.a, torch.cat(run.shards))
    # both tile widths, whichever the default call took: the same MMA chain for every element
    for tile_n in (256, 512):
        for mode in ("fused", "mm_only"):
            run.C.zero_()
            run(mode=mode, tile_n=tile_n, **(kw if mode == "fused" else {}))
            assert torch.equal(run.C, C_fused), (mode, tile_n)


def test_copy_engine_mode_back_to_back_with_other_modes():
    """FUSED_CE calls queued back to back behind other modes without a host synchronisation, as a
    benchmark's interleaved rounds do, on the large workload: the copies, which the runtime may
    run as a kernel of its own, find room beside the GEMM (the mode keeps 256-column tiles), so no
    flag wait expires, and C matches the plain GEMM bit for bit."""
    cfg, shards, B = _inputs("large_skewed")
    run = Run(cfg, shards, B)
    run(mode="unfused")   # gathers `a`, then the plain GEMM
    ref = run.C.clone()
    run.C.zero_()
    for mode in ("fused", "mm_only", "fused_ce", "fused_ce", "unfused", "fused_ce", "fused_ce"):
        run.epoch += 1
        tgc.tgc_ag_matmul_ex(run.shards, run.B, run.C, run.a, cfg.cb, mode=mode, progress=run.progress,
                             epoch=run.epoch, workspace=run.ws, sync=False, spin_timeout_ns=500_000_000)
    torch.cuda.synchronize()
    assert int(run.ws[:4].view(torch.int32)[0]) == 0, "a bounded wait expired"
    assert torch.equal(run.C, ref)
    assert torch.equal(run.a, torch.cat(run.shards))


# ----------------------------------------------------------------------------- CUDA graphs


def test_fused_call_replayed_from_a_cuda_graph():
    """tgc_ag_matmul_ex (sync = 0, no host order arrays) captured in a CUDA graph together with a
    reset of its progress entries, then replayed on new shard contents each time: every replay
    gives the oracle's C for the data it ran on, and the gathered `a`."""
    cfg, shards, B = _custom(4, 256, 512, 776, 64, seed=61)
    run = Run(cfg, shards, B)
    run()   # outside the capture: kernel attributes and the occupancy query are set up once
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run.progress.zero_()
            tgc.tgc_ag_matmul_ex(run.shards, run.B, run.C, run.a, cfg.cb, progress=run.progress, epoch=1,
                                 workspace=run.ws, stream=s, pivot="auto")
    torch.cuda.synchronize()
    gen = torch.Generator().manual_seed(62)
    for i in range(3):
        new = [torch.randn(cfg.H, cfg.K, generator=gen).to(torch.bfloat16) for _ in range(cfg.R)]
        for d, h in zip(run.shards, new):
            d.copy_(h)
        run.C.fill_(float("nan"))
        run.a.view(torch.int16).fill_(-1)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        C_ref, a_ref = _oracle_full(new, B)
        assert_within_tol(run.C, C_ref, f"replay {i}")
        assert np.array_equal(bits16(run.a), a_ref), f"replay {i}: gathered A"
        assert torch.all(_ws_zero(run) == 0), f"replay {i}: workspace counters"


def _ws_zero(run):
    # status word, ticket dispenser and per-block counters (the rest of the workspace holds
    # copies of host arrays and the ready ring, which every call rewrites)
    return torch.cat([run.ws[:4], run.ws[64:80], run.ws[128:128 + 4 * run.cfg.nblocks]])


# ----------------------------------------------------------------------------- edge cases


@pytest.mark.parametrize("R,H,K,N,cb", [
    (64, 16, 64, 64, 16),      # the maximum rank count, one block per rank
    (64, 8, 128, 24, 4),       # 64 ranks, blocks smaller than a tile, tiles straddling 32 ranks
    (1, 512, 64, 256, 64),     # a single rank: every tile local, nothing to wait for
    (2, 1024, 8, 8, 1),        # K = 8 (one 16-byte row), N = 8, one-row blocks: 2048 flags
    (4, 2048, 64, 264, 8),     # 1024 blocks of 8 rows, N not a multiple of the tile
])
def test_edge_shapes_full(R, H, K, N, cb):
    cfg, shards, B = _custom(R, H, K, N, cb, seed=R + H + K)
    C_ref, a_ref = _oracle_full(shards, B)
    run = Run(cfg, shards, B)
    for mode, pivot, rank in (("fused", "page", 0), ("fused", "ready_queue", R - 1), ("fused", "shard", R // 2),
                              ("unfused", "page", 0)):
        run.C.zero_()
        run.a.view(torch.int16).fill_(-1)
        run(mode=mode, pivot=pivot, rank=rank)
        assert_within_tol(run.C, C_ref, f"{mode} {pivot} rank {rank}")
        assert np.array_equal(bits16(run.a), a_ref)


def test_explicit_grid_sizes_give_identical_results():
    """Fewer persistent clusters than SMs (down to one) change only the schedule."""
    cfg, shards, B = _custom(4, 256, 128, 512, 64, seed=11)
    run = Run(cfg, shards, B)
    run(mode="unfused")
    ref = run.C.clone()
    for grid in (2, 6, 30):
        for pivot in ("page", "ready_queue"):
            for tile_n in (256, 512):
                run.C.zero_()
                run(grid=grid, pivot=pivot, tile_n=tile_n)
                assert torch.equal(run.C, ref), (grid, pivot, tile_n)


def test_trace_records_every_cta():
    cfg, shards, B = _custom(4, 512, 256, 1024, 64, seed=12)
    run = Run(cfg, shards, B)
    trace = trace_buffer(_lib.TRACE_WORDS)
    run(trace=trace)
    t = trace.view(-1, _lib.TRACE_WORDS).cpu()
    used = t[t[:, _lib.TRACE["start"]] > 0]
    assert used.shape[0] >= 2
    # both CTAs of a pair count each 256 x 256 tile they share (256-column tiles: K is short here)
    assert int(used[:, _lib.TRACE["tiles"]].sum()) == 2 * (cfg.M // 256) * (cfg.N // 256)
    trace512 = trace_buffer(_lib.TRACE_WORDS)
    run(trace=trace512, tile_n=512)   # the same call on 256 x 512 tiles
    t512 = trace512.view(-1, _lib.TRACE_WORDS).cpu()
    assert int(t512[:, _lib.TRACE["tiles"]].sum()) == 2 * (cfg.M // 256) * (cfg.N // 512)
    # every piece is copied once, by one of the producer warps
    copied = int(used[:, _lib.TRACE["pieces"]].sum())
    assert copied == _expected_pieces(cfg, used)
    assert torch.all(used[:, _lib.TRACE["end"]] >= used[:, _lib.TRACE["start"]])


def test_trace_size_is_checked_against_the_launched_ctas():
    """A trace must hold one record per CTA the call may launch: one per SM with grid 0, at most
    max(grid, 2) otherwise; a smaller buffer is refused before anything is enqueued."""
    cfg, shards, B = _custom(4, 256, 128, 512, 64, seed=13)
    run = Run(cfg, shards, B)
    nsm = torch.cuda.get_device_properties(0).multi_processor_count
    small = torch.zeros((nsm - 2) * _lib.TRACE_WORDS, dtype=torch.int64, device=DEV)
    assert run(trace=small, check=False) == _lib.TGC_ERR_INVALID_ARG
    run.epoch -= 1
    pair = torch.zeros(2 * _lib.TRACE_WORDS, dtype=torch.int64, device=DEV)
    assert run(trace=pair, grid=2, check=False) == _lib.TGC_OK
    assert run(trace=pair, grid=1, check=False) == _lib.TGC_OK      # one pair all the same
    assert run(trace=pair, grid=4, check=False) == _lib.TGC_ERR_INVALID_ARG
    t = pair.view(2, _lib.TRACE_WORDS).cpu()
    assert torch.all(t[:, _lib.TRACE["start"]] > 0)   # both CTAs of the one pair recorded
    C_ref, _ = _oracle_full(shards, B)
    run.epoch -= 1
    run(grid=2)
    assert_within_tol(run.C, C_ref, "one CTA pair")


def test_copy_intensity_follows_local_lead():
    """The producer runs on two warps when the caller's own tiles fill the first two waves of the
    tile order, and on every copy warp when the first waves reach remote rows; the piece size is
    the largest of 64 / 32 / 16 KiB that gives every copy warp two pieces; C is the same."""
    seen = {}
    for label, R, H, K, N in (("lead", 2, 4096, 64, 4096), ("urgent", 8, 512, 64, 4096),
                              ("lead_big_copy", 2, 4096, 4096, 2560)):
        cfg, shards, B = _custom(R, H, K, N, 256, seed=21)
        run = Run(cfg, shards, B)
        run(mode="unfused")
        ref = run.C.clone()
        trace = trace_buffer(_lib.TRACE_WORDS)
        run.C.zero_()
        run(trace=trace)
        assert torch.equal(run.C, ref), label
        t = trace.view(-1, _lib.TRACE_WORDS).cpu()
        used = t[t[:, _lib.TRACE["start"]] > 0]
        warps = set(int(w) for w in used[:, _lib.TRACE["copy_warps"]].tolist())
        assert len(warps) == 1, (label, warps)
        seen[label] = warps.pop()
        assert int(used[:, _lib.TRACE["pieces"]].sum()) == _expected_pieces(cfg, used)
        pb = int(used[0, _lib.TRACE["piece_bytes"]])
        warps_total = used.shape[0] * seen[label]
        pieces = lambda size: cfg.nblocks * -(-cfg.cb * cfg.K * 2 // size)
        expect = next((sz for sz in (65536, 32768) if pieces(sz) >= 2 * warps_total), 16384)
        assert pb == expect, (label, pb, expect)
    assert 1 <= seen["lead"] <= 2 and seen["lead_big_copy"] == seen["lead"]
    assert seen["urgent"] >= seen["lead"]


# ----------------------------------------------------------------------------- float8 e4m3 output


def _e4m3_ulp(v):
    """Spacing of e4m3 values at |v| (subnormal spacing 2^-9 below 2^-6)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0**-6)))
    return np.exp2(e - 3)


def _run_fp8(run, **kw):
    C8 = torch.zeros(run.cfg.M, run.cfg.N, dtype=torch.uint8, device=DEV)
    run.epoch += 1
    tgc.tgc_ag_matmul_ex(run.shards, run.B, C8, run.a, run.cfg.cb, progress=run.progress, epoch=run.epoch,
                         workspace=run.ws, sync=True, out_format="f8e4m3", **kw)
    return C8


def test_fp8_output_integer_exact():
    """Values in {-1, 0, 1}, K = 16: |C| <= 16, and integers up to 16 are exact in e4m3."""
    g = torch.Generator().manual_seed(31)
    R, H, K, N = 4, 64, 16, 272
    si = [torch.randint(-1, 2, (H, K), generator=g) for _ in range(R)]
    Bi = torch.randint(-1, 2, (N, K), generator=g)
    cfg = AGConfig("int8out", R=R, H=H, K=K, N=N, cb=32, b_sigma=1.0)
    run = Run(cfg, [s.to(torch.bfloat16) for s in si], Bi.to(torch.bfloat16))
    ref = (torch.cat(si) @ Bi.T).numpy().astype(np.float64)
    for mode, pivot in (("fused", "page"), ("unfused", "page"), ("fused", "ready_queue")):
        for tile_n in (256, 512):
            C8 = _run_fp8(run, mode=mode, pivot=pivot, tile_n=tile_n)
            assert np.array_equal(oracle.e4m3_to_f64(C8.cpu().numpy()), ref), (mode, tile_n)


def test_fp8_output_square_workload_within_one_step():
    """Sampled rows against the oracle's fp8 rows: the fp32 sums differ only by summation
    order, so the e4m3 results may differ by one step where a sum lies at a rounding boundary."""
    cfg, shards, B = _inputs("square")
    run = Run(cfg, shards, B)
    C8 = _run_fp8(run)
    rows = sample_rows(cfg, seed=0, per_block_random=1)
    ref = oracle.e4m3_to_f64(oracle.ag_matmul_rows_e4m3([bits16(s) for s in shards], bits16(B), rows))
    got = oracle.e4m3_to_f64(C8[rows].cpu().numpy())
    diff = np.abs(got - ref)
    assert np.all(diff <= _e4m3_ulp(ref) + 1e-12)
    assert (diff > 0).mean() < 0.01
    C8u = _run_fp8(run, mode="unfused")
    assert torch.equal(C8, C8u), "fused and unfused fp8 outputs differ"
    C8w = _run_fp8(run, tile_n=512)
    assert torch.equal(C8, C8w), "256- and 512-column tiles give different fp8 outputs"


def test_fp8_output_saturates():
    """Sums beyond 448 saturate to +-448 (0x7E / 0xFE) instead of becoming NaN."""
    g = torch.Generator().manual_seed(32)
    R, H, K, N = 2, 128, 64, 256
    si = [torch.ones(H, K) * 4 for _ in range(R)]
    Bm = torch.ones(N, K) * 4
    Bm[: N // 2] *= -1
    cfg = AGConfig("sat", R=R, H=H, K=K, N=N, cb=64, b_sigma=1.0)
    run = Run(cfg, [s.to(torch.bfloat16) for s in si], Bm.to(torch.bfloat16))
    for tile_n in (256, 512):
        C8 = _run_fp8(run, tile_n=tile_n).cpu().numpy()   # every sum is +-1024
        assert np.all(C8[:, : N // 2] == 0xFE) and np.all(C8[:, N // 2:] == 0x7E), tile_n


# ----------------------------------------------------------------------------- stress


def test_stress_random_orders_delays_pivots_bit_exact():
    """Many calls with random release orders, delays, tile orders, ranks and grid sizes on
    one workspace: every result bit-identical to the unfused path, `a` refilled with NaN
    before each call so that a tile reading a block before its flag would show up in C."""
    cfg, shards, B = _custom(4, 512, 256, 768, 64, seed=77)
    run = Run(cfg, shards, B)
    run(mode="unfused")
    ref = run.C.clone()
    g = torch.Generator().manual_seed(78)
    pivots = ["page", "shard", "none", "ready_queue", "auto"]
    for i in range(150):
        order = torch.randperm(cfg.nblocks, generator=g).tolist()
        delay = torch.randint(0, 5000, (cfg.nblocks,), generator=g).tolist() if i % 3 == 0 else None
        pivot = pivots[int(torch.randint(0, len(pivots), (1,), generator=g))]
        rank = int(torch.randint(0, cfg.R, (1,), generator=g))
        grid = [0, 2, 8, 40][int(torch.randint(0, 4, (1,), generator=g))]
        band_n = [0, -1, 1, 3][int(torch.randint(0, 4, (1,), generator=g))]
        tile_n = [0, 256, 512][int(torch.randint(0, 3, (1,), generator=g))]
        run.a.view(torch.int16).fill_(-1)
        run.C.zero_()
        run(order=order, delay_ns=delay, pivot=pivot, rank=rank, grid=grid, band_n=band_n, tile_n=tile_n)
        assert torch.equal(run.C, ref), (i, pivot, rank, grid, band_n, tile_n)
        assert torch.equal(run.a, torch.cat(run.shards)), i
    # status word, ticket dispenser and per-block counters are zero again (the workspace also
    # keeps the device copies of the last order / delay arrays, which need no clearing)
    ws = run.ws.cpu()
    assert torch.all(ws[:4] == 0) and torch.all(ws[64:80] == 0)
    assert torch.all(ws[128:128 + 4 * cfg.nblocks] == 0)


def test_random_shapes_against_oracle():
    """Seeded random problem shapes (ranks, shard rows, comm-block rows, K, N, rank, tile order,
    mode) compared with the oracle element by element; the fused paths also bit for bit with
    the unfused one and `a` with the concatenated shards."""
    g = torch.Generator().manual_seed(2026)
    pick = lambda seq: seq[int(torch.randint(0, len(seq), (1,), generator=g))]
    for i in range(24):
        R = pick([1, 2, 3, 4, 6, 8])
        cb = pick([8, 16, 40, 64, 128, 256])
        H = cb * pick([1, 2, 3, 5])
        K = 8 * pick([1, 3, 8, 17, 64])
        N = 8 * pick([1, 5, 32, 33, 96])
        cfg, shards, B = _custom(R, H, K, N, cb, seed=100 + i)
        C_ref, a_ref = _oracle_full(shards, B)
        run = Run(cfg, shards, B)
        run(mode="unfused")
        ref = run.C.clone()
        assert_within_tol(run.C, C_ref, f"shape {i}: R={R} H={H} cb={cb} K={K} N={N} unfused")
        for mode, pivot in (("fused", pick(["page", "shard", "ready_queue"])), ("fused_ce", "page")):
            rank = int(torch.randint(0, R, (1,), generator=g))
            tile_n = pick([256, 512]) if mode == "fused" else 0
            run.a.view(torch.int16).fill_(-1)
            run.C.fill_(float("nan"))
            run(mode=mode, pivot=pivot, rank=rank, tile_n=tile_n)
            assert torch.equal(run.C, ref), (i, R, H, cb, K, N, mode, pivot, rank, tile_n)
            assert np.array_equal(bits16(run.a), a_ref), (i, mode)


def test_soak_random_shapes_orders_modes_bit_exact():
    """Many calls over random shapes, release orders, delays, tile orders, ranks, grids and both
    fused producers: C bit-identical to the unfused path and `a` to the shards' concatenation,
    with `a` NaN-filled before every call so that a read ahead of a block's flag shows up."""
    g = torch.Generator().manual_seed(4242)
    pick = lambda seq: seq[int(torch.randint(0, len(seq), (1,), generator=g))]
    for shape_i in range(12):
        R = pick([1, 2, 4, 8])
        cb = pick([16, 64, 128, 256])
        cfg, shards, B = _custom(R, cb * pick([1, 2, 4]), 8 * pick([8, 32, 64]), 8 * pick([32, 64, 96]), cb,
                                 seed=500 + shape_i)
        run = Run(cfg, shards, B)
        run(mode="unfused")
        ref = run.C.clone()
        cat = torch.cat(run.shards)
        for it in range(20):
            mode = pick(["fused", "fused", "fused_ce"])
            order = torch.randperm(cfg.nblocks, generator=g).tolist() if mode == "fused" else None
            delay = (torch.randint(0, 3000, (cfg.nblocks,), generator=g).tolist()
                     if mode == "fused" and it % 2 else None)
            pivot = pick(["page", "shard", "none", "ready_queue"])
            rank = int(torch.randint(0, R, (1,), generator=g))
            grid = pick([0, 2, 16, 64])
            band_n = pick([0, -1, 2, 16])
            tile_n = pick([0, 256, 512]) if mode == "fused" else pick([0, 256])
            run.a.view(torch.int16).fill_(-1)
            run.C.zero_()
            run(mode=mode, order=order, delay_ns=delay, pivot=pivot, rank=rank, grid=grid, band_n=band_n,
                tile_n=tile_n)
            assert torch.equal(run.C, ref), (shape_i, it, mode, pivot, rank, grid, band_n, tile_n)
            assert torch.equal(run.a, cat), (shape_i, it)
