"""Ranks that are separate processes, on one GPU: two processes each hold one shard in their own
allocation, exchange IPC handles over gloo, and each runs the fused call as its own rank with the
peer's shard mapped into its address space (tile_gather_comm_gb300.ranks).  Every rank's C is
compared with the CPU oracle element by element, its gathered `a` bit for bit with the
concatenated shards, for the fused path (default order, page pivot, ready order), the
copy-engine producer and the unfused path.  Each rank has its own B, as in tensor parallelism.

The kernels of the two processes never wait on each other: each waits only on flags its own
producer sets, and a host barrier orders the shards' writes before any kernel reads them."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

from .helpers import requires_gpu

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist

    import oracle
    from tile_gather_comm_gb300.ranks import ProcessRanks
    from tile_gather_comm_gb300.workloads import AGConfig, make_ag_inputs
    from tests.helpers import assert_within_tol, bits16

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        oracle.build()
        cfg = AGConfig("ranks", R=world, H=384, K=512, N=776, cb=64, b_sigma=0.02)
        shards_h, _ = make_ag_inputs(cfg, seed=5)             # every rank draws the same shards
        _, B_h = make_ag_inputs(cfg, seed=100 + rank)         # and its own B
        shard = shards_h[rank].cuda()                         # but holds only its own on the device
        B = B_h.cuda()
        C_ref, a_ref = oracle.ag_matmul([bits16(s) for s in shards_h], bits16(B_h))
        pr = ProcessRanks(shard)
        C = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device="cuda")
        a = torch.empty(cfg.M, cfg.K, dtype=torch.bfloat16, device="cuda")
        cases = [dict(), dict(pivot="page", band_n=-1), dict(pivot="ready_queue", order=list(range(cfg.nblocks))[::-1]),
                 dict(mode="fused_ce"), dict(mode="unfused")]
        for kw in cases:
            C.fill_(float("nan"))
            a.view(torch.int16).fill_(-1)   # a read of `a` ahead of its flag shows up as NaN in C
            pr.ag_matmul(B, C, a, cfg.cb, **kw)
            assert_within_tol(C, C_ref, f"rank {rank} {kw}")
            assert np.array_equal(bits16(a), a_ref), f"rank {rank} {kw}: gathered A"
        pr.barrier()
        pr.close()
        pr.barrier()   # no rank frees its shard while a peer still has it mapped
        q.put((rank, "ok"))
    except BaseException as e:  # reported to the parent, which fails the test
        q.put((rank, f"{type(e).__name__}: {e}"))
        raise
    finally:
        dist.destroy_process_group()


def test_two_process_ranks_on_one_gpu_match_oracle():
    requires_gpu()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = []
    try:
        for _ in procs:
            results.append(q.get(timeout=300))
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
                p.join(timeout=30)
    assert sorted(results) == [(0, "ok"), (1, "ok")], results
    assert all(p.exitcode == 0 for p in procs)
