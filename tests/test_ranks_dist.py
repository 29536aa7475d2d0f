"""Ranks that are separate processes (tile_gather_comm_gb300.ranks), host logic on CPU:
two gloo ranks exchange their shard handles, each ends up with every rank's pointer in rank
order (its own at its own index), mismatched shards are refused, and closing unmaps exactly
what was opened.  The IPC calls are replaced by fakes here; the GPU test runs the real ones."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, rows, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    from tile_gather_comm_gb300.ranks import ProcessRanks

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        shard = torch.zeros(rows[rank], 64, dtype=torch.bfloat16)
        opened, closed = [], []
        exporter = lambda t: f"handle-of-rank-{rank}".encode()   # noqa: E731
        opener = lambda h: opened.append(h) or 1000 + int(h.decode().rsplit("-", 1)[1])   # noqa: E731
        closer = lambda p, h: closed.append((p, h))   # noqa: E731
        try:
            pr = ProcessRanks(shard, exporter=exporter, opener=opener, closer=closer)
        except ValueError as e:
            q.put((rank, "refused", str(e)))
            return
        pr.barrier()
        pr.close()
        q.put((rank, "ok", (pr.ptrs, shard.data_ptr(), pr.M, opened, closed)))
    finally:
        dist.destroy_process_group()


def _run(rows):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, len(rows), port, rows, q)) for r in range(len(rows))]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


def test_handles_exchanged_in_rank_order_gloo():
    out = _run([16, 16])
    for rank, status, (ptrs, own, M, opened, closed) in out:
        assert status == "ok"
        assert M == 32
        assert len(ptrs) == 2 and ptrs[rank] == own
        peer = 1 - rank
        assert ptrs[peer] == 1000 + peer                       # the peer's handle, opened
        assert opened == [f"handle-of-rank-{peer}".encode()]  # never its own
        assert closed == [(1000 + peer, f"handle-of-rank-{peer}".encode())]


def test_mismatched_shards_are_refused_gloo():
    out = _run([16, 8])
    assert [s for _, s, _ in out] == ["refused", "refused"]
    assert all("every shard must match" in msg for _, _, msg in out)
