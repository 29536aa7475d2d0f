"""Ranks that are separate processes: each holds its shard, the others address it.

"Triton第四课：基于对称内存融合 AllGather 与 MatMul，提速1.56倍", section
对称内存如何打通GPU间访问: every rank allocates its a_shard (M/W, K) in memory the
other ranks can address, and each rank's producer copies the others' shards into
its own aggregate buffer `a` before (or while) its MatMul reads it; section
数据搬运与细粒度同步: a rank's flags and its `a` are its own.

This module is host plumbing only.  It exports the caller's shard as an IPC handle
(tgc_ipc_export), exchanges the handles with the other ranks over a
torch.distributed process group (gloo is enough: only a few bytes per rank travel),
opens the peers' handles (tgc_ipc_open), and orders the ranks around each call
with barriers: every shard is complete before any rank's kernel may read it, and
no rank rewrites or frees its shard before every rank's kernel has finished.  All
bytes of the gather are moved by the library's kernels (tgc_ag_matmul_ex with the
peer pointers as a_shards and `rank` set to the caller).
"""
from __future__ import annotations

import torch

from . import _lib


class ProcessRanks:
    """The shard pointers of all ranks, as seen by this process.

    ``shard``: this rank's (M/W, K) bf16 shard, a device tensor whose memory comes
    from cudaMalloc (the default torch allocator).  ``group``: the process group of
    the ranks (default: the world), one process per rank, ranks in order.
    ``exporter`` / ``opener`` / ``closer`` default to the library's IPC calls; they
    are parameters so that the exchange can be exercised without a GPU.
    """

    def __init__(self, shard, group=None, exporter=None, opener=None, closer=None):
        import torch.distributed as dist

        self._dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self._open = opener or _lib.tgc_ipc_open
        self._close = closer or _lib.tgc_ipc_close
        handle = (exporter or _lib.tgc_ipc_export)(shard)
        meta = {"handle": bytes(handle), "shape": tuple(shard.shape), "dtype": str(shard.dtype)}
        metas = [None] * self.world
        dist.all_gather_object(metas, meta, group=group)
        for r, m in enumerate(metas):
            if m["shape"] != meta["shape"] or m["dtype"] != meta["dtype"]:
                raise ValueError(f"rank {r} holds a {m['dtype']} {m['shape']} shard, rank {self.rank} "
                                 f"a {meta['dtype']} {meta['shape']} one: every shard must match")
        self.rows_per_rank, self.K = meta["shape"]
        self.M = self.world * self.rows_per_rank
        self.ptrs = []
        self._opened = []
        try:
            for r, m in enumerate(metas):
                if r == self.rank:
                    self.ptrs.append(shard.data_ptr())
                else:
                    p = self._open(m["handle"])
                    self._opened.append((p, m["handle"]))
                    self.ptrs.append(p)
        except Exception:
            self.close()
            raise
        self._shard = shard  # keeps this rank's shard alive while peers may read it

    def barrier(self):
        """Every rank's device work enqueued so far has finished, on every rank."""
        if torch.cuda.is_available():
            torch.cuda.synchronize()
        self._dist.barrier(group=self.group)

    def ag_matmul(self, B, C, a_out, comm_block_rows: int, progress=None, workspace=None, epoch: int | None = None,
                  **kw) -> int:
        """C = gather(all ranks' shards) @ B^T on this rank: tgc_ag_matmul_ex with the peers' pointers,
        ``rank`` = this rank, mode FUSED and tile order AUTO unless ``kw`` says otherwise, between the
        barriers that make the peers' shards safe to read.  ``progress`` / ``workspace`` default to
        buffers this object keeps for the problem (zeroed once; each call publishes a new epoch)."""
        nblocks = self.M // comm_block_rows
        if progress is None or workspace is None:
            key = (nblocks, B.shape[0])
            if getattr(self, "_bufs_key", None) != key:
                dev = B.device
                nbytes = _lib.tgc_ag_matmul_workspace_bytes(self.world, self.M, self.K, B.shape[0], comm_block_rows)
                self._bufs = (torch.zeros(nblocks, dtype=torch.int32, device=dev),
                              torch.zeros(nbytes, dtype=torch.uint8, device=dev))
                self._bufs_key = key
                self._epoch = 0
            progress = self._bufs[0] if progress is None else progress
            workspace = self._bufs[1] if workspace is None else workspace
        if epoch is None:
            self._epoch = getattr(self, "_epoch", 0) + 1
            epoch = self._epoch
        kw.setdefault("pivot", "auto")
        self.barrier()
        try:
            rc = _lib.tgc_ag_matmul_ex(self.ptrs, B, C, a_out, comm_block_rows, M=self.M, rank=self.rank,
                                       progress=progress, workspace=workspace, epoch=epoch, sync=True, **kw)
        finally:
            self.barrier()
        return rc

    def close(self):
        """Unmap the peers' shards.  Call it on every rank after the last call, then barrier again
        before any rank frees its shard."""
        for p, h in self._opened:
            self._close(p, h)
        self._opened = []
