"""Seeded synthetic inputs for the chunked AllGather x MatMul path.

This module holds workload shapes and random-number recipes only; it performs
none of the method's arithmetic, so both the CUDA path and the CPU oracle may
take their inputs from it.

Recipe (every workload): one ``torch.Generator('cpu').manual_seed(seed)``;
draws are made in this order: the R bf16 shards (rank 0 first), then B, then
the TGATHER sources.  bf16 normals are ``randn(float32) * sigma`` rounded to
bf16 by torch.  The release schedule of the skewed workload (order and
delays) comes from a second generator seeded with ``seed``, so the data do
not depend on whether the schedule is drawn.

Shapes follow the pages' setting ("Triton第四课：基于对称内存融合
AllGather 与 MatMul", section 对称内存如何打通GPU间访问: a_shard (M/W, K) bf16,
b = randn(k, n).T.contiguous() stored (N, K); "CANN PTO-ISA TGATHER 指令深度解析",
§二 and §九: per-rank (D0, D1, D2, H, W) sources).
"""
from __future__ import annotations

import dataclasses

import torch


@dataclasses.dataclass(frozen=True)
class AGConfig:
    name: str
    R: int              # virtual ranks (separate shard allocations)
    H: int              # rows per shard (M / R)
    K: int
    N: int
    cb: int             # comm_block_rows
    b_sigma: float
    skewed: bool = False  # seeded release permutation + injected delays
    max_delay_ns: int = 20_000

    @property
    def M(self) -> int:
        return self.R * self.H

    @property
    def nblocks(self) -> int:
        return self.M // self.cb

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K


@dataclasses.dataclass(frozen=True)
class TGConfig:
    name: str
    nranks: int
    shape: tuple          # per-rank (D0, D1, D2, H, W)
    dtype: torch.dtype
    dist: str             # "uniform11", "normal", "int32full"

    @property
    def bytes_moved(self) -> int:
        """Algorithmic bytes: every source byte read once, every dst byte written once."""
        n = 1
        for s in self.shape:
            n *= s
        es = torch.empty((), dtype=self.dtype).element_size()
        return 2 * self.nranks * n * es


AG_CONFIGS = {
    "tiny": AGConfig("tiny", R=4, H=16, K=64, N=64, cb=8, b_sigma=1.0),
    "square": AGConfig("square", R=8, H=512, K=4096, N=4096, cb=128, b_sigma=0.02),
    "mlp_up": AGConfig("mlp_up", R=8, H=1024, K=4096, N=14336, cb=256, b_sigma=0.02),
    "large_skewed": AGConfig("large_skewed", R=4, H=8192, K=8192, N=8192, cb=512,
                             b_sigma=0.02, skewed=True),
}

TG_CONFIGS = {
    "tiny_f32": TGConfig("tiny_f32", 4, (1, 1, 1, 8, 32), torch.float32, "uniform11"),
    "bw_f16": TGConfig("bw_f16", 8, (2, 1, 1, 1024, 1024), torch.float16, "normal"),
    "ragged_i32": TGConfig("ragged_i32", 8, (1, 1, 1, 1000, 777), torch.int32, "int32full"),
}


def _bf16_normal(shape, sigma, g):
    return torch.randn(shape, generator=g, dtype=torch.float32).mul_(sigma).to(torch.bfloat16)


def make_ag_inputs(cfg: AGConfig, seed: int = 0, g: torch.Generator | None = None):
    """Return (shards, B): R CPU bf16 tensors (H, K) ~ N(0,1) and B (N, K) ~ N(0, sigma)."""
    if g is None:
        g = torch.Generator("cpu").manual_seed(seed)
    shards = [_bf16_normal((cfg.H, cfg.K), 1.0, g) for _ in range(cfg.R)]
    B = _bf16_normal((cfg.N, cfg.K), cfg.b_sigma, g)
    return shards, B


def make_tg_inputs(cfg: TGConfig, seed: int = 0, g: torch.Generator | None = None):
    """Return a list of nranks CPU tensors of shape cfg.shape."""
    if g is None:
        g = torch.Generator("cpu").manual_seed(seed)
    out = []
    for _ in range(cfg.nranks):
        if cfg.dist == "uniform11":
            t = torch.rand(cfg.shape, generator=g, dtype=torch.float32).mul_(2).sub_(1).to(cfg.dtype)
        elif cfg.dist == "normal":
            t = torch.randn(cfg.shape, generator=g, dtype=torch.float32).to(cfg.dtype)
        elif cfg.dist == "int32full":
            t = torch.randint(-2**31, 2**31, cfg.shape, generator=g, dtype=torch.int64).to(torch.int32)
        else:
            raise ValueError(cfg.dist)
        out.append(t)
    return out


def make_release_schedule(cfg: AGConfig, rank: int = 0, seed: int = 0):
    """Release order and per-block delays for the skewed workload.

    The rank's own blocks come first in increasing order (they need no
    communication); the remote blocks follow in a seeded random permutation.
    delay_ns[c] ~ U[0, max_delay_ns] for remote blocks, 0 for local ones.
    Returns (order int32 [nblocks], delay_ns uint32-valued int64 [nblocks]).
    """
    g = torch.Generator("cpu").manual_seed(seed)
    S = cfg.H // cfg.cb
    local = list(range(rank * S, (rank + 1) * S))
    remote = [c for c in range(cfg.nblocks) if not (rank * S <= c < (rank + 1) * S)]
    perm = torch.randperm(len(remote), generator=g).tolist()
    order = local + [remote[i] for i in perm]
    delay = torch.randint(0, cfg.max_delay_ns + 1, (cfg.nblocks,), generator=g, dtype=torch.int64)
    for c in local:
        delay[c] = 0
    return torch.tensor(order, dtype=torch.int32), delay


def sample_rows(cfg: AGConfig, seed: int = 0, per_block_random: int = 2):
    """Rows on which large outputs are checked against the oracle one by one:
    the first and last row of every comm block plus ``per_block_random`` seeded
    random rows of each block (so every block, rank and N-tile is covered)."""
    g = torch.Generator("cpu").manual_seed(seed + 12345)
    rows = []
    for c in range(cfg.nblocks):
        r0 = c * cfg.cb
        rows += [r0, r0 + cfg.cb - 1]
        if per_block_random:
            rows += (r0 + torch.randint(0, cfg.cb, (per_block_random,), generator=g)).tolist()
    return sorted(set(rows))
