"""GB300-native chunked AllGather x MatMul: TGATHER gather + flag-driven tcgen05 GEMM.

The compute lives in libtgc.so (hand-written sm_103a kernels behind a C ABI,
include/tgc.h); this package only builds it (``_build``), binds it with ctypes
(``_lib``), holds the seeded synthetic workloads (``workloads``) and the host
plumbing of ranks that are separate processes (``ranks``).
"""
from ._lib import (  # noqa: F401
    TGCError, lib, tgc_ag_matmul, tgc_ag_matmul_ex, tgc_ag_matmul_noalloc, tgc_ag_matmul_plan,
    tgc_ag_matmul_schedule,
    tgc_ag_matmul_workspace_bytes, tgc_gemm_tile_shape, tgc_ipc_close, tgc_ipc_export, tgc_ipc_open,
    tgc_last_cuda_error, tgc_status_string, tgc_tgather, tgc_tgather_ex, tgc_tgather_strided, tgc_version,
)
