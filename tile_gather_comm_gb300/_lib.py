"""ctypes binding of libtgc.so: argument marshalling only.

Every function here has the name of the C entry point it calls (include/tgc.h)
and does nothing but turn torch tensors / Python values into pointers and
integers; every step of the computation runs in the library's CUDA kernels.
Loading fails loudly if libtgc.so has not been built: there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libtgc.so")

TGC_OK = 0
TGC_ERR_INVALID_ARG = -1
TGC_ERR_DTYPE = -2
TGC_ERR_ALIGN = -3
TGC_ERR_CUDA = -5
TGC_ERR_TIMEOUT = -6
TGC_ERR_ABORTED = -7
TGC_ERR_WORKSPACE = -8
TGC_ERR_TOO_LARGE = -9
NOALLOC_MAX_BLOCKS = 2048      # TGC_NOALLOC_MAX_BLOCKS
NOALLOC_SCRATCH_BYTES = 65536  # TGC_NOALLOC_SCRATCH_BYTES

MODES = {"fused": 0, "unfused": 1, "mm_only": 2, "fused_ce": 3}
PIVOTS = {"page": 0, "shard": 1, "none": 2, "ready_queue": 3, "auto": 4}
OUT_FORMATS = {"bf16": 0, "f8e4m3": 1}
DTYPES = {
    torch.uint8: 0, torch.int8: 1, torch.float16: 2, torch.bfloat16: 3,
    torch.int32: 4, torch.float32: 5, torch.int64: 6, torch.float64: 7,
}
MAX_RANKS = 64
TRACE_WORDS = 16
TRACE = dict(start=0, wait_ns=1, waited_tiles=2, copy_first=3, copy_last=4, pieces=5, end=6, tiles=7,
             mma_stage_ns=8, mma_acc_ns=9, epi_wait_ns=10, load_stall_ns=11, piece_bytes=12,
             copy_warps=13)

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


class TgatherArgs(ctypes.Structure):
    _fields_ = [
        ("dst", _vp), ("srcs", ctypes.POINTER(_vp)), ("nranks", ctypes.c_int),
        ("D0", _i64), ("D1", _i64), ("D2", _i64), ("H", _i64), ("W", _i64),
        ("dtype", ctypes.c_int), ("dst_rows3", _i64),
        ("progress", _vp), ("counters", _vp), ("chunk_rows", _i64),
        ("epoch", ctypes.c_uint32), ("stream", _vp), ("spin_timeout_ns", ctypes.c_uint64),
    ]


class AgMatmulArgs(ctypes.Structure):
    _fields_ = [
        ("a_shards", ctypes.POINTER(_vp)), ("nranks", ctypes.c_int),
        ("B", _vp), ("C", _vp), ("a_out", _vp),
        ("M", _i64), ("K", _i64), ("N", _i64), ("comm_block_rows", _i64),
        ("rank", ctypes.c_int), ("mode", ctypes.c_int), ("pivot", ctypes.c_int),
        ("progress", _vp), ("epoch", ctypes.c_uint32),
        ("order", ctypes.POINTER(ctypes.c_int32)), ("n_order", _i64),
        ("delay_ns", ctypes.POINTER(ctypes.c_uint32)),
        ("spin_timeout_ns", ctypes.c_uint64), ("group_m", ctypes.c_int), ("grid", ctypes.c_int),
        ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("d_status", _vp),
        ("sync", ctypes.c_int), ("stream", _vp), ("trace", _vp), ("out_format", ctypes.c_int),
        ("trace_words", ctypes.c_size_t), ("band_n", ctypes.c_int), ("tile_n", ctypes.c_int),
    ]


class IpcHandle(ctypes.Structure):
    """tgc_ipc_handle: the CUDA IPC handle of an allocation and a buffer's offset inside it."""
    _fields_ = [("bytes", ctypes.c_ubyte * 64), ("offset", ctypes.c_uint64)]


class AgMatmulPlan(ctypes.Structure):
    _fields_ = [("pivot", ctypes.c_int), ("band_n", ctypes.c_int), ("group_m", ctypes.c_int),
                ("tile_n", ctypes.c_int)]


class TGCError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {tgc_status_string(status)} ({status})"
                         + (f", cuda error {tgc_last_cuda_error()}" if status == TGC_ERR_CUDA else ""))


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libtgc.so (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
    _lib = load_library(LIB_PATH)
    return _lib


def load_library(path: str) -> ctypes.CDLL:
    """Open a build of the library (the in-tree one, or one made by _build.build_variant)
    and declare the C prototypes of its entry points."""
    L = ctypes.CDLL(path)
    L.tgc_tgather.argtypes = [_vp, ctypes.POINTER(_vp), ctypes.c_int, _i64, _i64, _i64, _i64, _i64,
                              ctypes.c_int, _vp]
    L.tgc_tgather.restype = ctypes.c_int
    L.tgc_tgather_strided.argtypes = [_vp, ctypes.POINTER(_i64), ctypes.POINTER(_vp), ctypes.POINTER(_i64),
                                      ctypes.c_int, _i64, _i64, _i64, _i64, _i64, ctypes.c_int, _vp]
    L.tgc_tgather_strided.restype = ctypes.c_int
    L.tgc_tgather_ex.argtypes = [ctypes.POINTER(TgatherArgs)]
    L.tgc_tgather_ex.restype = ctypes.c_int
    L.tgc_ag_matmul.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, _vp, _vp, _i64, _i64, _i64, _i64, _vp]
    L.tgc_ag_matmul.restype = ctypes.c_int
    L.tgc_ag_matmul_ex.argtypes = [ctypes.POINTER(AgMatmulArgs)]
    L.tgc_ag_matmul_ex.restype = ctypes.c_int
    L.tgc_ag_matmul_plan.argtypes = [ctypes.POINTER(AgMatmulArgs), ctypes.POINTER(AgMatmulPlan)]
    L.tgc_ag_matmul_plan.restype = ctypes.c_int
    L.tgc_ag_matmul_noalloc.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, _vp, _vp, _vp, _i64, _i64, _i64,
                                         _i64, _vp]
    L.tgc_ag_matmul_noalloc.restype = ctypes.c_int
    L.tgc_ipc_export.argtypes = [_vp, ctypes.POINTER(IpcHandle)]
    L.tgc_ipc_export.restype = ctypes.c_int
    L.tgc_ipc_open.argtypes = [ctypes.POINTER(IpcHandle), ctypes.POINTER(_vp)]
    L.tgc_ipc_open.restype = ctypes.c_int
    L.tgc_ipc_close.argtypes = [_vp, ctypes.POINTER(IpcHandle)]
    L.tgc_ipc_close.restype = ctypes.c_int
    L.tgc_ag_matmul_workspace_bytes.argtypes = [ctypes.c_int, _i64, _i64, _i64, _i64]
    L.tgc_ag_matmul_workspace_bytes.restype = ctypes.c_size_t
    L.tgc_ag_matmul_schedule.argtypes = [_i64, _i64, _i64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.POINTER(_i64), _i64, ctypes.c_int]
    L.tgc_ag_matmul_schedule.restype = _i64
    L.tgc_gemm_tile_shape.argtypes = [ctypes.POINTER(ctypes.c_int)] * 3
    L.tgc_gemm_tile_shape.restype = None
    L.tgc_status_string.argtypes = [ctypes.c_int]
    L.tgc_status_string.restype = ctypes.c_char_p
    L.tgc_last_cuda_error.argtypes = []
    L.tgc_last_cuda_error.restype = ctypes.c_int
    L.tgc_version.argtypes = []
    L.tgc_version.restype = ctypes.c_char_p
    return L


# ----------------------------------------------------------------------------- helpers


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _ptrs(ts):
    return (_vp * len(ts))(*[_ptr(t) for t in ts])


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(rc: int, where: str) -> int:
    if rc != TGC_OK:
        raise TGCError(rc, where)
    return rc


# ----------------------------------------------------------------------------- API


def tgc_status_string(status: int) -> str:
    return lib().tgc_status_string(int(status)).decode()


def tgc_last_cuda_error() -> int:
    return lib().tgc_last_cuda_error()


def tgc_version() -> str:
    return lib().tgc_version().decode()


def tgc_gemm_tile_shape():
    v = [ctypes.c_int(0) for _ in range(3)]
    lib().tgc_gemm_tile_shape(*[ctypes.byref(x) for x in v])
    return tuple(x.value for x in v)


def tgc_tgather(dst, srcs, stream=None, check: bool = True) -> int:
    """dst[d0,d1,d2, r*H+i, j] = srcs[r][d0,d1,d2,i,j]; srcs are 5-D tensors of one shape."""
    D0, D1, D2, H, W = srcs[0].shape
    rc = lib().tgc_tgather(_ptr(dst), _ptrs(srcs), len(srcs), D0, D1, D2, H, W,
                           DTYPES[srcs[0].dtype], _stream(stream))
    return _check(rc, "tgc_tgather") if check else rc


def tgc_tgather_strided(dst, srcs, stream=None, check: bool = True) -> int:
    """TGATHER on strided 5-D views: srcs share one shape and one stride; dst is a
    (D0,D1,D2,>=N*H,W) view of any strides (rows r*H+i are written)."""
    D0, D1, D2, H, W = srcs[0].shape
    st = srcs[0].stride()
    if any(tuple(x.shape) != tuple(srcs[0].shape) or x.stride() != st for x in srcs):
        raise ValueError("all sources must share one shape and one stride")
    ss = (_i64 * 5)(*st)
    ds = (_i64 * 5)(*dst.stride())
    rc = lib().tgc_tgather_strided(_ptr(dst), ds, _ptrs(srcs), ss, len(srcs), D0, D1, D2, H, W,
                                   DTYPES[srcs[0].dtype], _stream(stream))
    return _check(rc, "tgc_tgather_strided") if check else rc


def tgc_tgather_ex(dst, srcs, dst_rows3: int = 0, progress=None, counters=None, chunk_rows: int = 0,
                   epoch: int = 0, stream=None, spin_timeout_ns: int = 0, check: bool = True) -> int:
    """TGATHER with the extended arguments of tgc_tgather_args: a taller destination
    (``dst_rows3``) and per-chunk progress release (``progress``, ``counters``, ``chunk_rows``,
    ``epoch``, ``spin_timeout_ns``), as include/tgc.h describes them.  Asynchronous on ``stream``."""
    D0, D1, D2, H, W = srcs[0].shape
    arr = _ptrs(srcs)
    a = TgatherArgs(dst=_ptr(dst), srcs=arr, nranks=len(srcs), D0=D0, D1=D1, D2=D2, H=H, W=W,
                    dtype=DTYPES[srcs[0].dtype], dst_rows3=dst_rows3, progress=_ptr(progress),
                    counters=_ptr(counters), chunk_rows=chunk_rows, epoch=epoch, stream=_stream(stream),
                    spin_timeout_ns=spin_timeout_ns)
    rc = lib().tgc_tgather_ex(ctypes.byref(a))
    return _check(rc, "tgc_tgather_ex") if check else rc


def tgc_ag_matmul(a_shards, B, C, comm_block_rows: int, stream=None, check: bool = True) -> int:
    """C = gather(a_shards) @ B^T (bf16); synchronizes the stream."""
    R = len(a_shards)
    H, K = a_shards[0].shape
    N = B.shape[0]
    rc = lib().tgc_ag_matmul(_ptrs(a_shards), R, _ptr(B), _ptr(C), R * H, K, N, comm_block_rows,
                             _stream(stream))
    return _check(rc, "tgc_ag_matmul") if check else rc


def tgc_ag_matmul_noalloc(a_shards, B, C, a_out, comm_block_rows: int, stream=None, check: bool = True) -> int:
    """Fused AllGather-MatMul without any device allocation (for callers that cannot allocate):
    the kernel's scratch is a fixed array inside the library; ``a_out`` receives the gathered A.
    Synchronizes the stream."""
    R = len(a_shards)
    H, K = a_shards[0].shape
    N = B.shape[0]
    rc = lib().tgc_ag_matmul_noalloc(_ptrs(a_shards), R, _ptr(B), _ptr(C), _ptr(a_out), R * H, K, N,
                                     comm_block_rows, _stream(stream))
    return _check(rc, "tgc_ag_matmul_noalloc") if check else rc


def tgc_ipc_export(buf) -> bytes:
    """The tgc_ipc_handle of a device buffer (tensor or address), as bytes to send to the other ranks."""
    h = IpcHandle()
    _check(lib().tgc_ipc_export(_ptr(buf), ctypes.byref(h)), "tgc_ipc_export")
    return bytes(h)


def tgc_ipc_open(handle: bytes) -> int:
    """Address, in this process, of a buffer another process exported."""
    h = IpcHandle.from_buffer_copy(handle)
    p = _vp()
    _check(lib().tgc_ipc_open(ctypes.byref(h), ctypes.byref(p)), "tgc_ipc_open")
    return int(p.value)


def tgc_ipc_close(ptr: int, handle: bytes) -> None:
    h = IpcHandle.from_buffer_copy(handle)
    _check(lib().tgc_ipc_close(ptr, ctypes.byref(h)), "tgc_ipc_close")


def tgc_ag_matmul_workspace_bytes(nranks: int, M: int, K: int, N: int, comm_block_rows: int) -> int:
    return lib().tgc_ag_matmul_workspace_bytes(nranks, M, K, N, comm_block_rows)


def _ag_args(a_shards, B, C, a_out, comm_block_rows: int, *, M: int | None = None, rank: int = 0,
             mode: str = "fused", pivot: str = "page", progress=None, epoch: int = 1, order=None,
             delay_ns=None, spin_timeout_ns: int = 0, group_m: int = 0, band_n: int = 0, grid: int = 0,
             workspace=None, d_status=None, sync: bool = False, stream=None, trace=None,
             out_format: str = "bf16", tile_n: int = 0) -> AgMatmulArgs:
    R = len(a_shards) if a_shards is not None else 1
    K = B.shape[1]
    N = B.shape[0]
    if M is None:
        M = R * a_shards[0].shape[0]
    shards = _ptrs(a_shards) if a_shards is not None else None
    order_arr = None
    n_order = 0
    if order is not None:
        order = [int(x) for x in order]
        order_arr = (ctypes.c_int32 * max(1, len(order)))(*order)
        n_order = len(order)
    delay_arr = None
    if delay_ns is not None:
        delay_arr = (ctypes.c_uint32 * len(delay_ns))(*[int(x) for x in delay_ns])
    a = AgMatmulArgs(
        a_shards=shards, nranks=R, B=_ptr(B), C=_ptr(C), a_out=_ptr(a_out), M=M, K=K, N=N,
        comm_block_rows=comm_block_rows, rank=rank, mode=MODES[mode], pivot=PIVOTS[pivot],
        progress=_ptr(progress), epoch=epoch, order=order_arr, n_order=n_order, delay_ns=delay_arr,
        spin_timeout_ns=spin_timeout_ns, group_m=group_m, band_n=band_n, grid=grid, workspace=_ptr(workspace),
        workspace_bytes=(workspace.numel() * workspace.element_size()) if workspace is not None else 0,
        d_status=_ptr(d_status), sync=1 if sync else 0, stream=_stream(stream), trace=_ptr(trace),
        out_format=OUT_FORMATS[out_format],
        trace_words=(trace.numel() * trace.element_size() // 8) if trace is not None else 0, tile_n=tile_n)
    a._keep = (shards, order_arr, delay_arr)  # the host arrays live as long as the struct
    return a


def tgc_ag_matmul_ex(a_shards, B, C, a_out, comm_block_rows: int, *, check: bool = True, **kw) -> int:
    """Extended AllGather-MatMul (see tgc.h).  ``order`` / ``delay_ns`` are host sequences."""
    a = _ag_args(a_shards, B, C, a_out, comm_block_rows, **kw)
    rc = lib().tgc_ag_matmul_ex(ctypes.byref(a))
    return _check(rc, "tgc_ag_matmul_ex") if check else rc


def tgc_ag_matmul_plan(a_shards, B, C, a_out, comm_block_rows: int, **kw) -> dict:
    """The tile order, raster and tile width tgc_ag_matmul_ex would run with these arguments."""
    a = _ag_args(a_shards, B, C, a_out, comm_block_rows, **kw)
    out = AgMatmulPlan()
    _check(lib().tgc_ag_matmul_plan(ctypes.byref(a), ctypes.byref(out)), "tgc_ag_matmul_plan")
    names = {v: k for k, v in PIVOTS.items()}
    return {"pivot": names.get(out.pivot, out.pivot), "band_n": out.band_n, "group_m": out.group_m,
            "tile_n": out.tile_n}


def tgc_ag_matmul_schedule(M: int, N: int, comm_block_rows: int, nranks: int, rank: int = 0,
                           pivot: str = "page", group_m: int = 0, grid: int = 1, cta: int = 0, band_n: int = 0,
                           tile_n: int = 256):
    """Tile sequence (pid_m, pid_n) of persistent CTA ``cta`` (host-side copy of the device schedule);
    ``band_n`` > 0 selects the band raster; tiles are ``tile_n`` columns wide."""
    n = lib().tgc_ag_matmul_schedule(M, N, comm_block_rows, nranks, rank, PIVOTS[pivot], group_m, band_n,
                                     grid, cta, None, 0, tile_n)
    _check(int(n) if n < 0 else 0, "tgc_ag_matmul_schedule")
    buf = (_i64 * max(1, 2 * n))()
    lib().tgc_ag_matmul_schedule(M, N, comm_block_rows, nranks, rank, PIVOTS[pivot], group_m, band_n, grid,
                                 cta, buf, n, tile_n)
    return [(buf[2 * i], buf[2 * i + 1]) for i in range(n)]
