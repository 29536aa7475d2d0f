"""CPU oracle for the chunked AllGather x MatMul path (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares
no code with the CUDA library in ``tile_gather_comm_gb300``; the arithmetic
lives in ``oracle.c`` (plain C, built with ``-ffp-contract=off``), and this
module only builds it and marshals numpy arrays through ctypes.

Sources:
  [TG]  "CANN PTO-ISA TGATHER 指令深度解析：跨 Rank 行拼接 Gather 的实现原理与开发指南"
  [AGM] "Triton第四课：基于对称内存融合 AllGather 与 MatMul，提速1.56倍"

bf16 values travel as numpy ``uint16`` bit patterns.

Parity status: every function is pinned in tests/test_oracle_pins.py.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP, no FMA contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-std=c11", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _bind(lib):
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    lib.oracle_tgather.argtypes = [vp, ctypes.POINTER(vp), ctypes.c_int,
                                   i64, i64, i64, i64, i64, i64, i64]
    lib.oracle_tgather.restype = ctypes.c_int
    lib.oracle_tgather_strided.argtypes = [vp, vp, ctypes.POINTER(vp), vp, ctypes.c_int,
                                           i64, i64, i64, i64, i64, i64]
    lib.oracle_tgather_strided.restype = ctypes.c_int
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_f32_to_bf16_rne.argtypes = [ctypes.c_float]
    lib.oracle_f32_to_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16_array.argtypes = [vp, vp, i64]
    lib.oracle_f32_to_bf16_array.restype = None
    lib.oracle_f32_to_e4m3_array.argtypes = [vp, vp, i64]
    lib.oracle_f32_to_e4m3_array.restype = None
    lib.oracle_ag_matmul_rows_e4m3.argtypes = [ctypes.POINTER(vp), ctypes.c_int, vp, i64, i64, i64, vp, i64, vp]
    lib.oracle_ag_matmul_rows_e4m3.restype = ctypes.c_int
    lib.oracle_ag_matmul.argtypes = [ctypes.POINTER(vp), ctypes.c_int, vp, vp, vp, i64, i64, i64]
    lib.oracle_ag_matmul.restype = ctypes.c_int
    lib.oracle_ag_matmul_rows.argtypes = [ctypes.POINTER(vp), ctypes.c_int, vp, i64, i64, i64,
                                          vp, i64, vp]
    lib.oracle_ag_matmul_rows.restype = ctypes.c_int
    lib.oracle_ag_matmul_chunked.argtypes = [ctypes.POINTER(vp), ctypes.c_int, vp, vp, vp,
                                             i64, i64, i64, i64, vp, i64]
    lib.oracle_ag_matmul_chunked.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_num_threads.restype = None
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = _bind(ctypes.CDLL(_LIB))
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _ptr_array(arrs):
    return (ctypes.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])


class Oracle:
    """The oracle's functions bound to one compiled copy of oracle.c (the
    default build, or a deliberately broken copy that a test compiles to show
    that the pins catch a planted mistake)."""

    def __init__(self, lib):
        self._L = lib

    def num_threads(self) -> int:
        return self._L.oracle_num_threads()

    def set_num_threads(self, n: int) -> None:
        self._L.oracle_set_num_threads(int(n))

    def tgather(self, srcs, dst_rows3: int | None = None, dst: np.ndarray | None = None) -> np.ndarray:
        """[TG] §二: dst[d0,d1,d2, r*H+i, j] = srcs[r][d0,d1,d2,i,j].

        ``srcs`` are N numpy arrays of identical 5-D shape (D0,D1,D2,H,W) and dtype.
        ``dst_rows3`` (>= N*H) gives dst's DIM_3 ([TG] §7.2); rows past N*H are left
        as they are in ``dst`` (zeros when ``dst`` is not given).
        """
        lib = self._L
        srcs = [np.ascontiguousarray(s) for s in srcs]
        n = len(srcs)
        if n == 0:
            raise ValueError("nranks must be > 0")
        shape, dt = srcs[0].shape, srcs[0].dtype
        if len(shape) != 5 or any(s.shape != shape or s.dtype != dt for s in srcs):
            raise ValueError("all sources must share one 5-D shape and dtype")
        D0, D1, D2, H, W = shape
        rows = n * H if dst_rows3 is None else int(dst_rows3)
        if dst is None:
            dst = np.zeros((D0, D1, D2, rows, W), dtype=dt)
        assert dst.shape == (D0, D1, D2, rows, W) and dst.dtype == dt
        rc = lib.oracle_tgather(_ptr(dst), _ptr_array(srcs), n, D0, D1, D2, H, W,
                                dt.itemsize, rows)
        if rc != 0:
            raise ValueError(f"oracle_tgather rejected the arguments (rc={rc})")
        return dst

    def tgather_strided(self, dst: np.ndarray, srcs) -> np.ndarray:
        """[TG] §7.3 / §8.1 strided views: writes srcs (numpy views of one shape and strides)
        into the view ``dst`` of shape (D0,D1,D2,>=N*H,W), rows r*H+i; returns dst."""
        n = len(srcs)
        shape = srcs[0].shape
        es = srcs[0].dtype.itemsize
        if len(shape) != 5 or any(x.shape != shape or x.strides != srcs[0].strides for x in srcs):
            raise ValueError("sources must share one 5-D shape and one stride")
        D0, D1, D2, H, W = shape
        sst = np.array([st // es for st in srcs[0].strides], dtype=np.int64)
        dstr = np.array([st // es for st in dst.strides], dtype=np.int64)
        ptrs = (ctypes.c_void_p * n)(*[x.ctypes.data for x in srcs])
        rc = self._L.oracle_tgather_strided(dst.ctypes.data, dstr.ctypes.data, ptrs, sst.ctypes.data, n,
                                            D0, D1, D2, H, W, es)
        if rc != 0:
            raise ValueError(f"oracle_tgather_strided rejected the arguments (rc={rc})")
        return dst

    def bf16_to_f32(self, bits: np.ndarray) -> np.ndarray:
        """Widen bf16 bit patterns (uint16) to float32: the bits go to the upper half."""
        bits = np.asarray(bits, dtype=np.uint16)
        return (bits.astype(np.uint32) << 16).view(np.float32)

    def f32_to_bf16(self, x: np.ndarray) -> np.ndarray:
        """float32 -> bf16 bit patterns (uint16), round to nearest even."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty(x.shape, dtype=np.uint16)
        self._L.oracle_f32_to_bf16_array(_ptr(x), _ptr(y), x.size)
        return y

    def f32_to_e4m3(self, x: np.ndarray) -> np.ndarray:
        """float32 -> float8 e4m3 (fn) bit patterns (uint8), RNE, saturating at +-448."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        y = np.empty(x.shape, dtype=np.uint8)
        self._L.oracle_f32_to_e4m3_array(_ptr(x), _ptr(y), x.size)
        return y

    @staticmethod
    def e4m3_to_f64(bits):
        return e4m3_to_f64(bits)

    def ag_matmul_rows_e4m3(self, a_shards, B: np.ndarray, rows) -> np.ndarray:
        """Sampled rows of C written as float8 e4m3 bit patterns (uint8)."""
        shards = [np.ascontiguousarray(s, dtype=np.uint16) for s in a_shards]
        R = len(shards)
        Hs, K = shards[0].shape
        B = np.ascontiguousarray(B, dtype=np.uint16)
        N = B.shape[0]
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((rows.size, N), dtype=np.uint8)
        rc = self._L.oracle_ag_matmul_rows_e4m3(_ptr_array(shards), R, _ptr(B), R * Hs, K, N,
                                                _ptr(rows), rows.size, _ptr(out))
        if rc != 0:
            raise ValueError(f"oracle_ag_matmul_rows_e4m3 rejected the arguments (rc={rc})")
        return out

    def f32_to_bf16_scalar(self, x: float) -> int:
        return int(self._L.oracle_f32_to_bf16_rne(ctypes.c_float(x)))

    def ag_matmul(self, a_shards, B: np.ndarray):
        """[AGM]: a = TGATHER(a_shards) (M,K); C = bf16(a @ B^T) with fp32 accumulation.

        ``a_shards``: R uint16 arrays (M/R, K); ``B``: uint16 (N, K).  Returns (C, a).
        """
        lib = self._L
        shards = [np.ascontiguousarray(s, dtype=np.uint16) for s in a_shards]
        R = len(shards)
        Hs, K = shards[0].shape
        M = R * Hs
        B = np.ascontiguousarray(B, dtype=np.uint16)
        N = B.shape[0]
        assert B.shape == (N, K)
        C = np.zeros((M, N), dtype=np.uint16)
        a = np.zeros((M, K), dtype=np.uint16)
        rc = lib.oracle_ag_matmul(_ptr_array(shards), R, _ptr(B), _ptr(C), _ptr(a), M, K, N)
        if rc != 0:
            raise ValueError(f"oracle_ag_matmul rejected the arguments (rc={rc})")
        return C, a

    def ag_matmul_rows(self, a_shards, B: np.ndarray, rows) -> np.ndarray:
        """The rows ``rows`` of C only (each computed exactly as in ag_matmul)."""
        lib = self._L
        shards = [np.ascontiguousarray(s, dtype=np.uint16) for s in a_shards]
        R = len(shards)
        Hs, K = shards[0].shape
        M = R * Hs
        B = np.ascontiguousarray(B, dtype=np.uint16)
        N = B.shape[0]
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        out = np.zeros((rows.size, N), dtype=np.uint16)
        rc = lib.oracle_ag_matmul_rows(_ptr_array(shards), R, _ptr(B), M, K, N,
                                       _ptr(rows), rows.size, _ptr(out))
        if rc != 0:
            raise ValueError(f"oracle_ag_matmul_rows rejected the arguments (rc={rc})")
        return out

    def ag_matmul_chunked(self, a_shards, B: np.ndarray, cb: int, order):
        """Block-by-block producer/consumer walk in release order ``order``; returns (C, a)."""
        lib = self._L
        shards = [np.ascontiguousarray(s, dtype=np.uint16) for s in a_shards]
        R = len(shards)
        Hs, K = shards[0].shape
        M = R * Hs
        B = np.ascontiguousarray(B, dtype=np.uint16)
        N = B.shape[0]
        order = np.ascontiguousarray(order, dtype=np.int64)
        C = np.zeros((M, N), dtype=np.uint16)
        a = np.zeros((M, K), dtype=np.uint16)
        rc = lib.oracle_ag_matmul_chunked(_ptr_array(shards), R, _ptr(B), _ptr(C), _ptr(a),
                                          M, K, N, int(cb), _ptr(order), order.size)
        if rc != 0:
            raise ValueError(f"oracle_ag_matmul_chunked rejected the arguments (rc={rc})")
        return C, a


def load_from(path: str) -> Oracle:
    """An Oracle over another compiled copy of oracle.c (used by the mutation tests)."""
    return Oracle(_bind(ctypes.CDLL(path)))


_default = None


def _oracle() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(_load())
    return _default


def num_threads() -> int:
    return _oracle().num_threads()


def set_num_threads(n: int) -> None:
    _oracle().set_num_threads(n)


def tgather(srcs, dst_rows3=None, dst=None):
    return _oracle().tgather(srcs, dst_rows3=dst_rows3, dst=dst)


def tgather_strided(dst, srcs):
    return _oracle().tgather_strided(dst, srcs)


def bf16_to_f32(bits):
    return _oracle().bf16_to_f32(bits)


def f32_to_bf16(x):
    return _oracle().f32_to_bf16(x)


def f32_to_bf16_scalar(x):
    return _oracle().f32_to_bf16_scalar(x)


def f32_to_e4m3(x):
    return _oracle().f32_to_e4m3(x)


def ag_matmul_rows_e4m3(a_shards, B, rows):
    return _oracle().ag_matmul_rows_e4m3(a_shards, B, rows)


def e4m3_to_f64(bits):
    """Decode float8 e4m3 (fn) bit patterns to float64 (exact; NaN for S.1111.111)."""
    b = np.asarray(bits, dtype=np.uint8).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = b & 0x7
    val = np.where(e == 0, m / 8.0 * 2.0**-6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((e == 0xF) & (m == 0x7), np.nan, val)
    return sign * val


def ag_matmul(a_shards, B):
    return _oracle().ag_matmul(a_shards, B)


def ag_matmul_rows(a_shards, B, rows):
    return _oracle().ag_matmul_rows(a_shards, B, rows)


def ag_matmul_chunked(a_shards, B, cb, order):
    return _oracle().ag_matmul_chunked(a_shards, B, cb, order)
