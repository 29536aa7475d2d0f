"""C-ABI boundary tests that need no GPU: the library loads, exports every
symbol include/tgc.h declares, rejects invalid arguments synchronously (before
any CUDA call), returns early on empty work, and its host-side copy of the
tile schedule has the properties the pages require of the pivot."""
import ctypes
import os
import re

import pytest

import tile_gather_comm_gb300 as tgc
from tile_gather_comm_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tgc.h")
FAKE = 1 << 20  # a 1 MiB-aligned fake device address: never dereferenced on these paths


@pytest.fixture(scope="module", autouse=True)
def built():
    from tile_gather_comm_gb300 import _build
    _build.build()


def _declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tgc_\w+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 10
    L = _lib.lib()
    for n in names:
        assert hasattr(L, n), n
        assert ctypes.cast(getattr(L, n), ctypes.c_void_p).value


@pytest.mark.parametrize("cls,cname", [(_lib.TgatherArgs, "tgc_tgather_args"),
                                       (_lib.AgMatmulArgs, "tgc_ag_matmul_args"),
                                       (_lib.AgMatmulPlan, "tgc_ag_matmul_plan_t"),
                                       (_lib.IpcHandle, "tgc_ipc_handle")])
def test_ctypes_structs_match_the_header(cls, cname, tmp_path):
    """The binding's argument structs have the header's size and every field at the header's
    offset (a C program compiled against include/tgc.h prints them)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    cuda_inc = "/usr/local/cuda/include"
    if gcc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("gcc or the CUDA headers are not available")
    names = [f[0] for f in cls._fields_]
    lines = [f'printf("%zu\\n", sizeof({cname}));']
    lines += [f'printf("%zu\\n", offsetof({cname}, {n}));' for n in names]
    src = tmp_path / "layout.c"
    src.write_text("#include <stdio.h>\n#include <stddef.h>\n#include \"tgc.h\"\nint main(void) {\n"
                   + "\n".join(lines) + "\nreturn 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-std=c11", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)],
                   check=True)
    out = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()]
    assert out[0] == ctypes.sizeof(cls), cname
    assert out[1:] == [getattr(cls, n).offset for n in names], cname


@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_compiles_cleanly_as_c_and_cpp(lang, tmp_path):
    """include/tgc.h is a C header usable from C11 and C++17 with strict warnings as errors."""
    import shutil
    import subprocess
    cc = shutil.which("gcc" if lang == "c" else "g++")
    cuda_inc = "/usr/local/cuda/include"
    if cc is None or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("compiler or CUDA headers not available")
    src = tmp_path / ("h.c" if lang == "c" else "h.cpp")
    init = "= {0}" if lang == "c" else "{}"   # zero-initialised, as the header asks
    src.write_text('#include "tgc.h"\nint main(void) { tgc_tgather_args a ' + init + '; tgc_ag_matmul_args b '
                   + init + '; (void)a; (void)b; return TGC_OK; }\n')
    std = "-std=c11" if lang == "c" else "-std=c++17"
    subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-isystem", cuda_inc, "-c", str(src), "-o", str(tmp_path / "h.o")], check=True)


def test_status_strings_and_version():
    assert tgc.tgc_status_string(0) == "ok"
    assert "wait" in tgc.tgc_status_string(_lib.TGC_ERR_TIMEOUT)
    assert tgc.tgc_status_string(12345) == "unknown status"
    assert tgc.tgc_version().count(".") == 2
    assert tgc.tgc_gemm_tile_shape() == (256, 256, 64)  # a CTA pair: 256 rows, 256-column MMA blocks


def _tg(dst, srcs, n, D0, D1, D2, H, W, dt=5):
    arr = (ctypes.c_void_p * max(1, n))(*srcs)
    return _lib.lib().tgc_tgather(dst, arr, n, D0, D1, D2, H, W, dt, None)


def test_tgather_invalid_arguments():
    E = _lib
    assert _tg(FAKE, [FAKE], 0, 1, 1, 1, 1, 1) == E.TGC_ERR_INVALID_ARG
    assert _tg(FAKE, [FAKE] * 65, 65, 1, 1, 1, 1, 1) == E.TGC_ERR_INVALID_ARG
    assert _tg(FAKE, [FAKE], 1, -1, 1, 1, 1, 1) == E.TGC_ERR_INVALID_ARG
    assert _tg(FAKE, [FAKE], 1, 1, 1, 1, 1, -4) == E.TGC_ERR_INVALID_ARG
    assert _tg(FAKE, [FAKE], 1, 1, 1, 1, 1, 1, dt=99) == E.TGC_ERR_DTYPE
    assert _tg(None, [FAKE], 1, 1, 1, 1, 4, 4) == E.TGC_ERR_INVALID_ARG
    assert _tg(FAKE, [None], 1, 1, 1, 1, 4, 4) == E.TGC_ERR_INVALID_ARG
    assert _tg(FAKE + 2, [FAKE], 1, 1, 1, 1, 4, 4, dt=5) == E.TGC_ERR_ALIGN   # f32 needs 4-byte alignment
    assert _tg(FAKE, [FAKE, FAKE + 6], 2, 1, 1, 1, 4, 4, dt=6) == E.TGC_ERR_ALIGN
    # sizes whose byte counts would overflow 64-bit offsets are refused before any launch
    big = 1 << 31
    assert _tg(FAKE, [FAKE], 1, big, big, 4, 4, 4) == E.TGC_ERR_INVALID_ARG
    assert _tg(FAKE, [FAKE], 1, 1, 1, 1, 1 << 40, 1 << 30) == E.TGC_ERR_INVALID_ARG
    assert _tg(FAKE, [FAKE] * 2, 2, 1, 1, 1, 1 << 60, 1) == E.TGC_ERR_INVALID_ARG


@pytest.mark.parametrize("shape", [(0, 1, 1, 4, 4), (1, 0, 1, 4, 4), (1, 1, 0, 4, 4), (1, 1, 1, 0, 4), (1, 1, 1, 4, 0)])
def test_tgather_empty_returns_ok_without_touching_memory(shape):
    # null pointers prove that nothing is dereferenced or launched
    assert _tg(None, [None, None], 2, *shape) == _lib.TGC_OK


def test_tgather_strided_invalid_and_empty():
    L = _lib.lib()
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    good = (ctypes.c_int64 * 5)(1, 1, 1, 4, 1)
    neg = (ctypes.c_int64 * 5)(1, 1, 1, 4, -1)
    args = lambda ds, ss, H=4: (FAKE, ds, arr, ss, 2, 1, 1, 1, H, 4, 5, None)
    assert L.tgc_tgather_strided(*args(good, neg)) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_tgather_strided(*args(neg, good)) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_tgather_strided(*args(None, good)) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_tgather_strided(FAKE + 2, good, arr, good, 2, 1, 1, 1, 4, 4, 5, None) == _lib.TGC_ERR_ALIGN
    # empty: returns before looking at any pointer
    assert L.tgc_tgather_strided(None, None, arr, None, 2, 1, 1, 1, 0, 4, 5, None) == _lib.TGC_OK
    # a view whose last element lies beyond 64-bit byte offsets is refused
    huge = (ctypes.c_int64 * 5)(1, 1, 1, 1 << 40, 1)
    assert L.tgc_tgather_strided(FAKE, good, arr, huge, 2, 1, 1, 1, 1 << 24, 4, 5, None) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_tgather_strided(FAKE, huge, arr, good, 2, 1, 1, 1, 1 << 24, 4, 5, None) == _lib.TGC_ERR_INVALID_ARG


def test_tgather_ex_rejects_short_dst_and_missing_counters():
    L = _lib.lib()
    arr = (ctypes.c_void_p * 2)(FAKE, FAKE)
    a = _lib.TgatherArgs(dst=FAKE, srcs=arr, nranks=2, D0=1, D1=1, D2=1, H=4, W=4, dtype=5, dst_rows3=7)
    assert L.tgc_tgather_ex(ctypes.byref(a)) == _lib.TGC_ERR_INVALID_ARG
    a = _lib.TgatherArgs(dst=FAKE, srcs=arr, nranks=2, D0=1, D1=1, D2=1, H=4, W=4, dtype=5,
                         progress=FAKE, counters=None, chunk_rows=2)
    assert L.tgc_tgather_ex(ctypes.byref(a)) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_tgather_ex(None) == _lib.TGC_ERR_INVALID_ARG


def _ag(**kw):
    R = kw.pop("R", 4)
    args = dict(a_shards=(ctypes.c_void_p * R)(*([FAKE] * R)), nranks=R, B=FAKE, C=FAKE, a_out=FAKE,
                M=64, K=64, N=64, comm_block_rows=8, rank=0, mode=0, pivot=0, progress=FAKE, epoch=1,
                workspace=FAKE, workspace_bytes=1 << 20, sync=0)
    args.update(kw)
    return _lib.lib().tgc_ag_matmul_ex(ctypes.byref(_lib.AgMatmulArgs(**args)))


def test_ag_matmul_invalid_arguments():
    E = _lib
    assert _ag(nranks=0) == E.TGC_ERR_INVALID_ARG
    assert _ag(M=66) == E.TGC_ERR_INVALID_ARG            # M % R != 0
    assert _ag(comm_block_rows=5) == E.TGC_ERR_INVALID_ARG  # cb does not divide M/R
    assert _ag(comm_block_rows=0) == E.TGC_ERR_INVALID_ARG
    assert _ag(rank=4) == E.TGC_ERR_INVALID_ARG
    assert _ag(rank=-1) == E.TGC_ERR_INVALID_ARG
    assert _ag(mode=7) == E.TGC_ERR_INVALID_ARG
    assert _ag(pivot=9) == E.TGC_ERR_INVALID_ARG
    assert _ag(K=60) == E.TGC_ERR_ALIGN                   # 16-byte rows for TMA
    assert _ag(N=60) == E.TGC_ERR_ALIGN
    assert _ag(K=0) == E.TGC_ERR_INVALID_ARG
    assert _ag(B=FAKE + 8) == E.TGC_ERR_ALIGN
    assert _ag(C=None) == E.TGC_ERR_INVALID_ARG
    assert _ag(progress=None) == E.TGC_ERR_INVALID_ARG
    assert _ag(workspace=None) == E.TGC_ERR_WORKSPACE
    assert _ag(workspace_bytes=16) == E.TGC_ERR_WORKSPACE
    R = 4
    bad = (ctypes.c_void_p * R)(FAKE, FAKE, FAKE + 4, FAKE)
    assert _ag(a_shards=bad) == E.TGC_ERR_ALIGN
    dup = (ctypes.c_int32 * 3)(0, 1, 1)
    assert _ag(order=dup, n_order=3) == E.TGC_ERR_INVALID_ARG
    oob = (ctypes.c_int32 * 2)(0, 8)
    assert _ag(order=oob, n_order=2) == E.TGC_ERR_INVALID_ARG
    assert _lib.lib().tgc_ag_matmul_ex(None) == E.TGC_ERR_INVALID_ARG
    assert _ag(out_format=1, N=72) == E.TGC_ERR_ALIGN       # fp8 C needs N % 16 == 0
    assert _ag(out_format=5) == E.TGC_ERR_INVALID_ARG
    # a trace must hold at least one CTA pair's records (the SM-count bound is checked on a GPU)
    assert _ag(trace=FAKE, trace_words=0) == E.TGC_ERR_INVALID_ARG
    assert _ag(trace=FAKE, trace_words=2 * E.TRACE_WORDS - 1) == E.TGC_ERR_INVALID_ARG
    assert _ag(trace=FAKE + 4, trace_words=1 << 16) == E.TGC_ERR_ALIGN


def test_status_codes_match_header_and_unused_code_is_unknown():
    """Every status the header declares has its own string; -4 (once "not resident") is unused:
    the persistent grids are sized from the device's reported occupancy, so no path returns it."""
    hdr = open(HEADER, encoding="utf-8").read()
    codes = {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(TGC_(?:OK|ERR_\w+))\s*=\s*(-?\d+)", hdr)}
    assert "TGC_ERR_NOT_RESIDENT" not in codes and -4 not in codes.values()
    for name, code in codes.items():
        assert getattr(_lib, name) == code, name
        assert tgc.tgc_status_string(code) != "unknown status", name
    assert tgc.tgc_status_string(-4) == "unknown status"


def _plan(**kw):
    R = kw.pop("R", 4)
    args = dict(a_shards=(ctypes.c_void_p * R)(*([FAKE] * R)), nranks=R, B=FAKE, C=FAKE, a_out=FAKE,
                M=64, K=64, N=64, comm_block_rows=8, rank=0, mode=0, pivot=4, progress=FAKE, epoch=1,
                workspace=FAKE, workspace_bytes=1 << 30, sync=0)
    args.update(kw)
    out = _lib.AgMatmulPlan()
    rc = _lib.lib().tgc_ag_matmul_plan(ctypes.byref(_lib.AgMatmulArgs(**args)), ctypes.byref(out))
    return rc, (out.pivot, out.band_n, out.group_m), out.tile_n


def test_auto_order_and_raster_follow_the_measured_rule():
    """AUTO and band_n = 0, resolved without a GPU: bands of 16 tile columns for the fused modes when
    a shard holds fewer 256-row tile rows than a group (8), the group raster otherwise; the ready
    order only with an explicit release order on the band raster, the page pivot otherwise."""
    P = _lib.PIVOTS
    order = (ctypes.c_int32 * 2)(1, 0)
    square = dict(R=8, M=4096, K=4096, N=4096, comm_block_rows=128)
    mlp_up = dict(R=8, M=8192, K=4096, N=14336, comm_block_rows=256)
    large = dict(R=4, M=32768, K=8192, N=8192, comm_block_rows=512)
    assert _plan(**square)[:2] == (0, (P["page"], 16, 8))
    assert _plan(**mlp_up)[:2] == (0, (P["page"], 16, 8))
    assert _plan(**large)[:2] == (0, (P["page"], 0, 8))
    assert _plan(**square, order=order, n_order=2)[:2] == (0, (P["ready_queue"], 16, 8))
    assert _plan(**large, order=order, n_order=2)[:2] == (0, (P["page"], 0, 8))   # group raster: page
    assert _plan(**square, group_m=2)[:2] == (0, (P["page"], 0, 2))               # 2 tile rows, not < 2
    assert _plan(**square, band_n=-1)[:2] == (0, (P["page"], 0, 8))
    assert _plan(**large, band_n=5)[:2] == (0, (P["page"], 5, 8))
    assert _plan(**square, mode=_lib.MODES["fused_ce"], order=order, n_order=2)[:2] == (0, (P["page"], 16, 8))
    for mode in ("unfused", "mm_only"):
        assert _plan(**square, mode=_lib.MODES[mode])[:2] == (0, (P["none"], 0, 8))
        assert _plan(**square, mode=_lib.MODES[mode], pivot=P["ready_queue"])[:2] == (0, (P["none"], 0, 8))
    assert _plan(**square, pivot=P["shard"])[:2] == (0, (P["shard"], 16, 8))
    # the same argument checks as the call itself
    assert _plan(**dict(square, M=4097))[0] == _lib.TGC_ERR_INVALID_ARG
    assert _plan(**dict(square, tile_n=384))[0] == _lib.TGC_ERR_INVALID_ARG
    assert _plan(**dict(square, tile_n=-256))[0] == _lib.TGC_ERR_INVALID_ARG
    assert _plan(**dict(square, K=60))[0] == _lib.TGC_ERR_ALIGN
    assert _lib.lib().tgc_ag_matmul_plan(None, None) == _lib.TGC_ERR_INVALID_ARG


def test_tile_width_follows_the_measured_rule():
    """tile_n = 0: 512-column tiles when K >= 8192 and a shard holds at least group_m tile rows,
    in every mode but FUSED_CE; 256 otherwise; an explicit width is taken as given, except 512
    with FUSED_CE, which is refused."""
    square = dict(R=8, M=4096, K=4096, N=4096, comm_block_rows=128)
    mlp_up = dict(R=8, M=8192, K=4096, N=14336, comm_block_rows=256)
    large = dict(R=4, M=32768, K=8192, N=8192, comm_block_rows=512)
    for mode in ("fused", "fused_ce", "unfused", "mm_only"):
        m = _lib.MODES[mode]
        # the copy-engine producer keeps 256 columns: its copies may need room on the GEMM's SMs
        assert _plan(**large, mode=m)[2] == (256 if mode == "fused_ce" else 512), mode
        assert _plan(**square, mode=m)[2] == 256, mode
        assert _plan(**mlp_up, mode=m)[2] == 256, mode
    assert _plan(**large, mode=_lib.MODES["fused_ce"], tile_n=512)[0] == _lib.TGC_ERR_INVALID_ARG
    rc, _, width = _plan(**large, mode=_lib.MODES["fused_ce"], tile_n=256)
    assert (rc, width) == (0, 256)
    assert _plan(**dict(large, K=4096))[2] == 256                      # short K
    assert _plan(**dict(large, R=8, comm_block_rows=256))[2] == 512    # 16 tile rows per shard
    assert _plan(**dict(large, R=32, comm_block_rows=256))[2] == 256   # 4 tile rows per shard
    assert _plan(**dict(mlp_up, K=8192))[2] == 256                     # long K, short shards
    assert _plan(**dict(large, group_m=64))[2] == 256                  # a group longer than a shard
    assert _plan(**large, tile_n=256)[2] == 256
    assert _plan(**square, tile_n=512)[2] == 512


def test_ag_matmul_empty_problem_is_ok():
    assert _ag(M=0, B=None, C=None, a_out=None) == _lib.TGC_OK
    assert _ag(N=0, B=None, C=None, a_out=None) == _lib.TGC_OK
    arr = (ctypes.c_void_p * 2)(None, None)
    assert _lib.lib().tgc_ag_matmul(arr, 2, None, None, 0, 64, 64, 8, None) == _lib.TGC_OK


def test_plain_ag_matmul_validates_before_allocating():
    arr = (ctypes.c_void_p * 4)(*([FAKE] * 4))
    L = _lib.lib()
    assert L.tgc_ag_matmul(arr, 4, FAKE, FAKE, 66, 64, 64, 8, None) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_ag_matmul(arr, 4, FAKE, FAKE, 64, 60, 64, 8, None) == _lib.TGC_ERR_ALIGN


def test_ipc_calls_reject_null_arguments_before_any_cuda_call():
    L = _lib.lib()
    h = _lib.IpcHandle()
    p = ctypes.c_void_p()
    assert ctypes.sizeof(_lib.IpcHandle) == 72   # 64-byte CUDA IPC handle + 8-byte offset
    assert L.tgc_ipc_export(None, ctypes.byref(h)) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_ipc_export(FAKE, None) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_ipc_open(None, ctypes.byref(p)) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_ipc_open(ctypes.byref(h), None) == _lib.TGC_ERR_INVALID_ARG
    assert L.tgc_ipc_close(None, ctypes.byref(h)) == _lib.TGC_ERR_INVALID_ARG
    h.offset = FAKE + 1                            # an offset beyond the address itself
    assert L.tgc_ipc_close(FAKE, ctypes.byref(h)) == _lib.TGC_ERR_INVALID_ARG


def test_workspace_bytes_grows_with_blocks():
    a = tgc.tgc_ag_matmul_workspace_bytes(4, 64, 64, 64, 8)
    b = tgc.tgc_ag_matmul_workspace_bytes(4, 32768, 8192, 8192, 512)
    c = tgc.tgc_ag_matmul_workspace_bytes(8, 1 << 20, 64, 64, 8)
    assert 256 <= a <= b < c


# ----------------------------------------------------------------------------- schedule


def _all_tiles(M, N, cb, R, rank, pivot, grid, group_m=0, band_n=0, tile_n=256):
    seqs = [tgc.tgc_ag_matmul_schedule(M, N, cb, R, rank, pivot, group_m, grid, c, band_n=band_n, tile_n=tile_n)
            for c in range(grid)]
    return seqs


@pytest.mark.parametrize("M,N,cb,R", [(4096, 4096, 128, 8), (8192, 14336, 256, 8), (32768, 8192, 512, 4),
                                      (64, 64, 8, 4), (1000 * 8, 1000, 1000, 8)])
@pytest.mark.parametrize("pivot", ["page", "shard", "none"])
@pytest.mark.parametrize("band_n", [0, 16, 3])
@pytest.mark.parametrize("tile_n", [256, 512])
def test_schedule_is_a_permutation(M, N, cb, R, pivot, band_n, tile_n):
    bm = tgc.tgc_gemm_tile_shape()[0]
    npm, npn = -(-M // bm), -(-N // tile_n)
    for rank in sorted({0, 1, R - 1}):
        seqs = _all_tiles(M, N, cb, R, rank, pivot, grid=148, band_n=band_n, tile_n=tile_n)
        tiles = [t for s in seqs for t in s]
        assert len(tiles) == npm * npn
        assert len(set(tiles)) == npm * npn
        assert all(0 <= pm < npm and 0 <= pn < npn for pm, pn in tiles)


@pytest.mark.parametrize("M,N,cb,R", [(4096, 4096, 512, 8), (32768, 8192, 8192, 4)])
@pytest.mark.parametrize("tile_n", [256, 512])
def test_page_pivot_matches_formula_and_starts_on_local_shard_when_one_block_per_rank(M, N, cb, R, tile_n):
    """Triton第四课 (融合后的流水线): pid_m = (pid_m + NUM_PID_M_PER_COMM_BLOCK*RANK) % num_pid_m
    after the GROUP_SIZE_M swizzle; with one comm block per rank every rank begins on its own
    shard."""
    bm = tgc.tgc_gemm_tile_shape()[0]
    npm, npn = M // bm, -(-N // tile_n)
    tpb = cb // bm
    G = 8
    for rank in range(R):
        seq = tgc.tgc_ag_matmul_schedule(M, N, cb, R, rank, "page", G, 1, 0, tile_n=tile_n)
        for t, (pm, pn) in enumerate(seq):
            group = t // (G * npn)
            first = group * G
            gsz = min(npm - first, G)
            pm0 = first + (t % (G * npn)) % gsz
            pn0 = (t % (G * npn)) // gsz
            assert (pm, pn) == ((pm0 + tpb * rank) % npm, pn0)
        assert seq[0][0] * bm // (M // R) == rank


@pytest.mark.parametrize("M,N,cb,R,band_n", [(8192, 14336, 256, 8, 16), (32768, 8192, 512, 4, 16),
                                             (4096, 4096, 128, 8, 5), (1000 * 8, 1000, 1000, 8, 2)])
@pytest.mark.parametrize("tile_n", [256, 512])
def test_band_raster_walks_rows_in_order_within_each_band(M, N, cb, R, band_n, tile_n):
    """Band raster: tiles in bands of band_n x 256 columns (ceil(band_n x 256 / tile_n) tiles),
    row-major inside a band, the rank rotation applied to the rows after it; with the page pivot,
    rank r's walk starts on the row the page's formula gives and every band visits the rows in
    that rotated order."""
    bm, bn, _ = tgc.tgc_gemm_tile_shape()
    npm, npn = -(-M // bm), -(-N // tile_n)
    bt = -(-band_n * bn // tile_n)  # band width in tiles
    for rank in sorted({0, R - 1}):
        seq = tgc.tgc_ag_matmul_schedule(M, N, cb, R, rank, "page", 8, 1, 0, band_n=band_n, tile_n=tile_n)
        assert len(seq) == npm * npn
        off = (rank * cb // bm) % npm
        for t, (pm, pn) in enumerate(seq):
            band, r = divmod(t, bt * npm)
            bw = min(npn - band * bt, bt)
            assert (pm, pn) == ((r // bw + off) % npm, band * bt + r % bw)


def test_shard_pivot_starts_every_rank_on_its_shard():
    M, N, cb, R = 8192, 14336, 256, 8
    bm = tgc.tgc_gemm_tile_shape()[0]
    for rank in range(R):
        seq = tgc.tgc_ag_matmul_schedule(M, N, cb, R, rank, "shard", 8, 1, 0)
        assert seq[0][0] * bm // (M // R) == rank


def test_schedule_rejects_bad_arguments():
    for dynamic in ("ready_queue", "auto"):  # no static order past the local prefix
        with pytest.raises(tgc.TGCError):
            tgc.tgc_ag_matmul_schedule(64, 64, 8, 4, 0, dynamic, 8, 1, 0)
    with pytest.raises(tgc.TGCError):
        tgc.tgc_ag_matmul_schedule(64, 64, 8, 4, 4, "page", 8, 1, 0)
    with pytest.raises(tgc.TGCError):
        tgc.tgc_ag_matmul_schedule(64, 64, 8, 4, 0, "page", 8, 2, 2)
    for width in (0, 128, 1024):
        with pytest.raises(tgc.TGCError):
            tgc.tgc_ag_matmul_schedule(64, 64, 8, 4, 0, "page", 8, 1, 0, tile_n=width)


def test_trace_word_indices_match_header():
    import re
    from tile_gather_comm_gb300 import _lib
    hdr = open(os.path.join(ROOT, "include", "tgc.h"), encoding="utf-8").read()
    defs = {m.group(1).lower(): int(m.group(2)) for m in re.finditer(r"#define TGC_TRACE_([A-Z_]+)\s+(\d+)", hdr)}
    words = defs.pop("words")
    assert words == _lib.TRACE_WORDS
    assert defs == _lib.TRACE
    assert max(defs.values()) < words
