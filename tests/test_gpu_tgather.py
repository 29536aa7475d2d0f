"""TGATHER on the GPU against the CPU oracle, bit for bit.

Covers the pages' workloads (tiny fp32, 8 x fp16 (2,1,1,1024,1024), ragged
int32 (1000, 777)), the TGATHER page's test table (§九), element sizes 1..8,
D0..D2 > 1, misaligned sources (narrower vectors and peeled heads/tails), a
destination with DIM_3 > N*H (§7.2), empty inputs (§七) and per-chunk
progress release.
"""
import numpy as np
import pytest
import torch

import oracle
import tile_gather_comm_gb300 as tgc
from tile_gather_comm_gb300.workloads import TG_CONFIGS, make_tg_inputs

from .helpers import requires_gpu
from .test_oracle_pins import _golden_cases, _tagged_sources

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(autouse=True)
def _gpu():
    requires_gpu()


def _bytes(t):
    return t.detach().cpu().contiguous().numpy().tobytes()


@pytest.mark.parametrize("name", list(TG_CONFIGS))
def test_workloads_bit_exact(name):
    cfg = TG_CONFIGS[name]
    srcs = make_tg_inputs(cfg, seed=0)
    D0, D1, D2, H, W = cfg.shape
    d_srcs = [s.to(DEV) for s in srcs]
    dst = torch.empty((D0, D1, D2, cfg.nranks * H, W), dtype=cfg.dtype, device=DEV)
    dst.view(torch.uint8).fill_(0xA5)
    tgc.tgc_tgather(dst, d_srcs)
    ref = oracle.tgather([s.numpy() for s in srcs])
    assert _bytes(dst) == ref.tobytes()


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
@pytest.mark.parametrize("nranks", [1, 2, 4, 8])
def test_page_test_table(case, nranks):
    name, dt, rows, cols, _ = case
    srcs = _tagged_sources(dt, rows, cols, nranks)
    d_srcs = [torch.from_numpy(s).to(DEV) for s in srcs]
    # two spare destination rows (DIM_3 > N*H) must keep their -1 fill in every case,
    # including the empty one, where nothing at all may be written
    rows3 = nranks * rows + 2
    prefill = np.full((1, 1, 1, rows3, cols), -1).astype(srcs[0].dtype)
    dst = torch.from_numpy(prefill.copy()).to(DEV)
    tgc.tgc_tgather_ex(dst, d_srcs, dst_rows3=rows3)
    ref = oracle.tgather(srcs, dst_rows3=rows3, dst=prefill)
    assert _bytes(dst) == ref.tobytes()
    assert np.all(dst.cpu().numpy()[0, 0, 0, nranks * rows:].astype(np.int64) % 256 == 255)


@pytest.mark.parametrize("case", [c for c in _golden_cases() if c[4] > 0], ids=lambda c: c[0])
@pytest.mark.parametrize("nranks", [2, 8])
def test_page_chunk_cases_with_release(case, nranks):
    """The page's chunked scenarios (rows moved tile by tile, `page_tile_rows` rows at a time):
    here each tile of rows is one progress chunk, released once its bytes are in place."""
    name, dt, rows, cols, tile_rows = case
    srcs = _tagged_sources(dt, rows, cols, nranks)
    S = rows // tile_rows
    progress = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    counters = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    dst = torch.full((1, 1, 1, nranks * rows, cols), -1, dtype=torch.from_numpy(srcs[0]).dtype, device=DEV)
    for epoch in (1, 2):  # a second call over the same flags and counters
        dst.fill_(-1)
        tgc.tgc_tgather_ex(dst, [torch.from_numpy(s).to(DEV) for s in srcs], progress=progress,
                           counters=counters, chunk_rows=tile_rows, epoch=epoch)
        torch.cuda.synchronize()
        assert _bytes(dst) == oracle.tgather(srcs).tobytes(), (name, epoch)
        assert torch.all(progress == epoch) and torch.all(counters == 0)


@pytest.mark.parametrize("shape", [(2, 3, 2, 5, 7), (1, 1, 1, 1, 1), (3, 1, 2, 33, 65), (1, 2, 1, 257, 129),
                                   (2, 1, 1, 1024, 24)])
@pytest.mark.parametrize("dtype", [torch.uint8, torch.float16, torch.int32, torch.float64])
@pytest.mark.parametrize("nranks", [1, 3, 8])
def test_shapes_and_dtypes(shape, dtype, nranks):
    es = torch.empty((), dtype=dtype).element_size()
    g = torch.Generator().manual_seed(nranks * 7 + es)
    srcs = [torch.randint(0, 256, shape + (es,), generator=g, dtype=torch.uint8).view(dtype).reshape(shape)
            for _ in range(nranks)]
    d_srcs = [s.to(DEV) for s in srcs]
    dst = torch.zeros(shape[:3] + (nranks * shape[3], shape[4]), dtype=dtype, device=DEV)
    tgc.tgc_tgather(dst, d_srcs)
    assert _bytes(dst) == _bytes(torch.cat(srcs, dim=3))


@pytest.mark.parametrize("src_off,dst_off", [(1, 0), (0, 3), (2, 6), (5, 1), (4, 4)])
def test_misaligned_pointers(src_off, dst_off):
    """Sources and destination at element offsets that break 16-byte alignment."""
    shape = (2, 1, 1, 37, 41)
    nranks = 4
    n = int(np.prod(shape))
    g = torch.Generator().manual_seed(src_off * 10 + dst_off)
    bufs = [torch.randint(-2**31, 2**31, (n + 16,), generator=g, dtype=torch.int64).to(torch.int32).to(DEV)
            for _ in range(nranks)]
    srcs = [b[src_off + r:src_off + r + n].view(shape) for r, b in enumerate(bufs)]
    big = torch.zeros(nranks * n + 16, dtype=torch.int32, device=DEV)
    dst = big[dst_off:dst_off + nranks * n].view(shape[:3] + (nranks * shape[3], shape[4]))
    tgc.tgc_tgather(dst, srcs)
    ref = oracle.tgather([s.cpu().numpy() for s in srcs])
    assert _bytes(dst) == ref.tobytes()
    assert torch.all(big[:dst_off] == 0) and torch.all(big[dst_off + nranks * n:] == 0)


def test_dst_rows3_larger_leaves_rest():
    shape = (2, 1, 2, 30, 17)
    srcs = [torch.randn(shape) for _ in range(3)]
    rows3 = 3 * 30 + 11
    dst = torch.full(shape[:3] + (rows3, 17), -7.0, device=DEV)
    tgc.tgc_tgather_ex(dst, [s.to(DEV) for s in srcs], dst_rows3=rows3)
    ref = oracle.tgather([s.numpy() for s in srcs], dst_rows3=rows3,
                         dst=np.full(shape[:3] + (rows3, 17), -7.0, dtype=np.float32))
    assert _bytes(dst) == ref.tobytes()


@pytest.mark.parametrize("shape", [(1, 1, 1, 0, 8), (1, 1, 1, 8, 0), (0, 1, 1, 8, 8)])
def test_empty_leaves_dst(shape):
    D0, D1, D2, H, W = shape
    srcs = [torch.zeros(shape, device=DEV) for _ in range(2)]
    dst = torch.full((max(D0, 1), D1, D2, max(2 * H, 1), max(W, 1)), -1.0, device=DEV)
    tgc.tgc_tgather(dst, srcs)
    torch.cuda.synchronize()
    assert torch.all(dst == -1)


@pytest.mark.parametrize("H,W,chunk_rows,D0", [(1024, 1024, 128, 2), (1000, 777, 96, 1), (64, 32, 7, 3),
                                               (1024, 64, 8, 2),    # 1024 chunks: the counting CTAs publish
                                               (300, 40, 1, 1),     # 2400 one-row chunks
                                               (5, 3, 8, 1)])       # chunk_rows > H: one chunk per rank
def test_progress_release(H, W, chunk_rows, D0):
    nranks = 8
    shape = (D0, 1, 1, H, W)
    g = torch.Generator().manual_seed(H + W)
    srcs = [torch.randint(-2**31, 2**31, shape, generator=g, dtype=torch.int64).to(torch.int32)
            for _ in range(nranks)]
    S = -(-H // chunk_rows)
    progress = torch.full((nranks * S,), 6, dtype=torch.int32, device=DEV)   # stale epoch
    counters = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    dst = torch.zeros((D0, 1, 1, nranks * H, W), dtype=torch.int32, device=DEV)
    tgc.tgc_tgather_ex(dst, [s.to(DEV) for s in srcs], progress=progress, counters=counters,
                       chunk_rows=chunk_rows, epoch=7)
    torch.cuda.synchronize()
    assert _bytes(dst) == oracle.tgather([s.numpy() for s in srcs]).tobytes()
    assert torch.all(progress == 7)
    assert torch.all(counters == 0)


@pytest.mark.parametrize("src_off,dst_off,es", [(8, 8, 2), (4, 12, 4), (2, 6, 2), (16, 48, 4), (1, 3, 1)])
def test_progress_release_misaligned_views(src_off, dst_off, es):
    """Per-chunk release with sources and destination at byte offsets that allow 16-byte
    vectors only, 8-byte ones, or element copies, ragged rows: bytes and flags exact."""
    nranks, D0, H, W, chunk_rows = 4, 2, 203, 131, 40
    dt = {1: torch.uint8, 2: torch.float16, 4: torch.int32}[es]  # compared as raw bytes
    g = torch.Generator().manual_seed(src_off * 31 + dst_off)
    n = D0 * H * W
    srcs_h = [torch.randint(0, 256, (n * es,), generator=g, dtype=torch.int64).to(torch.uint8)
              for _ in range(nranks)]
    srcs = []
    for sh in srcs_h:
        buf = torch.zeros(n * es + 64, dtype=torch.uint8, device=DEV)
        buf[src_off:src_off + n * es].copy_(sh.to(DEV))
        srcs.append(buf[src_off:src_off + n * es].view(dt).view(D0, 1, 1, H, W))
    dbuf = torch.zeros(nranks * n * es + 64, dtype=torch.uint8, device=DEV)
    dst = dbuf[dst_off:dst_off + nranks * n * es].view(dt).view(D0, 1, 1, nranks * H, W)
    S = -(-H // chunk_rows)
    progress = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    counters = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    tgc.tgc_tgather_ex(dst, srcs, progress=progress, counters=counters, chunk_rows=chunk_rows, epoch=5)
    torch.cuda.synchronize()
    ref = oracle.tgather([sh.numpy().view({1: np.uint8, 2: np.uint16, 4: np.int32}[es]).reshape(D0, 1, 1, H, W)
                          for sh in srcs_h])
    assert _bytes(dst) == ref.tobytes()
    assert torch.all(dbuf[:dst_off] == 0) and torch.all(dbuf[dst_off + nranks * n * es:] == 0)
    assert torch.all(progress == 5) and torch.all(counters == 0)


@pytest.mark.parametrize("H,chunk_rows,epochs", [(4096, 128, 1), (3000, 64, 3)])
def test_progress_release_many_items_per_cta(H, chunk_rows, epochs):
    """Per-chunk release with far more items than resident CTAs (each CTA walks several items,
    counting each), over several epochs on the same flags: bytes exact against the oracle,
    every flag at the last epoch, every counter back at 0."""
    nranks, D0, W = 8, 2, 1024
    shape = (D0, 1, 1, H, W)
    g = torch.Generator().manual_seed(H + chunk_rows)
    srcs_h = [torch.randint(-2**15, 2**15, shape, generator=g, dtype=torch.int32).to(torch.int16)
              .view(torch.float16) for _ in range(nranks)]   # random bit patterns, compared as bytes
    srcs = [s.to(DEV) for s in srcs_h]
    S = -(-H // chunk_rows)
    progress = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    counters = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    dst = torch.zeros((D0, 1, 1, nranks * H, W), dtype=torch.float16, device=DEV)
    ref = oracle.tgather([s.numpy() for s in srcs_h]).tobytes()
    for e in range(1, epochs + 1):
        dst.zero_()
        tgc.tgc_tgather_ex(dst, srcs, progress=progress, counters=counters, chunk_rows=chunk_rows, epoch=10 + e)
        torch.cuda.synchronize()
        assert _bytes(dst) == ref
        assert torch.all(progress == 10 + e)
        assert torch.all(counters == 0)


@pytest.mark.parametrize("chunk_rows", [16, 1])   # 64 chunks (publisher block), 1024 (completing block)
def test_progress_release_with_taller_destination(chunk_rows):
    """Per-chunk release into a destination with DIM_3 > nranks*H ([TG] §7.2): the gathered rows
    exact, the rows past them in every slab untouched, every flag published."""
    nranks, D0, H, W = 8, 3, 128, 96
    shape = (D0, 1, 1, H, W)
    g = torch.Generator().manual_seed(chunk_rows)
    srcs = [torch.randint(-2**31, 2**31, shape, generator=g, dtype=torch.int64).to(torch.int32)
            for _ in range(nranks)]
    rows3 = nranks * H + 37
    prefill = np.full((D0, 1, 1, rows3, W), -5, dtype=np.int32)
    dst = torch.from_numpy(prefill.copy()).to(DEV)
    S = -(-H // chunk_rows)
    progress = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    counters = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    tgc.tgc_tgather_ex(dst, [s.to(DEV) for s in srcs], dst_rows3=rows3, progress=progress, counters=counters,
                       chunk_rows=chunk_rows, epoch=4)
    torch.cuda.synchronize()
    ref = oracle.tgather([s.numpy() for s in srcs], dst_rows3=rows3, dst=prefill)
    assert _bytes(dst) == ref.tobytes()
    assert torch.all(dst[:, :, :, nranks * H:] == -5)
    assert torch.all(progress == 4) and torch.all(counters == 0)


def test_progress_release_marks_chunks_whose_count_never_completes():
    """The publisher's wait is bounded: with counters that were not zero on entry (a caller
    error), no chunk's count ever equals its item count, so after spin_timeout_ns every entry
    gets ~epoch (never taken for the flag), the rows are still copied, the counters keep what
    the copying blocks added, and the context stays usable for the next call."""
    nranks, D0, H, W, chunk_rows = 4, 2, 256, 512, 64
    shape = (D0, 1, 1, H, W)
    g = torch.Generator().manual_seed(11)
    srcs_h = [torch.randint(-2**31, 2**31, shape, generator=g, dtype=torch.int64).to(torch.int32)
              for _ in range(nranks)]
    srcs = [s.to(DEV) for s in srcs_h]
    S = H // chunk_rows
    progress = torch.zeros(nranks * S, dtype=torch.int32, device=DEV)
    counters = torch.full((nranks * S,), -2**31, dtype=torch.int32, device=DEV)  # 2^31: never a count
    dst = torch.zeros((D0, 1, 1, nranks * H, W), dtype=torch.int32, device=DEV)
    tgc.tgc_tgather_ex(dst, srcs, progress=progress, counters=counters, chunk_rows=chunk_rows, epoch=7,
                       spin_timeout_ns=20_000_000)
    torch.cuda.synchronize()
    ref = oracle.tgather([s.numpy() for s in srcs_h]).tobytes()
    assert _bytes(dst) == ref
    assert torch.all(progress == ~7)
    assert torch.all(counters > -2**31)   # every chunk was counted on top of the bad start
    # the same flags, cleared, then a correct call: published as usual
    counters.zero_()
    dst.zero_()
    tgc.tgc_tgather_ex(dst, srcs, progress=progress, counters=counters, chunk_rows=chunk_rows, epoch=8)
    torch.cuda.synchronize()
    assert _bytes(dst) == ref
    assert torch.all(progress == 8) and torch.all(counters == 0)


@pytest.mark.parametrize("nranks,shape,dtype", [
    (64, (1, 1, 1, 3, 5), torch.int32),       # the maximum rank count
    (64, (2, 1, 1, 17, 128), torch.float16),
    (1, (1, 1, 1, 1, 1), torch.uint8),        # one element
    (3, (4, 3, 2, 1, 9), torch.float64),      # many slabs, one row each
])
def test_edge_counts(nranks, shape, dtype):
    es = torch.empty((), dtype=dtype).element_size()
    g = torch.Generator().manual_seed(nranks + es)
    srcs = [torch.randint(0, 256, shape + (es,), generator=g, dtype=torch.uint8).view(dtype).reshape(shape)
            for _ in range(nranks)]
    dst = torch.zeros(shape[:3] + (nranks * shape[3], shape[4]), dtype=dtype, device=DEV)
    tgc.tgc_tgather(dst, [s.to(DEV) for s in srcs])
    assert _bytes(dst) == _bytes(torch.cat(srcs, dim=3))


# ----------------------------------------------------------------------------- strided views


def _strided_case(case, nranks, dtype, g):
    es = torch.empty((), dtype=dtype).element_size()

    def rnd(shape):
        return torch.randint(0, 256, shape + (es,), generator=g, dtype=torch.uint8).view(dtype).reshape(shape)
    if case == "slices":
        bases = [rnd((3, 2, 4, 40, 300)) for _ in range(nranks)]
        srcs = [b[1:3, :1, 1:4, 3:35, 8:264] for b in bases]          # offset rows/cols, padded pitch
        big = torch.zeros((2, 1, 3, nranks * 32 + 5, 300), dtype=dtype)
        dst = big[:, :, :, 2:2 + nranks * 32, 16:272]
    elif case == "transposed":
        bases = [rnd((2, 1, 1, 24, 10)) for _ in range(nranks)]
        srcs = [b.transpose(3, 4) for b in bases]                      # inner stride != 1
        big = torch.zeros((2, 1, 1, nranks * 10, 24), dtype=dtype)
        dst = big
    elif case == "odd_offsets":
        bases = [rnd((1, 1, 1, 17, 41)) for _ in range(nranks)]
        srcs = [b[:, :, :, 1:16, 1:40] for b in bases]                # unaligned starts, odd widths
        big = torch.zeros((1, 1, 1, nranks * 15 + 2, 45), dtype=dtype)
        dst = big[:, :, :, 1:1 + nranks * 15, 3:42]
    else:
        raise ValueError(case)
    return srcs, big, dst


def _same_view_on_device(x):
    """The same strided view (shape, strides, offset) over a device copy of x's whole storage."""
    flat = torch.empty(0, dtype=x.dtype).set_(x.untyped_storage())
    return flat.to(DEV).as_strided(x.shape, x.stride(), x.storage_offset())


@pytest.mark.parametrize("case", ["slices", "transposed", "odd_offsets"])
@pytest.mark.parametrize("dtype", [torch.uint8, torch.float16, torch.int32, torch.float64])
@pytest.mark.parametrize("nranks", [1, 4])
def test_strided_views(case, dtype, nranks):
    g = torch.Generator().manual_seed(nranks * 31 + len(case))
    srcs, big, dst = _strided_case(case, nranks, dtype, g)
    ref_big = big.clone()
    ref_dst_view = ref_big.as_strided(dst.shape, dst.stride(), dst.storage_offset())
    oracle.tgather_strided(ref_dst_view.numpy(), [s.numpy() for s in srcs])
    assert _bytes(ref_dst_view) == _bytes(torch.cat(srcs, dim=3))  # the oracle agrees with torch.cat (raw bits)
    d_big = big.to(DEV)
    d_dst = d_big.as_strided(dst.shape, dst.stride(), dst.storage_offset())
    d_srcs = [_same_view_on_device(x) for x in srcs]
    assert all(x.stride() == srcs[0].stride() for x in d_srcs)
    tgc.tgc_tgather_strided(d_dst, d_srcs)
    assert _bytes(d_big) == _bytes(ref_big)  # view written, everything around it untouched


def test_strided_views_of_device_buffers():
    """Sources that are strided views of device buffers (not copies)."""
    g = torch.Generator().manual_seed(5)
    bases = [torch.randint(-2**31, 2**31, (2, 1, 2, 50, 130), generator=g, dtype=torch.int64).to(torch.int32)
             for _ in range(3)]
    d_bases = [b.to(DEV) for b in bases]
    views = [b[:, :, :, 5:45, 2:130] for b in d_bases]
    assert views[0].stride()[3] == 130
    dst = torch.zeros((2, 1, 2, 3 * 40, 128), dtype=torch.int32, device=DEV)
    tgc.tgc_tgather_strided(dst, views)
    ref = torch.cat([b[:, :, :, 5:45, 2:130] for b in bases], dim=3)
    assert torch.equal(dst.cpu(), ref)
