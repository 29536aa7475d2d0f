"""Pins for the CPU oracle: checks against what the pages and mathematics fix.

Each test compares the oracle with something other than itself:
  * the TGATHER closed form's consequences (the page's rank-tagged value scheme,
    torch.cat along DIM_3, N=1 as a plain copy, untouched extra rows, early
    return on empty input, raw-bit copying);
  * bf16 round-to-nearest-even against torch's conversion on random bit patterns;
  * integer-exact GEMM special cases against an int64 matmul;
  * general GEMM against a float64 matmul and against exact rational brute force,
    within the fp32 accumulation error bound;
  * chunked producer/consumer execution against gather-then-MatMul (bit-exact).

Sources:
  [TG]  "CANN PTO-ISA TGATHER 指令深度解析：跨 Rank 行拼接 Gather 的实现原理与开发指南"
  [AGM] "Triton第四课：基于对称内存融合 AllGather 与 MatMul，提速1.56倍"
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tgather_npu_cases.txt")
NP_DT = {"float32": np.float32, "int32": np.int32, "uint8": np.uint8}


def _golden_cases():
    cases = []
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, dt, rows, cols, tile = line.split()
            cases.append((name, dt, int(rows), int(cols), int(tile)))
    return cases


def _tagged_sources(dt, rows, cols, nranks):
    """[TG] §九: element i of rank r holds i + r*10000 (uint8: modulo 256)."""
    out = []
    for r in range(nranks):
        v = np.arange(rows * cols, dtype=np.int64) + r * 10000
        if dt == "uint8":
            v = v % 256
        out.append(v.astype(NP_DT[dt]).reshape(1, 1, 1, rows, cols))
    return out


# ----------------------------------------------------------------------------- TGATHER


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
@pytest.mark.parametrize("nranks", [1, 2, 4, 8])
def test_tgather_page_value_scheme(oracle_mod, case, nranks):
    """[TG] §九 value scheme: dst row r*H+i, col j must hold (i*W+j) + r*10000."""
    name, dt, rows, cols, _ = case
    srcs = _tagged_sources(dt, rows, cols, nranks)
    prefill = np.full((1, 1, 1, nranks * rows, cols), -1).astype(NP_DT[dt])
    dst = oracle_mod.tgather(srcs, dst=prefill.copy())
    assert dst.shape == (1, 1, 1, nranks * rows, cols)  # [TG] §二 output shape
    for r in range(nranks):
        for i in range(rows):
            expect = np.arange(cols, dtype=np.int64) + i * cols + r * 10000
            if dt == "uint8":
                expect = expect % 256
            got = dst[0, 0, 0, r * rows + i].astype(np.int64)
            assert np.array_equal(got, expect), (name, r, i)
    if rows == 0:  # [TG] §7.4 / §九 empty case: the destination keeps its -1 fill
        assert np.array_equal(dst, prefill)


@pytest.mark.parametrize("shape", [(1, 1, 1, 8, 32), (2, 3, 2, 5, 7), (3, 1, 2, 1, 1),
                                   (1, 2, 1, 13, 33), (2, 1, 1, 64, 16)])
@pytest.mark.parametrize("dtype", [torch.uint8, torch.float16, torch.int32, torch.float64])
@pytest.mark.parametrize("nranks", [1, 3, 8])
def test_tgather_equals_torch_cat_dim3(oracle_mod, shape, dtype, nranks):
    """[TG] §二: concatenation along DIM_3, other dims unchanged == torch.cat(dim=3)."""
    g = torch.Generator().manual_seed(hash((shape, str(dtype), nranks)) % 2**31)
    srcs = [torch.randint(0, 256, shape + (torch.empty((), dtype=dtype).element_size(),),
                          generator=g, dtype=torch.uint8).view(dtype).reshape(shape)
            for _ in range(nranks)]
    ref = torch.cat(srcs, dim=3)
    got = oracle_mod.tgather([s.numpy() for s in srcs])
    assert got.shape == tuple(ref.shape)
    assert got.tobytes() == ref.contiguous().numpy().tobytes()


def test_tgather_single_rank_is_plain_copy(oracle_mod):
    x = np.random.default_rng(1).standard_normal((2, 2, 3, 9, 11)).astype(np.float32)
    assert oracle_mod.tgather([x]).tobytes() == x.tobytes()


def test_tgather_dst_rows3_larger_leaves_rest(oracle_mod):
    """[TG] §7.2: dst DIM_3 > N*H -> only the first N*H rows of every slab are written."""
    rng = np.random.default_rng(2)
    srcs = [rng.integers(-1000, 1000, (2, 1, 2, 3, 5)).astype(np.int32) for _ in range(4)]
    dst = np.full((2, 1, 2, 15, 5), -7, dtype=np.int32)
    out = oracle_mod.tgather(srcs, dst_rows3=15, dst=dst.copy())
    for r in range(4):
        assert np.array_equal(out[:, :, :, r * 3:(r + 1) * 3, :], srcs[r])
    assert np.all(out[:, :, :, 12:, :] == -7)


@pytest.mark.parametrize("shape", [(1, 1, 1, 0, 8), (1, 1, 1, 8, 0), (0, 1, 1, 8, 8), (1, 1, 0, 4, 4)])
def test_tgather_empty_returns_without_writes(oracle_mod, shape):
    """[TG] §七 / §6.1: empty data returns before any transfer."""
    srcs = [np.zeros(shape, dtype=np.float32) for _ in range(3)]
    D0, D1, D2, H, W = shape
    dst = np.full((D0, D1, D2, 3 * H, W), -1.0, dtype=np.float32)
    out = oracle_mod.tgather(srcs, dst=dst.copy())
    assert np.array_equal(out, dst)


def test_tgather_rejects_short_dst(oracle_mod):
    with pytest.raises(ValueError):
        oracle_mod.tgather([np.zeros((1, 1, 1, 4, 4), np.float32)] * 2, dst_rows3=7)


def test_tgather_copies_raw_bits(oracle_mod):
    """NaN payloads, signalling NaNs and -0 must survive (a byte copy, no float conversion)."""
    bits = np.array([0x7FC00001, 0xFFA00000, 0x80000000, 0x7F800001, 0x00000001, 0xFF800000],
                    dtype=np.uint32)
    srcs = [(bits + r).view(np.float32).reshape(1, 1, 1, 1, 6) for r in range(3)]
    out = oracle_mod.tgather(srcs)
    for r in range(3):
        assert np.array_equal(out[0, 0, 0, r].view(np.uint32), bits + r)


# ----------------------------------------------------------------------------- bf16


def _torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_bf16_rne_matches_torch_on_random_bit_patterns(oracle_mod):
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 2**32, 2_000_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    ours = oracle_mod.f32_to_bf16(x)
    ref = _torch_bf16_bits(x)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    # NaN must stay NaN (payload is implementation-chosen): exponent all ones, mantissa != 0
    assert np.all((ours[nan] & 0x7F80) == 0x7F80) and np.all((ours[nan] & 0x7F) != 0)


def test_bf16_rne_edge_cases(oracle_mod):
    cases = {
        0x3F808000: 0x3F80,  # tie, kept part even -> stays
        0x3F818000: 0x3F82,  # tie, kept part odd -> rounds up to even
        0x3F808001: 0x3F81,  # just above half -> up
        0x3F807FFF: 0x3F80,  # just below half -> down
        0x00000000: 0x0000, 0x80000000: 0x8000,  # +-0
        0x00000001: 0x0000, 0x80000001: 0x8000,  # tiny subnormals -> signed zero
        0x00008000: 0x0000, 0x00018000: 0x0002,  # subnormal ties
        0x7F7FFFFF: 0x7F80,  # max finite float rounds to +Inf
        0x7F7F7FFF: 0x7F7F,  # max finite bf16 stays
        0xFF7FFFFF: 0xFF80,
        0x7F800000: 0x7F80, 0xFF800000: 0xFF80,  # +-Inf
    }
    for inp, want in cases.items():
        x = np.array([inp], dtype=np.uint32).view(np.float32)
        assert int(oracle_mod.f32_to_bf16(x)[0]) == want, hex(inp)
        assert int(_torch_bf16_bits(x)[0]) == want, hex(inp)  # the table itself is right
    for nan in (0x7FC00000, 0xFFC00000, 0x7F800001, 0xFF800001):
        x = np.array([nan], dtype=np.uint32).view(np.float32)
        y = int(oracle_mod.f32_to_bf16(x)[0])
        assert (y & 0x7F80) == 0x7F80 and (y & 0x7F) != 0
        assert (y >> 15) == (nan >> 31)  # sign kept


def test_bf16_widen_matches_torch(oracle_mod):
    bits = np.arange(0, 2**16, dtype=np.uint32).astype(np.uint16)
    ours = oracle_mod.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    assert np.array_equal(ours.view(np.uint32), ref.view(np.uint32))


# ----------------------------------------------------------------------------- AG-MatMul


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _from_bits(b: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("R,H,K,N", [(4, 16, 64, 40), (2, 24, 64, 96), (8, 4, 32, 8), (1, 8, 64, 24)])
def test_ag_matmul_integer_exact(oracle_mod, R, H, K, N):
    """Small-integer bf16 inputs: every product and partial sum is an exact fp32 integer
    and |C| <= 2*2*64 = 256 is exact in bf16, so C must equal an int64 matmul exactly.
    N != K catches a transposed B; R > 1 with distinct shards catches a wrong gather."""
    g = torch.Generator().manual_seed(R * 1000 + N)
    shards_i = [torch.randint(-2, 3, (H, K), generator=g) for _ in range(R)]
    B_i = torch.randint(-2, 3, (N, K), generator=g)
    shards = [_bf16_bits(s.to(torch.bfloat16)) for s in shards_i]
    Bb = _bf16_bits(B_i.to(torch.bfloat16))
    C, a = oracle_mod.ag_matmul(shards, Bb)
    A_i = torch.cat(shards_i, 0)
    ref = (A_i.to(torch.int64) @ B_i.to(torch.int64).T)
    assert int(ref.abs().max()) <= 256
    got = _from_bits(C).to(torch.float64)
    assert torch.equal(got, ref.to(torch.float64))
    assert np.array_equal(a, np.concatenate(shards, 0))  # a == the gather (closed form, D0=D1=D2=1)


def _fp32_sum_bound(A64, B64):
    """|fl32(sum) - sum| <= (K-1) u sum|a_k b_k|, u = 2^-24 (recursive summation)."""
    K = A64.shape[1]
    return (K - 1) * 2.0**-24 * (np.abs(A64) @ np.abs(B64).T)


def _bf16_half_ulp(x):
    x = np.abs(x)
    e = np.floor(np.log2(np.maximum(x, 2.0**-133)))
    return 2.0 ** (np.maximum(e, -126) - 7) / 2


@pytest.mark.parametrize("R,H,K,N,sigma", [(4, 16, 64, 64, 1.0), (8, 16, 256, 48, 0.02), (2, 32, 512, 16, 0.5)])
def test_ag_matmul_vs_float64(oracle_mod, R, H, K, N, sigma):
    g = torch.Generator().manual_seed(K + N)
    shards_t = [torch.randn(H, K, generator=g).to(torch.bfloat16) for _ in range(R)]
    B_t = (torch.randn(N, K, generator=g) * sigma).to(torch.bfloat16)
    C, _ = oracle_mod.ag_matmul([_bf16_bits(s) for s in shards_t], _bf16_bits(B_t))
    A64 = torch.cat(shards_t, 0).to(torch.float64).numpy()
    B64 = B_t.to(torch.float64).numpy()
    exact = A64 @ B64.T
    got = _from_bits(C).to(torch.float64).numpy()
    bound = _fp32_sum_bound(A64, B64) + 2 * _bf16_half_ulp(np.abs(exact) + _fp32_sum_bound(A64, B64))
    assert np.all(np.abs(got - exact) <= bound + 1e-300)
    # the benchmark spec's tolerance against the float64 reference holds with a wide margin
    assert np.all(np.abs(got - exact) <= 0.02 + 0.01 * np.abs(exact))


def test_ag_matmul_bruteforce_exact_rationals(oracle_mod):
    """Tiny case (the tiny workload's shape, first rows): exact rational dot products.
    The oracle's bf16 output must be within half a bf16 ulp of the fp32-rounded sum,
    and the fp32 sum within the recursive-summation bound of the exact sum."""
    from tile_gather_comm_gb300.workloads import AG_CONFIGS, make_ag_inputs
    cfg = AG_CONFIGS["tiny"]
    shards_t, B_t = make_ag_inputs(cfg, seed=0)
    shards = [_bf16_bits(s) for s in shards_t]
    Bb = _bf16_bits(B_t)
    C, _ = oracle_mod.ag_matmul(shards, Bb)
    A = torch.cat(shards_t, 0).to(torch.float64).numpy()
    Bm = B_t.to(torch.float64).numpy()
    got = _from_bits(C).to(torch.float64).numpy()
    K = cfg.K
    for m in range(0, cfg.M, 5):
        for n in range(cfg.N):
            exact = sum((Fraction(A[m, k]) * Fraction(Bm[n, k]) for k in range(K)), Fraction(0))
            absum = sum(abs(Fraction(A[m, k]) * Fraction(Bm[n, k])) for k in range(K))
            err32 = (K - 1) * Fraction(1, 2**24) * absum
            e = float(exact)
            tol = float(err32) + 2 * _bf16_half_ulp(abs(e) + float(err32))
            assert abs(Fraction(got[m, n]) - exact) <= Fraction(tol), (m, n)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_chunked_equals_gather_then_matmul(oracle_mod, seed):
    """[AGM] 融合后的流水线: after every chunk is consumed the result equals a full
    AllGather followed by MatMul -- bit for bit, in any release order."""
    R, H, K, N, cb = 4, 32, 64, 48, 8
    g = torch.Generator().manual_seed(seed)
    shards = [_bf16_bits(torch.randn(H, K, generator=g).to(torch.bfloat16)) for _ in range(R)]
    Bb = _bf16_bits(torch.randn(N, K, generator=g).to(torch.bfloat16))
    C, a = oracle_mod.ag_matmul(shards, Bb)
    order = torch.randperm(R * H // cb, generator=g).numpy()
    C2, a2 = oracle_mod.ag_matmul_chunked(shards, Bb, cb, order)
    assert np.array_equal(C, C2) and np.array_equal(a, a2)


def test_chunked_rejects_non_permutation(oracle_mod):
    shards = [np.zeros((8, 16), np.uint16)] * 2
    Bb = np.zeros((4, 16), np.uint16)
    with pytest.raises(ValueError):
        oracle_mod.ag_matmul_chunked(shards, Bb, 4, np.array([0, 1, 1, 3]))
    with pytest.raises(ValueError):
        oracle_mod.ag_matmul_chunked(shards, Bb, 4, np.array([0, 1, 2]))


def test_rows_variant_matches_full(oracle_mod):
    g = torch.Generator().manual_seed(7)
    shards = [_bf16_bits(torch.randn(24, 64, generator=g).to(torch.bfloat16)) for _ in range(3)]
    Bb = _bf16_bits(torch.randn(40, 64, generator=g).to(torch.bfloat16))
    C, _ = oracle_mod.ag_matmul(shards, Bb)
    rows = np.array([0, 5, 23, 24, 47, 48, 71])
    assert np.array_equal(oracle_mod.ag_matmul_rows(shards, Bb, rows), C[rows])


# ----------------------------------------------------------------------------- strided TGATHER


@pytest.mark.parametrize("nranks", [1, 3, 8])
def test_tgather_strided_dense_equals_dense_form(oracle_mod, nranks):
    """With dense strides the strided form is the dense formula."""
    rng = np.random.default_rng(nranks)
    srcs = [rng.integers(-2**31, 2**31, (2, 3, 1, 5, 7)).astype(np.int32) for _ in range(nranks)]
    ref = oracle_mod.tgather(srcs)
    out = np.zeros_like(ref)
    oracle_mod.tgather_strided(out, srcs)
    assert np.array_equal(out, ref)


@pytest.mark.parametrize("case", ["slices", "transposed_w", "padded_dst"])
def test_tgather_strided_views_equal_torch_cat(oracle_mod, case):
    """[TG] §7.3: GlobalTensor views with strides; torch.cat of the same views along DIM_3."""
    g = torch.Generator().manual_seed(len(case))
    nranks, shape = 4, (2, 1, 3, 6, 10)
    if case == "transposed_w":
        bases = [torch.randint(-1000, 1000, (2, 1, 3, 10, 6), generator=g, dtype=torch.int32) for _ in range(nranks)]
        srcs = [b.transpose(3, 4) for b in bases]        # inner stride != 1
    else:
        bases = [torch.randint(-1000, 1000, (3, 2, 4, 9, 17), generator=g, dtype=torch.int32) for _ in range(nranks)]
        srcs = [b[1:3, :1, ::1][:, :, 1:4, 2:8, 3:13] for b in bases]   # offset slices, padded rows
    assert tuple(srcs[0].shape) == shape
    ref = torch.cat(srcs, dim=3)
    if case == "padded_dst":
        big = torch.full((2, 1, 3, nranks * 6 + 3, 15), -5, dtype=torch.int32)
        dst = big[:, :, :, 1:1 + nranks * 6, 2:12]
    else:
        big = torch.full((2, 1, 3, nranks * 6, 10), -5, dtype=torch.int32)
        dst = big
    out = oracle_mod.tgather_strided(dst.numpy(), [s.numpy() for s in srcs])
    assert np.array_equal(np.asarray(dst.numpy()), ref.numpy())
    if case == "padded_dst":
        mask = torch.ones_like(big, dtype=torch.bool)
        mask[:, :, :, 1:1 + nranks * 6, 2:12] = False
        assert torch.all(big[mask] == -5)  # everything outside the destination view untouched


# ----------------------------------------------------------------------------- float8 e4m3 output


def _torch_e4m3_bits(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_rne_matches_torch_inside_range(oracle_mod):
    """Inside the finite range torch's float8_e4m3fn cast is round-to-nearest-even."""
    rng = np.random.default_rng(11)
    x = np.concatenate([
        rng.uniform(-448, 448, 400_000), rng.uniform(-1, 1, 200_000),
        rng.uniform(-2**-5, 2**-5, 200_000),  # subnormals and the smallest normals
        np.exp2(rng.uniform(-12, 8.8, 200_000)) * rng.choice([-1, 1], 200_000),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    assert np.array_equal(oracle_mod.f32_to_e4m3(x), _torch_e4m3_bits(x))


def test_e4m3_grid_points_ties_and_saturation(oracle_mod):
    grid = oracle_mod.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    finite = ~np.isnan(grid)
    codes = np.arange(256, dtype=np.uint8)[finite]
    # every representable value converts to itself (0x80 is -0)
    assert np.array_equal(oracle_mod.f32_to_e4m3(grid[finite].astype(np.float32)), codes)
    # midpoints between neighbours round to the even code
    pos = np.sort(np.unique(grid[finite & (grid >= 0)]))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    lo = oracle_mod.f32_to_e4m3(pos[:-1].astype(np.float32))
    hi = oracle_mod.f32_to_e4m3(pos[1:].astype(np.float32))
    got = oracle_mod.f32_to_e4m3(mids)
    assert np.all(np.where(lo % 2 == 0, got == lo, got == hi))
    # saturation: the largest finite magnitude is 448 = 0x7E; everything beyond clamps there
    big = np.array([448, 449, 464, 465, 480, 1e6, np.inf], dtype=np.float32)
    assert np.all(oracle_mod.f32_to_e4m3(big) == 0x7E)
    assert np.all(oracle_mod.f32_to_e4m3(-big) == 0xFE)
    assert oracle_mod.f32_to_e4m3(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_ag_matmul_e4m3_rows_integer_exact(oracle_mod):
    """Values in {-1, 0, 1} with K = 16: |C| <= 16, and integers up to 16 are exact in e4m3."""
    g = torch.Generator().manual_seed(21)
    R, H, K, N = 4, 8, 16, 24
    si = [torch.randint(-1, 2, (H, K), generator=g) for _ in range(R)]
    Bi = torch.randint(-1, 2, (N, K), generator=g)
    rows = np.arange(R * H)
    got = oracle_mod.ag_matmul_rows_e4m3([_bf16_bits(s.to(torch.bfloat16)) for s in si],
                                         _bf16_bits(Bi.to(torch.bfloat16)), rows)
    ref = (torch.cat(si) @ Bi.T).numpy().astype(np.float64)
    assert np.array_equal(oracle_mod.e4m3_to_f64(got), ref)
