/*
 * oracle.c -- plain, slow CPU oracle for the chunked AllGather x MatMul path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file.  It is used by tests/, by __graft_entry__.smoke() and by the
 * cpu_baseline / --impl reference legs of bench.py, and it shares no code,
 * header, table or helper with the CUDA library under tile_gather_comm_gb300/.
 *
 * Sources (web pages; each function cites the section it follows):
 *   [TG]  "CANN PTO-ISA TGATHER 指令深度解析：跨 Rank 行拼接 Gather 的实现原理与开发指南"
 *   [AGM] "Triton第四课：基于对称内存融合 AllGather 与 MatMul，提速1.56倍"
 *
 * Every function is the plain definition written out: no blocking, no
 * reordering of any output's arithmetic.  OpenMP only splits independent
 * output rows across threads; each output is computed by exactly the same
 * sequence of operations as in a single-threaded run.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (see oracle/__init__.py).
 *
 * Parity status: every function below is pinned by tests/test_oracle_pins.py
 * (closed forms, library special cases, integer-exact cases, brute force).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* TGATHER                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * [TG] §二 数学语义: with N ranks each holding src^(r) of shape
 * (D0, D1, D2, H, W), the root's destination satisfies
 *     dst[d0, d1, d2, r*H + i, j] = src^(r)[d0, d1, d2, i, j]
 * for r in [0,N), i in [0,H), j in [0,W); every dimension other than DIM_3 is
 * unchanged.  [TG] §7.2: dst DIM_3 may be larger than N*H, in which case only
 * the first N*H rows are written and the rest stay untouched -> dst_rows3.
 * [TG] §七 (7.4) and §6.3: empty data (D0*D1*D2*H == 0 or W == 0) returns at
 * once without touching dst.  [TG] §6.3: the CPU simulation copies element by
 * element; so does this oracle, as raw bytes of size `es` (no float
 * conversion, so NaN payloads and -0 survive).
 *
 * Arrays are dense row-major.  srcs is a host array of nranks pointers.
 * dst_rows3 = 0 means N*H.  Returns 0, or -1 if dst_rows3 < N*H or nranks<=0.
 */
int oracle_tgather(void *dst, const void *const *srcs, int nranks,
                   int64_t D0, int64_t D1, int64_t D2, int64_t H, int64_t W,
                   int64_t es, int64_t dst_rows3)
{
    if (nranks <= 0 || es <= 0)
        return -1;
    if (dst_rows3 == 0)
        dst_rows3 = (int64_t)nranks * H;
    if (dst_rows3 < (int64_t)nranks * H)
        return -1;
    if (D0 * D1 * D2 * H == 0 || W == 0)
        return 0;
    unsigned char *d = (unsigned char *)dst;
    for (int r = 0; r < nranks; ++r) {
        const unsigned char *s = (const unsigned char *)srcs[r];
        for (int64_t d0 = 0; d0 < D0; ++d0)
            for (int64_t d1 = 0; d1 < D1; ++d1)
                for (int64_t d2 = 0; d2 < D2; ++d2)
                    for (int64_t i = 0; i < H; ++i)
                        for (int64_t j = 0; j < W; ++j) {
                            int64_t slab = (d0 * D1 + d1) * D2 + d2;
                            int64_t src_idx = (slab * H + i) * W + j;
                            int64_t dst_idx = (slab * dst_rows3 + (int64_t)r * H + i) * W + j;
                            memcpy(d + dst_idx * es, s + src_idx * es, (size_t)es);
                        }
    }
    return 0;
}

/*
 * Strided form of the same formula ([TG] §7.3 and §8.1: sources are
 * GlobalTensor views with a shape and a stride, all sources sharing both).
 * Element (d0,d1,d2,i,j) of source r lives at srcs[r] + es * sum(idx * src_strides),
 * destination element (d0,d1,d2,r*H+i,j) at dst + es * sum(idx * dst_strides);
 * strides are in elements and non-negative.  Empty input returns at once.
 */
int oracle_tgather_strided(void *dst, const int64_t *dst_strides, const void *const *srcs,
                           const int64_t *src_strides, int nranks, int64_t D0, int64_t D1,
                           int64_t D2, int64_t H, int64_t W, int64_t es)
{
    if (nranks <= 0 || es <= 0)
        return -1;
    for (int k = 0; k < 5; ++k)
        if (dst_strides[k] < 0 || src_strides[k] < 0)
            return -1;
    if (D0 * D1 * D2 * H == 0 || W == 0)
        return 0;
    unsigned char *d = (unsigned char *)dst;
    for (int r = 0; r < nranks; ++r) {
        const unsigned char *s = (const unsigned char *)srcs[r];
        for (int64_t d0 = 0; d0 < D0; ++d0)
            for (int64_t d1 = 0; d1 < D1; ++d1)
                for (int64_t d2 = 0; d2 < D2; ++d2)
                    for (int64_t i = 0; i < H; ++i)
                        for (int64_t j = 0; j < W; ++j) {
                            int64_t so = d0 * src_strides[0] + d1 * src_strides[1] + d2 * src_strides[2] +
                                         i * src_strides[3] + j * src_strides[4];
                            int64_t row = (int64_t)r * H + i;
                            int64_t dd = d0 * dst_strides[0] + d1 * dst_strides[1] + d2 * dst_strides[2] +
                                         row * dst_strides[3] + j * dst_strides[4];
                            memcpy(d + dd * es, s + so * es, (size_t)es);
                        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* bf16 <-> fp32                                                             */
/* ------------------------------------------------------------------------ */

/* bf16 is the upper half of an IEEE-754 binary32 word, so widening is a shift. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Narrowing with IEEE-754 round-to-nearest, ties-to-even, written from the
 * definition: the 16 discarded bits are compared with the halfway point
 * 0x8000; adding 0x7FFF plus the lowest kept bit carries into the kept part
 * exactly when the discarded part is above half, or equal to half with an odd
 * kept part.  The carry may ripple into the exponent, which is the correct
 * rounding up to the next binade and, from the largest finite values, to Inf.
 * NaN is returned as a quiet NaN with its sign kept (IEEE-754 §6.2 requires a
 * NaN; the payload is implementation-chosen).
 */
uint16_t oracle_f32_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void oracle_f32_to_bf16_array(const float *x, uint16_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = oracle_f32_to_bf16_rne(x[i]);
}

/*
 * float32 -> float8 e4m3 ("fn" variant: 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities, S.1111.111 is NaN, so the largest finite
 * magnitude is 1.110b * 2^8 = 448), round to nearest even, saturating: every
 * finite or infinite input of magnitude >= 448 becomes +-448.  [AGM] section
 * MatMul 按需等待远端分片: the kernel takes FP8_OUTPUT and writes C as
 * float8_e4m3fn; the saturating conversion is the reading taken here.  Written
 * from the format definition: subnormals are k * 2^-9 (k = 0..7), normals
 * (1 + m/8) * 2^e with e in [-6, 8].  NaN -> 0x7F with the sign kept.
 */
uint8_t oracle_f32_to_e4m3_sat(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    const uint8_t sign = (uint8_t)((u >> 24) & 0x80u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint8_t)(sign | 0x7Fu);
    double a = fabs((double)f);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7Eu);
    if (a < ldexp(1.0, -6)) {                 /* subnormal range: multiples of 2^-9 */
        double q = a * 512.0;                  /* exact: a is a float, 512 a power of 2 */
        double k = floor(q);
        double rem = q - k;
        if (rem > 0.5 || (rem == 0.5 && fmod(k, 2.0) != 0.0))
            k += 1.0;
        /* k == 8 is the smallest normal 2^-6, whose encoding is 0x08 as well */
        return (uint8_t)(sign | (uint8_t)k);
    }
    int e;
    double m = frexp(a, &e);                   /* a = m * 2^e, m in [0.5, 1) */
    e -= 1;                                     /* a = (2m) * 2^e, 2m in [1, 2) */
    double frac = (2.0 * m - 1.0) * 8.0;       /* mantissa in units of 1/8, exact */
    double k = floor(frac);
    double rem = frac - k;
    if (rem > 0.5 || (rem == 0.5 && fmod(k, 2.0) != 0.0))
        k += 1.0;
    if (k == 8.0) {
        k = 0.0;
        e += 1;
    }
    if (e > 8 || (e == 8 && k > 6.0))
        return (uint8_t)(sign | 0x7Eu);        /* rounded past 448: saturate */
    return (uint8_t)(sign | (uint8_t)(((e + 7) << 3) | (int)k));
}

void oracle_f32_to_e4m3_array(const float *x, uint8_t *y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        y[i] = oracle_f32_to_e4m3_sat(x[i]);
}

/* ------------------------------------------------------------------------ */
/* AllGather then MatMul                                                     */
/* ------------------------------------------------------------------------ */

/*
 * One output: C[m][n] = bf16_rne( sum_{k=0}^{K-1} a[m][k] * B[n][k] ), the sum
 * taken in fp32 in increasing k.  B is stored (N, K) row-major: [AGM]
 * "对称内存如何打通GPU间访问" builds b as randn(k, n).T.contiguous(), i.e. the
 * GEMM is C = a * B^T with both operands K-contiguous.  bf16*bf16 products
 * are exact in fp32 (8+8 significand bits), so the only roundings are the K
 * fp32 additions and the final bf16 rounding.
 */
static uint16_t dot_row(const uint16_t *arow, const uint16_t *brow, int64_t K)
{
    float acc = 0.0f;
    for (int64_t k = 0; k < K; ++k)
        acc += oracle_bf16_to_f32(arow[k]) * oracle_bf16_to_f32(brow[k]);
    return oracle_f32_to_bf16_rne(acc);
}

/*
 * [AGM] "为什么要融合 AllGather 与 MatMul": the unfused reference is "gather
 * every shard, then run the MatMul on the concatenated tensor".  [AGM]
 * "融合后的流水线": once every chunk is consumed, the fused result equals that
 * of a complete AllGather followed by MatMul.  So the oracle for the fused
 * path is exactly this:
 *   a = TGATHER(a_shards) with D0=D1=D2=1, H = M/R, W = K      -> (M, K)
 *   C = a * B^T, fp32 accumulation, bf16 output               -> (M, N)
 * a_out receives `a` (may be NULL).  Requires M % R == 0.  Returns 0 / -1.
 */
int oracle_ag_matmul(const uint16_t *const *a_shards, int R, const uint16_t *B,
                     uint16_t *C, uint16_t *a_out, int64_t M, int64_t K, int64_t N)
{
    if (R <= 0 || M < 0 || K < 0 || N < 0 || M % R != 0)
        return -1;
    if (M == 0 || N == 0)
        return 0;
    uint16_t *a = a_out;
    if (a == NULL)
        return -1;
    oracle_tgather(a, (const void *const *)a_shards, R, 1, 1, 1, M / R, K, 2, 0);
    int64_t m;
#pragma omp parallel for schedule(dynamic, 1)
    for (m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            C[m * N + n] = dot_row(a + m * K, B + n * K, K);
    return 0;
}

/*
 * The same outputs for a chosen list of rows only (the rows are computed one
 * by one, as in oracle_ag_matmul).  Row m of `a` is located through the
 * TGATHER closed form with H = M/R: it is row (m mod H) of shard (m div H).
 * C_rows is (nrows, N).
 */
int oracle_ag_matmul_rows(const uint16_t *const *a_shards, int R, const uint16_t *B,
                          int64_t M, int64_t K, int64_t N,
                          const int64_t *rows, int64_t nrows, uint16_t *C_rows)
{
    if (R <= 0 || M % R != 0)
        return -1;
    int64_t H = M / R;
    for (int64_t t = 0; t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= M)
            return -1;
    int64_t t;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < nrows; ++t) {
        int64_t m = rows[t];
        const uint16_t *arow = a_shards[m / H] + (m % H) * K;
        for (int64_t n = 0; n < N; ++n)
            C_rows[t * N + n] = dot_row(arow, B + n * K, K);
    }
    return 0;
}

/*
 * The same sampled rows with C written as float8 e4m3 (the FP8_OUTPUT variant
 * of [AGM]'s kernel): identical fp32 sums, converted by oracle_f32_to_e4m3_sat.
 */
int oracle_ag_matmul_rows_e4m3(const uint16_t *const *a_shards, int R, const uint16_t *B,
                               int64_t M, int64_t K, int64_t N,
                               const int64_t *rows, int64_t nrows, uint8_t *C_rows)
{
    if (R <= 0 || M % R != 0)
        return -1;
    int64_t H = M / R;
    for (int64_t t = 0; t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= M)
            return -1;
    int64_t t;
#pragma omp parallel for schedule(dynamic, 1)
    for (t = 0; t < nrows; ++t) {
        int64_t m = rows[t];
        const uint16_t *arow = a_shards[m / H] + (m % H) * K;
        for (int64_t n = 0; n < N; ++n) {
            float acc = 0.0f;
            const uint16_t *brow = B + n * K;
            for (int64_t k = 0; k < K; ++k)
                acc += oracle_bf16_to_f32(arow[k]) * oracle_bf16_to_f32(brow[k]);
            C_rows[t * N + n] = oracle_f32_to_e4m3_sat(acc);
        }
    }
    return 0;
}

/*
 * [AGM] "融合后的流水线" and "数据搬运与细粒度同步": the gather is cut into
 * communication blocks of `cb` rows (S = (M/R)/cb per rank, block id
 * c = src_rank * S + split_id).  The producer copies one block into the
 * aggregate buffer and publishes it; the MatMul consumes the output rows of
 * that block as soon as it is published.  This oracle walks the blocks in the
 * given release order, copies block c into `a`, then computes the C rows of
 * block c.  Its result must equal oracle_ag_matmul bit for bit, which is the
 * pages' claim that chunked consumption equals gather-then-MatMul.
 * `order` must be a permutation of [0, M/cb); returns -1 otherwise.
 */
int oracle_ag_matmul_chunked(const uint16_t *const *a_shards, int R, const uint16_t *B,
                             uint16_t *C, uint16_t *a_out, int64_t M, int64_t K, int64_t N,
                             int64_t cb, const int64_t *order, int64_t norder)
{
    if (R <= 0 || cb <= 0 || M % R != 0 || (M / R) % cb != 0 || a_out == NULL)
        return -1;
    int64_t H = M / R, S = H / cb, nblocks = M / cb;
    if (norder != nblocks)
        return -1;
    /* order must be a permutation */
    for (int64_t p = 0; p < norder; ++p) {
        if (order[p] < 0 || order[p] >= nblocks)
            return -1;
        for (int64_t q = 0; q < p; ++q)
            if (order[q] == order[p])
                return -1;
    }
    for (int64_t p = 0; p < norder; ++p) {
        int64_t c = order[p];
        int64_t src_rank = c / S, split_id = c % S;
        int64_t row0 = src_rank * H + split_id * cb;
        /* producer: copy block c of shard src_rank into a */
        memcpy(a_out + row0 * K, a_shards[src_rank] + split_id * cb * K,
               (size_t)(cb * K) * sizeof(uint16_t));
        /* consumer: the output rows that depend only on block c */
        int64_t m;
#pragma omp parallel for schedule(dynamic, 1)
        for (m = row0; m < row0 + cb; ++m)
            for (int64_t n = 0; n < N; ++n)
                C[m * N + n] = dot_row(a_out + m * K, B + n * K, K);
    }
    return 0;
}

/* Threads the OpenMP runtime will use (1 when built without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
void oracle_set_num_threads(int n) { omp_set_num_threads(n); }
#else
int oracle_num_threads(void) { return 1; }
void oracle_set_num_threads(int n) { (void)n; }
#endif
