/*
 * tgc.h -- C ABI of libtgc.so: TGATHER row-concat gather and chunked
 * AllGather fused with a bf16 MatMul, for one sm_103a GPU.
 *
 * Sources (web pages):
 *   [TG]  "CANN PTO-ISA TGATHER 指令深度解析：跨 Rank 行拼接 Gather 的实现原理与开发指南"
 *   [AGM] "Triton第四课：基于对称内存融合 AllGather 与 MatMul，提速1.56倍"
 *
 * Conventions for every entry point
 *   - Pointers named d_* or documented as "device" are device addresses in the
 *     current CUDA device; the caller owns them.  Arrays of source pointers
 *     (srcs, a_shards) are HOST arrays of device pointers; they are copied into
 *     kernel parameters, so the host array may be freed after the call returns.
 *   - All work is enqueued on `stream` (cudaStream_t; NULL = legacy default
 *     stream) and is asynchronous unless stated; device buffers must stay alive
 *     until the stream has passed the call.
 *   - Tensors are dense and row-major (C order).
 *   - Argument errors are reported synchronously as a negative tgc_status
 *     before anything is enqueued.  Errors detected on the device (a bounded
 *     wait that expired) are written to a device status word; the synchronous
 *     entry points read it back and return it.
 *   - The library keeps no per-problem state between calls: tensor
 *     descriptors are encoded per call on the host, and what it keeps per
 *     device (the allocating entry point's memory pool, the copy-engine
 *     mode's side streams, kernel attributes and SM counts) does not depend
 *     on the problem.  It is safe to call from several host threads.
 *   - A "virtual rank" is one of `nranks` separate allocations in the same
 *     GPU's memory standing for the shard a rank holds ([AGM] section
 *     对称内存如何打通GPU间访问: every rank holds a_shard of shape (M/W, K)).
 */
#ifndef TGC_H
#define TGC_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TGC_MAX_RANKS 64

typedef enum tgc_status {
    TGC_OK = 0,
    TGC_ERR_INVALID_ARG = -1,  /* null pointer, bad count or shape, bad mode   */
    TGC_ERR_DTYPE = -2,        /* unknown dtype                               */
    TGC_ERR_ALIGN = -3,        /* pointer or row pitch misaligned for the path */
    /* -4 is not used: the persistent grids are sized from the occupancy the
       device reports, and no kernel needs more of its CTAs resident at once
       than that (copy work is handed out by tickets), so a grid that cannot
       launch is a launch error (TGC_ERR_CUDA). */
    TGC_ERR_CUDA = -5,         /* a CUDA call failed: see tgc_last_cuda_error */
    TGC_ERR_TIMEOUT = -6,      /* a bounded device wait expired               */
    TGC_ERR_ABORTED = -7,      /* the kernel stopped because another CTA timed out */
    TGC_ERR_WORKSPACE = -8,    /* workspace missing or too small              */
    TGC_ERR_TOO_LARGE = -9     /* problem exceeds tgc_ag_matmul_noalloc's fixed scratch */
} tgc_status;

/* Element types.  TGATHER only uses the element size ([TG] §7.1: source,
 * destination and staging tile share one type; the copy is type-agnostic). */
typedef enum tgc_dtype {
    TGC_U8 = 0, TGC_I8 = 1, TGC_F16 = 2, TGC_BF16 = 3,
    TGC_I32 = 4, TGC_F32 = 5, TGC_I64 = 6, TGC_F64 = 7
} tgc_dtype;

/* ------------------------------------------------------------------------ */
/* TGATHER                                                                   */
/* ------------------------------------------------------------------------ */

/*
 * tgc_tgather -- [TG] §二 数学语义:
 *     dst[d0, d1, d2, r*H + i, j] = srcs[r][d0, d1, d2, i, j]
 *     for r in [0, nranks), i in [0, H), j in [0, W), every (d0, d1, d2).
 *
 * dst     device, (D0, D1, D2, nranks*H, W) elements of `dtype`, written.
 * srcs    host array of nranks device pointers, each (D0, D1, D2, H, W),
 *         read.  All sources share shape and layout ([TG] §7.3).
 * dtype   element type (only its size matters).
 * Alignment: every pointer must be aligned to the element size.  Any H and W
 * are accepted (non-tile-multiple tails are handled; [TG] §7.4's divisibility
 * rule for static tiles does not apply).
 * Empty input (any of D0, D1, D2, H, W == 0) returns TGC_OK and writes
 * nothing ([TG] §七: empty data returns before any transfer).
 * Errors: TGC_ERR_INVALID_ARG (nranks not in [1, TGC_MAX_RANKS], negative
 * extent, null pointer, or a destination of 2^62 bytes or more),
 * TGC_ERR_DTYPE, TGC_ERR_ALIGN, TGC_ERR_CUDA.
 * Asynchronous on `stream`.
 */
int tgc_tgather(void *dst, const void *const *srcs, int nranks,
                int64_t D0, int64_t D1, int64_t D2, int64_t H, int64_t W,
                tgc_dtype dtype, cudaStream_t stream);

/*
 * tgc_tgather_strided -- the same gather on strided views ([TG] §7.3: every
 * source is a view with one shape and one stride, shared by all sources;
 * §8.1: GlobalTensor<T, Shape<5>, Stride, Layout::ND>):
 *     dst[d0, d1, d2, r*H + i, j] = srcs[r][d0, d1, d2, i, j]
 * Element (d0,d1,d2,i,j) of a source lives at
 *     srcs[r] + es * (d0*ss[0] + d1*ss[1] + d2*ss[2] + i*ss[3] + j*ss[4]),
 * destination element (d0,d1,d2,row,j) at
 *     dst + es * (d0*ds[0] + d1*ds[1] + d2*ds[2] + row*ds[3] + j*ds[4]),
 * with ss = src_strides, ds = dst_strides: host arrays of 5 element strides,
 * each >= 0.  Only the view is written; memory between its rows and columns is
 * left as it is.  The destination view must not overlap itself or a source
 * (undefined otherwise).  Rows that are contiguous in both source and
 * destination (ss[4] == ds[4] == 1) are copied with the widest vector every
 * start address and stride allows; otherwise element by element.  Errors and
 * the empty-input rule as tgc_tgather; a negative stride, or a view whose last
 * element lies 2^62 bytes or more from its base, is TGC_ERR_INVALID_ARG.
 * Asynchronous on `stream`.
 */
int tgc_tgather_strided(void *dst, const int64_t *dst_strides, const void *const *srcs,
                        const int64_t *src_strides, int nranks,
                        int64_t D0, int64_t D1, int64_t D2, int64_t H, int64_t W,
                        tgc_dtype dtype, cudaStream_t stream);

/*
 * Extended TGATHER.  Zero-initialise the struct (`tgc_tgather_args a = {0};`,
 * `tgc_tgather_args a{};` in C++):
 * every field below means its default at 0 or a null pointer.  Adds:
 *   dst_rows3  dst's DIM_3; 0 means nranks*H.  [TG] §7.2: it may exceed
 *              nranks*H, in which case only the first nranks*H rows of each
 *              (d0, d1, d2) slab are written and the rest are left unchanged.
 *   progress   optional device uint32 array of nranks*S entries,
 *              S = ceil(H / chunk_rows).  Entry c = r*S + s refers to rows
 *              [s*chunk_rows, min((s+1)*chunk_rows, H)) of rank r in every
 *              slab.  When all those rows are in dst, the kernel stores
 *              `epoch` there with a gpu-scope release ([AGM] section
 *              数据搬运与细粒度同步: one progress entry per (src_rank,
 *              split_id) at offset src_rank*splits_per_rank + split_id; the
 *              data must be visible before the flag).  A reader that loads the
 *              entry with gpu-scope acquire and sees `epoch` may read the rows.
 *   counters   device uint32 array of nranks*S entries, required with
 *              progress; must be zero on entry and is zero again when the
 *              kernel ends.
 *   chunk_rows rows per progress chunk (> 0 when progress is given).
 *   epoch      the value published; must differ from every value the
 *              progress entries hold on entry ([AGM] same section, last
 *              paragraph: versioned progress values keep a previous round's
 *              flag from passing as a new one).
 *   spin_timeout_ns  (with progress) bound on the kernel's one wait, 0 = 10 s.
 *              With up to 512 chunks (nranks*S), the copying blocks count each
 *              piece of a chunk and never wait; one block publishes every chunk
 *              whose count is complete, and waits for the counts.  Those always
 *              complete while the GPU runs the grid, but should a chunk's count
 *              not complete within this bound (for example, counters that were
 *              not zero on entry), its entry receives ~epoch instead of epoch
 *              (an error mark no reader takes for the flag) and its counter is
 *              left as it is; its rows are still copied.  With more chunks the
 *              block whose count completes a chunk publishes it, nothing waits,
 *              and this bound is unused.
 */
typedef struct tgc_tgather_args {
    void *dst;
    const void *const *srcs;
    int nranks;
    int64_t D0, D1, D2, H, W;
    tgc_dtype dtype;
    int64_t dst_rows3;
    uint32_t *progress;
    uint32_t *counters;
    int64_t chunk_rows;
    uint32_t epoch;
    cudaStream_t stream;
    uint64_t spin_timeout_ns;
} tgc_tgather_args;

int tgc_tgather_ex(const tgc_tgather_args *args);

/* ------------------------------------------------------------------------ */
/* AllGather fused with MatMul                                               */
/* ------------------------------------------------------------------------ */

/*
 * tgc_ag_matmul -- [AGM]: gather nranks shards along M into `a` and compute
 *     C = a * B^T   (a: (M, K), B stored (N, K), C: (M, N); bf16 in and out,
 *                    fp32 accumulation)
 * with the gather cut into communication blocks of comm_block_rows rows, each
 * published through a progress flag, and the MatMul tiles consuming each
 * block as soon as its flag is set ([AGM] sections 融合后的流水线 and
 * MatMul 按需等待远端分片).  The result equals gather-then-MatMul.  Runs as
 * tgc_ag_matmul_ex with mode FUSED, rank 0, tile order TGC_PIVOT_AUTO.
 *
 * a_shards        host array of nranks device pointers, each (M/nranks, K)
 *                 bf16, 16-byte aligned.
 * B               device (N, K) bf16, 16-byte aligned.
 * C               device (M, N) bf16, written.
 * comm_block_rows must divide M/nranks.
 * Requirements: M % nranks == 0, K % 8 == 0 and N % 8 == 0 (16-byte rows for
 * TMA), K > 0.
 * Temporaries (`a`, progress flags, workspace) are allocated stream-ordered
 * from a memory pool the library creates per device (cudaMallocFromPoolAsync)
 * and freed the same way.  The pool keeps up to TGC_POOL_KEEP_BYTES of freed
 * memory mapped for the next call and returns the rest to the device when
 * the stream synchronizes, so a large call does not pin its `a` (M*K*2 bytes)
 * for the life of the process.  This entry point synchronizes `stream` before
 * returning so that it can report a device-side error.
 * M == 0 or N == 0: returns TGC_OK, nothing written.
 */
int tgc_ag_matmul(const void *const *a_shards, int nranks, const void *B, void *C,
                  int64_t M, int64_t K, int64_t N, int64_t comm_block_rows,
                  cudaStream_t stream);
#define TGC_POOL_KEEP_BYTES ((uint64_t)256 << 20)

typedef enum tgc_mode {
    TGC_MODE_FUSED = 0,    /* one kernel: copy blocks into a_out + flag-waiting GEMM */
    TGC_MODE_UNFUSED = 1,  /* tgather kernel into a_out, then the GEMM kernel on a_out */
    TGC_MODE_MM_ONLY = 2,  /* GEMM kernel on a_out as it is (every block taken as ready) */
    TGC_MODE_FUSED_CE = 3  /* copy engines fill a_out block by block on a library-owned
                              side stream, each block followed by a stream write of its
                              progress flag; the flag-waiting GEMM kernel runs at the same
                              time with no producer warps ([AGM] section
                              数据搬运与细粒度同步: the backend stream copies every
                              (src_rank, split_id) chunk and then stream_write_value32's
                              its progress entry).  delay_ns is ignored and READY_QUEUE
                              behaves as PAGE in this mode.  The runtime may carry a
                              device-to-device cudaMemcpyAsync out with a kernel of its
                              own rather than a copy engine; that kernel must then find
                              room on SMs the persistent GEMM kernel already occupies.
                              So this mode always runs 256-column tiles (256 threads
                              and about 27 K registers per SM, leaving room for such a
                              copy kernel beside each GEMM CTA); tile_n = 512 is
                              TGC_ERR_INVALID_ARG here.  Should the copies still find
                              no room, the GEMM's flag waits would expire and the call
                              would return TGC_ERR_TIMEOUT (after spin_timeout_ns)
                              instead of a result: measured with 512-column tiles,
                              whose consumer kernel takes 168 registers x 384 threads
                              of each SM's 65536. */
} tgc_mode;

/*
 * Tile order.  Tiles are first grouped along M in groups of `group_m` tile
 * rows (the usual L2-friendly swizzle), then pid_m is rotated
 * ([AGM] section 融合后的流水线: the pivot is applied after the swizzle):
 *   PAGE : pid_m = (pid_m + floor(rank*comm_block_rows / BM)) % num_pid_m,
 *          the page's (pid_m + NUM_PID_M_PER_COMM_BLOCK*RANK) % num_pid_m
 *          whenever BM divides comm_block_rows;
 *   SHARD: pid_m = (pid_m + floor(rank*(M/nranks) / BM)) % num_pid_m, which
 *          starts every rank on its own shard;
 *   NONE : no rotation.
 *   READY_QUEUE (FUSED only; the other modes treat it as NONE): the tile rows
 *          lying entirely inside the caller's shard come first (they wait for
 *          nothing); every other tile row is handed out in the order in which
 *          its data becomes complete -- the producer that completes a tile row
 *          appends it to a device ring, and the i-th position after the local
 *          prefix takes the i-th row appended ([AGM] section 融合后的流水线:
 *          tiles are processed "in their ready order").
 * The order only changes which tile runs when; C does not depend on it.
 */
typedef enum tgc_pivot {
    TGC_PIVOT_PAGE = 0,
    TGC_PIVOT_SHARD = 1,
    TGC_PIVOT_NONE = 2,
    TGC_PIVOT_READY_QUEUE = 3,
    TGC_PIVOT_AUTO = 4  /* the library's choice.  FUSED: READY_QUEUE when the caller passes
                           a release `order` and the band raster is in use (blocks then
                           arrive out of tile order while rows are walked one at a time),
                           PAGE otherwise (with the default release order the two orders
                           coincide).  FUSED_CE: PAGE.  UNFUSED and MM_ONLY: NONE (no tile
                           waits there).  The order tgc_ag_matmul and
                           tgc_ag_matmul_noalloc use. */
} tgc_pivot;

/* Element type of C.  F8E4M3: float8 e4m3 ("fn": bias 7, no infinities,
 * largest finite 448), round to nearest even and saturating at +-448 ([AGM]
 * section MatMul 按需等待远端分片: the kernel's FP8_OUTPUT argument writes C
 * as float8_e4m3fn).  Needs N % 16 == 0. */
typedef enum tgc_out_format {
    TGC_OUT_BF16 = 0,
    TGC_OUT_F8E4M3 = 1
} tgc_out_format;

/*
 * Extended AllGather-MatMul.  Zero-initialise the struct, as for
 * tgc_tgather_args; each field's description below says what 0 or a null
 * pointer means (pivot 0 is TGC_PIVOT_PAGE, not the plain call's AUTO).
 * Fields beyond tgc_ag_matmul's:
 *   a_out        device (M, K) bf16: the gathered A.  FUSED and UNFUSED write
 *                it completely (local shard included); MM_ONLY reads it.
 *   rank         the calling virtual rank, 0 <= rank < nranks.  Tiles whose
 *                rows lie inside shard `rank` read a_shards[rank] directly
 *                and wait for nothing; all other tiles wait for the flags of
 *                every block they cover and read a_out.
 *   progress     device uint32 array of M/comm_block_rows entries; block
 *                c = src_rank*S + split_id, S = (M/nranks)/comm_block_rows.
 *                FUSED stores `epoch` into entry c with a gpu-scope release
 *                once block c is in a_out.  Unused by UNFUSED/MM_ONLY.
 *   epoch        must differ from every value progress holds on entry.
 *   order        optional HOST int32 array of n_order distinct block ids in
 *                [0, M/comm_block_rows): the order in which the producer
 *                copies and releases blocks (copied into the workspace).
 *                NULL: the order in which the tile schedule first reaches the
 *                blocks' rows, the caller's own shard last (its tiles read the
 *                shard directly).  Blocks missing from `order` are never
 *                released: their tiles wait until spin_timeout_ns and the call
 *                fails with TGC_ERR_TIMEOUT (host-side fault injection).
 *   delay_ns     optional HOST uint32 array, one entry per block: the
 *                producer that completes a block busy-waits that many ns on
 *                %globaltimer before it publishes the block (injected arrival
 *                skew).
 *   spin_timeout_ns  limit for every device wait; 0 = 2 s.
 *   group_m      tile rows per swizzle group of the group raster; 0 = default (8).
 *   band_n       tile raster.  > 0: band raster -- the tiles are taken in bands
 *                of band_n tile columns, each band walking the tile rows in
 *                order (the rank rotation still applies to the rows), which
 *                keeps the band's columns of B in L2 and asks for the rows of
 *                `a` in the order the producer publishes them; < 0: group
 *                raster (group_m tile rows per group, column-major inside a
 *                group: the page's GROUP_SIZE_M swizzle); 0: the library's
 *                choice -- for FUSED and FUSED_CE, bands of TGC_DEFAULT_BAND_N
 *                columns when one shard holds fewer whole tile rows (256 rows
 *                each) than group_m, else the group raster; the group raster
 *                for UNFUSED and MM_ONLY.  Band widths count 256-column
 *                blocks whatever the tile width.
 *   tile_n       output columns of a GEMM tile: 256 (two TMEM accumulators per
 *                CTA, so a tile's epilogue overlaps the next tile's MMAs) or 512
 *                (two 256-column MMA blocks side by side on one accumulator:
 *                a quarter fewer operand bytes per flop and less power, but the
 *                epilogue no longer overlaps); 0 = the library's choice: 512
 *                when K >= 8192 and one shard holds at least group_m tile rows
 *                (the group raster case), else 256; always 256 for FUSED_CE (see
 *                TGC_MODE_FUSED_CE), where 512 is TGC_ERR_INVALID_ARG.  Other
 *                values are TGC_ERR_INVALID_ARG.  The result does not depend on it: every
 *                element of C is the same chain of 16-deep MMA steps over K.
 *   grid         persistent CTAs (used in pairs); 0 = every SM.
 *   workspace    device memory of tgc_ag_matmul_workspace_bytes() bytes,
 *                128-byte aligned, zero-filled once by the caller before first
 *                use; every call that succeeds leaves its counters and status
 *                zeroed again (after an error, zero it again).  Required by
 *                FUSED; optional otherwise.
 *   d_status     optional device int32, zeroed by the call, then set by the
 *                kernel to a tgc_status code if a device wait fails.  When
 *                NULL the status word lives in the workspace (FUSED) or is
 *                not kept (UNFUSED / MM_ONLY without workspace).
 *   sync         nonzero: synchronize `stream` and return the device status.
 *   out_format   element type of C (tgc_out_format; 0 = bf16).
 *   trace        optional device uint64 array of trace_words words: per
 *                launched CTA, TGC_TRACE_WORDS words of %globaltimer stamps
 *                and signal-wait totals, laid out as the TGC_TRACE_* indices
 *                below (CTA i at word i*TGC_TRACE_WORDS).  NULL records
 *                nothing.  The page's evaluation advice asks for the time
 *                spent waiting on signals to be reported separately.
 *   trace_words  words of `trace`.  The kernels launch CTAs in pairs, at
 *                most one per SM, and no more than max(grid, 2) when grid is
 *                nonzero, so with a trace this must be at least
 *                TGC_TRACE_WORDS * min(max(grid, 2), SM count of the current
 *                device) -- the SM count when grid is 0; a smaller value is
 *                TGC_ERR_INVALID_ARG.
 * Calls that share a workspace or progress array must not overlap on the GPU.
 * With sync = 0 and without `order` / `delay_ns` a call can be captured in a
 * CUDA graph (make one uncaptured call first on the device, so that kernel
 * attributes are set outside the capture).  The epoch is fixed in the graph,
 * so capture a reset of the progress entries (for instance a memset to 0)
 * before the call: each replay then publishes its blocks afresh.
 */
typedef struct tgc_ag_matmul_args {
    const void *const *a_shards;
    int nranks;
    const void *B;
    void *C;
    void *a_out;
    int64_t M, K, N;
    int64_t comm_block_rows;
    int rank;
    tgc_mode mode;
    tgc_pivot pivot;
    uint32_t *progress;
    uint32_t epoch;
    const int32_t *order;
    int64_t n_order;
    const uint32_t *delay_ns;
    uint64_t spin_timeout_ns;
    int group_m;
    int grid;
    void *workspace;
    size_t workspace_bytes;
    int32_t *d_status;
    int sync;
    cudaStream_t stream;
    uint64_t *trace;
    tgc_out_format out_format;
    size_t trace_words;
    int band_n;
    int tile_n;
} tgc_ag_matmul_args;

int tgc_ag_matmul_ex(const tgc_ag_matmul_args *args);

#define TGC_DEFAULT_BAND_N 16

/* Per-CTA trace words (times in ns of %globaltimer). */
#define TGC_TRACE_WORDS 16
#define TGC_TRACE_START 0        /* CTA start                                        */
#define TGC_TRACE_WAIT_NS 1      /* tile scheduler: time spent waiting on flags/ring */
#define TGC_TRACE_WAITED_TILES 2 /* tiles that found their data not yet published    */
#define TGC_TRACE_COPY_FIRST 3   /* producer: first piece handed out                 */
#define TGC_TRACE_COPY_LAST 4    /* producer: last piece of this CTA retired         */
#define TGC_TRACE_PIECES 5       /* producer: pieces copied by this CTA              */
#define TGC_TRACE_END 6          /* epilogue: last tile of this CTA stored           */
#define TGC_TRACE_TILES 7        /* tiles computed by this CTA                       */
#define TGC_TRACE_MMA_STAGE_NS 8 /* MMA issuer: time waiting for operand stages     */
#define TGC_TRACE_MMA_ACC_NS 9   /* MMA issuer: time waiting for a free accumulator  */
#define TGC_TRACE_EPI_WAIT_NS 10 /* epilogue (first warp): time waiting for results  */
#define TGC_TRACE_LOAD_STALL_NS 11 /* TMA issuer: time waiting for free stages       */
#define TGC_TRACE_PIECE_BYTES 12 /* producer: copy piece size chosen for the call    */
#define TGC_TRACE_COPY_WARPS 13  /* producer: warps of this CTA that took pieces     */

/*
 * The tile order and raster a call to tgc_ag_matmul_ex with these arguments runs,
 * with TGC_PIVOT_AUTO, band_n = 0 and tile_n = 0 resolved as described above: pivot
 * is PAGE, SHARD, NONE or READY_QUEUE; band_n > 0 means the band raster of bands of
 * band_n x 256 columns, 0 the group raster of group_m tile rows; tile_n is 256 or 512.  The arguments are checked as
 * tgc_ag_matmul_ex checks them (the same negative status for invalid ones), but
 * nothing is enqueued and no pointer is dereferenced: placeholders will do.  Needs
 * no GPU.
 */
typedef struct tgc_ag_matmul_plan_t {
    tgc_pivot pivot;
    int band_n;
    int group_m;
    int tile_n;
} tgc_ag_matmul_plan_t;

int tgc_ag_matmul_plan(const tgc_ag_matmul_args *args, tgc_ag_matmul_plan_t *out);

/*
 * tgc_ag_matmul_noalloc -- the fused AllGather-MatMul of tgc_ag_matmul with
 * no device allocation.  No counterpart on the pages: this is a library
 * convenience for callers that cannot call cudaMalloc -- for instance code
 * running under a memory manager that owns all device memory and forbids raw
 * allocations, or a latency-critical path on which no allocation may happen
 * after start-up.
 *
 * Arguments as in tgc_ag_matmul, plus
 *   a_out   device (M, K) bf16 output: the gathered A (as in tgc_ag_matmul_ex).
 * The scratch the fused kernel needs (status word, ticket dispenser, per-block
 * counters and progress flags, per-tile-row counters and ready ring) lives in
 * a fixed array of TGC_NOALLOC_SCRATCH_BYTES of device memory declared
 * statically in the library, one per GPU that loads the library and held
 * until the process exits.  Limits, both checked before anything is
 * enqueued, TGC_ERR_TOO_LARGE otherwise:
 *   - M / comm_block_rows <= TGC_NOALLOC_MAX_BLOCKS comm blocks;
 *   - the scratch bytes fit the array: 16 bytes per comm block (counter,
 *     flag, two host-array copies) plus 12 bytes per 256-row tile row of M
 *     plus a few hundred bytes of fixed fields, each region rounded up to
 *     128 bytes.  With 2048 blocks this caps M at about 700,000 rows.
 * Each call looks up the array's device address on the current device
 * (cudaGetSymbolAddress, which allocates nothing), so the address stays
 * right after a device reset; make the first call on a device before any
 * stream capture, since that lookup may load the library's module.
 * Every call on a device shares the same array, which keeps the previous
 * call's contents: each call clears the part it uses (cudaMemsetAsync on
 * `stream`) before launching.  Calls that overlap on the GPU -- on different
 * streams or from different host threads -- race on the array and must not be
 * issued.  Calls no cudaMalloc, cudaFree or other allocating routine.
 * Synchronizes `stream` and returns the device status, like tgc_ag_matmul.
 */
#define TGC_NOALLOC_MAX_BLOCKS 2048
#define TGC_NOALLOC_SCRATCH_BYTES 65536
int tgc_ag_matmul_noalloc(const void *const *a_shards, int nranks, const void *B, void *C, void *a_out,
                          int64_t M, int64_t K, int64_t N, int64_t comm_block_rows,
                          cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Ranks in separate processes                                               */
/* ------------------------------------------------------------------------ */

/*
 * [AGM] section 对称内存如何打通GPU间访问: every rank allocates its a_shard (M/W, K) in
 * memory the other ranks can address, and each rank's producer copies the other ranks'
 * shards into its own `a` ([AGM] section 数据搬运与细粒度同步).  With one process per
 * rank, a rank exports the device buffer holding its shard as an IPC handle
 * (tgc_ipc_export), the ranks exchange the handles by any host transport, and each
 * rank opens the others' (tgc_ipc_open) to obtain device pointers it passes, in rank
 * order with its own shard's pointer at its own index, as a_shards[] to
 * tgc_ag_matmul_ex with `rank` set to itself.  Every rank computes C = a * B_r^T with
 * its own B_r and publishes its own progress flags; nothing is written into another
 * rank's memory.  Peer bytes are moved only by the kernels' own loads and stores (the
 * register-copy producer of FUSED, the TGATHER kernel of UNFUSED) or, in FUSED_CE, by
 * device-to-device copies; tile loads (TMA) read the caller's own shard, `a` and B,
 * all local.  The library build that copies with bulk asynchronous copies
 * (TGC_COPY_LSU=0) would read peer memory with them and must not be used with peer
 * pointers.
 *
 * The caller orders the ranks: a peer's shard must be complete before a rank's call
 * is enqueued (for instance: every rank synchronizes its writes, then a barrier), and
 * must not be freed or rewritten until every rank's call has completed.
 */
typedef struct tgc_ipc_handle {
    unsigned char bytes[64];  /* the CUDA IPC handle of the allocation holding the buffer */
    uint64_t offset;          /* byte offset of the buffer inside that allocation          */
} tgc_ipc_handle;

/* Fills *out for the device buffer at d_ptr (any address inside an allocation made
 * with cudaMalloc, in the current device).  TGC_ERR_INVALID_ARG for null arguments,
 * TGC_ERR_CUDA if the runtime cannot export the allocation (for instance memory from
 * a virtual-memory or pool allocator). */
int tgc_ipc_export(const void *d_ptr, tgc_ipc_handle *out);
/* Maps another process's exported buffer into this process (current device; peer
 * access enabled lazily when it lives on another device) and returns its address in
 * *d_ptr_out.  A handle exported by this same process cannot be opened here. */
int tgc_ipc_open(const tgc_ipc_handle *h, void **d_ptr_out);
/* Unmaps a buffer opened by tgc_ipc_open: d_ptr as returned there, h as passed there. */
int tgc_ipc_close(void *d_ptr, const tgc_ipc_handle *h);

/* Bytes of workspace tgc_ag_matmul_ex needs for this problem (>= 256). */
size_t tgc_ag_matmul_workspace_bytes(int nranks, int64_t M, int64_t K, int64_t N,
                                     int64_t comm_block_rows);

/*
 * Host-side copy of the tile schedule the GEMM kernels run (the same code the
 * device uses).  A tile is BM x tile_n outputs (BM from tgc_gemm_tile_shape;
 * tile_n 256 or 512, as tgc_ag_matmul_plan reports for a call), computed by one
 * persistent cluster (a pair of CTAs on two SMs).  Writes, for cluster `cta` of
 * `grid` persistent clusters, the sequence of (pid_m, pid_n) pairs it processes
 * (pid_n counts tiles of tile_n columns; band_n > 0: bands of band_n x 256
 * columns; band_n <= 0: group raster of group_m tile rows, 0 = 8) into out[2*t],
 * out[2*t+1], at most max_tiles pairs; returns the number of tiles of that
 * cluster, or a negative tgc_status.  Needs no GPU.  READY_QUEUE has no static
 * order past its local prefix, and AUTO may choose it: both are
 * TGC_ERR_INVALID_ARG here, as is a tile_n other than 256 or 512.
 */
int64_t tgc_ag_matmul_schedule(int64_t M, int64_t N, int64_t comm_block_rows, int nranks,
                               int rank, tgc_pivot pivot, int group_m, int band_n, int grid,
                               int cta, int64_t *out, int64_t max_tiles, int tile_n);

/* Tile shape used by the GEMM kernels (BM, BN, BK): BM rows are shared by a
 * pair of CTAs (128 each), BN is the width of one MMA column block (a tile is
 * one or two blocks wide, see tile_n), BK is the K depth of one pipeline stage. */
void tgc_gemm_tile_shape(int *bm, int *bn, int *bk);

/* ------------------------------------------------------------------------ */
/* Misc                                                                      */
/* ------------------------------------------------------------------------ */

const char *tgc_status_string(int status);
/* Last CUDA error seen by this thread inside the library (cudaSuccess if none). */
int tgc_last_cuda_error(void);
/* Library version, e.g. "0.1.0". */
const char *tgc_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TGC_H */
