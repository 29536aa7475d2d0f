// internal.h -- host-side declarations shared by the translation units of
// libtgc.so (not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/tgc.h"

#ifndef TGC_DEFAULT_GROUP_M
#define TGC_DEFAULT_GROUP_M 8  // tile rows per swizzle group when the caller passes 0
#endif

namespace tgc {

constexpr int kBN = 256;     // columns of one tcgen05.mma (N); a tile is one or two such blocks wide
constexpr int kBK = 64;      // bf16 elements per 128-byte swizzled row
constexpr int kTileM = 256;  // GEMM tile rows: a pair of CTAs, 128 rows each (tcgen05 cta_group::2)
// Fused producer: the unit of the ticket dispenser and of block completion is a
// piece of kMinPieceBytes..kMaxPieceBytes, chosen per call (a power of two).
#ifndef TGC_MIN_PIECE_BYTES
#define TGC_MIN_PIECE_BYTES 16384
#endif
constexpr int kMaxPieceBytes = 65536;
constexpr int kMinPieceBytes = TGC_MIN_PIECE_BYTES;
static_assert(kMinPieceBytes >= 4096 && kMinPieceBytes <= kMaxPieceBytes && kMinPieceBytes % 16 == 0, "piece size");

// Records a CUDA error for tgc_last_cuda_error() and maps it to a status.
int cuda_fail(cudaError_t e);
int sm_count(int device);

// Launch the TGATHER kernel; arguments already validated.
struct TGatherLaunch {
    const void *srcs[TGC_MAX_RANKS];
    void *dst;
    int nranks;
    int64_t nslab, run_bytes, dst_slab_bytes, seg_bytes, nseg;
    int es;
    uint32_t *progress;
    uint32_t *counters;
    uint32_t epoch;
    uint64_t spin_timeout_ns;  // the publisher's bound (0: default)
};
int launch_tgather(const TGatherLaunch &L, cudaStream_t stream);
int launch_tgather_strided(const void *const *srcs, void *dst, int nranks, int64_t D0, int64_t D1, int64_t D2,
                           int64_t H, int64_t W, int es, const int64_t *src_strides, const int64_t *dst_strides,
                           cudaStream_t stream);

// Launch one of the GEMM kernels; arguments already validated.
struct GemmLaunch {
    bool fused;        // tiles wait on progress flags
    bool producer;     // (fused) the kernel's own warps copy the blocks
    const void *shards[TGC_MAX_RANKS];
    int nranks;
    const void *B;
    void *C;
    void *a;           // gathered A (written by the fused producer, read by tiles)
    int64_t M, K, N;
    int64_t cb;        // comm_block_rows
    int rank;
    int pivot;
    int group_m;
    int band_n;        // > 0: band raster, bands of band_n x 256 columns; otherwise the group raster
    int tile_n;        // output columns of a tile: 256 or 512
    int grid;
    uint32_t *progress;
    uint32_t epoch;
    const int32_t *order;
    int64_t n_order;
    const uint32_t *delay_ns;
    uint64_t timeout_ns;
    uint32_t *ws_counters;  // nblocks
    uint32_t *ws_tickets;   // [0] piece ticket, [1] finished producers, [2] ready-ring tail, [3] finished CTAs
    uint32_t *ws_rowcnt;    // tile rows (READY_QUEUE)
    uint64_t *ws_ring;      // tile rows (READY_QUEUE)
    int32_t *status;
    uint64_t *trace;        // optional, kTraceWords per CTA
    int out_fp8;            // C as float8 e4m3 (saturating) instead of bf16
};
int launch_gemm(const GemmLaunch &L, cudaStream_t stream);

// Argument check shared by the AllGather-MatMul entry points: returns a
// negative tgc_status, 0 when there is work, 1 when the problem is empty.
struct AGCheck {
    int64_t nblocks;
    int64_t rows_per_rank;
};
int ag_validate(const tgc_ag_matmul_args &a, AGCheck &out);

// Workspace layout of tgc_ag_matmul_ex.
struct WorkspaceLayout {
    size_t status_off;    // int32 status word
    size_t tickets_off;   // uint32 x 4: piece ticket, finished producers, ready-ring tail, finished CTAs
    size_t counters_off;  // nblocks x uint32 piece counters
    size_t order_off;     // nblocks x int32: device copy of the release order
    size_t delay_off;     // nblocks x uint32: device copy of the release delays
    size_t rowcnt_off;    // tile_rows x uint32: released blocks per tile row
    size_t ring_off;      // tile_rows x uint64: ready ring, (epoch << 32) | (row + 1)
    size_t total;
};
WorkspaceLayout workspace_layout(int64_t nblocks, int64_t tile_rows);

}  // namespace tgc
