// gemm.cu -- persistent, warp-specialised bf16 GEMM C = a * B^T on tcgen05 /
// TMEM / TMA for sm_103a, in two variants:
//   FUSED = true : the AllGather is produced inside the kernel.  Producer
//                  warps copy communication blocks of the shards into `a` and
//                  publish progress[block] = epoch; tiles that need remote
//                  rows wait on exactly the blocks they cover.
//   FUSED = false: plain GEMM over `a` (the unfused path's second kernel and
//                  the "mm_only" ceiling).
//
// Source: "Triton第四课：基于对称内存融合 AllGather 与 MatMul，提速1.56倍":
//   融合后的流水线 -- tiles pivoted by rank; a tile whose comm block belongs to
//       the caller reads a_shard directly, any other tile waits for
//       progress[comm_block_id] and reads the aggregate buffer a;
//   数据搬运与细粒度同步 -- progress entry src_rank*splits_per_rank+split_id
//       is set once the block's data is in place; data before flag;
//   wait_signal 的实现与语义 -- one thread polls the flag, then the CTA
//       proceeds; here one warp polls (one lane per covered block) with
//       ld.acquire.gpu and the wait is bounded.
//
// Tile order (schedule.h): the group raster (the page's GROUP_SIZE_M swizzle) or
// a band raster (bands of tile columns, rows walked in order), then the rank
// rotation of the tile row; or the ready order, built on the device from the
// order in which the producer completes tile rows.  The host picks the raster
// and, for TGC_PIVOT_AUTO, the order (api.cu).
//
// Tiles are 256 rows by 256 or 512 columns (template parameter TN, chosen per
// call), computed by a CTA pair (a cluster of 2 CTAs on two SMs, tcgen05
// cta_group::2): each CTA holds 128 rows of A and, per 256-column block, 128 of
// the block's columns of B per stage; the even CTA issues the 256 x 256 x 16
// MMAs for both (two per K step at TN = 512, sharing the A tile), and each CTA's
// TMEM receives its 128 rows of the accumulator.  At TN = 256 two accumulators
// alternate, so a tile's epilogue overlaps the next tile's MMAs; at TN = 512 one
// accumulator fills TMEM, the operand bytes per flop drop by a quarter and the
// epilogue hands the accumulator back as soon as its last columns are in
// registers.  A single-CTA variant (128-row tiles, cta_group::1) is kept behind
// the CG template parameter.
//
// CTA anatomy (one CTA per SM, persistent over tiles; 256 threads, 384 for
// the fused kernel with its extra copy warps):
//   warp 0     scheduler + flag wait + TMA loads of this CTA's A (128x64) and
//              B (128x64 per CTA of a pair and 256-column block, 256x64
//              alone) into a multi-stage shared-memory ring (128-byte swizzle)
//   warp 1     TMEM owner; one lane (of the even CTA) issues tcgen05.mma into
//              a TMEM accumulator (2 x 256 or 1 x 512 fp32 columns)
//   warps 2, 3, 8..11  (FUSED) copy producer: 16-64 KiB pieces of comm blocks,
//              handed out by a global ticket so any resident CTA can copy any
//              block, moved with 16-byte register loads and stores (or, with
//              TGC_COPY_LSU=0, by warp 2 alone with bulk async copies through
//              shared memory); the piece that completes a block publishes its
//              flag
//   warps 4..7 epilogue: tcgen05.ld of the accumulator (one TMEM lane quarter
//              per warp), fp32 -> bf16 round-to-nearest-even, stores to C;
//              with 512-column tiles warps 8..11 are a second epilogue group
//              for columns 256..511 (and only warps 2, 3 copy)
// With 256-column tiles the two TMEM accumulators let the epilogue of tile i
// overlap the mainloop of tile i+1.  All waits are bounded; on expiry the
// kernel records a status, lets its in-flight copies and MMAs land, frees TMEM
// and returns.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "prims.cuh"
#include "schedule.h"

namespace tgc {

// Compile-time tuning (defaults chosen by measurement on GB300).
#ifndef TGC_PAIR_STAGES
#define TGC_PAIR_STAGES 6        // pipeline stages of the GEMM on CTA pairs, 256-column tiles
#endif
#ifndef TGC_PAIR_FUSED_STAGES
#define TGC_PAIR_FUSED_STAGES 6  // the same when the copy producer also needs shared memory
#endif
#ifndef TGC_WIDE_STAGES
#define TGC_WIDE_STAGES 4        // pipeline stages with 512-column tiles (48 KiB each)
#endif
#ifndef TGC_COPY_SLOTS
#define TGC_COPY_SLOTS 4         // staging slots of the copy producer
#endif
// Copy producer: 0 = bulk async copies through shared-memory slots (the TMA
// unit), 1 = 16-byte vector loads and stores through registers (the load/store
// units) by warps 2 and 3.
#ifndef TGC_COPY_LSU
#define TGC_COPY_LSU 1
#endif
#ifndef TGC_COPY_VEC
#define TGC_COPY_VEC 32          // vectors per lane in flight in the register copy
#endif
#ifndef TGC_COPY_WARPS
#define TGC_COPY_WARPS 6         // register-copy warps: 2 and 3, then extra warps 8, 9, ...
#endif
#ifndef TGC_COPY_LEAD_WAVES
#define TGC_COPY_LEAD_WAVES 2    // waves of local tiles up front that let the copy run on two warps
#endif
// L2 policies: 0 = default, 1 = evict_first, 2 = evict_last, 3 = evict_normal
#ifndef TGC_COPY_HINT
#define TGC_COPY_HINT 0          // producer's bulk loads of the shards and stores into `a`
#endif
#ifndef TGC_TMA_STORE_C
#define TGC_TMA_STORE_C 1        // bf16 C leaves through shared memory and TMA stores
#endif
// 512-column tiles: convert a warp's whole share of the accumulator before
// handing it back (1), or hand it back after the last TMEM load (0).
#ifndef TGC_EPI_PACK_ALL
#define TGC_EPI_PACK_ALL 1
#endif
#ifndef TGC_A_HINT
#define TGC_A_HINT 0             // tile loads of A
#endif
#ifndef TGC_B_HINT
#define TGC_B_HINT 0             // tile loads of B
#endif

__device__ __forceinline__ uint64_t make_policy(int kind) {
    return kind == 1 ? policy_evict_first() : kind == 2 ? policy_evict_last() : policy_evict_normal();
}

constexpr int kThreads = 256;  // warps 0..7: tile loads, MMA, copy (2, 3), epilogue (4..7)
constexpr int kCopyWarps = TGC_COPY_LSU ? TGC_COPY_WARPS : 1;
static_assert(kCopyWarps >= 1 && kCopyWarps <= 8, "copy warps");
// Register-copy warps of a kernel: 2 and 3, then 8, 9, ... -- only 2 and 3 with
// 512-column tiles, whose warps 8..11 are a second epilogue group.
template <int TN>
constexpr int kCopyWarpsOf = TN == 512 && kCopyWarps > 2 ? 2 : kCopyWarps;
// Threads per CTA: the fused kernel with a register copy adds warps 8.. when it
// runs more than two copy warps; 512-column tiles add warps 8..11 for the
// epilogue.
template <bool FUSED, bool PROD, int TN>
constexpr int kThreadsOf = TN == 512 ? 384
                         : (FUSED && PROD && TGC_COPY_LSU && kCopyWarps > 2) ? 32 * (6 + kCopyWarps) : kThreads;
constexpr int kSlots = TGC_COPY_SLOTS;
constexpr int kSlotBytes = 8192;        // one bulk sub-copy through a staging slot
constexpr uint32_t kTmemCols = 512;     // two accumulators of 256 fp32 columns x 128 lanes
constexpr uint64_t kDrainTimeoutNs = 200ull * 1000 * 1000;

// Per-CTA-group configuration.  CG = number of CTAs sharing one MMA tile.
#ifndef TGC_C_BUFS
#define TGC_C_BUFS 4  // staging buffers per epilogue warp (TMA stores in flight), 256-column tiles
#endif
constexpr int kCBufs = TGC_C_BUFS;
static_assert(kCBufs == 2 || kCBufs == 4, "C staging buffers");

// TN: output columns of a tile, 256 (one MMA column block, two TMEM accumulators) or 512
// (two blocks side by side, one accumulator).
template <int CG, bool SLOTS, int TN>  // SLOTS: the copy producer's staging slots share shared memory
struct Cfg {
    static_assert(TN == 256 || TN == 512, "tile width");
    static constexpr int kTN = TN;
    static constexpr int kTileM = 128 * CG;             // output rows per (cluster) tile
    static constexpr int kRowsCta = 128;                // rows of A per CTA
    static constexpr int kNH = TN / kBN;                // MMA column blocks side by side in a tile
    static constexpr int kHalfN = kBN / CG;             // rows of B each CTA stages per column block
    static constexpr int kAStage = kRowsCta * kBK * 2;  // 16 KiB
    static constexpr int kBBox = kHalfN * kBK * 2;      // one column block: 32 KiB alone, 16 KiB in a pair
    static constexpr int kBStage = kNH * kBBox;
    static constexpr int kAccs = (int)kTmemCols / TN;   // TMEM accumulators per CTA (2, or 1 at 512)
    static constexpr int kStages = CG == 1 ? 4 : TN == 512 ? TGC_WIDE_STAGES
                                                  : (SLOTS ? TGC_PAIR_FUSED_STAGES : TGC_PAIR_STAGES);
    static constexpr uint32_t kIdesc = make_idesc_bf16_f32(kTileM, kBN);
    static constexpr uint32_t kStageTx = CG * (kAStage + kBStage);  // bytes landing per stage
    static constexpr int kEpiGroups = TN == 512 ? 2 : 1;  // groups of 4 epilogue warps, one per 256 columns
    static constexpr uint32_t kEpiArrivals = 4 * kEpiGroups * CG;  // warps that release an accumulator
    static constexpr int kCBufsWarp = TN == 512 ? 2 : kCBufs;      // C staging buffers per epilogue warp
};

// Only the bulk copy producer stages through shared memory.
template <bool FUSED, bool PROD>
constexpr bool kUsesSlots = FUSED && PROD && !TGC_COPY_LSU;

// Epilogue staging for TMA stores of C: per epilogue warp, two buffers of 32
// rows x 32 bf16 columns (64 bytes a row, 64-byte swizzle).  The bulk copy
// producer's slots leave no room for it; that kernel stores C directly.
constexpr int kCBoxCols = 32, kCBoxRows = 32;
constexpr int kCBufBytes = kCBoxCols * kCBoxRows * 2;  // 2 KiB
constexpr int kCStageBytes = 4 * kCBufs * kCBufBytes;  // 4 warps x kCBufs buffers (or 8 x 2 at 512 columns)
static_assert(kCStageBytes >= 8 * 2 * kCBufBytes, "C staging of the 512-column epilogue");
template <bool SLOTS>
constexpr bool kTmaC = TGC_TMA_STORE_C && !SLOTS;

template <int CG, bool SLOTS, int TN>
constexpr int smem_bytes() {
    using C = Cfg<CG, SLOTS, TN>;
    return 1024 /* alignment slack */ + C::kStages * (C::kAStage + C::kBStage) +
           (SLOTS ? kSlots * kSlotBytes : 0) + (kTmaC<SLOTS> ? kCStageBytes : 0) + 512 /* barriers + TMEM address */;
}

static_assert(smem_bytes<2, true, 256>() <= 232448 && smem_bytes<2, false, 256>() <= 232448 &&
                  smem_bytes<2, true, 512>() <= 232448 && smem_bytes<2, false, 512>() <= 232448,
              "shared memory per CTA");
static_assert((2 * 8 + 4 + kSlots + 1) * 8 + 4 <= 512, "barrier area");

struct GemmParams {
    int M, N, K;
    int num_kb;
    TileSchedule sched;
    uint16_t *C;
    int out_fp8;  // C as float8 e4m3 (N bytes per row) instead of bf16
    int *status;
    uint64_t timeout_ns;       // flag waits
    uint64_t mbar_timeout_ns;  // pipeline waits
    // fused-only
    int cb;
    int nblocks;
    int blocks_per_rank;
    int rows_per_rank;
    int local_row0, local_row1;
    int local_b0, local_b1;
    int first_block;
    int n_order;
    int pieces_per_block;
    int piece_bytes;      // copy piece size of this call
    int64_t row_bytes;
    int64_t block_bytes;
    const uint8_t *shards[TGC_MAX_RANKS];
    uint8_t *a;
    uint32_t *progress;
    uint32_t epoch;
    const int32_t *order;      // device copy in the workspace, or null
    const uint32_t *delay_ns;  // device copy in the workspace, or null
    uint32_t *counters;
    uint32_t *tickets;   // [0] piece ticket, [1] finished producers, [2] ready-ring tail, [3] finished CTAs
    int copy_warps;      // register copy: warps that take pieces (the others idle)
    uint64_t *trace;  // optional: kTraceWords per CTA
    // ready-queue order (FUSED only)
    int rq;               // nonzero: READY_QUEUE tile order
    int rq_local_row0;    // first tile row lying entirely inside the caller's shard
    int rq_local_rows;    // number of such tile rows (they come first)
    int tile_m;           // rows per tile (cluster)
    uint32_t *rowcnt;     // released blocks per tile row
    uint64_t *ring;       // tile rows in the order they became complete
};

// Trace word indices (mirrors TGC_TRACE_* in tgc.h).
constexpr int kTraceWords = 16;
enum : int {
    kTrStart = 0, kTrWaitNs, kTrWaitedTiles, kTrCopyFirst, kTrCopyLast, kTrPieces, kTrEnd, kTrTiles,
    kTrMmaStageNs, kTrMmaAccNs, kTrEpiWaitNs, kTrLoadStallNs, kTrPieceBytes, kTrCopyWarps
};

// mbar_wait that adds the time it blocked to *acc (only when tracing).
__device__ __forceinline__ bool mbar_wait_timed(uint64_t *bar, uint32_t parity, int *status, uint64_t timeout_ns,
                                                bool trace, uint64_t *acc) {
    if (!trace) return mbar_wait(bar, parity, status, timeout_ns);
    if (mbar_try_wait(smem_addr(bar), parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait(bar, parity, status, timeout_ns);
    *acc += globaltimer_ns() - t0;
    return ok;
}

// ---------------------------------------------------------------- flag wait

// Warp-collective: wait until progress[b] == epoch for every b in [b0, b1].
// Lane i polls block b0 + i (+32, ...) with gpu-scope acquire loads.
// Returns -1 if the wait was abandoned (timeout or abort), 0 if every flag was
// already set at the first poll, 1 if the warp had to spin.
__device__ int wait_blocks(const GemmParams &p, int b0, int b1, int lane) {
    int waited = 0;
    for (int base = b0; base <= b1; base += 32) {
        const int b = base + lane;
        const bool need = b <= b1;
        const uint64_t t0 = globaltimer_ns();
        for (uint64_t iter = 0;; ++iter) {
            const bool ready = !need || ld_acquire_gpu(p.progress + b) == p.epoch;
            if (__all_sync(0xffffffffu, ready)) break;
            waited = 1;
            if ((iter & 7) == 7) {
                const bool bad = ld_status(p.status) != 0;
                bool late = (globaltimer_ns() - t0 > p.timeout_ns) || iter > (1ull << 36);
                late = __shfl_sync(0xffffffffu, late, 0);
                if (late && lane == 0) raise_status(p.status, kStatusTimeout);
                if (__any_sync(0xffffffffu, bad || late)) return -1;
            }
            __nanosleep(32);
        }
    }
    __syncwarp();
    fence_proxy_async_global();  // the TMA loads that follow read what the flags published
    return waited;
}

// ---------------------------------------------------------------- tile order

// Position `pos` of the persistent walk -> tile.  Static orders map it with
// the swizzle + pivot of TileSchedule.  READY_QUEUE maps the first
// rq_local_rows * num_pid_n positions to the rows inside the caller's shard
// (swizzled), and position q past that prefix to column-major chunks of
// group_m ready-ring rows: ring slot `ring_idx` then names the tile row, known
// only once the producer has appended it.
struct TilePos {
    int pid_m, pid_n;
    int ring_idx;  // >= 0: pid_m comes from ring[ring_idx]
};

__device__ __forceinline__ TilePos tile_at(const GemmParams &p, int pos) {
    TilePos r;
    r.ring_idx = -1;
    if (!p.rq) {
        p.sched.tile(pos, r.pid_m, r.pid_n);
        return r;
    }
    const int npn = p.sched.num_pid_n;
    if (p.sched.band_n > 0) {
        // band raster: every band walks the caller's own rows, then the ready ring in order
        const int bn = p.sched.band_n;
        const int in_band = bn * p.sched.num_pid_m;
        const int band_id = pos / in_band;
        const int first_n = band_id * bn;
        const int bw = (npn - first_n) < bn ? (npn - first_n) : bn;
        const int rr = pos - band_id * in_band;
        const int row_idx = rr / bw;
        r.pid_n = first_n + rr % bw;
        if (row_idx < p.rq_local_rows) {
            r.pid_m = p.rq_local_row0 + row_idx;
        } else {
            r.ring_idx = row_idx - p.rq_local_rows;
            r.pid_m = -1;
        }
        return r;
    }
    const int n_local = p.rq_local_rows * npn;
    if (pos < n_local) {
        TileSchedule s = p.sched;
        s.num_pid_m = p.rq_local_rows;
        s.pivot_off = 0;
        s.tile(pos, r.pid_m, r.pid_n);
        r.pid_m += p.rq_local_row0;
        return r;
    }
    const int q = pos - n_local;
    const int G = p.sched.group_m;
    const int nrem = p.sched.num_pid_m - p.rq_local_rows;
    const int chunk = q / (G * npn);
    const int rows = (nrem - chunk * G) < G ? (nrem - chunk * G) : G;
    const int rr = q - chunk * G * npn;
    r.ring_idx = chunk * G + rr % rows;
    r.pid_n = rr / rows;
    r.pid_m = -1;
    return r;
}

// Warp-collective: tile row stored in ring[idx] for this call's epoch, or -1
// if the wait was abandoned (timeout or abort).  Sets *waited if it spun.
__device__ int ring_row(const GemmParams &p, int idx, int lane, bool *waited) {
    int row = -1;
    if (lane == 0) {
        const uint64_t t0 = globaltimer_ns();
        for (uint64_t it = 0; it < (1ull << 36); ++it) {
            const uint64_t e = ld_acquire_gpu_u64(p.ring + idx);
            if ((uint32_t)(e >> 32) == p.epoch && (uint32_t)e != 0u) {
                row = (int)(uint32_t)e - 1;
                break;
            }
            *waited = true;
            if ((it & 7) == 7) {
                if (ld_status(p.status) != 0) break;
                if (globaltimer_ns() - t0 > p.timeout_ns) {
                    raise_status(p.status, kStatusTimeout);
                    break;
                }
            }
            __nanosleep(32);
        }
    }
    return __shfl_sync(0xffffffffu, row, 0);
}

// ---------------------------------------------------------------- roles

// Cluster-tile index space: cluster c of nclusters persistent clusters (a
// "cluster" is a single CTA when CG == 1).
template <int CG>
__device__ __forceinline__ int cluster_id() { return (int)blockIdx.x / CG; }
template <int CG>
__device__ __forceinline__ int num_clusters() { return (int)gridDim.x / CG; }

template <int CG, bool FUSED, bool PROD, int TN>
__device__ void role_tma(const CUtensorMap *tmA, const CUtensorMap *tmL, const CUtensorMap *tmB,
                         const GemmParams &p, uint8_t *sA, uint8_t *sB, uint64_t *full, uint64_t *empty,
                         uint32_t crank, int lane) {
    using C = Cfg<CG, kUsesSlots<FUSED, PROD>, TN>;
    uint32_t it = 0;
    bool ok = true;
    uint64_t wait_ns = 0, waited_tiles = 0, load_stall_ns = 0;
    // completion of every stage is counted on the even CTA's full barrier
    const uint32_t full0 = CG == 2 ? mapa_shared(smem_addr(full), 0) : smem_addr(full);
    const uint64_t polA = make_policy(TGC_A_HINT), polB = make_policy(TGC_B_HINT);
    for (int t = cluster_id<CG>(); t < p.sched.num_tiles; t += num_clusters<CG>()) {
        TilePos tp = tile_at(p, t);
        if (tp.ring_idx >= 0) {
            bool spun = false;
            const uint64_t w0 = p.trace != nullptr ? globaltimer_ns() : 0;
            tp.pid_m = ring_row(p, tp.ring_idx, lane, &spun);
            if (tp.pid_m < 0) { ok = false; break; }
            if (p.trace != nullptr && spun) {
                wait_ns += globaltimer_ns() - w0;
                ++waited_tiles;
            }
        }
        const int pid_m = tp.pid_m, pid_n = tp.pid_n;
        const int m0 = pid_m * C::kTileM + (int)crank * C::kRowsCta;  // this CTA's 128 rows
        const int nb = pid_n * C::kTN + (int)crank * C::kHalfN;       // this CTA's B rows (first block)
        const CUtensorMap *mapA = tmA;
        int arow = m0;
        if (FUSED) {
            if (m0 >= p.local_row0 && m0 + C::kRowsCta <= p.local_row1) {
                mapA = tmL;               // rows of the caller's own shard: no wait
                arow = m0 - p.local_row0;
            } else if (m0 < p.M) {
                const int m1 = (m0 + C::kRowsCta) < p.M ? (m0 + C::kRowsCta) : p.M;
                const uint64_t w0 = p.trace != nullptr ? globaltimer_ns() : 0;
                const int w = wait_blocks(p, m0 / p.cb, (m1 - 1) / p.cb, lane);
                if (w < 0) { ok = false; break; }
                if (p.trace != nullptr && w > 0) {
                    wait_ns += globaltimer_ns() - w0;
                    ++waited_tiles;
                }
            }
        }
        if (lane == 0) {
            for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
                const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                if (!mbar_wait_timed(&empty[s], ph ^ 1u, p.status, p.mbar_timeout_ns, p.trace != nullptr,
                                     &load_stall_ns)) { ok = false; break; }
                if (CG == 1) {
                    mbar_arrive_expect_tx(&full[s], C::kStageTx);
                    if (TGC_A_HINT) tma_load_2d_hint(sA + s * C::kAStage, mapA, &full[s], kb * kBK, arow, polA);
                    else tma_load_2d(sA + s * C::kAStage, mapA, &full[s], kb * kBK, arow);
#pragma unroll
                    for (int h = 0; h < C::kNH; ++h) {
                        uint8_t *dstB = sB + s * C::kBStage + h * C::kBBox;
                        if (TGC_B_HINT) tma_load_2d_hint(dstB, tmB, &full[s], kb * kBK, nb + h * kBN, polB);
                        else tma_load_2d(dstB, tmB, &full[s], kb * kBK, nb + h * kBN);
                    }
                } else {
                    if (crank == 0) mbar_arrive_expect_tx(&full[s], C::kStageTx);  // both CTAs' bytes
                    const uint32_t bar = full0 + s * 8u;
                    if (TGC_A_HINT) tma_load_2d_pair_hint(sA + s * C::kAStage, mapA, bar, kb * kBK, arow, polA);
                    else tma_load_2d_pair(sA + s * C::kAStage, mapA, bar, kb * kBK, arow);
#pragma unroll
                    for (int h = 0; h < C::kNH; ++h) {
                        uint8_t *dstB = sB + s * C::kBStage + h * C::kBBox;
                        if (TGC_B_HINT) tma_load_2d_pair_hint(dstB, tmB, bar, kb * kBK, nb + h * kBN, polB);
                        else tma_load_2d_pair(dstB, tmB, bar, kb * kBK, nb + h * kBN);
                    }
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
    }
    if (p.trace != nullptr && lane == 0) {
        p.trace[blockIdx.x * kTraceWords + kTrWaitNs] = wait_ns;
        p.trace[blockIdx.x * kTraceWords + kTrWaitedTiles] = waited_tiles;
        p.trace[blockIdx.x * kTraceWords + kTrLoadStallNs] = load_stall_ns;
    }
    if (!ok && lane == 0) {
        if (CG == 1 || crank == 0) {
            // let every stage this CTA expected land before shared memory is given up
            for (uint32_t s = 0; s < (uint32_t)C::kStages; ++s) {
                const uint32_t n_s = it / C::kStages + (s < it % C::kStages ? 1u : 0u);
                if (n_s > 0) mbar_drain_wait(&full[s], (n_s - 1) & 1u, kDrainTimeoutNs);
            }
        } else {
            // the odd CTA cannot observe the even CTA's barrier: give its own
            // in-flight tile loads ample time to land
            spin_for_ns(200000);
        }
    }
    __syncwarp();
}

template <int CG, bool FUSED, bool PROD, int TN>
__device__ void role_mma(const GemmParams &p, uint8_t *sA, uint8_t *sB, uint64_t *full, uint64_t *empty,
                         uint64_t *tfull, uint64_t *tempty, uint64_t *drain, uint32_t tmem_base, uint32_t crank,
                         int lane) {
    using C = Cfg<CG, kUsesSlots<FUSED, PROD>, TN>;
    if (lane == 0 && crank == 0) {  // in a pair only the even CTA issues MMAs
        uint32_t it = 0, tc = 0;
        bool ok = true;
        uint64_t stage_ns = 0, acc_ns = 0;
        const bool tr = p.trace != nullptr;
        const uint32_t a_base = smem_addr(sA), b_base = smem_addr(sB);
        for (int t = cluster_id<CG>(); t < p.sched.num_tiles && ok; t += num_clusters<CG>(), ++tc) {
            const uint32_t acc = tc % (uint32_t)C::kAccs, aph = (tc / (uint32_t)C::kAccs) & 1u;
            if (!mbar_wait_timed(&tempty[acc], aph ^ 1u, p.status, p.mbar_timeout_ns, tr, &acc_ns)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem_base + acc * (uint32_t)C::kTN;
            for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
                const uint32_t s = it % C::kStages, ph = (it / C::kStages) & 1u;
                if (!mbar_wait_timed(&full[s], ph, p.status, p.mbar_timeout_ns, tr, &stage_ns)) { ok = false; break; }
                tc_fence_after();
                const uint64_t ad = make_sw128_kmajor_desc(a_base + s * C::kAStage);
                const uint64_t bd = make_sw128_kmajor_desc(b_base + s * C::kBStage);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k) {
#pragma unroll
                    for (int h = 0; h < C::kNH; ++h) {  // column block h: accumulator columns h*BN..
                        const uint64_t bdh = bd + (uint64_t)(h * (C::kBBox >> 4)) + 2u * k;
                        if (CG == 1)
                            mma_bf16_ss(d + h * kBN, ad + 2u * k, bdh, C::kIdesc, (kb | k) != 0 ? 1u : 0u);
                        else
                            mma_bf16_ss_pair(d + h * kBN, ad + 2u * k, bdh, C::kIdesc, (kb | k) != 0 ? 1u : 0u);
                    }
                }
                // frees the stage (in both CTAs of a pair) once these MMAs have read it
                if (CG == 1) mma_commit(&empty[s]);
                else mma_commit_pair_mc(&empty[s], (uint16_t)0x3);
            }
            if (ok) {
                if (CG == 1) mma_commit(&tfull[acc]);
                else mma_commit_pair_mc(&tfull[acc], (uint16_t)0x3);
            }
        }
        if (CG == 1) mma_commit(drain);  // every MMA issued above has completed once this arrives
        else mma_commit_pair_mc(drain, (uint16_t)0x1);
        mbar_drain_wait(drain, 0, kDrainTimeoutNs);
        if (tr) {
            p.trace[blockIdx.x * kTraceWords + kTrMmaStageNs] = stage_ns;
            p.trace[blockIdx.x * kTraceWords + kTrMmaAccNs] = acc_ns;
        }
    }
    __syncwarp();
}

// 2-D tiled TMA store of a box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *smem_src, int c0, int c1) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 ::"l"(map), "r"(smem_addr(smem_src)), "r"(c0), "r"(c1)
                 : "memory");
}

template <int CG, bool FUSED, bool PROD, int TN>
__device__ void role_epilogue(const GemmParams &p, const CUtensorMap *tmC, uint8_t *sC, uint64_t *tfull,
                              uint64_t *tempty, uint32_t tmem_base, uint32_t crank, int warp, int lane) {
    using C = Cfg<CG, kUsesSlots<FUSED, PROD>, TN>;
    constexpr bool kTma = kTmaC<kUsesSlots<FUSED, PROD>>;
    const bool tma_c = kTma && !p.out_fp8;
    constexpr int kBufs = C::kCBufsWarp;
    const int ew = warp - 4;                          // index among the epilogue warps
    const int col0 = (ew >> 2) * kBN;                 // this warp's group's first column of a tile
    constexpr int kCols = C::kTN / C::kEpiGroups;     // columns of a tile this warp's group stores
    uint8_t *stg = sC + ew * kBufs * kCBufBytes;      // this warp's staging buffers
    uint32_t stores = 0;                              // TMA stores this warp has issued
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    // the accumulator is released on the even CTA's barrier
    const uint32_t tempty0 = CG == 2 ? mapa_shared(smem_addr(tempty), 0) : smem_addr(tempty);
    uint32_t tc = 0;
    uint64_t epi_ns = 0;
    for (int t = cluster_id<CG>(); t < p.sched.num_tiles; t += num_clusters<CG>(), ++tc) {
        TilePos tp = tile_at(p, t);
        const uint32_t acc = tc % (uint32_t)C::kAccs, aph = (tc / (uint32_t)C::kAccs) & 1u;
        bool ok = true;
        if (lane == 0)
            ok = mbar_wait_timed(&tfull[acc], aph, p.status, p.mbar_timeout_ns, p.trace != nullptr, &epi_ns);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;  // warp-uniform: tcgen05.ld is .sync.aligned
        if (!ok) break;
        if (tp.ring_idx >= 0) {  // already published: the loads of this tile waited for it
            bool spun = false;
            tp.pid_m = ring_row(p, tp.ring_idx, lane, &spun);
            if (tp.pid_m < 0) break;
        }
        const int pid_m = tp.pid_m, pid_n = tp.pid_n;
        tc_fence_after();
        const int m = pid_m * C::kTileM + (int)crank * C::kRowsCta + row;
        const int n0 = pid_n * C::kTN + col0;
        uint16_t *crow = p.C + (int64_t)m * p.N;
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * (uint32_t)C::kTN + (uint32_t)col0;
        // Stores one 32-column chunk (fp32 bit patterns in v) of this lane's row to C.
        auto emit = [&](int j, const uint32_t(&v)[32]) {
            if (p.out_fp8) {
                // 32 columns -> 32 bytes: two 16-byte stores (N % 16 == 0)
                if (m < p.M) {
                    uint8_t *crow8 = reinterpret_cast<uint8_t *>(p.C) + (int64_t)m * p.N;
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int n = n0 + j * 32 + c * 16;
                        if (n < p.N) {
                            uint32_t w[4];
#pragma unroll
                            for (int q4 = 0; q4 < 4; ++q4) {
                                const int b = c * 16 + q4 * 4;
                                w[q4] = (uint32_t)pack_e4m3x2(v[b + 0], v[b + 1]) |
                                        ((uint32_t)pack_e4m3x2(v[b + 2], v[b + 3]) << 16);
                            }
                            *reinterpret_cast<uint4 *>(crow8 + n) = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                return;
            }
            if (kTma && tma_c) {
                // Row `lane` of a 32 x 32 box goes to shared memory in the 64-byte swizzle
                // (16-byte chunk c of row r at chunk c ^ ((r >> 1) & 3)), then one lane stores
                // the box with TMA; the tensor map clips rows >= M and columns >= N.
                uint8_t *buf = stg + (stores % (uint32_t)kBufs) * kCBufBytes;
                if (stores >= (uint32_t)kBufs) {
                    if (lane == 0) bulk_wait_read<kBufs - 1>();  // this buffer's previous store has read it
                    __syncwarp();
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint4 o;
                    o.x = pack_bf16x2(v[c * 8 + 0], v[c * 8 + 1]);
                    o.y = pack_bf16x2(v[c * 8 + 2], v[c * 8 + 3]);
                    o.z = pack_bf16x2(v[c * 8 + 4], v[c * 8 + 5]);
                    o.w = pack_bf16x2(v[c * 8 + 6], v[c * 8 + 7]);
                    const int cs = c ^ ((lane >> 1) & 3);
                    *reinterpret_cast<uint4 *>(buf + lane * 64 + cs * 16) = o;
                }
                fence_proxy_async_shared();  // the box is visible to the TMA unit
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(tmC, buf, n0 + j * 32, m - lane);
                    bulk_commit();
                }
                ++stores;
                return;
            }
            if (m < p.M) {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int n = n0 + j * 32 + c * 8;
                    if (n < p.N) {
                        uint4 o;
                        o.x = pack_bf16x2(v[c * 8 + 0], v[c * 8 + 1]);
                        o.y = pack_bf16x2(v[c * 8 + 2], v[c * 8 + 3]);
                        o.z = pack_bf16x2(v[c * 8 + 4], v[c * 8 + 5]);
                        o.w = pack_bf16x2(v[c * 8 + 6], v[c * 8 + 7]);
                        *reinterpret_cast<uint4 *>(crow + n) = o;
                    }
                }
            }
        };
        // 512-column tiles, bf16 C through TMA: the MMA issuer waits for this accumulator, so
        // the whole of this warp's 256 columns is converted to packed bf16 in registers first
        // (128 per lane), the accumulator handed back, and only then staged and stored.
        if (TGC_EPI_PACK_ALL && C::kTN == 512 && kTma && tma_c) {
            uint32_t pk[kCols / 32][16];
#pragma unroll
            for (int j = 0; j < kCols / 32; j += 2) {
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v0);
                tmem_ld_32x32b_x32(taddr + (uint32_t)((j + 1) * 32), v1);
                tmem_wait_ld();
#pragma unroll
                for (int c = 0; c < 16; ++c) {
                    pk[j][c] = pack_bf16x2(v0[2 * c], v0[2 * c + 1]);
                    pk[j + 1][c] = pack_bf16x2(v1[2 * c], v1[2 * c + 1]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (CG == 1) mbar_arrive(&tempty[acc]);
                else mbar_arrive_cluster(tempty0 + acc * 8u);
            }
#pragma unroll
            for (int j = 0; j < kCols / 32; ++j) {
                // the box's rows in the 64-byte swizzle, then one TMA store (as in emit)
                uint8_t *buf = stg + (stores % (uint32_t)kBufs) * kCBufBytes;
                if (stores >= (uint32_t)kBufs) {
                    if (lane == 0) bulk_wait_read<kBufs - 1>();
                    __syncwarp();
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int cs = c ^ ((lane >> 1) & 3);
                    *reinterpret_cast<uint4 *>(buf + lane * 64 + cs * 16) =
                        make_uint4(pk[j][4 * c], pk[j][4 * c + 1], pk[j][4 * c + 2], pk[j][4 * c + 3]);
                }
                fence_proxy_async_shared();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(tmC, buf, n0 + j * 32, m - lane);
                    bulk_commit();
                }
                ++stores;
            }
            continue;
        }
        // The same for float8 C (32 bytes per 32 columns: 64 words per lane), stored per thread.
        if (TGC_EPI_PACK_ALL && C::kTN == 512 && p.out_fp8) {
            uint32_t pk[kCols / 32][8];
#pragma unroll
            for (int j = 0; j < kCols / 32; j += 2) {
                uint32_t v0[32], v1[32];
                tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v0);
                tmem_ld_32x32b_x32(taddr + (uint32_t)((j + 1) * 32), v1);
                tmem_wait_ld();
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    pk[j][w] = (uint32_t)pack_e4m3x2(v0[4 * w], v0[4 * w + 1]) |
                               ((uint32_t)pack_e4m3x2(v0[4 * w + 2], v0[4 * w + 3]) << 16);
                    pk[j + 1][w] = (uint32_t)pack_e4m3x2(v1[4 * w], v1[4 * w + 1]) |
                                   ((uint32_t)pack_e4m3x2(v1[4 * w + 2], v1[4 * w + 3]) << 16);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (CG == 1) mbar_arrive(&tempty[acc]);
                else mbar_arrive_cluster(tempty0 + acc * 8u);
            }
            if (m < p.M) {
                uint8_t *crow8 = reinterpret_cast<uint8_t *>(p.C) + (int64_t)m * p.N;
#pragma unroll
                for (int j = 0; j < kCols / 32; ++j) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const int n = n0 + j * 32 + c * 16;  // N % 16 == 0
                        if (n < p.N)
                            *reinterpret_cast<uint4 *>(crow8 + n) =
                                make_uint4(pk[j][4 * c], pk[j][4 * c + 1], pk[j][4 * c + 2], pk[j][4 * c + 3]);
                    }
                }
            }
            continue;
        }
        // Two chunks per TMEM round trip; the accumulator goes back to the MMA issuer as soon as
        // its last columns are in registers, before they are converted and stored.
#pragma unroll 1
        for (int j = 0; j < kCols / 32; j += 2) {
            uint32_t v0[32], v1[32];
            tmem_ld_32x32b_x32(taddr + (uint32_t)(j * 32), v0);
            tmem_ld_32x32b_x32(taddr + (uint32_t)((j + 1) * 32), v1);
            tmem_wait_ld();
            if (j + 2 >= kCols / 32) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (CG == 1) mbar_arrive(&tempty[acc]);
                    else mbar_arrive_cluster(tempty0 + acc * 8u);
                }
            }
            emit(j, v0);
            emit(j + 1, v1);
        }
    }
    if (kTma && lane == 0) bulk_wait<0>();  // every store of C has landed and read its buffer
    __syncwarp();
    if (p.trace != nullptr && warp == 4 && lane == 0) {
        p.trace[blockIdx.x * kTraceWords + kTrEnd] = globaltimer_ns();
        p.trace[blockIdx.x * kTraceWords + kTrTiles] = tc;
        p.trace[blockIdx.x * kTraceWords + kTrEpiWaitNs] = epi_ns;
    }
}

struct Piece {
    const uint8_t *src;
    uint8_t *dst;
    uint32_t bytes;
    int block;
};

__device__ __forceinline__ Piece piece_of(const GemmParams &p, uint32_t ticket) {
    const int pos = (int)(ticket / (uint32_t)p.pieces_per_block);
    const int j = (int)(ticket % (uint32_t)p.pieces_per_block);
    const int c = p.order != nullptr
                      ? p.order[pos]
                      : default_release_block(pos, p.nblocks, p.first_block, p.local_b0, p.local_b1);
    const int r = c / p.blocks_per_rank, s = c % p.blocks_per_rank;
    const int64_t off = (int64_t)j * p.piece_bytes;
    const int64_t rem = p.block_bytes - off;
    Piece pc;
    pc.src = p.shards[r] + (int64_t)s * p.block_bytes + off;
    pc.dst = p.a + ((int64_t)r * p.rows_per_rank + (int64_t)s * p.cb) * p.row_bytes + off;
    pc.bytes = (uint32_t)(rem < p.piece_bytes ? rem : p.piece_bytes);
    pc.block = c;
    return pc;
}

// A piece's bytes are globally written: count it; the block's last piece publishes the block.
__device__ __forceinline__ void retire_piece(const GemmParams &p, uint32_t ticket) {
    const Piece pc = piece_of(p, ticket);
    const uint32_t old = atom_add_acq_rel_gpu(p.counters + pc.block, 1u);
    if (old + 1 == (uint32_t)p.pieces_per_block) {
        st_relaxed_gpu(p.counters + pc.block, 0u);  // every piece of this block is counted
        if (p.delay_ns != nullptr) spin_for_ns(p.delay_ns[pc.block]);
        st_release_gpu(p.progress + pc.block, p.epoch);
        if (p.rq) {
            // tile rows this block completes go to the ready ring (rows inside
            // the caller's shard are never queued: they come first anyway)
            const int64_t b_row0 = (int64_t)pc.block * p.cb;
            const int r0 = (int)(b_row0 / p.tile_m);
            const int r1 = (int)((b_row0 + p.cb - 1) / p.tile_m);
            for (int r = r0; r <= r1 && r < p.sched.num_pid_m; ++r) {
                if (r >= p.rq_local_row0 && r < p.rq_local_row0 + p.rq_local_rows) continue;
                const int64_t lo = (int64_t)r * p.tile_m;
                const int64_t hi = (lo + p.tile_m < p.M ? lo + p.tile_m : p.M) - 1;
                const uint32_t need = (uint32_t)(hi / p.cb - lo / p.cb + 1);  // blocks covering row r
                const uint32_t o = atom_add_acq_rel_gpu(p.rowcnt + r, 1u);
                if (o + 1 == need) {
                    st_relaxed_gpu(p.rowcnt + r, 0u);
                    const uint32_t slot = atom_add_relaxed_gpu(p.tickets + 2, 1u);
                    st_release_gpu_u64(p.ring + slot, ((uint64_t)p.epoch << 32) | (uint64_t)(r + 1));
                }
            }
        }
    }
}

// Bulk copy loop (one lane; TGC_COPY_LSU=0).  Work arrives in pieces of up to
// p.piece_bytes, handed out by a global ticket (any resident CTA can copy any
// block), and flows through NSLOT shared-memory slots of kSlotBytes as
// sub-copies: bulk load global -> slot, then bulk store slot -> `a`.  A slot
// is reused as soon as its store has finished READING shared memory, while the
// store's global writes may still be in flight.  A piece is retired -- counted
// toward its block, and the block published by the piece that completes it --
// once the writes of its last sub-copy have landed, which may lag up to
// kStoreLag stores behind, so loads, stores in flight and retirement overlap.
// Once no ticket is left the loop finishes the pieces it holds, waits for all
// its copies, retires them and returns the number of pieces it retired.  *ok
// becomes false if a wait was abandoned.
constexpr int kStoreLag = 6;
constexpr int kPieceRing = 16;  // pieces loaded but not yet retired

template <int NSLOT>
__device__ uint32_t copy_loop(const GemmParams &p, uint8_t *slots, uint64_t *bars, bool *ok_out) {
    const uint32_t total = (uint32_t)p.n_order * (uint32_t)p.pieces_per_block;
    // sub-copy sequence numbers: [0, tail) loads issued, [0, head) stores issued
    uint32_t head = 0, tail = 0;
    uint32_t slot_piece[NSLOT];   // piece ring index of the sub-copy in each slot
    uint32_t slot_off[NSLOT];     // byte offset of that sub-copy within its piece
    // piece ring: [pret, pload) pieces with sub-copies in flight or unretired
    uint32_t ring_ticket[kPieceRing];
    uint32_t ring_last_store[kPieceRing];  // store sequence number of the piece's last sub-copy (+1)
    uint32_t pret = 0, pload = 0;
    Piece cur{};
    uint32_t cur_off = 0, cur_ring = 0;
    bool have_cur = false, nomore = false, ok = true;
    const uint64_t pol = make_policy(TGC_COPY_HINT);
    for (;;) {
        // issue loads while a slot is free (its previous store has read it)
        while (tail - head < (uint32_t)NSLOT) {
            if (!have_cur) {
                if (nomore || pload - pret >= (uint32_t)kPieceRing) break;
                const uint32_t tk = atom_add_relaxed_gpu(p.tickets, 1u);
                if (tk >= total) { nomore = true; break; }
                cur = piece_of(p, tk);
                cur_off = 0;
                cur_ring = pload % kPieceRing;
                ring_ticket[cur_ring] = tk;
                ring_last_store[cur_ring] = 0;  // unknown yet
                ++pload;
                have_cur = true;
            }
            const uint32_t slot = tail % NSLOT;
            const uint32_t left = cur.bytes - cur_off;
            const uint32_t nb = left < (uint32_t)kSlotBytes ? left : (uint32_t)kSlotBytes;
            slot_piece[slot] = cur_ring;
            slot_off[slot] = cur_off;
            mbar_arrive_expect_tx(&bars[slot], nb);
            if (TGC_COPY_HINT) bulk_g2s_hint(slots + slot * kSlotBytes, cur.src + cur_off, nb, &bars[slot], pol);
            else bulk_g2s(slots + slot * kSlotBytes, cur.src + cur_off, nb, &bars[slot]);
            cur_off += nb;
            if (cur_off == cur.bytes) have_cur = false;
            ++tail;
        }
        if (head == tail) {
            if (nomore && !have_cur) break;
            if (pload - pret >= (uint32_t)kPieceRing) {  // ring full: retire what has landed
                bulk_wait<0>();
                fence_proxy_async_global();
                while (pret < pload && ring_last_store[pret % kPieceRing] != 0) {
                    retire_piece(p, ring_ticket[pret % kPieceRing]);
                    ++pret;
                }
            }
            continue;
        }
        {
            const uint32_t slot = head % NSLOT;
            if (!mbar_wait(&bars[slot], (head / NSLOT) & 1u, p.status, p.mbar_timeout_ns)) { ok = false; break; }
            fence_proxy_async_shared();
            const uint32_t pr = slot_piece[slot];
            const Piece pc = piece_of(p, ring_ticket[pr]);
            const uint32_t off = slot_off[slot];
            const uint32_t left = pc.bytes - off;
            const uint32_t nb = left < (uint32_t)kSlotBytes ? left : (uint32_t)kSlotBytes;
            if (TGC_COPY_HINT) bulk_s2g_hint(pc.dst + off, slots + slot * kSlotBytes, nb, pol);
            else bulk_s2g(pc.dst + off, slots + slot * kSlotBytes, nb);
            bulk_commit();
            ++head;
            if (off + nb == pc.bytes) ring_last_store[pr] = head;  // stores [0, head) cover this piece
        }
        bulk_wait_read<0>();  // the store just issued has read its slot
        // retire the oldest pieces whose last store is older than the newest kStoreLag
        if (pret < pload) {
            const uint32_t ls = ring_last_store[pret % kPieceRing];
            if (ls != 0 && head - ls >= (uint32_t)kStoreLag) {
                bulk_wait<kStoreLag>();  // all but the newest kStoreLag stores have landed
                fence_proxy_async_global();
                while (pret < pload) {
                    const uint32_t l2 = ring_last_store[pret % kPieceRing];
                    if (l2 == 0 || head - l2 < (uint32_t)kStoreLag) break;
                    retire_piece(p, ring_ticket[pret % kPieceRing]);
                    ++pret;
                }
            }
        }
    }
    bulk_wait<0>();
    if (ok) {
        fence_proxy_async_global();
        while (pret < pload) { retire_piece(p, ring_ticket[pret % kPieceRing]); ++pret; }
    } else {
        for (uint32_t i = head; i < tail; ++i) mbar_drain_wait(&bars[i % NSLOT], (i / NSLOT) & 1u, kDrainTimeoutNs);
    }
    *ok_out = ok;
    return pret;
}

// The copy producer role (warp 2, one lane): the copy loop over the kSlots
// slots reserved for it, until no ticket is left.
__device__ void role_copy(const GemmParams &p, uint8_t *sSlot, uint64_t *slotbar, int lane) {
    if (lane != 0) return;
    const uint64_t t_first = p.trace != nullptr ? globaltimer_ns() : 0;
    bool ok = true;
    const uint32_t pieces = copy_loop<kSlots>(p, sSlot, slotbar, &ok);
    if (p.trace != nullptr) {
        p.trace[blockIdx.x * kTraceWords + kTrCopyFirst] = t_first;
        p.trace[blockIdx.x * kTraceWords + kTrCopyLast] = globaltimer_ns();
        p.trace[blockIdx.x * kTraceWords + kTrPieces] = pieces;
        p.trace[blockIdx.x * kTraceWords + kTrCopyWarps] = 1;
        p.trace[blockIdx.x * kTraceWords + kTrPieceBytes] = (uint64_t)p.piece_bytes;
    }
}

constexpr int kCopyVec = TGC_COPY_VEC;

// 16-byte load through the non-coherent path without L1 allocation: the shards
// are read-only while the kernel runs and every byte is read once.
__device__ __forceinline__ uint4 ld_nc_v4(const uint4 *ptr) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(ptr));
    return v;
}

// The register copy producer (warps 2, 3 and 8.., TGC_COPY_LSU): each warp takes
// pieces from the same ticket dispenser as the bulk producer and moves them
// with coalesced 16-byte loads into registers and stores out of them,
// kCopyVec vectors per lane in flight.  The tile loads keep the SM's TMA unit
// busy; these copies bypass it.  After its stores every lane fences at gpu
// scope (and for the async proxy that the consumers' tile loads use); lane 0
// then retires the piece, and the piece that completes its block publishes it.
template <int NCW>  // copy warps of the kernel
__device__ void role_copy_lsu(const GemmParams &p, int warp, int lane) {
    __shared__ uint32_t s_pieces[NCW];
    __shared__ uint64_t s_last[NCW];
    const int cw = warp < 4 ? warp - 2 : warp - 6;  // index among the copy warps
    const uint32_t total = (uint32_t)p.n_order * (uint32_t)p.pieces_per_block;
    const uint64_t t_first = p.trace != nullptr ? globaltimer_ns() : 0;
    uint32_t pieces = 0;
    for (;;) {
        if (cw >= p.copy_warps) break;
        uint32_t tk = total;
        if (lane == 0 && ld_status(p.status) == 0) tk = atom_add_relaxed_gpu(p.tickets, 1u);
        tk = __shfl_sync(0xffffffffu, tk, 0);
        if (tk >= total) break;
        const Piece pc = piece_of(p, tk);
        const uint4 *src = reinterpret_cast<const uint4 *>(pc.src);
        uint4 *dst = reinterpret_cast<uint4 *>(pc.dst);
        const int nvec = (int)(pc.bytes / 16u);  // block bytes are a multiple of 16 (K % 8 == 0)
        for (int base = 0; base < nvec; base += 32 * kCopyVec) {
            uint4 r[kCopyVec];
#pragma unroll
            for (int j = 0; j < kCopyVec; ++j) {
                const int v = base + j * 32 + lane;
                if (v < nvec) r[j] = ld_nc_v4(src + v);
            }
#pragma unroll
            for (int j = 0; j < kCopyVec; ++j) {
                const int v = base + j * 32 + lane;
                if (v < nvec) dst[v] = r[j];
            }
        }
        fence_proxy_async_global();
        __threadfence();
        __syncwarp();
        if (lane == 0) retire_piece(p, tk);
        ++pieces;
    }
    if (p.trace != nullptr) {
        if (lane == 0) {
            s_pieces[cw] = pieces;
            s_last[cw] = globaltimer_ns();
        }
        asm volatile("bar.sync 1, %0;" ::"r"(32 * NCW) : "memory");  // the copy warps only
        if (cw == 0 && lane == 0) {
            uint64_t last = 0;
            uint32_t sum = 0;
            for (int i = 0; i < NCW; ++i) {
                last = s_last[i] > last ? s_last[i] : last;
                sum += s_pieces[i];
            }
            p.trace[blockIdx.x * kTraceWords + kTrCopyFirst] = t_first;
            p.trace[blockIdx.x * kTraceWords + kTrCopyLast] = last;
            p.trace[blockIdx.x * kTraceWords + kTrPieces] = sum;
            p.trace[blockIdx.x * kTraceWords + kTrCopyWarps] = (uint64_t)p.copy_warps;
            p.trace[blockIdx.x * kTraceWords + kTrPieceBytes] = (uint64_t)p.piece_bytes;
        }
    }
}

// ---------------------------------------------------------------- kernel

template <int CG, bool FUSED, bool PROD, int TN>
__global__ void __launch_bounds__(kThreadsOf<FUSED, PROD, TN>, 1)
    ag_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmL,
                   const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmC,
                   const GemmParams p) {
    using C = Cfg<CG, kUsesSlots<FUSED, PROD>, TN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    uint8_t *sA = smem;
    uint8_t *sB = smem + C::kStages * C::kAStage;
    uint8_t *sSlot = sB + C::kStages * C::kBStage;
    uint8_t *sC = sSlot + (kUsesSlots<FUSED, PROD> ? kSlots * kSlotBytes : 0);  // 2 KiB-aligned
    uint64_t *bars = reinterpret_cast<uint64_t *>(sC + (kTmaC<kUsesSlots<FUSED, PROD>> ? kCStageBytes : 0));
    uint64_t *full = bars;
    uint64_t *empty = full + C::kStages;
    uint64_t *tfull = empty + C::kStages;
    uint64_t *tempty = tfull + 2;
    uint64_t *slotbar = tempty + 2;
    uint64_t *drain = slotbar + kSlots;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(drain + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = CG == 2 ? cluster_ctarank() : 0u;
    if (threadIdx.x == 0) {
        if (p.trace != nullptr) p.trace[blockIdx.x * kTraceWords + kTrStart] = globaltimer_ns();
        for (int s = 0; s < C::kStages; ++s) { mbar_init(&full[s], 1); mbar_init(&empty[s], 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(&tfull[a], 1); mbar_init(&tempty[a], C::kEpiArrivals); }
        for (int i = 0; i < kSlots; ++i) mbar_init(&slotbar[i], 1);
        mbar_init(drain, 1);
        fence_mbarrier_init();
        fence_proxy_async_shared();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
        if (FUSED) prefetch_tensormap(&tmL);
    }
    if (warp == 1) {
        if (CG == 1) { tmem_alloc(tmem_holder, kTmemCols); tmem_relinquish(); }
        else { tmem_alloc_pair(tmem_holder, kTmemCols); tmem_relinquish_pair(); }
    }
    tc_fence_before();
    if (CG == 1) __syncthreads(); else cluster_sync();  // barriers initialised in both CTAs before any remote use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        role_tma<CG, FUSED, PROD, TN>(&tmA, &tmL, &tmB, p, sA, sB, full, empty, crank, lane);
    } else if (warp == 1) {
        role_mma<CG, FUSED, PROD, TN>(p, sA, sB, full, empty, tfull, tempty, drain, tmem_base, crank, lane);
    } else if (TN == 512 && warp >= 8) {
        role_epilogue<CG, FUSED, PROD, TN>(p, &tmC, sC, tfull, tempty, tmem_base, crank, warp, lane);
    } else if (warp == 2 || warp == 3 || warp >= 8) {
        if (FUSED && PROD) {
            if (TGC_COPY_LSU) {
                if (warp < 4 ? warp - 2 < kCopyWarpsOf<TN> : true) role_copy_lsu<kCopyWarpsOf<TN>>(p, warp, lane);
            } else if (warp == 2) {
                role_copy(p, sSlot, slotbar, lane);
            }
        }
    } else {
        role_epilogue<CG, FUSED, PROD, TN>(p, &tmC, sC, tfull, tempty, tmem_base, crank, warp, lane);
    }

    // In a pair, the even CTA's MMAs read the odd CTA's shared memory and write
    // its TMEM, and its commits arrive on the odd CTA's barriers: neither CTA
    // leaves (or frees TMEM) before both are done.
    __syncwarp();  // reconverge each warp before the aligned barrier
    tc_fence_before();
    if (CG == 1) __syncthreads(); else cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if (CG == 1) tmem_dealloc(tmem_base, kTmemCols);
        else tmem_dealloc_pair(tmem_base, kTmemCols);
    }
    if (FUSED && PROD && threadIdx.x == 0 && ld_status(p.status) == 0) {
        // Every warp of this CTA is past its last ticket and ring access; the
        // last CTA to get here rewinds the ticket dispenser and the ring so that
        // the workspace is zero again for the next call.
        const uint32_t done = atom_add_acq_rel_gpu(p.tickets + 3, 1u);
        if (done + 1 == gridDim.x) {
            st_relaxed_gpu(p.tickets, 0u);
            st_relaxed_gpu(p.tickets + 1, 0u);
            st_relaxed_gpu(p.tickets + 2, 0u);
            if (p.rq)
                for (int r = 0; r < p.sched.num_pid_m; ++r) p.ring[r] = 0ull;
            st_relaxed_gpu(p.tickets + 3, 0u);
        }
    }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 2-D bf16 row-major (rows x cols) with a (box_rows x 64) box, 128-byte swizzle.
// C (rows x cols bf16, row-major) for TMA stores of 32 x 32 boxes, 64-byte swizzle.
static bool make_map_c(CUtensorMap *m, const void *base, int64_t rows, int64_t cols) {
    auto enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kCBoxCols, (cuuint32_t)kCBoxRows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static bool make_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t box_rows) {
    auto enc = encode_fn();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// CTAs that share one MMA tile in the launched kernels.
constexpr int kCG = 2;
constexpr int kMaxDevices = 64;

template <int CG, bool FUSED, bool PROD, int TN>
static int set_smem_attr(int dev) {
    // a kernel's attributes belong to the device's context: set once per device
    static std::mutex mu;
    static cudaError_t err[kMaxDevices];
    static bool done[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return TGC_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
        err[dev] = cudaFuncSetAttribute(ag_gemm_kernel<CG, FUSED, PROD, TN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem_bytes<CG, kUsesSlots<FUSED, PROD>, TN>());
        done[dev] = true;
    }
    return err[dev] == cudaSuccess ? TGC_OK : cuda_fail(err[dev]);
}

// Persistent clusters that can be resident at once (one CTA per SM).
template <int CG, bool FUSED, bool PROD, int TN>
static int max_clusters(int dev, int sms) {
    if (CG == 1) return sms;
    static std::mutex mu;
    static int cached[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return sms / CG;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CG;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3((unsigned)(sms / CG * CG), 1, 1);
        cfg.blockDim = dim3(kThreadsOf<FUSED, PROD, TN>, 1, 1);
        cfg.dynamicSmemBytes = smem_bytes<CG, kUsesSlots<FUSED, PROD>, TN>();
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, ag_gemm_kernel<CG, FUSED, PROD, TN>, &cfg) != cudaSuccess || n <= 0)
            n = sms / CG;
        cached[dev] = n;
    }
    return cached[dev];
}

template <int CG, bool FUSED, bool PROD, int TN>
static int launch(const CUtensorMap &tmA, const CUtensorMap &tmL, const CUtensorMap &tmB, const CUtensorMap &tmC,
                  const GemmParams &p,
                  int nclusters, cudaStream_t stream) {
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return cuda_fail(de);
    int rc = set_smem_attr<CG, FUSED, PROD, TN>(dev);
    if (rc != TGC_OK) return rc;
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3((unsigned)(nclusters * CG), 1, 1);
    cfg.blockDim = dim3(kThreadsOf<FUSED, PROD, TN>, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<CG, kUsesSlots<FUSED, PROD>, TN>();
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, ag_gemm_kernel<CG, FUSED, PROD, TN>, tmA, tmL, tmB, tmC, p);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? TGC_OK : cuda_fail(e);
}

// Copy intensity of the register copy.  While the first TGC_COPY_LEAD_WAVES
// waves of the tile order reach rows outside the caller's shard, tiles wait
// for the copy, and every copy warp runs.  When the caller's own rows keep
// every cluster busy for that long, two warps deliver the remote blocks in
// time, and a faster copy would only compete with the GEMM's operand loads
// for HBM.
static int copy_warps_for(const GemmParams &p, int nclusters) {
    using C = Cfg<kCG, false, 256>;  // tile rows do not depend on the width
    const int horizon = TGC_COPY_LEAD_WAVES * nclusters;
    bool urgent = false;
    if (p.rq) {
        // positions of the caller's own rows at the head of the order (of the first band)
        const int cols = p.sched.band_n > 0 && p.sched.band_n < p.sched.num_pid_n ? p.sched.band_n
                                                                                 : p.sched.num_pid_n;
        urgent = p.rq_local_rows * cols < horizon;
    } else {
        for (int t = 0; t < horizon && t < p.sched.num_tiles && !urgent; ++t) {
            int pm = 0, pn = 0;
            p.sched.tile(t, pm, pn);
            const int m0 = pm * C::kTileM;
            const int m1 = m0 + C::kTileM < p.M ? m0 + C::kTileM : p.M;
            urgent = m0 < p.local_row0 || m1 > p.local_row1;
        }
    }
    return urgent || kCopyWarps < 2 ? kCopyWarps : 2;
}

// Copy piece size: the largest power of two from kMaxPieceBytes down to
// kMinPieceBytes that still gives every copy warp of the grid two pieces.  A
// small gather spread over many warps then finishes in a few round trips
// instead of one long piece per warp; a large one keeps the per-piece fence
// and counter traffic low.
#ifndef TGC_PIECES_PER_WARP
#define TGC_PIECES_PER_WARP 2
#endif
static int piece_bytes_for(const GemmParams &p, int64_t copy_warps_total) {
    int pb = kMaxPieceBytes;
    while (pb > kMinPieceBytes) {
        const int64_t pieces = (int64_t)p.n_order * ((p.block_bytes + pb - 1) / pb);
        if (pieces >= TGC_PIECES_PER_WARP * copy_warps_total) break;
        pb /= 2;
    }
    return pb;
}

template <int TN>
static int launch_gemm_tn(const GemmLaunch &L, cudaStream_t stream) {
    using C = Cfg<kCG, false, TN>;  // tile geometry does not depend on FUSED
    GemmParams p;
    std::memset(&p, 0, sizeof p);
    p.M = (int)L.M;
    p.N = (int)L.N;
    p.K = (int)L.K;
    p.num_kb = (int)((L.K + kBK - 1) / kBK);
    p.sched.num_pid_m = (int)((L.M + C::kTileM - 1) / C::kTileM);
    p.sched.num_pid_n = (int)((L.N + TN - 1) / TN);
    p.sched.num_tiles = p.sched.num_pid_m * p.sched.num_pid_n;
    p.sched.group_m = L.group_m;
    // band widths are given in columns of one MMA block (256)
    p.sched.band_n = L.band_n > 0 ? (int)(((int64_t)L.band_n * kBN + TN - 1) / TN) : L.band_n;
    const int64_t rows_per_rank = L.M / L.nranks;
    p.sched.pivot_off = pivot_offset(L.pivot, L.rank, L.cb, rows_per_rank, C::kTileM, p.sched.num_pid_m);
    p.C = static_cast<uint16_t *>(L.C);
    p.out_fp8 = L.out_fp8;
    p.status = L.status;
    p.timeout_ns = L.timeout_ns;
    p.mbar_timeout_ns = 4 * L.timeout_ns + 100ull * 1000 * 1000;
    p.trace = L.trace;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const int sms = sm_count(dev);

    CUtensorMap tmA, tmL, tmB, tmC;
    std::memset(&tmC, 0, sizeof tmC);
    if (!make_map(&tmA, L.a, L.M, L.K, C::kRowsCta) || !make_map(&tmB, L.B, L.N, L.K, C::kHalfN))
        return TGC_ERR_CUDA;
    // bf16 C leaves through TMA stores; float8 C is stored by the epilogue itself (no map)
    if (!L.out_fp8 && !make_map_c(&tmC, L.C, L.M, L.N)) return TGC_ERR_CUDA;
    if (L.fused) {
        if (!make_map(&tmL, L.shards[L.rank], rows_per_rank, L.K, C::kRowsCta)) return TGC_ERR_CUDA;
        p.cb = (int)L.cb;
        p.nblocks = (int)(L.M / L.cb);
        p.blocks_per_rank = (int)(rows_per_rank / L.cb);
        p.rows_per_rank = (int)rows_per_rank;
        p.local_row0 = (int)(L.rank * rows_per_rank);
        p.local_row1 = (int)((L.rank + 1) * rows_per_rank);
        p.local_b0 = L.rank * p.blocks_per_rank;
        p.local_b1 = (L.rank + 1) * p.blocks_per_rank;
        p.first_block = (int)(((int64_t)p.sched.pivot_off * C::kTileM) / L.cb);
        p.n_order = (int)L.n_order;
        p.row_bytes = L.K * 2;
        p.block_bytes = L.cb * L.K * 2;
        for (int r = 0; r < L.nranks; ++r) p.shards[r] = static_cast<const uint8_t *>(L.shards[r]);
        p.a = static_cast<uint8_t *>(L.a);
        p.progress = L.progress;
        p.epoch = L.epoch;
        p.order = L.order;
        p.delay_ns = L.delay_ns;
        p.counters = L.ws_counters;
        p.tickets = L.ws_tickets;
        p.tile_m = C::kTileM;
        p.rowcnt = L.ws_rowcnt;
        p.ring = L.ws_ring;
        if (L.pivot == TGC_PIVOT_READY_QUEUE && L.producer) {
            p.rq = 1;
            p.sched.pivot_off = 0;
            // tile rows lying entirely inside [local_row0, local_row1)
            const int64_t r0 = (p.local_row0 + C::kTileM - 1) / C::kTileM;
            int64_t r1 = p.local_row1 / C::kTileM;  // exclusive
            if (p.local_row1 == p.M) r1 = p.sched.num_pid_m;  // a partial last row inside the shard
            p.rq_local_row0 = (int)r0;
            p.rq_local_rows = (int)(r1 > r0 ? r1 - r0 : 0);
            if (p.rq_local_rows == 0) p.rq_local_row0 = 0;
            // releases follow the ring's natural consumer: rows after the local prefix, in order
            p.first_block = (int)((r1 < p.sched.num_pid_m ? r1 : 0) * C::kTileM / L.cb);
        }
    } else {
        tmL = tmA;
    }

    // persistent clusters: every SM busy; for the plain GEMM no more clusters than tiles
    // (the shared-memory attribute must be set before the occupancy query)
    const int variant = !L.fused ? 0 : (L.producer ? 1 : 2);
    int rc = variant == 0 ? set_smem_attr<kCG, false, false, TN>(dev)
           : variant == 1 ? set_smem_attr<kCG, true, true, TN>(dev) : set_smem_attr<kCG, true, false, TN>(dev);
    if (rc != TGC_OK) return rc;
    int nclusters = variant == 0 ? max_clusters<kCG, false, false, TN>(dev, sms)
                  : variant == 1 ? max_clusters<kCG, true, true, TN>(dev, sms)
                                 : max_clusters<kCG, true, false, TN>(dev, sms);
    if (L.grid > 0 && L.grid / kCG < nclusters) nclusters = L.grid / kCG;
    if (!L.fused && nclusters > p.sched.num_tiles) nclusters = p.sched.num_tiles;
    if (nclusters < 1) nclusters = 1;
    if (variant == 1) {
        p.copy_warps = copy_warps_for(p, nclusters);
        if (p.copy_warps > kCopyWarpsOf<TN>) p.copy_warps = kCopyWarpsOf<TN>;  // the kernel's copy warps
        p.piece_bytes = piece_bytes_for(p, (int64_t)nclusters * kCG * p.copy_warps);
    } else {
        p.piece_bytes = kMaxPieceBytes;
    }
    if (L.fused) p.pieces_per_block = (int)((p.block_bytes + p.piece_bytes - 1) / p.piece_bytes);
    return variant == 0 ? launch<kCG, false, false, TN>(tmA, tmL, tmB, tmC, p, nclusters, stream)
         : variant == 1 ? launch<kCG, true, true, TN>(tmA, tmL, tmB, tmC, p, nclusters, stream)
                        : launch<kCG, true, false, TN>(tmA, tmL, tmB, tmC, p, nclusters, stream);
}

int launch_gemm(const GemmLaunch &L, cudaStream_t stream) {
    if (L.tile_n == 512) return launch_gemm_tn<512>(L, stream);
    if (L.tile_n == 256) return launch_gemm_tn<256>(L, stream);
    return TGC_ERR_INVALID_ARG;
}

}  // namespace tgc
