// schedule.h -- tile order of the persistent GEMM kernels, shared by the
// device code and the host-side enumeration entry point (tgc_ag_matmul_schedule),
// so host tests check exactly what the kernels run.
//
// Source: "Triton第四课：基于对称内存融合 AllGather 与 MatMul，提速1.56倍",
// section 融合后的流水线: tiles are swizzled first (GROUP_SIZE_M grouping), then
// pid_m is rotated by the rank so that M tiles are visited in the order their
// data becomes ready ("this pivot preserves the prior swizzling").
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define TGC_HD __host__ __device__ __forceinline__
#else
#define TGC_HD inline
#endif

namespace tgc {

enum PivotMode : int { kPivotPage = 0, kPivotShard = 1, kPivotNone = 2 };

struct TileSchedule {
    int num_pid_m;
    int num_pid_n;
    int num_tiles;
    int group_m;
    int pivot_off;  // in tile rows, already reduced mod num_pid_m
    int band_n;     // > 0: band raster of band_n tile columns (group_m unused)

    // Linear tile index -> (pid_m, pid_n), then the rank rotation of pid_m.
    //   group raster (band_n <= 0): group_m tile rows per group, column-major
    //       inside a group -- the page's GROUP_SIZE_M swizzle;
    //   band raster (band_n > 0): band_n tile columns per band, row-major inside
    //       a band -- every band walks the tile rows in order while its columns
    //       of B stay in L2, so the rows are needed in the order a producer
    //       releases them.
    TGC_HD void tile(int t, int &pid_m, int &pid_n) const {
        if (band_n > 0) {
            const int in_band = band_n * num_pid_m;
            const int band_id = t / in_band;
            const int first_n = band_id * band_n;
            const int bw = (num_pid_n - first_n) < band_n ? (num_pid_n - first_n) : band_n;
            const int r = t - band_id * in_band;
            pid_m = r / bw + pivot_off;
            pid_n = first_n + r % bw;
            if (pid_m >= num_pid_m) pid_m -= num_pid_m;
            return;
        }
        const int in_group = group_m * num_pid_n;
        const int group_id = t / in_group;
        const int first_m = group_id * group_m;
        const int gsz = (num_pid_m - first_m) < group_m ? (num_pid_m - first_m) : group_m;
        const int r = t - group_id * in_group;
        pid_m = first_m + r % gsz;
        pid_n = r / gsz;
        pid_m += pivot_off;
        if (pid_m >= num_pid_m) pid_m -= num_pid_m;
    }
};

// Rotation in tile rows for each pivot mode:
//   page : floor(rank * cb / BM)      (= NUM_PID_M_PER_COMM_BLOCK * RANK when BM | cb)
//   shard: floor(rank * (M/R) / BM)   (the first tile row of the rank's shard)
TGC_HD int pivot_offset(int mode, int64_t rank, int64_t cb, int64_t rows_per_rank, int bm, int num_pid_m) {
    int64_t off = 0;
    if (mode == kPivotPage) off = (rank * cb) / bm;
    else if (mode == kPivotShard) off = (rank * rows_per_rank) / bm;
    if (num_pid_m <= 0) return 0;
    return (int)(off % num_pid_m);
}

// Default release order of the in-kernel producer (no explicit order given):
// the blocks in the order the schedule first reaches their rows -- starting at
// the block holding the first pivoted row and wrapping around -- with the
// caller's own shard moved to the end, since its tiles read the shard
// directly and do not wait for these copies.
TGC_HD int default_release_block(int pos, int nblocks, int first_block, int local_b0, int local_b1) {
    const int nlocal = local_b1 - local_b0;
    const int nremote = nblocks - nlocal;
    if (pos < nremote) {
        // walk remote blocks from first_block, skipping the local range
        int start = first_block;
        if (start >= local_b0 && start < local_b1) start = local_b1 % nblocks;
        // index of `start` among remote blocks
        int start_idx = start < local_b0 ? start : start - nlocal;
        int idx = start_idx + pos;
        if (idx >= nremote) idx -= nremote;
        return idx < local_b0 ? idx : idx + nlocal;
    }
    return local_b0 + (pos - nremote);
}

}  // namespace tgc
