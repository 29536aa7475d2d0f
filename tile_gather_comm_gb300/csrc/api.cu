// api.cu -- the C ABI of libtgc.so (declared in include/tgc.h): argument
// validation, workspace layout, and the launch sequence of each mode.
// Every check runs before anything is enqueued, so invalid calls return
// synchronously and touch no device state.
#include <cstdint>
#include <cstring>
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "schedule.h"

namespace tgc {

static thread_local int g_last_cuda_error = 0;

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = (int)e;
    return TGC_ERR_CUDA;
}

int sm_count(int device) {
    constexpr int kMaxDevices = 64;
    static int cache[kMaxDevices] = {0};
    static std::mutex mu;
    auto query = [](int d) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess || n <= 0) n = 1;
        return n;
    };
    if (device < 0 || device >= kMaxDevices) return query(device);
    std::lock_guard<std::mutex> lock(mu);
    if (cache[device] == 0) cache[device] = query(device);
    return cache[device];
}

WorkspaceLayout workspace_layout(int64_t nblocks, int64_t tile_rows) {
    WorkspaceLayout w{};
    auto up = [](size_t x, size_t a) { return (x + a - 1) / a * a; };
    w.status_off = 0;
    w.tickets_off = 64;
    w.counters_off = 128;
    size_t off = w.counters_off + up((size_t)nblocks * 4, 128);
    w.order_off = off;
    off += up((size_t)nblocks * 4, 128);
    w.delay_off = off;
    off += up((size_t)nblocks * 4, 128);
    w.rowcnt_off = off;
    off += up((size_t)tile_rows * 4, 128);
    w.ring_off = off;
    off += up((size_t)tile_rows * 8, 128);
    w.total = off < 256 ? 256 : off;
    return w;
}

static int64_t tile_rows_of(int64_t M) { return M > 0 ? (M + kTileM - 1) / kTileM : 0; }

static int elem_size(tgc_dtype dt) {
    switch (dt) {
        case TGC_U8: case TGC_I8: return 1;
        case TGC_F16: case TGC_BF16: return 2;
        case TGC_I32: case TGC_F32: return 4;
        case TGC_I64: case TGC_F64: return 8;
        default: return 0;
    }
}

static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// *acc = *acc * b for non-negative operands, unless the product reaches 2^62: every element
// count and byte offset the kernels form from it then fits int64 with room to spare.
static bool mul_fits(int64_t *acc, int64_t b) {
    int64_t r = 0;
    if (__builtin_mul_overflow(*acc, b, &r) || r >= (int64_t(1) << 62)) return false;
    *acc = r;
    return true;
}

// Memory pool of the allocating entry point, one per device, owned by the
// library so that its release threshold does not change the device's default
// pool.  Up to TGC_POOL_KEEP_BYTES of memory freed back to it stays mapped for
// the next call; the rest goes back to the device at the next synchronization.
static cudaError_t library_pool(int device, cudaMemPool_t *out) {
    static std::mutex mu;
    static std::vector<cudaMemPool_t> pools;
    std::lock_guard<std::mutex> lock(mu);
    if ((int)pools.size() <= device) pools.resize(device + 1, nullptr);
    if (pools[device] == nullptr) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = device;
        cudaMemPool_t pool = nullptr;
        cudaError_t e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = TGC_POOL_KEEP_BYTES;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) return e;
        pools[device] = pool;
    }
    *out = pools[device];
    return cudaSuccess;
}

// ------------------------------------------------------------------ TGATHER

static int tgather_impl(const tgc_tgather_args &a) {
    if (a.nranks <= 0 || a.nranks > TGC_MAX_RANKS) return TGC_ERR_INVALID_ARG;
    if (a.D0 < 0 || a.D1 < 0 || a.D2 < 0 || a.H < 0 || a.W < 0 || a.dst_rows3 < 0) return TGC_ERR_INVALID_ARG;
    const int es = elem_size(a.dtype);
    if (es == 0) return TGC_ERR_DTYPE;
    if (a.H >= (int64_t(1) << 56)) return TGC_ERR_INVALID_ARG;  // nranks * H must fit
    const int64_t rows3 = a.dst_rows3 == 0 ? (int64_t)a.nranks * a.H : a.dst_rows3;
    if (rows3 < (int64_t)a.nranks * a.H) return TGC_ERR_INVALID_ARG;
    if (a.progress != nullptr && (a.counters == nullptr || a.chunk_rows <= 0)) return TGC_ERR_INVALID_ARG;
    if (a.D0 == 0 || a.D1 == 0 || a.D2 == 0 || a.H == 0 || a.W == 0) return TGC_OK;  // empty: nothing written
    int64_t nslab = a.D0, dst_bytes = 0;
    if (!mul_fits(&nslab, a.D1) || !mul_fits(&nslab, a.D2)) return TGC_ERR_INVALID_ARG;
    dst_bytes = nslab;  // the destination holds every source byte (rows3 >= nranks * H)
    if (!mul_fits(&dst_bytes, rows3) || !mul_fits(&dst_bytes, a.W) || !mul_fits(&dst_bytes, es))
        return TGC_ERR_INVALID_ARG;
    if (a.dst == nullptr || a.srcs == nullptr) return TGC_ERR_INVALID_ARG;
    for (int r = 0; r < a.nranks; ++r)
        if (a.srcs[r] == nullptr) return TGC_ERR_INVALID_ARG;
    if (!aligned(a.dst, es)) return TGC_ERR_ALIGN;
    for (int r = 0; r < a.nranks; ++r)
        if (!aligned(a.srcs[r], es)) return TGC_ERR_ALIGN;
    if (a.progress != nullptr && (!aligned(a.progress, 4) || !aligned(a.counters, 4))) return TGC_ERR_ALIGN;

    TGatherLaunch L{};
    for (int r = 0; r < a.nranks; ++r) L.srcs[r] = a.srcs[r];
    L.dst = a.dst;
    L.nranks = a.nranks;
    L.es = es;
    L.nslab = nslab;
    L.run_bytes = a.H * a.W * es;
    L.dst_slab_bytes = rows3 * a.W * es;
    if (a.progress != nullptr) {
        const int64_t cr = a.chunk_rows < a.H ? a.chunk_rows : a.H;
        L.seg_bytes = cr * a.W * es;
        L.nseg = (a.H + cr - 1) / cr;
        L.progress = a.progress;
        L.counters = a.counters;
        L.epoch = a.epoch;
        L.spin_timeout_ns = a.spin_timeout_ns;
    } else {
        L.seg_bytes = L.run_bytes;
        L.nseg = 1;
    }
    return launch_tgather(L, a.stream);
}

// ------------------------------------------------------------------ AG-MatMul

int ag_validate(const tgc_ag_matmul_args &a, AGCheck &out) {
    if (a.nranks <= 0 || a.nranks > TGC_MAX_RANKS) return TGC_ERR_INVALID_ARG;
    if (a.M < 0 || a.K < 0 || a.N < 0) return TGC_ERR_INVALID_ARG;
    if (a.mode != TGC_MODE_FUSED && a.mode != TGC_MODE_UNFUSED && a.mode != TGC_MODE_MM_ONLY &&
        a.mode != TGC_MODE_FUSED_CE)
        return TGC_ERR_INVALID_ARG;
    const bool flagged = a.mode == TGC_MODE_FUSED || a.mode == TGC_MODE_FUSED_CE;
    if (a.pivot != TGC_PIVOT_PAGE && a.pivot != TGC_PIVOT_SHARD && a.pivot != TGC_PIVOT_NONE &&
        a.pivot != TGC_PIVOT_READY_QUEUE && a.pivot != TGC_PIVOT_AUTO)
        return TGC_ERR_INVALID_ARG;
    if (a.M % a.nranks != 0) return TGC_ERR_INVALID_ARG;
    const int64_t rows_per_rank = a.M / a.nranks;
    if (flagged) {
        if (a.comm_block_rows <= 0) return TGC_ERR_INVALID_ARG;
        if (rows_per_rank % a.comm_block_rows != 0) return TGC_ERR_INVALID_ARG;
    }
    if (a.rank < 0 || a.rank >= a.nranks) return TGC_ERR_INVALID_ARG;
    if (a.group_m < 0 || a.grid < 0) return TGC_ERR_INVALID_ARG;
    if (a.tile_n != 0 && a.tile_n != 256 && a.tile_n != 512) return TGC_ERR_INVALID_ARG;
    // the copy-engine producer's copies may run as a runtime kernel beside the GEMM CTAs, which
    // the 512-column kernel (168 registers x 384 threads per SM) leaves no room for
    if (a.mode == TGC_MODE_FUSED_CE && a.tile_n == 512) return TGC_ERR_INVALID_ARG;
    // sizes the kernels index with 32-bit integers
    if (a.M >= (int64_t(1) << 31) || a.N >= (int64_t(1) << 31) || a.K >= (int64_t(1) << 31))
        return TGC_ERR_INVALID_ARG;
    out.rows_per_rank = rows_per_rank;
    out.nblocks = flagged ? a.M / a.comm_block_rows : 0;
    if (a.M == 0 || a.N == 0) return 1;  // nothing to do
    if (a.K == 0) return TGC_ERR_INVALID_ARG;
    if (a.out_format != TGC_OUT_BF16 && a.out_format != TGC_OUT_F8E4M3) return TGC_ERR_INVALID_ARG;
    if (a.K % 8 != 0 || a.N % 8 != 0) return TGC_ERR_ALIGN;
    if (a.out_format == TGC_OUT_F8E4M3 && a.N % 16 != 0) return TGC_ERR_ALIGN;
    if (a.B == nullptr || a.C == nullptr || a.a_out == nullptr) return TGC_ERR_INVALID_ARG;
    if (!aligned(a.B, 16) || !aligned(a.C, 16) || !aligned(a.a_out, 16)) return TGC_ERR_ALIGN;
    if (a.mode != TGC_MODE_MM_ONLY) {
        if (a.a_shards == nullptr) return TGC_ERR_INVALID_ARG;
        for (int r = 0; r < a.nranks; ++r) {
            if (a.a_shards[r] == nullptr) return TGC_ERR_INVALID_ARG;
            if (!aligned(a.a_shards[r], 16)) return TGC_ERR_ALIGN;
        }
    }
    if (flagged) {
        if (out.nblocks >= (int64_t(1) << 24)) return TGC_ERR_INVALID_ARG;
        if (a.progress == nullptr || !aligned(a.progress, 4)) return TGC_ERR_INVALID_ARG;
        if (a.workspace == nullptr) return TGC_ERR_WORKSPACE;
        if (a.workspace_bytes < workspace_layout(out.nblocks, tile_rows_of(a.M)).total) return TGC_ERR_WORKSPACE;
        if (!aligned(a.workspace, 128)) return TGC_ERR_ALIGN;
        if (a.order != nullptr) {
            if (a.n_order < 0 || a.n_order > out.nblocks) return TGC_ERR_INVALID_ARG;
            std::vector<char> seen((size_t)out.nblocks, 0);
            for (int64_t i = 0; i < a.n_order; ++i) {
                const int32_t c = a.order[i];
                if (c < 0 || c >= out.nblocks || seen[(size_t)c]) return TGC_ERR_INVALID_ARG;
                seen[(size_t)c] = 1;
            }
        }
        // pieces per block * blocks must fit the 32-bit ticket dispenser (with room for
        // the one ticket each copy warp draws past the end)
        const int64_t pieces = (a.comm_block_rows * a.K * 2 + kMinPieceBytes - 1) / kMinPieceBytes;
        if (pieces * out.nblocks >= (int64_t(1) << 31)) return TGC_ERR_INVALID_ARG;
    }
    if (a.d_status != nullptr && !aligned(a.d_status, 4)) return TGC_ERR_ALIGN;
    if (a.trace != nullptr && !aligned(a.trace, 8)) return TGC_ERR_ALIGN;
    // a trace holds at least one CTA pair's records (the full bound needs the SM count)
    if (a.trace != nullptr && a.trace_words < 2 * (size_t)TGC_TRACE_WORDS) return TGC_ERR_INVALID_ARG;
    return 0;
}

// The tile order and raster a call runs (the resolution of AUTO and of band_n = 0).
struct OrderPlan {
    int pivot;    // PAGE / SHARD / NONE / READY_QUEUE as the kernel takes it
    int band_n;   // > 0: band raster, bands of band_n x 256 columns; 0: group raster
    int group_m;  // tile rows per group of the group raster
    int tile_n;   // output columns of a tile: 256 or 512
};

static OrderPlan resolve_order(const tgc_ag_matmul_args &a, const AGCheck &chk) {
    OrderPlan o{};
    const bool flagged = a.mode == TGC_MODE_FUSED || a.mode == TGC_MODE_FUSED_CE;
    o.group_m = a.group_m > 0 ? a.group_m : TGC_DEFAULT_GROUP_M;
    // Raster.  The fused modes take the band raster when the caller's shard holds fewer tile
    // rows than one group of the group raster: that raster's first group would already wait
    // on remote rows all at once, while bands ask for them one tile row at a time.  With a
    // longer local lead the group raster consumes remote rows slowly enough for the copy to
    // stay ahead, and keeps its operand reuse.
    if (a.band_n > 0) o.band_n = a.band_n;
    else if (a.band_n < 0 || !flagged) o.band_n = 0;
    else o.band_n = chk.rows_per_rank / kTileM < o.group_m ? TGC_DEFAULT_BAND_N : 0;
    // Tile width.  512 columns read a quarter fewer operand bytes per flop from L2, which
    // draws less power and lets the capped clock rise, but their single accumulator leaves the
    // epilogue exposed, and their first wave reaches twice as many tile rows.  They win where
    // K is long (the epilogue is then a small part of a tile) and a shard's own rows keep the
    // first waves busy (the group raster's case); 256 elsewhere.
    if (a.tile_n > 0) o.tile_n = a.tile_n;
    else if (a.mode == TGC_MODE_FUSED_CE) o.tile_n = 256;  // room for a runtime copy kernel per SM
    else o.tile_n = (a.K >= 8192 && chk.rows_per_rank / kTileM >= o.group_m) ? 512 : 256;
    // Tile order.  AUTO: the ready order for FUSED when the caller gives a release order and
    // the band raster walks rows soon enough to meet it out of order; the page's rank pivot
    // otherwise (with the default release order both orders coincide, and the ready order
    // only adds its ring lookups).
    tgc_pivot pivot = a.pivot;
    if (pivot == TGC_PIVOT_AUTO)
        pivot = a.mode == TGC_MODE_FUSED ? (a.order != nullptr && o.band_n > 0 ? TGC_PIVOT_READY_QUEUE
                                                                                : TGC_PIVOT_PAGE)
              : a.mode == TGC_MODE_FUSED_CE ? TGC_PIVOT_PAGE
                                            : TGC_PIVOT_NONE;
    // the ready order needs the in-kernel producer: the copy-engine mode takes the page pivot,
    // the plain GEMM no rotation
    o.pivot = (pivot == TGC_PIVOT_READY_QUEUE && a.mode != TGC_MODE_FUSED)
                  ? (a.mode == TGC_MODE_FUSED_CE ? (int)TGC_PIVOT_PAGE : (int)TGC_PIVOT_NONE)
                  : (int)pivot;
    return o;
}

// ------------------------------------------------------------------ copy-engine producer

using WriteValue32Fn = PFN_cuStreamWriteValue32_v11070;

static WriteValue32Fn write_value32_fn() {
    static WriteValue32Fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &f, 11070, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<WriteValue32Fn>(f);
    });
    return fn;
}

#ifndef TGC_CE_STREAMS
#define TGC_CE_STREAMS 4  // side streams of the copy-engine producer (blocks round-robin)
#endif
constexpr int kCeStreams = TGC_CE_STREAMS;

// Per-device side streams and events of the copy-engine producer.
struct CeState {
    std::mutex mu;
    cudaStream_t side[kCeStreams] = {};
    cudaEvent_t start = nullptr;
    cudaEvent_t done[kCeStreams] = {};
    bool ready = false;
};

static int ce_state(int device, CeState **out) {
    constexpr int kMaxDevices = 64;
    static CeState states[kMaxDevices];
    if (device < 0 || device >= kMaxDevices) return TGC_ERR_INVALID_ARG;
    CeState &st = states[device];
    std::lock_guard<std::mutex> lock(st.mu);
    if (!st.ready) {
        int lo = 0, hi = 0;
        cudaError_t e = cudaDeviceGetStreamPriorityRange(&lo, &hi);
        for (int i = 0; i < kCeStreams && e == cudaSuccess; ++i) {
            e = cudaStreamCreateWithPriority(&st.side[i], cudaStreamNonBlocking, hi);
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st.done[i], cudaEventDisableTiming);
        }
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st.start, cudaEventDisableTiming);
        if (e != cudaSuccess) return cuda_fail(e);
        st.ready = true;
    }
    *out = &st;
    return TGC_OK;
}

// The gather of FUSED_CE: on the side streams, after everything enqueued on
// `stream` so far, one device-to-device copy per comm block in release order
// (blocks dealt round-robin to the side streams, so several copy engines run
// at once), each followed by a stream write of `epoch` into its progress entry
// (the write's default memory barrier orders the block's bytes before the
// flag).  `launch` enqueues the consumer kernel on `stream`; `stream` then
// waits for every side stream, so the call completes only when `a_out` is whole.
template <class LaunchFn>
static int ce_fused(const tgc_ag_matmul_args &a, const AGCheck &chk, int64_t first_block, LaunchFn launch) {
    auto wv = write_value32_fn();
    if (wv == nullptr) return TGC_ERR_CUDA;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    CeState *st = nullptr;
    int rc = ce_state(dev, &st);
    if (rc != TGC_OK) return rc;
    std::lock_guard<std::mutex> lock(st->mu);
    e = cudaEventRecord(st->start, a.stream);
    for (int i = 0; i < kCeStreams && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(st->side[i], st->start, 0);
    if (e != cudaSuccess) return cuda_fail(e);
    const int64_t S = chk.rows_per_rank / a.comm_block_rows;
    const int64_t nb = chk.nblocks;
    const int local_b0 = (int)(a.rank * S), local_b1 = (int)((a.rank + 1) * S);
    const int64_t n = a.order != nullptr ? a.n_order : nb;
    const size_t block_bytes = (size_t)a.comm_block_rows * (size_t)a.K * 2;
    for (int64_t pos = 0; pos < n; ++pos) {
        const int64_t c = a.order != nullptr ? a.order[pos]
                                            : default_release_block((int)pos, (int)nb, (int)first_block, local_b0,
                                                                    local_b1);
        const int64_t r = c / S, sidx = c % S;
        const uint8_t *src = static_cast<const uint8_t *>(a.a_shards[r]) + (size_t)sidx * block_bytes;
        uint8_t *dst = static_cast<uint8_t *>(a.a_out) +
                       ((size_t)(r * chk.rows_per_rank + sidx * a.comm_block_rows)) * (size_t)a.K * 2;
        cudaStream_t side = st->side[pos % kCeStreams];
        e = cudaMemcpyAsync(dst, src, block_bytes, cudaMemcpyDeviceToDevice, side);
        if (e != cudaSuccess) return cuda_fail(e);
        CUresult cr = wv(reinterpret_cast<CUstream>(side), reinterpret_cast<CUdeviceptr>(a.progress + c), a.epoch, 0);
        if (cr != CUDA_SUCCESS) return TGC_ERR_CUDA;
    }
    for (int i = 0; i < kCeStreams && e == cudaSuccess; ++i) e = cudaEventRecord(st->done[i], st->side[i]);
    if (e != cudaSuccess) return cuda_fail(e);
    rc = launch();
    // even if the launch failed: keep stream order
    for (int i = 0; i < kCeStreams && e == cudaSuccess; ++i) e = cudaStreamWaitEvent(a.stream, st->done[i], 0);
    if (rc != TGC_OK) return rc;
    return e == cudaSuccess ? TGC_OK : cuda_fail(e);
}

static int ag_ex_impl(const tgc_ag_matmul_args &a) {
    AGCheck chk{};
    int rc = ag_validate(a, chk);
    if (rc < 0) return rc;
    if (rc == 1) return TGC_OK;  // empty problem
    cudaError_t e;
    cudaStream_t st = a.stream;
    const uint64_t timeout = a.spin_timeout_ns ? a.spin_timeout_ns : 2000000000ull;

    if (a.trace != nullptr) {
        // one trace record per launched CTA: CTAs come in pairs, at most one per SM, and no
        // more than `grid` (at least one pair) when the caller sets it
        int dev = 0;
        e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return cuda_fail(e);
        const int sms = sm_count(dev);
        const int want = a.grid > 0 ? (a.grid < 2 ? 2 : a.grid) : sms;
        const int ctas = want < sms ? want : sms;
        if (a.trace_words < (size_t)ctas * TGC_TRACE_WORDS) return TGC_ERR_INVALID_ARG;
    }
    int32_t *status = a.d_status;
    WorkspaceLayout wl = workspace_layout(chk.nblocks, tile_rows_of(a.M));
    uint8_t *ws = static_cast<uint8_t *>(a.workspace);
    if (status == nullptr && ws != nullptr) status = reinterpret_cast<int32_t *>(ws + wl.status_off);
    if (a.d_status != nullptr) {
        e = cudaMemsetAsync(a.d_status, 0, sizeof(int32_t), st);
        if (e != cudaSuccess) return cuda_fail(e);
    }

    GemmLaunch G{};
    G.nranks = a.nranks;
    G.B = a.B;
    G.C = a.C;
    G.a = a.a_out;
    G.M = a.M;
    G.K = a.K;
    G.N = a.N;
    G.cb = a.comm_block_rows;
    G.rank = a.rank;
    const OrderPlan plan = resolve_order(a, chk);
    G.group_m = plan.group_m;
    G.band_n = plan.band_n;
    G.tile_n = plan.tile_n;
    G.pivot = plan.pivot;
    G.grid = a.grid;
    G.timeout_ns = timeout;
    G.status = status;
    G.trace = a.trace;
    G.out_fp8 = a.out_format == TGC_OUT_F8E4M3 ? 1 : 0;
    if (a.mode != TGC_MODE_MM_ONLY)
        for (int r = 0; r < a.nranks; ++r) G.shards[r] = a.a_shards[r];

    if (a.mode == TGC_MODE_FUSED || a.mode == TGC_MODE_FUSED_CE) {
        G.fused = true;
        G.producer = a.mode == TGC_MODE_FUSED;
        G.progress = a.progress;
        G.epoch = a.epoch;
        G.ws_counters = reinterpret_cast<uint32_t *>(ws + wl.counters_off);
        G.ws_tickets = reinterpret_cast<uint32_t *>(ws + wl.tickets_off);
        G.ws_rowcnt = reinterpret_cast<uint32_t *>(ws + wl.rowcnt_off);
        G.ws_ring = reinterpret_cast<uint64_t *>(ws + wl.ring_off);
        G.n_order = chk.nblocks;
        if (a.order != nullptr) {
            e = cudaMemcpyAsync(ws + wl.order_off, a.order, (size_t)a.n_order * 4, cudaMemcpyHostToDevice, st);
            if (e != cudaSuccess) return cuda_fail(e);
            G.order = reinterpret_cast<const int32_t *>(ws + wl.order_off);
            G.n_order = a.n_order;
        }
        if (a.delay_ns != nullptr) {
            e = cudaMemcpyAsync(ws + wl.delay_off, a.delay_ns, (size_t)chk.nblocks * 4, cudaMemcpyHostToDevice, st);
            if (e != cudaSuccess) return cuda_fail(e);
            G.delay_ns = reinterpret_cast<const uint32_t *>(ws + wl.delay_off);
        }
        if (status == nullptr) return TGC_ERR_WORKSPACE;
        if (a.mode == TGC_MODE_FUSED_CE) {
            const int64_t tiles_m = tile_rows_of(a.M);
            const int64_t off = pivot_offset(G.pivot, a.rank, a.comm_block_rows, chk.rows_per_rank, kTileM,
                                             (int)tiles_m);
            rc = ce_fused(a, chk, off * kTileM / a.comm_block_rows, [&] { return launch_gemm(G, st); });
        } else {
            rc = launch_gemm(G, st);
        }
        if (rc != TGC_OK) return rc;
    } else {
        if (a.mode == TGC_MODE_UNFUSED) {
            TGatherLaunch T{};
            for (int r = 0; r < a.nranks; ++r) T.srcs[r] = a.a_shards[r];
            T.dst = a.a_out;
            T.nranks = a.nranks;
            T.es = 2;
            T.nslab = 1;
            T.run_bytes = chk.rows_per_rank * a.K * 2;
            T.dst_slab_bytes = a.M * a.K * 2;
            T.seg_bytes = T.run_bytes;
            T.nseg = 1;
            if (T.run_bytes > 0) {
                rc = launch_tgather(T, st);
                if (rc != TGC_OK) return rc;
            }
        }
        G.fused = false;
        rc = launch_gemm(G, st);
        if (rc != TGC_OK) return rc;
    }

    if (a.sync) {
        if (status == nullptr) {
            e = cudaStreamSynchronize(st);
            return e == cudaSuccess ? TGC_OK : cuda_fail(e);
        }
        int32_t h = 0;
        e = cudaMemcpyAsync(&h, status, sizeof h, cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return cuda_fail(e);
        e = cudaStreamSynchronize(st);
        if (e != cudaSuccess) return cuda_fail(e);
        return h;
    }
    return TGC_OK;
}

}  // namespace tgc

using namespace tgc;

extern "C" {

int tgc_tgather(void *dst, const void *const *srcs, int nranks, int64_t D0, int64_t D1, int64_t D2, int64_t H,
                int64_t W, tgc_dtype dtype, cudaStream_t stream) {
    tgc_tgather_args a{};
    a.dst = dst;
    a.srcs = srcs;
    a.nranks = nranks;
    a.D0 = D0;
    a.D1 = D1;
    a.D2 = D2;
    a.H = H;
    a.W = W;
    a.dtype = dtype;
    a.stream = stream;
    return tgather_impl(a);
}

int tgc_tgather_strided(void *dst, const int64_t *dst_strides, const void *const *srcs, const int64_t *src_strides,
                        int nranks, int64_t D0, int64_t D1, int64_t D2, int64_t H, int64_t W, tgc_dtype dtype,
                        cudaStream_t stream) {
    if (nranks <= 0 || nranks > TGC_MAX_RANKS) return TGC_ERR_INVALID_ARG;
    if (D0 < 0 || D1 < 0 || D2 < 0 || H < 0 || W < 0) return TGC_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    if (es == 0) return TGC_ERR_DTYPE;
    if (D0 == 0 || D1 == 0 || D2 == 0 || H == 0 || W == 0) return TGC_OK;  // empty: nothing written
    if (dst == nullptr || srcs == nullptr || dst_strides == nullptr || src_strides == nullptr)
        return TGC_ERR_INVALID_ARG;
    for (int k = 0; k < 5; ++k)
        if (dst_strides[k] < 0 || src_strides[k] < 0) return TGC_ERR_INVALID_ARG;
    // the largest element offset of each view, in bytes, must fit
    {
        int64_t rows = nranks;
        if (!mul_fits(&rows, H)) return TGC_ERR_INVALID_ARG;
        const int64_t dst_ext[5] = {D0, D1, D2, rows, W}, src_ext[5] = {D0, D1, D2, H, W};
        for (int v = 0; v < 2; ++v) {
            const int64_t *ext = v == 0 ? dst_ext : src_ext;
            const int64_t *str = v == 0 ? dst_strides : src_strides;
            int64_t last = 0;
            for (int k = 0; k < 5; ++k) {
                int64_t term = ext[k] - 1;
                if (!mul_fits(&term, str[k])) return TGC_ERR_INVALID_ARG;
                last += term;  // five terms below 2^62 each: no overflow
                if (last >= (int64_t(1) << 62)) return TGC_ERR_INVALID_ARG;
            }
            if (!mul_fits(&last, es)) return TGC_ERR_INVALID_ARG;
        }
    }
    for (int r = 0; r < nranks; ++r)
        if (srcs[r] == nullptr) return TGC_ERR_INVALID_ARG;
    if (!aligned(dst, es)) return TGC_ERR_ALIGN;
    for (int r = 0; r < nranks; ++r)
        if (!aligned(srcs[r], es)) return TGC_ERR_ALIGN;
    return launch_tgather_strided(srcs, dst, nranks, D0, D1, D2, H, W, es, src_strides, dst_strides, stream);
}

int tgc_tgather_ex(const tgc_tgather_args *args) {
    if (args == nullptr) return TGC_ERR_INVALID_ARG;
    return tgather_impl(*args);
}

size_t tgc_ag_matmul_workspace_bytes(int nranks, int64_t M, int64_t K, int64_t N, int64_t comm_block_rows) {
    (void)K;
    (void)N;
    int64_t nblocks = 0;
    if (nranks > 0 && comm_block_rows > 0 && M > 0) nblocks = M / comm_block_rows;
    return workspace_layout(nblocks, tile_rows_of(M)).total;
}

int tgc_ag_matmul_ex(const tgc_ag_matmul_args *args) {
    if (args == nullptr) return TGC_ERR_INVALID_ARG;
    return ag_ex_impl(*args);
}

int tgc_ag_matmul_plan(const tgc_ag_matmul_args *args, tgc_ag_matmul_plan_t *out) {
    if (args == nullptr || out == nullptr) return TGC_ERR_INVALID_ARG;
    AGCheck chk{};
    const int rc = ag_validate(*args, chk);
    if (rc < 0) return rc;
    const OrderPlan o = resolve_order(*args, chk);
    out->pivot = (tgc_pivot)o.pivot;
    out->band_n = o.band_n;
    out->group_m = o.group_m;
    out->tile_n = o.tile_n;
    return TGC_OK;
}

int tgc_ag_matmul(const void *const *a_shards, int nranks, const void *B, void *C, int64_t M, int64_t K, int64_t N,
                  int64_t comm_block_rows, cudaStream_t stream) {
    tgc_ag_matmul_args a{};
    a.a_shards = a_shards;
    a.nranks = nranks;
    a.B = B;
    a.C = C;
    a.M = M;
    a.K = K;
    a.N = N;
    a.comm_block_rows = comm_block_rows;
    a.mode = TGC_MODE_FUSED;
    a.pivot = TGC_PIVOT_AUTO;
    a.epoch = 1;
    a.stream = stream;
    a.sync = 1;
    // validate with placeholder temporaries before allocating anything
    {
        tgc_ag_matmul_args probe = a;
        alignas(256) static const uint64_t fake[64] = {0};
        probe.a_out = const_cast<uint64_t *>(fake);
        probe.progress = reinterpret_cast<uint32_t *>(const_cast<uint64_t *>(fake));
        probe.workspace = const_cast<uint64_t *>(fake);
        probe.workspace_bytes = (size_t)-1;
        AGCheck chk{};
        int rc = ag_validate(probe, chk);
        if (rc < 0) return rc;
        if (rc == 1) return TGC_OK;
    }
    const int64_t nblocks = M / comm_block_rows;
    const size_t a_bytes = (size_t)M * (size_t)K * 2;
    const size_t p_bytes = (size_t)nblocks * 4;
    const size_t w_bytes = workspace_layout(nblocks, tile_rows_of(M)).total;
    void *d_a = nullptr, *d_p = nullptr, *d_w = nullptr;
    int dev = 0;
    cudaMemPool_t pool = nullptr;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = library_pool(dev, &pool);
    if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&d_a, a_bytes, pool, stream);
    if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&d_p, p_bytes, pool, stream);
    if (e == cudaSuccess) e = cudaMallocFromPoolAsync(&d_w, w_bytes, pool, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_p, 0, p_bytes, stream);
    if (e == cudaSuccess) e = cudaMemsetAsync(d_w, 0, w_bytes, stream);
    int rc = TGC_OK;
    if (e != cudaSuccess) {
        rc = cuda_fail(e);
    } else {
        a.a_out = d_a;
        a.progress = static_cast<uint32_t *>(d_p);
        a.workspace = d_w;
        a.workspace_bytes = w_bytes;
        rc = ag_ex_impl(a);  // synchronizes and returns the device status
    }
    if (d_a) cudaFreeAsync(d_a, stream);
    if (d_p) cudaFreeAsync(d_p, stream);
    if (d_w) cudaFreeAsync(d_w, stream);
    e = cudaStreamSynchronize(stream);
    if (rc == TGC_OK && e != cudaSuccess) rc = cuda_fail(e);
    return rc;
}

int64_t tgc_ag_matmul_schedule(int64_t M, int64_t N, int64_t comm_block_rows, int nranks, int rank,
                               tgc_pivot pivot, int group_m, int band_n, int grid, int cta, int64_t *out,
                               int64_t max_tiles, int tile_n) {
    if (M <= 0 || N <= 0 || nranks <= 0 || M % nranks != 0 || rank < 0 || rank >= nranks || grid <= 0 ||
        cta < 0 || cta >= grid || group_m < 0 || comm_block_rows <= 0)
        return TGC_ERR_INVALID_ARG;
    if (pivot != TGC_PIVOT_PAGE && pivot != TGC_PIVOT_SHARD && pivot != TGC_PIVOT_NONE) return TGC_ERR_INVALID_ARG;  // READY_QUEUE is dynamic
    if (tile_n != 256 && tile_n != 512) return TGC_ERR_INVALID_ARG;
    TileSchedule s{};
    s.num_pid_m = (int)((M + kTileM - 1) / kTileM);
    s.num_pid_n = (int)((N + tile_n - 1) / tile_n);
    s.num_tiles = s.num_pid_m * s.num_pid_n;
    s.group_m = group_m > 0 ? group_m : TGC_DEFAULT_GROUP_M;
    s.band_n = band_n > 0 ? (int)(((int64_t)band_n * kBN + tile_n - 1) / tile_n) : 0;  // given in 256 columns
    s.pivot_off = pivot_offset((int)pivot, rank, comm_block_rows, M / nranks, kTileM, s.num_pid_m);
    int64_t n = 0;
    for (int t = cta; t < s.num_tiles; t += grid, ++n) {
        if (out != nullptr && n < max_tiles) {
            int pm, pn;
            s.tile(t, pm, pn);
            out[2 * n] = pm;
            out[2 * n + 1] = pn;
        }
    }
    return n;
}

void tgc_gemm_tile_shape(int *bm, int *bn, int *bk) {
    if (bm) *bm = kTileM;
    if (bn) *bn = kBN;
    if (bk) *bk = kBK;
}

const char *tgc_status_string(int status) {
    switch (status) {
        case TGC_OK: return "ok";
        case TGC_ERR_INVALID_ARG: return "invalid argument";
        case TGC_ERR_DTYPE: return "unsupported dtype";
        case TGC_ERR_ALIGN: return "misaligned pointer or row pitch";
        case TGC_ERR_CUDA: return "CUDA error (see tgc_last_cuda_error)";
        case TGC_ERR_TIMEOUT: return "bounded device wait expired";
        case TGC_ERR_ABORTED: return "kernel aborted after another CTA failed";
        case TGC_ERR_WORKSPACE: return "workspace missing or too small";
        case TGC_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of tgc_ag_matmul_noalloc";
        default: return "unknown status";
    }
}

int tgc_last_cuda_error(void) { return g_last_cuda_error; }

const char *tgc_version(void) { return "0.1.0"; }

}  // extern "C"
