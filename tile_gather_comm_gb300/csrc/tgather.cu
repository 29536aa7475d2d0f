// tgather.cu -- TGATHER row-concatenation gather for sm_103a.
//
// Source: "CANN PTO-ISA TGATHER 指令深度解析：跨 Rank 行拼接 Gather 的实现原理与开发指南"
//   §二 数学语义: dst[d0,d1,d2, r*H+i, j] = src^(r)[d0,d1,d2,i,j].
//   §6.1: the NPU version stages tiles through its unified buffer with a 2-D
//   sliding window and masks for ragged tiles.
//
// GPU design.  With dense tensors, the H*W elements of rank r in slab
// (d0,d1,d2) are ONE contiguous run in the source and ONE contiguous run in
// the destination, so the whole gather is nranks*D0*D1*D2 contiguous copies.
// Without progress release (tgather_flat_kernel) each CTA of a grid of 8 per SM
// copies an equal byte share of the concatenated runs.  With progress release
// (tgather_kernel) each run is cut into segments, one per progress chunk, each
// segment into tiles of kTGThreads*kTGUnroll vectors, and the grid's CTAs walk
// the (segment, tile) items.  Copies go through registers with VW-byte vectors
// (16 bytes whenever the source and destination agree modulo 16), coalesced:
// consecutive threads touch consecutive vectors.  The unaligned head and the
// ragged tail of a segment (fewer than VW bytes each) are copied element by
// element by the segment's first tile -- this replaces the page's dynamic
// ValidRow/ValidCol masks, so any H and W work.
//
// Per-chunk release: when progress is given, every item of chunk (r, s) is
// counted with a gpu-scope release add once its bytes are stored, and
// `epoch` goes into progress[r*S + s] with st.release.gpu once the chunk's
// count is complete ("Triton第四课：基于对称内存融合 AllGather 与 MatMul，
// 提速1.56倍", section 数据搬运与细粒度同步: data visible before the flag) --
// stored by CTA 0, which watches the counts, for up to 512 chunks, else by the
// CTA whose add (returning the count) completes the chunk.
#include <cstdint>
#include <cuda_runtime.h>

#include "internal.h"
#include "prims.cuh"

namespace tgc {

// Compile-time tuning (defaults chosen by measurement on GB300).
#ifndef TGC_TG_THREADS
#define TGC_TG_THREADS 256   // threads per CTA
#endif
#ifndef TGC_TG_UNROLL
#define TGC_TG_UNROLL 8      // vectors in flight per thread
#endif
#ifndef TGC_TG_FLAT
#define TGC_TG_FLAT 1        // equal byte shares per CTA (1) or 16 KiB items (0)
#endif
#ifndef TGC_TG_PDL
#define TGC_TG_PDL 1         // programmatic dependent launch for the flat kernel
#endif
#ifndef TGC_TG_MIN_SHARE
#define TGC_TG_MIN_SHARE 4096  // smallest byte share per CTA of the flat kernel
#endif
#ifndef TGC_TG_CTAS_PER_SM
#define TGC_TG_CTAS_PER_SM 8   // CTAs per SM in the grid (5 of them resident at once at 46-47 registers)
#endif
#ifndef TGC_TG_VW32
#define TGC_TG_VW32 1          // flat kernel: 32-byte vectors when every address allows them
#endif
#ifndef TGC_TG_REL_PDL
#define TGC_TG_REL_PDL 1       // release kernel: programmatic dependent launch, as the flat kernel
#endif
#ifndef TGC_TG_REL_ATOM
#define TGC_TG_REL_ATOM 1      // release kernel: thread 0 counts an item with one release atomic (1),
                               // or with a gpu-scope fence followed by an acq_rel atomic (0)
#endif
#ifndef TGC_TG_REL_POLL
#define TGC_TG_REL_POLL 1      // release kernel: copying CTAs count items with a release reduction that
                               // returns nothing and CTA 0 publishes each completed chunk (1), or the
                               // CTA whose returned count completes a chunk publishes it (0)
#endif
#ifndef TGC_TG_PUBLISH_MAX_CHUNKS
#define TGC_TG_PUBLISH_MAX_CHUNKS 512  // publisher only up to this many chunks (two per publisher thread):
                                       // it publishes a thread's chunks one after another, one poll each
#endif
#ifndef TGC_TG_PUBLISH_SLEEP_NS
#define TGC_TG_PUBLISH_SLEEP_NS 128  // release kernel: the publisher's pause between polls of a count
#endif
#ifndef TGC_TG_CHUNK
#define TGC_TG_CHUNK 32768     // flat kernel: shares above this many bytes are cut into chunks
                               // dealt round-robin over the CTAs (0: one contiguous share each)
#endif

constexpr int kTGThreads = TGC_TG_THREADS;
constexpr int kTGUnroll = TGC_TG_UNROLL;

struct TGParams {
    const uint8_t *srcs[TGC_MAX_RANKS];
    uint8_t *dst;
    int nranks;
    int es;
    int64_t nslab;
    int64_t run_bytes;       // H*W*es: one (rank, slab) run; also the source slab stride
    int64_t dst_slab_bytes;  // dst_rows3*W*es
    int64_t seg_bytes;       // bytes per segment (chunk_rows*W*es, or run_bytes)
    int64_t nseg;            // segments per run
    int64_t tiles_per_seg;   // upper bound, identical for every segment
    int64_t total_items;
    uint32_t *progress;
    uint32_t *counters;
    uint32_t epoch;
    uint64_t publish_timeout_ns;  // publisher CTA's bound on waiting for a chunk's count
    int publish;                  // 1: CTA 0 publishes the chunks, the others count without waiting
};

struct alignas(32) Vec32 { uint32_t w[8]; };

template <int VW> struct VecT;
template <> struct VecT<32> { using T = Vec32; };
template <> struct VecT<16> { using T = uint4; };
template <> struct VecT<8> { using T = uint2; };
template <> struct VecT<4> { using T = uint32_t; };
template <> struct VecT<2> { using T = uint16_t; };
template <> struct VecT<1> { using T = uint8_t; };

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}
__device__ __forceinline__ Vec32 ld_stream(const Vec32 *p) {
    Vec32 v;
    asm volatile("ld.global.nc.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v.w[0]), "=r"(v.w[1]), "=r"(v.w[2]), "=r"(v.w[3]), "=r"(v.w[4]), "=r"(v.w[5]),
                   "=r"(v.w[6]), "=r"(v.w[7])
                 : "l"(p));
    return v;
}
template <typename T>
__device__ __forceinline__ T ld_stream(const T *p) { return __ldg(p); }

__device__ __forceinline__ void st_vec(Vec32 *p, const Vec32 &v) {
    asm volatile("st.global.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(v.w[0]), "r"(v.w[1]),
                 "r"(v.w[2]), "r"(v.w[3]), "r"(v.w[4]), "r"(v.w[5]), "r"(v.w[6]), "r"(v.w[7])
                 : "memory");
}
template <typename T>
__device__ __forceinline__ void st_vec(T *p, const T &v) { *p = v; }

// Element-wise copy of `n` bytes (n and both addresses multiples of es).
__device__ __forceinline__ void copy_elems(uint8_t *d, const uint8_t *s, int64_t n, int es, int tid, int nt) {
    switch (es) {
        case 8: for (int64_t i = tid; i < n / 8; i += nt) reinterpret_cast<uint64_t *>(d)[i] = reinterpret_cast<const uint64_t *>(s)[i]; break;
        case 4: for (int64_t i = tid; i < n / 4; i += nt) reinterpret_cast<uint32_t *>(d)[i] = reinterpret_cast<const uint32_t *>(s)[i]; break;
        case 2: for (int64_t i = tid; i < n / 2; i += nt) reinterpret_cast<uint16_t *>(d)[i] = reinterpret_cast<const uint16_t *>(s)[i]; break;
        default: for (int64_t i = tid; i < n; i += nt) d[i] = s[i]; break;
    }
}

// CTA 0 of the release kernel with a publisher: publishes each chunk once all its items are
// counted.  Thread t watches chunks t, t + kTGThreads, ... in turn (items are chunk-major, so
// chunks complete in about that order) with gpu-scope acquire loads, TGC_TG_PUBLISH_SLEEP_NS
// apart: the value that completes the count was written by the last of a chain of release adds,
// so every counted item's bytes are visible to the thread, which then resets the counter and
// stores `epoch` with a release.
// The copying CTAs never wait, so the counts always complete while the GPU runs the grid; the
// wait is still bounded: a chunk not counted within publish_timeout_ns of the start gets
// ~epoch (never equal to epoch) in its progress entry instead, and its counter is left as is.
__device__ __forceinline__ void tg_publish(const TGParams &p, int tid) {
    const uint32_t target = (uint32_t)(p.nslab * p.tiles_per_seg);
    const int64_t nch = (int64_t)p.nranks * p.nseg;
    const uint64_t t0 = globaltimer_ns();
    bool late = false;
    for (int64_t c = tid; c < nch; c += kTGThreads) {
        uint32_t spins = 0;
        while (!late && ld_acquire_gpu(p.counters + c) != target) {
            if ((++spins & 15u) == 0 && globaltimer_ns() - t0 > p.publish_timeout_ns) late = true;
            else if (TGC_TG_PUBLISH_SLEEP_NS > 0) __nanosleep(TGC_TG_PUBLISH_SLEEP_NS);
        }
        if (late) {
            st_relaxed_gpu(p.progress + c, ~p.epoch);
            continue;
        }
        st_relaxed_gpu(p.counters + c, 0u);  // every item of this chunk is counted
        st_release_gpu(p.progress + c, p.epoch);
    }
}

template <int VW>
__global__ void __launch_bounds__(kTGThreads) tgather_kernel(const TGParams p) {
    using V = typename VecT<VW>::T;
    constexpr int U = VW == 32 ? kTGUnroll / 2 : kTGUnroll;  // the same bytes in flight per thread
    constexpr int64_t kTileVecs = (int64_t)kTGThreads * U;
#if TGC_TG_REL_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
    const int tid = threadIdx.x;
    const bool poll = p.publish != 0;  // set by the host only with progress
    if (poll && blockIdx.x == 0) {
        tg_publish(p, tid);
        return;
    }
    // with a publisher, CTAs 1.. copy
    const int64_t first = poll ? (int64_t)blockIdx.x - 1 : (int64_t)blockIdx.x;
    const int64_t step = poll ? (int64_t)gridDim.x - 1 : (int64_t)gridDim.x;

    for (int64_t item = first; item < p.total_items; item += step) {
        // item = ((s * nranks + r) * nslab + slab) * tiles_per_seg + tile
        const int64_t tile = item % p.tiles_per_seg;
        int64_t rest = item / p.tiles_per_seg;
        const int64_t slab = rest % p.nslab;
        rest /= p.nslab;
        const int r = (int)(rest % p.nranks);
        const int64_t s = rest / p.nranks;

        const int64_t seg_off = s * p.seg_bytes;
        const int64_t len0 = p.run_bytes - seg_off;
        const int64_t len = len0 < p.seg_bytes ? len0 : p.seg_bytes;
        const uint8_t *src = p.srcs[r] + slab * p.run_bytes + seg_off;
        uint8_t *dst = p.dst + slab * p.dst_slab_bytes + (int64_t)r * p.run_bytes + seg_off;

        // Split [0, len) into head (to VW alignment of src), vector body, tail.
        int64_t head = (int64_t)((VW - (reinterpret_cast<uintptr_t>(src) % VW)) % VW);
        if (head > len) head = len;
        const int64_t nvec = (len - head) / VW;
        const int64_t body_end = head + nvec * VW;

        const int64_t v0 = tile * kTileVecs;
        if (v0 < nvec) {
            const V *vs = reinterpret_cast<const V *>(src + head) + v0;
            V *vd = reinterpret_cast<V *>(dst + head) + v0;
            const int64_t n = (nvec - v0) < kTileVecs ? (nvec - v0) : kTileVecs;
            V reg[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int64_t idx = tid + (int64_t)k * kTGThreads;
                if (idx < n) reg[k] = ld_stream(vs + idx);
            }
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const int64_t idx = tid + (int64_t)k * kTGThreads;
                if (idx < n) st_vec(vd + idx, reg[k]);
            }
        }
        if (tile == 0) {
            if (head > 0) copy_elems(dst, src, head, p.es, tid, kTGThreads);
            if (len > body_end) copy_elems(dst + body_end, src + body_end, len - body_end, p.es, tid, kTGThreads);
        }

        if (p.progress != nullptr) {
            // Count the item towards chunk (r, s), whose nslab*tiles_per_seg items publish it.  The
            // barrier orders every thread's stores of this item before thread 0's count; the other
            // threads go on to their next item instead of each waiting for its own stores.
            __syncthreads();
            if (tid == 0 && poll) {
                // counted without waiting for the add to land: CTA 0 publishes the chunk
                red_add_release_gpu(p.counters + ((int64_t)r * p.nseg + s), 1u);
            } else if (tid == 0) {
                const int64_t c = (int64_t)r * p.nseg + s;
                const uint32_t target = (uint32_t)(p.nslab * p.tiles_per_seg);
#if TGC_TG_REL_ATOM
                // the release add makes the item's bytes visible before the count (measured
                // 4.7% faster on the TGATHER workload than a separate fence and acq_rel add)
                const uint32_t old = atom_add_release_gpu(p.counters + c, 1u);
#else
                __threadfence();
                const uint32_t old = atom_add_acq_rel_gpu(p.counters + c, 1u);
#endif
                if (old + 1 == target) {
                    // acquire side: the other items' bytes, released by their counts, are
                    // visible to this thread before it publishes the chunk
                    __threadfence();
                    st_relaxed_gpu(p.counters + c, 0u);  // no other item of this chunk remains
                    st_release_gpu(p.progress + c, p.epoch);
                }
            }
        }
    }
}

// Flat variant (no progress release): the work space is the concatenation of
// all (slab, rank) runs, cut into gridDim.x equal, 32-byte-aligned shares --
// every CTA of the grid moves the same number of bytes, so the SMs get even
// loads.  A share larger than TGC_TG_CHUNK is dealt as chunks
// instead: CTA c copies chunks c, c + gridDim.x, ..., so at any moment the
// grid works on one compact window of memory rather than on gridDim.x far-apart
// streams (measured: 6.38 vs 6.02 TB/s on 537 MB, unchanged on 67 MB).  A
// range may span several runs; each (run, range) intersection is copied with
// VW-byte vectors between element-wise heads and tails.  The kernel is launched with programmatic
// stream serialization: it lets the next launch in the stream be scheduled as
// soon as every CTA has started, and waits for the previous grid's completion
// (griddepcontrol.wait) before touching memory.
template <int VW>
__global__ void __launch_bounds__(kTGThreads) tgather_flat_kernel(const TGParams p, int64_t share, int64_t stride) {
    using V = typename VecT<VW>::T;
    constexpr int U = VW == 32 ? kTGUnroll / 2 : kTGUnroll;  // the same bytes in flight per thread
#if TGC_TG_PDL
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
    const int tid = threadIdx.x;
    const int64_t total = p.nslab * p.nranks * p.run_bytes;
    // ranges [first, first + share), then every `stride` bytes (stride 0: one range)
    for (int64_t first = (int64_t)blockIdx.x * share; first < total; first += stride) {
        int64_t lo = first;
        const int64_t hi = lo + share < total ? lo + share : total;
        while (lo < hi) {
            const int64_t run = lo / p.run_bytes;         // run = slab * nranks + r
            const int64_t off = lo - run * p.run_bytes;   // offset inside the run
            const int64_t end_in_run = (hi - run * p.run_bytes) < p.run_bytes ? (hi - run * p.run_bytes) : p.run_bytes;
            const int64_t len = end_in_run - off;
            const int64_t slab = run / p.nranks;
            const int r = (int)(run - slab * p.nranks);
            const uint8_t *src = p.srcs[r] + slab * p.run_bytes + off;
            uint8_t *dst = p.dst + slab * p.dst_slab_bytes + (int64_t)r * p.run_bytes + off;

            int64_t head = (int64_t)((VW - (reinterpret_cast<uintptr_t>(src) % VW)) % VW);
            if (head > len) head = len;
            const int64_t nvec = (len - head) / VW;
            const int64_t body_end = head + nvec * VW;
            const V *vs = reinterpret_cast<const V *>(src + head);
            V *vd = reinterpret_cast<V *>(dst + head);
            for (int64_t base = 0; base < nvec; base += (int64_t)kTGThreads * U) {
                V reg[U];
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const int64_t idx = base + tid + (int64_t)k * kTGThreads;
                    if (idx < nvec) reg[k] = ld_stream(vs + idx);
                }
#pragma unroll
                for (int k = 0; k < U; ++k) {
                    const int64_t idx = base + tid + (int64_t)k * kTGThreads;
                    if (idx < nvec) st_vec(vd + idx, reg[k]);
                }
            }
            if (head > 0) copy_elems(dst, src, head, p.es, tid, kTGThreads);
            if (len > body_end) copy_elems(dst + body_end, src + body_end, len - body_end, p.es, tid, kTGThreads);
            lo += len;
        }
        if (stride == 0) break;
    }
}

// Strided views ("CANN PTO-ISA TGATHER 指令深度解析", §7.3 and §8.1: GlobalTensor
// views with a shape and a stride, shared by every source).  Rows are ordered
// (rank, d0, d1, d2, i).  When rows are contiguous in source and destination
// they are copied with VW-byte vectors by tgather_strided_rows_kernel (below);
// otherwise tgather_strided_elems_kernel copies every element on its own with
// both inner strides, thread g of the grid taking element g of the flattened
// (row, element) space.
struct TGStridedParams {
    const uint8_t *srcs[TGC_MAX_RANKS];
    uint8_t *dst;
    int nranks;
    int64_t D0, D1, D2, H;
    int64_t ss[5], ds[5];  // byte strides
    int64_t rows;          // nranks * D0 * D1 * D2 * H
    int64_t nv;            // vectors (contiguous rows) or elements per row
};

template <int ES>
__global__ void __launch_bounds__(256) tgather_strided_elems_kernel(const TGStridedParams p) {
    using V = typename VecT<ES>::T;
    const int64_t total = p.rows * p.nv;
    for (int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = g / p.nv, v = g - row * p.nv;
        int64_t t = row / p.H;
        const int64_t i = row - t * p.H;
        const int64_t d2 = t % p.D2;
        t /= p.D2;
        const int64_t d1 = t % p.D1;
        t /= p.D1;
        const int64_t d0 = t % p.D0;
        const int r = (int)(t / p.D0);
        const uint8_t *s = p.srcs[r] + d0 * p.ss[0] + d1 * p.ss[1] + d2 * p.ss[2] + i * p.ss[3];
        uint8_t *d = p.dst + d0 * p.ds[0] + d1 * p.ds[1] + d2 * p.ds[2] + ((int64_t)r * p.H + i) * p.ds[3];
        *reinterpret_cast<V *>(d + v * p.ds[4]) = *reinterpret_cast<const V *>(s + v * p.ss[4]);
    }
}

// Strided views whose rows are contiguous in source and destination: one warp
// copies one segment of one row, 32 x kTGUnroll vectors, with all its loads in
// flight before its stores.  The row coordinates (rank, d0, d1, d2, i) are
// decoded once per segment rather than once per vector.
template <int VW>
__global__ void __launch_bounds__(256) tgather_strided_rows_kernel(const TGStridedParams p, int64_t nseg) {
    using V = typename VecT<VW>::T;
    constexpr int U = VW == 32 ? kTGUnroll / 2 : kTGUnroll;  // the same bytes in flight per lane
    constexpr int kSeg = 32 * U;                              // vectors per segment
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t items = p.rows * nseg;
    for (int64_t it = (((int64_t)blockIdx.x * blockDim.x) + threadIdx.x) >> 5; it < items; it += nwarps) {
        const int64_t row = it / nseg;
        const int64_t v0 = (it - row * nseg) * kSeg;
        int64_t t = row / p.H;
        const int64_t i = row - t * p.H;
        const int64_t d2 = t % p.D2;
        t /= p.D2;
        const int64_t d1 = t % p.D1;
        t /= p.D1;
        const int64_t d0 = t % p.D0;
        const int r = (int)(t / p.D0);
        const V *s = reinterpret_cast<const V *>(p.srcs[r] + d0 * p.ss[0] + d1 * p.ss[1] + d2 * p.ss[2] +
                                                 i * p.ss[3]);
        V *d = reinterpret_cast<V *>(p.dst + d0 * p.ds[0] + d1 * p.ds[1] + d2 * p.ds[2] +
                                     ((int64_t)r * p.H + i) * p.ds[3]);
        V reg[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int64_t v = v0 + j * 32 + lane;
            if (v < p.nv) reg[j] = ld_stream(s + v);
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            const int64_t v = v0 + j * 32 + lane;
            if (v < p.nv) st_vec(d + v, reg[j]);
        }
    }
}

int launch_tgather_strided(const void *const *srcs, void *dst, int nranks, int64_t D0, int64_t D1, int64_t D2,
                           int64_t H, int64_t W, int es, const int64_t *src_strides, const int64_t *dst_strides,
                           cudaStream_t stream) {
    TGStridedParams p{};
    for (int r = 0; r < nranks; ++r) p.srcs[r] = static_cast<const uint8_t *>(srcs[r]);
    p.dst = static_cast<uint8_t *>(dst);
    p.nranks = nranks;
    p.D0 = D0;
    p.D1 = D1;
    p.D2 = D2;
    p.H = H;
    for (int k = 0; k < 5; ++k) {
        p.ss[k] = src_strides[k] * es;
        p.ds[k] = dst_strides[k] * es;
    }
    p.rows = (int64_t)nranks * D0 * D1 * D2 * H;
    const bool inner = p.ss[4] == es && p.ds[4] == es;
    int vw = es;
    if (inner) {
        // widest vector every row start (source and destination) and the row length allow
        uint64_t g = TGC_TG_VW32 ? 32 : 16;
        auto fold = [&](uint64_t x) { while (g > (uint64_t)es && (x % g) != 0) g >>= 1; };
        for (int r = 0; r < nranks; ++r) fold(reinterpret_cast<uintptr_t>(srcs[r]));
        fold(reinterpret_cast<uintptr_t>(dst));
        const int64_t ext[4] = {D0, D1, D2, H};
        for (int k = 0; k < 4; ++k)
            if (ext[k] > 1) { fold((uint64_t)p.ss[k]); fold((uint64_t)p.ds[k]); }
        if ((int64_t)nranks * H > 1) fold((uint64_t)p.ds[3]);
        fold((uint64_t)(W * es));
        vw = (int)g;
    }
    p.nv = inner ? W * es / vw : W;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const int64_t cap = (int64_t)sm_count(dev) * 8;
    if (inner) {
        const int64_t seg = 32 * (vw == 32 ? kTGUnroll / 2 : kTGUnroll);  // the kernel's kSeg
        const int64_t nseg = (p.nv + seg - 1) / seg;
        int64_t grid = (p.rows * nseg + 7) / 8;  // 8 warps per CTA, one item each per pass
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
        const dim3 gd((unsigned)grid), bd(256);
        switch (vw) {
            case 32: tgather_strided_rows_kernel<32><<<gd, bd, 0, stream>>>(p, nseg); break;
            case 16: tgather_strided_rows_kernel<16><<<gd, bd, 0, stream>>>(p, nseg); break;
            case 8: tgather_strided_rows_kernel<8><<<gd, bd, 0, stream>>>(p, nseg); break;
            case 4: tgather_strided_rows_kernel<4><<<gd, bd, 0, stream>>>(p, nseg); break;
            case 2: tgather_strided_rows_kernel<2><<<gd, bd, 0, stream>>>(p, nseg); break;
            default: tgather_strided_rows_kernel<1><<<gd, bd, 0, stream>>>(p, nseg); break;
        }
    } else {
        const int64_t total = p.rows * p.nv;
        int64_t grid = (total + 255) / 256;
        if (grid > cap) grid = cap;
        if (grid < 1) grid = 1;
        const dim3 gd((unsigned)grid), bd(256);
        switch (es) {
            case 8: tgather_strided_elems_kernel<8><<<gd, bd, 0, stream>>>(p); break;
            case 4: tgather_strided_elems_kernel<4><<<gd, bd, 0, stream>>>(p); break;
            case 2: tgather_strided_elems_kernel<2><<<gd, bd, 0, stream>>>(p); break;
            default: tgather_strided_elems_kernel<1><<<gd, bd, 0, stream>>>(p); break;
        }
    }
    e = cudaGetLastError();
    return e == cudaSuccess ? TGC_OK : cuda_fail(e);
}

static int pick_vw(const TGatherLaunch &L, uint64_t widest = 16) {
    // Largest power of two <= widest dividing every (src - dst) address difference;
    // then source and destination share their alignment modulo VW everywhere.
    uint64_t g = widest;
    const uint64_t slab_delta = (uint64_t)(L.dst_slab_bytes - L.run_bytes);
    auto fold = [&](uint64_t x) {
        while (g > 1 && (x % g) != 0) g >>= 1;
    };
    for (int r = 0; r < L.nranks; ++r) {
        const uint64_t d = reinterpret_cast<uintptr_t>(L.dst) + (uint64_t)r * (uint64_t)L.run_bytes;
        fold(reinterpret_cast<uintptr_t>(L.srcs[r]) - d);
    }
    if (L.nslab > 1) fold(slab_delta);
    if ((int)g < L.es) g = (uint64_t)L.es;  // cannot happen for element-aligned pointers
    return (int)g;
}

int launch_tgather(const TGatherLaunch &L, cudaStream_t stream) {
    TGParams p{};
    for (int r = 0; r < L.nranks; ++r) p.srcs[r] = static_cast<const uint8_t *>(L.srcs[r]);
    p.dst = static_cast<uint8_t *>(L.dst);
    p.nranks = L.nranks;
    p.es = L.es;
    p.nslab = L.nslab;
    p.run_bytes = L.run_bytes;
    p.dst_slab_bytes = L.dst_slab_bytes;
    p.seg_bytes = L.seg_bytes;
    p.nseg = L.nseg;
    p.progress = L.progress;
    p.counters = L.counters;
    p.epoch = L.epoch;
    p.publish_timeout_ns = L.spin_timeout_ns > 0 ? L.spin_timeout_ns : 10000000000ull;

    const int vw = pick_vw(L);
    const int64_t tile_vecs = (int64_t)kTGThreads * (vw == 32 ? kTGUnroll / 2 : kTGUnroll);  // the kernel's kTileVecs
    const int64_t max_vecs = L.seg_bytes / vw;
    p.tiles_per_seg = max_vecs > 0 ? (max_vecs + tile_vecs - 1) / tile_vecs : 1;
    if (p.tiles_per_seg < 1) p.tiles_per_seg = 1;
    p.total_items = L.nseg * (int64_t)L.nranks * L.nslab * p.tiles_per_seg;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    const int64_t slots = (int64_t)sm_count(dev) * TGC_TG_CTAS_PER_SM;

    if (TGC_TG_FLAT && L.progress == nullptr) {
        // equal 32-byte-aligned shares over 8 CTAs per SM (fewer CTAs only for small copies)
        const int64_t total = L.nslab * L.nranks * L.run_bytes;
        const int64_t min_share = TGC_TG_MIN_SHARE;
        int64_t grid = (total + min_share - 1) / min_share;
        if (grid > slots) grid = slots;
        if (grid < 1) grid = 1;
        int64_t share = (total + grid - 1) / grid;
        const int vwf = TGC_TG_VW32 && vw == 16 ? pick_vw(L, 32) : vw;  // 32 only where 16 already holds
        share = (share + 31) / 32 * 32;
        int64_t stride = 0;
        if (TGC_TG_CHUNK > 0 && share > TGC_TG_CHUNK) {
            share = (TGC_TG_CHUNK + 31) / 32 * 32;
            stride = grid * share;
        }
        grid = (total + share - 1) / share;
        if (stride > 0 && grid > stride / share) grid = stride / share;
        cudaLaunchConfig_t cfg{};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3(kTGThreads, 1, 1);
        cfg.stream = stream;
        cfg.attrs = attr;
        cfg.numAttrs = TGC_TG_PDL ? 1 : 0;
        switch (vwf) {
            case 32: e = cudaLaunchKernelEx(&cfg, tgather_flat_kernel<32>, p, share, stride); break;
            case 16: e = cudaLaunchKernelEx(&cfg, tgather_flat_kernel<16>, p, share, stride); break;
            case 8: e = cudaLaunchKernelEx(&cfg, tgather_flat_kernel<8>, p, share, stride); break;
            case 4: e = cudaLaunchKernelEx(&cfg, tgather_flat_kernel<4>, p, share, stride); break;
            case 2: e = cudaLaunchKernelEx(&cfg, tgather_flat_kernel<2>, p, share, stride); break;
            default: e = cudaLaunchKernelEx(&cfg, tgather_flat_kernel<1>, p, share, stride); break;
        }
        if (e == cudaSuccess) e = cudaGetLastError();
        return e == cudaSuccess ? TGC_OK : cuda_fail(e);
    }
    const int64_t waves = (p.total_items + slots - 1) / slots;
    int64_t grid = (p.total_items + waves - 1) / waves;
    // CTA 0 publishes when the chunks are few enough for its threads to watch them without
    // falling behind; otherwise the CTA whose count completes a chunk publishes it
    p.publish = TGC_TG_REL_POLL && L.progress != nullptr &&
                (int64_t)L.nranks * L.nseg <= (int64_t)TGC_TG_PUBLISH_MAX_CHUNKS;
    if (p.publish) ++grid;

    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kTGThreads, 1, 1);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = TGC_TG_REL_PDL ? 1 : 0;
    switch (vw) {
        case 16: e = cudaLaunchKernelEx(&cfg, tgather_kernel<16>, p); break;
        case 8: e = cudaLaunchKernelEx(&cfg, tgather_kernel<8>, p); break;
        case 4: e = cudaLaunchKernelEx(&cfg, tgather_kernel<4>, p); break;
        case 2: e = cudaLaunchKernelEx(&cfg, tgather_kernel<2>, p); break;
        default: e = cudaLaunchKernelEx(&cfg, tgather_kernel<1>, p); break;
    }
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? TGC_OK : cuda_fail(e);
}

}  // namespace tgc
