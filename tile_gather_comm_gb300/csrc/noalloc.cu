// noalloc.cu -- tgc_ag_matmul_noalloc: the fused AllGather-MatMul with no
// device allocation at all.
//
// Some callers cannot call cudaMalloc: code that runs under a memory manager
// which owns every byte of device memory and forbids raw allocations, code on
// a latency-critical path where an allocation (and the implicit
// synchronisation some allocators perform) is not allowed after start-up, and
// host threads that must never touch the allocator while another thread holds
// it.  tgc_ag_matmul allocates its temporaries and tgc_ag_matmul_ex needs a
// caller-allocated workspace and flag array; this entry point instead keeps
// that scratch -- status word, ticket dispenser, per-block piece counters,
// per-block progress flags, per-tile-row counters and the ready ring -- in one
// fixed array in device memory that the library declares statically.  The
// caller passes only inputs and outputs.
//
// The array is a property of the loaded module: every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits, and every
// call on a device shares that device's copy.
#include <cstdint>

#include <cuda_runtime.h>

#include "internal.h"

namespace tgc {

constexpr size_t kNoAllocScratchBytes = TGC_NOALLOC_SCRATCH_BYTES;
constexpr int64_t kNoAllocMaxBlocks = TGC_NOALLOC_MAX_BLOCKS;

// The scratch.  Host code must not use this name as an address (on the host
// it is only a stand-in for the device symbol); it takes the device address
// from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

// Device address of the scratch on the current device.  It is looked up on
// every call (with the caller's device current) rather than cached: the lookup
// allocates nothing, and a cached address would go stale if the device were
// reset and the module loaded again.
int scratch_address(uint8_t **out) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    *out = static_cast<uint8_t *>(p);
    return TGC_OK;
}

struct ScratchLayout {
    size_t ws_bytes;      // workspace of the fused kernel (status, tickets, counters)
    size_t progress_off;  // progress flags, one uint32 per comm block
    size_t total;
};

ScratchLayout scratch_layout(int64_t nblocks, int64_t M) {
    ScratchLayout l{};
    l.ws_bytes = workspace_layout(nblocks, M > 0 ? (M + kTileM - 1) / kTileM : 0).total;
    l.progress_off = (l.ws_bytes + 255) / 256 * 256;
    l.total = l.progress_off + (size_t)nblocks * 4;
    return l;
}

}  // namespace
}  // namespace tgc

using namespace tgc;

extern "C" int tgc_ag_matmul_noalloc(const void *const *a_shards, int nranks, const void *B, void *C, void *a_out,
                                     int64_t M, int64_t K, int64_t N, int64_t comm_block_rows,
                                     cudaStream_t stream) {
    tgc_ag_matmul_args a{};
    a.a_shards = a_shards;
    a.nranks = nranks;
    a.B = B;
    a.C = C;
    a.a_out = a_out;
    a.M = M;
    a.K = K;
    a.N = N;
    a.comm_block_rows = comm_block_rows;
    a.rank = 0;
    a.mode = TGC_MODE_FUSED;
    a.pivot = TGC_PIVOT_AUTO;
    a.epoch = 1;
    a.sync = 1;
    a.stream = stream;

    // Host-side checks first, with placeholder scratch pointers: nothing is
    // enqueued for an invalid or oversized call.
    {
        tgc_ag_matmul_args probe = a;
        alignas(256) static const uint64_t placeholder[32] = {0};
        probe.progress = reinterpret_cast<uint32_t *>(const_cast<uint64_t *>(placeholder));
        probe.workspace = const_cast<uint64_t *>(placeholder);
        probe.workspace_bytes = kNoAllocScratchBytes;
        AGCheck chk{};
        const int rc = ag_validate(probe, chk);
        if (rc == 1) return TGC_OK;  // empty problem
        if (rc < 0 && rc != TGC_ERR_WORKSPACE) return rc;
        if (rc == TGC_ERR_WORKSPACE || chk.nblocks > kNoAllocMaxBlocks ||
            scratch_layout(chk.nblocks, M).total > kNoAllocScratchBytes)
            return TGC_ERR_TOO_LARGE;
    }
    const int64_t nblocks = M / comm_block_rows;
    const ScratchLayout l = scratch_layout(nblocks, M);

    uint8_t *base = nullptr;
    int rc = scratch_address(&base);
    if (rc != TGC_OK) return rc;
    // The scratch keeps whatever the previous call left (a failed call may
    // leave counters or flags set): clear the part this call uses, so the
    // counters, ticket dispenser and status start at zero and no flag equals
    // the epoch (1) this call publishes.
    cudaError_t e = cudaMemsetAsync(base, 0, l.total, stream);
    if (e != cudaSuccess) return cuda_fail(e);
    a.workspace = base;
    a.workspace_bytes = l.ws_bytes;
    a.progress = reinterpret_cast<uint32_t *>(base + l.progress_off);
    return tgc_ag_matmul_ex(&a);  // fused kernel on the scratch; synchronizes and returns the device status
}
