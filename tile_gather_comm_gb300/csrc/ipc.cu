// ipc.cu -- device buffers shared between the processes of a multi-process rank
// set: export a buffer as a CUDA IPC handle plus its offset inside its allocation,
// open another process's buffer, close it again (declared in include/tgc.h).
//
// Source: "Triton第四课：基于对称内存融合 AllGather 与 MatMul，提速1.56倍",
// section 对称内存如何打通GPU间访问: every rank's a_shard lives in memory the other
// ranks can address; the producer of each rank copies the others' shards into its
// own aggregate buffer.  Here a rank is a process and "addressable" means mapped
// through an IPC handle; the library keeps no table of what it opened (the caller
// hands the handle back to close).
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace tgc {

static_assert(sizeof(cudaIpcMemHandle_t) == sizeof(((tgc_ipc_handle *)nullptr)->bytes), "IPC handle size");

using AddressRangeFn = PFN_cuMemGetAddressRange_v3020;

// Base of the allocation holding an address (driver entry point, looked up once).
static AddressRangeFn address_range_fn() {
    static AddressRangeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &f, 3020, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<AddressRangeFn>(f);
    });
    return fn;
}

}  // namespace tgc

using namespace tgc;

extern "C" {

int tgc_ipc_export(const void *d_ptr, tgc_ipc_handle *out) {
    if (d_ptr == nullptr || out == nullptr) return TGC_ERR_INVALID_ARG;
    auto range = address_range_fn();
    if (range == nullptr) return TGC_ERR_CUDA;
    CUdeviceptr base = 0;
    size_t size = 0;
    if (range(&base, &size, reinterpret_cast<CUdeviceptr>(d_ptr)) != CUDA_SUCCESS) return TGC_ERR_CUDA;
    cudaIpcMemHandle_t h{};
    const cudaError_t e = cudaIpcGetMemHandle(&h, reinterpret_cast<void *>(base));
    if (e != cudaSuccess) return cuda_fail(e);
    std::memset(out, 0, sizeof *out);
    std::memcpy(out->bytes, &h, sizeof h);
    out->offset = (uint64_t)(reinterpret_cast<uintptr_t>(d_ptr) - (uintptr_t)base);
    return TGC_OK;
}

int tgc_ipc_open(const tgc_ipc_handle *h, void **d_ptr_out) {
    if (h == nullptr || d_ptr_out == nullptr) return TGC_ERR_INVALID_ARG;
    cudaIpcMemHandle_t ch{};
    std::memcpy(&ch, h->bytes, sizeof ch);
    void *base = nullptr;
    const cudaError_t e = cudaIpcOpenMemHandle(&base, ch, cudaIpcMemLazyEnablePeerAccess);
    if (e != cudaSuccess) return cuda_fail(e);
    *d_ptr_out = static_cast<uint8_t *>(base) + h->offset;
    return TGC_OK;
}

int tgc_ipc_close(void *d_ptr, const tgc_ipc_handle *h) {
    if (d_ptr == nullptr || h == nullptr) return TGC_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(d_ptr) < h->offset) return TGC_ERR_INVALID_ARG;
    const cudaError_t e = cudaIpcCloseMemHandle(static_cast<uint8_t *>(d_ptr) - h->offset);
    return e == cudaSuccess ? TGC_OK : cuda_fail(e);
}

}  // extern "C"
