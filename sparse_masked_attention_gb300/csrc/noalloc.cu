// noalloc.cu -- flashmask_fwd_noalloc: the forward pass for callers that
// cannot allocate device memory.
//
// flashmask_fwd needs a caller-provided workspace: the normalised mask
// boundaries, the tile map, and the per-query-tile lists of key tiles.  Some
// callers have no way to obtain one.  Examples: a plugin host that hands out
// only its tensors, code running where cudaMalloc is forbidden or would
// synchronise, or an embedding with no allocator of its own.  This entry
// point takes the workspace from a fixed array compiled into the library
// instead, so the call itself allocates nothing.
//
// The array is a file-scope __device__ variable of FM_NOALLOC_SCRATCH_BYTES
// (16 MiB).  Every GPU that loads this library keeps its own copy until the
// process exits.  In host code the array's name is only a host-side stand-in
// and never a device address.  On the first call on a device, with that
// device current, cudaGetSymbolAddress resolves the real address once.  That
// first call should therefore come before any stream capture on that device.
//
// All calls on a device share the one array, and it keeps whatever the last
// call wrote.  Nothing in it has to start at zero: the tile-map kernel
// rewrites every entry the forward kernels read, on every call.  Calls whose
// work overlaps on the GPU (different streams, or different host threads
// without ordering) race on the array and give wrong results.  Order them on
// one stream, or synchronise between them.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "fm_internal.h"

namespace fm {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FM_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;

struct DeviceScratch {
    std::once_flag once;
    void *ptr = nullptr;
    cudaError_t err = cudaSuccess;
};
DeviceScratch g_devices[MAX_DEVICES];

// Device that owns `p` (device memory), made current for this library.
cudaError_t bind_owner(const void *p, int *dev) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) return e;
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return cudaErrorInvalidDevicePointer;
    *dev = attr.device;
    return cudaSetDevice(attr.device);
}

}  // namespace
}  // namespace fm

extern "C" fm_status flashmask_fwd_noalloc(const fm_problem *p, const fm_options *opt,
                                           const void *q, const void *k, const void *v,
                                           const int32_t *lts, const int32_t *lte,
                                           const int32_t *uts, const int32_t *ute, void *o,
                                           float *lse, void *stream) {
    using namespace fm;
    const size_t need = flashmask_workspace_size(p, opt, 0);
    if (need == 0)  // invalid problem: let the regular entry point name the error
        return flashmask_fwd(p, opt, q, k, v, lts, lte, uts, ute, o, lse, nullptr, 0, stream);
    if (need > FM_NOALLOC_SCRATCH_BYTES) {
        char msg[200];
        snprintf(msg, sizeof(msg),
                 "flashmask_fwd_noalloc: this problem needs %zu bytes of scratch; the static "
                 "scratch holds %zu (use flashmask_fwd with a workspace)",
                 need, static_cast<size_t>(FM_NOALLOC_SCRATCH_BYTES));
        set_error_detail(msg);
        return FM_ERR_WORKSPACE;
    }
    if (!q || !o) return FM_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = bind_owner(q, &dev);
    if (e != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        set_error_detail("flashmask_fwd_noalloc: q is not device memory of a usable device");
        return FM_ERR_INVALID_ARG;
    }
    DeviceScratch &ds = g_devices[dev];
    std::call_once(ds.once, [&ds] {
        ds.err = cudaGetSymbolAddress(&ds.ptr, g_noalloc_scratch);
    });
    if (ds.err != cudaSuccess || !ds.ptr) {
        char msg[160];
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the static scratch: %s",
                 cudaGetErrorString(ds.err));
        set_error_detail(msg);
        return FM_ERR_CUDA;
    }
    return flashmask_fwd(p, opt, q, k, v, lts, lte, uts, ute, o, lse, ds.ptr,
                         FM_NOALLOC_SCRATCH_BYTES, stream);
}
