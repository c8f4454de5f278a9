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
// device current, cudaGetSymbolAddress resolves the real address, which is
// then kept for that device's context (a cudaDeviceReset gives a new context,
// and its first call looks the address up again; a failed lookup is retried
// on the next call).  The first call on a device should therefore come before
// any stream capture on that device.
//
// All calls on a device share the one array, and it keeps whatever the last
// call wrote.  Nothing in it has to start at zero: every call runs the
// tile-map and list kernels, which rewrite every entry the forward kernel
// reads.  For that reason the entry point refuses fm_options.reuse_tile_map:
// the array may hold another problem's lists.  Calls whose work overlaps on
// the GPU (different streams, or different host threads without ordering)
// race on the array and give wrong results.  Order them on one stream, or
// synchronise between them.
#include <cuda_runtime.h>
#include <stdio.h>

#include <mutex>

#include "fm_internal.h"

namespace fm {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[FM_NOALLOC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;

// Device address of the array, per device, with the unique id of the context
// it was looked up in: a new primary context (after cudaDeviceReset) may
// place the array elsewhere, so a changed id means a fresh lookup.  Only a
// successful lookup is kept; a failed one is tried again on the next call.
struct DeviceScratch {
    void *ptr = nullptr;
    unsigned long long ctx_id = 0;
};
DeviceScratch g_devices[MAX_DEVICES];
std::mutex g_devices_mu;

using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
using CtxGetCurrentFn = CUresult (*)(CUcontext *);

// Unique id of the calling thread's current context (0 if unknown).
unsigned long long current_context_id() {
    static CtxGetIdFn get_id = nullptr;
    static CtxGetCurrentFn get_cur = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &a, 12000, cudaEnableDefault, &qa) ==
                cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &b, 12000, cudaEnableDefault,
                                             &qb) == cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_id = reinterpret_cast<CtxGetIdFn>(a);
            get_cur = reinterpret_cast<CtxGetCurrentFn>(b);
        }
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_id && get_cur && get_cur(&ctx) == CUDA_SUCCESS && ctx &&
        get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// The array's device address on `dev`, which must be current.  The lookup
// (cudaGetSymbolAddress) runs on the first call in a context only.
cudaError_t scratch_address(int dev, void **out) {
    std::lock_guard<std::mutex> lock(g_devices_mu);
    DeviceScratch &ds = g_devices[dev];
    const unsigned long long id = current_context_id();
    if (ds.ptr && id != 0 && id == ds.ctx_id) {
        *out = ds.ptr;
        return cudaSuccess;
    }
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) return e != cudaSuccess ? e : cudaErrorInvalidSymbol;
    ds.ptr = p;
    ds.ctx_id = id;
    *out = p;
    return cudaSuccess;
}

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
    // The array may hold another problem's tile map and lists: a reused map
    // could walk lists of the wrong length.  Refused before anything else.
    if (opt && opt->reuse_tile_map != 0) {
        set_error_detail("flashmask_fwd_noalloc: reuse_tile_map is not accepted (the static "
                         "scratch is shared by every call)");
        return FM_ERR_INVALID_ARG;
    }
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
    CallerContext keep;
    int dev = 0;
    cudaError_t e = bind_owner(q, &dev);
    if (e != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
        set_error_detail("flashmask_fwd_noalloc: q is not device memory of a usable device");
        return FM_ERR_INVALID_ARG;
    }
    void *scratch = nullptr;
    e = scratch_address(dev, &scratch);
    if (e != cudaSuccess) {
        char msg[160];
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the static scratch: %s",
                 cudaGetErrorString(e));
        set_error_detail(msg);
        return FM_ERR_CUDA;
    }
    return flashmask_fwd(p, opt, q, k, v, lts, lte, uts, ute, o, lse, scratch,
                         FM_NOALLOC_SCRATCH_BYTES, stream);
}
