// api.cu -- the C ABI of libflashmask (declared in include/flashmask.h):
// argument checks, workspace layout, TMA tensor maps and kernel launches.
// Nothing here computes attention; every step runs in the CUDA kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "fm_internal.h"

namespace fm {
namespace {

constexpr uint64_t DEFAULT_TIMEOUT_NS = 1000000000ull;
constexpr size_t WS_ALIGN = 256;
constexpr unsigned long long MAX_SELFTEST_NS = 10000000000ull;  // 10 s

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool supported_dims(int d, int dv) {
    return (d == 64 && dv == 64) || (d == 128 && dv == 128) || (d == 192 && dv == 128) ||
           (d == 256 && dv == 256);
}

fm_status make_geometry(const fm_problem *p, const fm_options *opt, Geometry *g) {
    if (!p) return FM_ERR_INVALID_ARG;
    if (p->B < 1 || p->H < 1 || p->N < 1 || p->N > (1 << 24) || p->d < 1 || p->dv < 1)
        return FM_ERR_INVALID_ARG;
    if (!(p->Hm == 1 || p->Hm == p->H)) return FM_ERR_INVALID_ARG;
    if (p->causal != 0 && p->causal != 1) return FM_ERR_INVALID_ARG;
    if (!isfinite(p->scale)) return FM_ERR_INVALID_ARG;
    if (opt && opt->debug_bounds != 0 && opt->debug_bounds != 1) return FM_ERR_INVALID_ARG;
    if (!supported_dims(p->d, p->dv)) return FM_ERR_UNSUPPORTED;
    // Grid limits: H and B are grid dimensions y and z.
    if (p->H > 65535 || p->B > 65535) return FM_ERR_INVALID_ARG;
    g->B = p->B;
    g->H = p->H;
    g->Hm = p->Hm;
    g->N = p->N;
    g->d = p->d;
    g->dv = p->dv;
    g->T = (p->N + TILE - 1) / TILE;
    g->Npad = g->T * TILE;
    g->scale = p->scale > 0.f ? p->scale : 1.0f / sqrtf(static_cast<float>(p->d));
    g->causal = p->causal;
    g->timeout_ns =
        (opt && opt->wait_timeout_ns) ? static_cast<uint64_t>(opt->wait_timeout_ns) : DEFAULT_TIMEOUT_NS;
    g->deterministic = opt ? opt->deterministic : 0;
    g->sink = opt ? opt->sink : nullptr;
    g->dsink = opt ? opt->dsink : nullptr;
    if (g->dsink && !g->sink) return FM_ERR_INVALID_ARG;  // a gradient needs its logits
    g->reuse_map = opt ? opt->reuse_tile_map : 0;
    if (g->reuse_map != 0 && g->reuse_map != 1) return FM_ERR_INVALID_ARG;
    g->debug_bounds = opt ? opt->debug_bounds : 0;
    g->acc32 = opt ? opt->accumulate_f32 : 0;
    if (g->acc32 != 0 && g->acc32 != 1) return FM_ERR_INVALID_ARG;
    g->drop_load = opt ? opt->debug_drop_load : 0;
    if (g->drop_load < 0) return FM_ERR_INVALID_ARG;
    // The list and map sizes must fit the int indexing of the kernels.
    const double entries = static_cast<double>(g->B) * g->Hm * g->T * g->T;
    if (entries > 2.0e9) return FM_ERR_INVALID_ARG;
    return FM_OK;
}

fm_status check_mask(const MaskPtrs &m) {
    if ((m.lts == nullptr) != (m.lte == nullptr)) return FM_ERR_INVALID_ARG;
    if ((m.uts == nullptr) != (m.ute == nullptr)) return FM_ERR_INVALID_ARG;
    const int32_t *v[4] = {m.lts, m.lte, m.uts, m.ute};
    for (auto x : v)
        if (x && !aligned16(x)) return FM_ERR_INVALID_ARG;
    return FM_OK;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// cuCtxGetCurrent / cuCtxSetCurrent through the same route.
using CtxGetFn = CUresult (*)(CUcontext *);
using CtxSetFn = CUresult (*)(CUcontext);
struct CtxFns {
    CtxGetFn get = nullptr;
    CtxSetFn set = nullptr;
};

const CtxFns &ctx_fns() {
    static CtxFns fns;
    static std::once_flag once;
    std::call_once(once, [] {
        void *g = nullptr, *s = nullptr;
        cudaDriverEntryPointQueryResult qg, qs;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &g, 12000, cudaEnableDefault,
                                             &qg) == cudaSuccess &&
            qg == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxSetCurrent", &s, 12000, cudaEnableDefault,
                                             &qs) == cudaSuccess &&
            qs == cudaDriverEntryPointSuccess) {
            fns.get = reinterpret_cast<CtxGetFn>(g);
            fns.set = reinterpret_cast<CtxSetFn>(s);
        }
    });
    return fns;
}

// Tensor [B, N, H, dim] bf16 seen by TMA as 4-D (dim, H, N, B), box
// (64, 1, rows, 1), 128-byte swizzle; rows past N read as zeros.
// Last encoder failure on this thread: which tensor and the driver's code.
thread_local char g_encode_detail[160] = "";

bool encode_bnhd(CUtensorMap *map, const void *base, int B, int N, int H, int dim, int rows,
                 bool fp16 = false) {
    EncodeTiledFn enc = get_encoder();
    if (!enc) {
        snprintf(g_encode_detail, sizeof(g_encode_detail), "driver entry point not found");
        return false;
    }
    cuuint64_t gdim[4] = {static_cast<cuuint64_t>(dim), static_cast<cuuint64_t>(H),
                          static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(B)};
    cuuint64_t gstride[3] = {static_cast<cuuint64_t>(dim) * 2,
                             static_cast<cuuint64_t>(H) * dim * 2,
                             static_cast<cuuint64_t>(N) * H * dim * 2};
    cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(rows), 1};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    CUresult r = enc(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     4, const_cast<void *>(base), gdim,
                     gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        snprintf(g_encode_detail, sizeof(g_encode_detail),
                 "CUresult %d for base %p dims (%d,%d,%d,%d) rows %d", static_cast<int>(r), base,
                 dim, H, N, B, rows);
    return r == CUDA_SUCCESS;
}

// Makes the device that owns `anchor` (device memory of the caller) current
// for this library on the calling thread, which also binds its primary
// context there (the tensor-map encoder is a driver call and needs one), then
// checks that it is an sm_103 part.  Threads the library has not seen before,
// such as an autograd worker, have no context bound otherwise.
bool device_ok(const void *anchor) {
    int dev = 0;
    cudaPointerAttributes attr;
    if (anchor && cudaPointerGetAttributes(&attr, anchor) == cudaSuccess &&
        (attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged))
        dev = attr.device;
    else if (cudaGetDevice(&dev) != cudaSuccess)
        return false;
    if (cudaSetDevice(dev) != cudaSuccess) return false;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
        return false;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return false;
    return major == 10 && minor == 3;
}

}  // namespace

size_t carve_workspace(const Geometry &g, bool bwd, void *base, Workspace *ws) {
    size_t off = 0;
    auto take = [&](size_t bytes) -> void * {
        void *p = base ? static_cast<char *>(base) + off : nullptr;
        off = align_up(off + bytes, WS_ALIGN);
        return p;
    };
    const size_t BM = static_cast<size_t>(g.B) * g.Hm;
    const size_t TT = static_cast<size_t>(g.T) * g.T;
    Workspace w;
    w.vec = static_cast<int4 *>(take(BM * g.Npad * sizeof(int4)));
    w.cls = static_cast<uint8_t *>(take(BM * TT));
    w.fwd_list = static_cast<int *>(take(BM * TT * sizeof(int)));
    w.fwd_cnt = static_cast<int *>(take(BM * g.T * sizeof(int)));
    w.bwd_list = static_cast<int *>(take(BM * TT * sizeof(int)));
    w.bwd_cnt = static_cast<int *>(take(BM * g.T * sizeof(int)));
    const size_t TP = (static_cast<size_t>(g.T) + 1) / 2;
    w.pair_list = static_cast<int *>(take(BM * TP * g.T * sizeof(int)));
    w.pair_cnt = static_cast<int *>(take(BM * TP * sizeof(int)));
    w.pair_order = static_cast<int *>(take(BM * TP * sizeof(int)));
    w.lse2 = nullptr;
    w.delta = nullptr;
    w.v16 = nullptr;
    w.do16 = nullptr;
    w.sink_part = nullptr;
    w.range_part = nullptr;
    w.scales = nullptr;
    w.dqacc = nullptr;
    if (bwd) {
        const size_t rows = static_cast<size_t>(g.B) * g.H * g.Npad;
        w.lse2 = static_cast<float *>(take(rows * sizeof(float)));
        w.delta = static_cast<float *>(take(rows * sizeof(float)));
        const size_t vbytes = static_cast<size_t>(g.B) * g.N * g.H * g.dv * 2;
        w.v16 = fused_dq(g) ? nullptr : take(vbytes);  // the one-pass kernel converts V itself
        w.do16 = take(vbytes);
        w.sink_part = static_cast<float *>(take(rows / 16 * sizeof(float)));
        const size_t bht = static_cast<size_t>(g.B) * g.H * g.T;
        w.range_part = static_cast<uint2 *>(take(bht * sizeof(uint2)));
        w.scales = static_cast<float4 *>(take(static_cast<size_t>(g.B) * g.H * sizeof(float4)));
        if (fused_dq(g))
            w.dqacc = static_cast<float4 *>(take(rows * g.d * sizeof(float)));
    }
    if (ws) *ws = w;
    return off;
}

}  // namespace fm

using namespace fm;

namespace {

fm_status prepare(const fm_problem *p, const fm_options *opt, bool bwd, const MaskPtrs &m,
                  void *workspace, size_t ws_bytes, Geometry *g, Workspace *ws) {
    fm_status s = make_geometry(p, opt, g);
    if (s != FM_OK) return s;
    s = check_mask(m);
    if (s != FM_OK) return s;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % WS_ALIGN) != 0)
        return FM_ERR_WORKSPACE;
    if (carve_workspace(*g, bwd, nullptr, nullptr) > ws_bytes) return FM_ERR_WORKSPACE;
    carve_workspace(*g, bwd, workspace, ws);
    if (!device_ok(workspace)) return FM_ERR_UNSUPPORTED;
    return FM_OK;
}

thread_local char g_detail[256] = "";

fm_status fail(cudaError_t e, const char *what) {
    snprintf(g_detail, sizeof(g_detail), "%s: %s (%d)", what, cudaGetErrorString(e),
             static_cast<int>(e));
    return FM_ERR_CUDA;
}

fm_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FM_OK : fail(e, "launch"); }

Recorder recorder(const fm_options *opt) {
    Recorder r;
    if (opt && opt->kernel_events && opt->n_kernel_events > 0) {
        r.ev = reinterpret_cast<cudaEvent_t *>(opt->kernel_events);
        r.n = opt->n_kernel_events;
    }
    return r;
}

// Tile map, then the per-query-tile lists of kept key tiles.
cudaError_t map_and_lists(const Geometry &g, const MaskPtrs &m, const Workspace &ws,
                          cudaStream_t st, Recorder &rec) {
    rec.before(st);
    cudaError_t e = launch_classify(g, m, ws, st);
    rec.after(st);
    if (e != cudaSuccess) return e;
    rec.before(st);
    e = launch_fwd_lists(g, ws, st);
    rec.after(st);
    return e;
}

}  // namespace

namespace fm {
// Sets the text flashmask_last_error_detail returns on this thread.
void set_error_detail(const char *msg) { snprintf(g_detail, sizeof(g_detail), "%s", msg); }
// Makes the device owning `anchor` current for this thread and checks it.
bool bind_device(const void *anchor) { return device_ok(anchor); }

CallerContext::CallerContext() {
    const CtxFns &f = ctx_fns();
    valid_ = f.get && f.set && f.get(&saved_) == CUDA_SUCCESS;
}

CallerContext::~CallerContext() {
    if (!valid_) return;
    const CtxFns &f = ctx_fns();
    CUcontext now = nullptr;
    if (f.get(&now) == CUDA_SUCCESS && now != saved_) f.set(saved_);
}
}  // namespace fm

extern "C" {

size_t flashmask_workspace_size(const fm_problem *p, const fm_options *opt, int is_bwd) {
    Geometry g;
    if (make_geometry(p, opt, &g) != FM_OK) return 0;
    return carve_workspace(g, is_bwd != 0, nullptr, nullptr);
}

fm_status flashmask_classify(const fm_problem *p, const int32_t *lts, const int32_t *lte,
                             const int32_t *uts, const int32_t *ute, uint8_t *tile_class,
                             void *workspace, size_t ws_bytes, void *stream) {
    CallerContext keep;
    Geometry g;
    Workspace ws;
    MaskPtrs m{lts, lte, uts, ute};
    fm_status s = prepare(p, nullptr, false, m, workspace, ws_bytes, &g, &ws);
    if (s != FM_OK) return s;
    if (!tile_class) return FM_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_classify(g, m, ws, st);
    if (e != cudaSuccess) return fail(e, "classify launch");
    const size_t bytes = static_cast<size_t>(g.B) * g.Hm * g.T * g.T;
    return cuda_status(
        cudaMemcpyAsync(tile_class, ws.cls, bytes, cudaMemcpyDeviceToDevice, st));
}

fm_status flashmask_count_unmasked(const fm_problem *p, const int32_t *lts, const int32_t *lte,
                                   const int32_t *uts, const int32_t *ute,
                                   unsigned long long *counts, void *stream) {
    CallerContext keep;
    Geometry g;
    fm_status s = make_geometry(p, nullptr, &g);
    if (s != FM_OK) return s;
    MaskPtrs m{lts, lte, uts, ute};
    s = check_mask(m);
    if (s != FM_OK) return s;
    if (!counts || (reinterpret_cast<uintptr_t>(counts) & 7u)) return FM_ERR_INVALID_ARG;
    if (!device_ok(counts)) return FM_ERR_UNSUPPORTED;
    return cuda_status(launch_count(g, m, counts, static_cast<cudaStream_t>(stream)));
}

fm_status flashmask_fwd(const fm_problem *p, const fm_options *opt, const void *q, const void *k,
                        const void *v, const int32_t *lts, const int32_t *lte,
                        const int32_t *uts, const int32_t *ute, void *o, float *lse,
                        void *workspace, size_t ws_bytes, void *stream) {
    CallerContext keep;
    Geometry g;
    Workspace ws;
    MaskPtrs m{lts, lte, uts, ute};
    const void *ptrs[] = {q, k, v, o, lse};
    for (auto x : ptrs)
        if (!x || !aligned16(x)) return FM_ERR_INVALID_ARG;
    fm_status s = prepare(p, opt, false, m, workspace, ws_bytes, &g, &ws);
    if (s != FM_OK) return s;
    CUtensorMap tq, tk, tv, to;
    const int kr = fwd_key_rows(g.d, g.dv);
    if (!encode_bnhd(&tq, q, g.B, g.N, g.H, g.d, 128) ||
        !encode_bnhd(&tk, k, g.B, g.N, g.H, g.d, kr) ||
        !encode_bnhd(&tv, v, g.B, g.N, g.H, g.dv, kr) ||
        !encode_bnhd(&to, o, g.B, g.N, g.H, g.dv, 128))
        return fail(cudaErrorInvalidValue, g_encode_detail);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Recorder rec = recorder(opt);
    cudaError_t e = g.reuse_map ? cudaSuccess : map_and_lists(g, m, ws, st, rec);
    if (e == cudaSuccess && g.debug_bounds) e = launch_validate_lists(g, ws, st);
    if (e == cudaSuccess) {
        FwdArgs a{&tq, &tk, &tv, kr, &to, o, lse};
        rec.before(st);
        e = launch_fwd(g, ws, a, st);
        rec.after(st);
    }
    return cuda_status(e);
}

fm_status flashmask_bwd(const fm_problem *p, const fm_options *opt, const void *q, const void *k,
                        const void *v, const void *o, const float *lse, const void *dout,
                        const int32_t *lts, const int32_t *lte, const int32_t *uts,
                        const int32_t *ute, void *dq, void *dk, void *dv, void *workspace,
                        size_t ws_bytes, void *stream) {
    CallerContext keep;
    Geometry g;
    Workspace ws;
    MaskPtrs m{lts, lte, uts, ute};
    const void *ptrs[] = {q, k, v, o, lse, dout, dq, dk, dv};
    for (auto x : ptrs)
        if (!x || !aligned16(x)) return FM_ERR_INVALID_ARG;
    fm_status s = prepare(p, opt, true, m, workspace, ws_bytes, &g, &ws);
    if (s != FM_OK) return s;
    CUtensorMap tq_q, tk_k, tv_k, tdo_q;  // maps for the dq kernel (query-side)
    CUtensorMap tq_k, tk_kv, tv_kv, tdo_k;  // maps for the dkdv kernel (key-side)
    CUtensorMap tdq_o, tdk_o, tdv_o;        // the gradients, stored by TMA
    const int dq_kr = dq_key_rows(g.d, g.dv), kv_qr = dkdv_query_rows(g.d, g.dv);
    // dO and V enter the dP and dV products through their fp16 copies (made by
    // the preprocess kernel); Q and K stay bf16.  The one-pass backward loads
    // the bf16 V instead and converts its tile in shared memory (its query-side
    // maps go unused).
    const bool fused = fused_dq(g);
    const void *v_src = fused ? v : ws.v16;
    if (!encode_bnhd(&tq_q, q, g.B, g.N, g.H, g.d, 128) ||
        !encode_bnhd(&tdo_q, ws.do16, g.B, g.N, g.H, g.dv, 128, true) ||
        !encode_bnhd(&tk_k, k, g.B, g.N, g.H, g.d, dq_kr) ||
        !encode_bnhd(&tv_k, v_src, g.B, g.N, g.H, g.dv, dq_kr, !fused) ||
        !encode_bnhd(&tq_k, q, g.B, g.N, g.H, g.d, kv_qr) ||
        !encode_bnhd(&tdo_k, ws.do16, g.B, g.N, g.H, g.dv, kv_qr, true) ||
        !encode_bnhd(&tk_kv, k, g.B, g.N, g.H, g.d, 128) ||
        !encode_bnhd(&tv_kv, v_src, g.B, g.N, g.H, g.dv, 128, !fused))
        return fail(cudaErrorInvalidValue, g_encode_detail);
    // bf16 outputs are stored by TMA; fp32 accumulation (acc32) adds to them
    // with plain loads and stores, and the maps stay unused.
    memset(&tdq_o, 0, sizeof(tdq_o));
    memset(&tdk_o, 0, sizeof(tdk_o));
    memset(&tdv_o, 0, sizeof(tdv_o));
    if (!g.acc32 && (!encode_bnhd(&tdq_o, dq, g.B, g.N, g.H, g.d, 128) ||
                     !encode_bnhd(&tdk_o, dk, g.B, g.N, g.H, g.d, 128) ||
                     !encode_bnhd(&tdv_o, dv, g.B, g.N, g.H, g.dv, 128)))
        return fail(cudaErrorInvalidValue, g_encode_detail);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    Recorder rec = recorder(opt);
    cudaError_t e = g.reuse_map ? cudaSuccess : map_and_lists(g, m, ws, st, rec);
    if (e == cudaSuccess && g.debug_bounds) e = launch_validate_lists(g, ws, st);
    if (e == cudaSuccess) {
        BwdArgs a;
        a.dq_k_rows = dq_kr;
        a.kv_q_rows = kv_qr;
        a.tm_q = &tq_k;
        a.tm_k = &tk_kv;
        a.tm_v = &tv_kv;
        a.tm_do = &tdo_k;
        a.tm_q_dq = &tq_q;
        a.tm_k_dq = &tk_k;
        a.tm_v_dq = &tv_k;
        a.tm_do_dq = &tdo_q;
        a.tm_dq_out = &tdq_o;
        a.tm_dk_out = &tdk_o;
        a.tm_dv_out = &tdv_o;
        a.o = o;
        a.v = v;
        a.dout = dout;
        a.lse = lse;
        a.dq = dq;
        a.dk = dk;
        a.dv = dv;
        e = launch_bwd(g, ws, a, st, rec);
    }
    return cuda_status(e);
}

fm_status flashmask_selftest_wait(unsigned long long timeout_ns, void *stream) {
    CallerContext keep;
    if (timeout_ns == 0 || timeout_ns > MAX_SELFTEST_NS) return FM_ERR_INVALID_ARG;
    if (!device_ok(nullptr)) return FM_ERR_UNSUPPORTED;
    return cuda_status(launch_wait_selftest(timeout_ns, static_cast<cudaStream_t>(stream)));
}

fm_status flashmask_get_error(void *stream) {
    CallerContext keep;
    // The error words read below are those of the stream's device.
    int dev = 0;
    cudaError_t e = cudaStreamGetDevice(static_cast<cudaStream_t>(stream), &dev);
    if (e != cudaSuccess) return fail(e, "cudaStreamGetDevice");
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return fail(e, "cudaSetDevice");
    e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(e, "cudaStreamSynchronize");
    unsigned err = read_clear_error_classify() | read_clear_error_fwd() | read_clear_error_bwd();
    if (err & ERR_BOUNDS) return FM_ERR_DEVICE_BOUNDS;
    return err ? FM_ERR_DEVICE_TIMEOUT : FM_OK;
}

const char *flashmask_last_error_detail(void) { return g_detail; }

const char *flashmask_error_string(fm_status s) {
    switch (s) {
        case FM_OK: return "ok";
        case FM_ERR_INVALID_ARG: return "invalid argument";
        case FM_ERR_UNSUPPORTED: return "unsupported head dims or device";
        case FM_ERR_WORKSPACE: return "workspace missing, unaligned or too small";
        case FM_ERR_CUDA: return "CUDA call failed";
        case FM_ERR_DEVICE_TIMEOUT: return "a kernel gave up on a bounded wait";
        case FM_ERR_DEVICE_BOUNDS: return "a kernel found a work list out of bounds";
    }
    return "unknown status";
}

}  // extern "C"
