// chunks.cu -- context-parallel chunks on one GPU.
//
// "FlashMask-3: Efficient and Expressive Mask-Aware Distributed Attention"
// (abstract): under any multi-chunk context-parallel assignment, per-rank mask
// localization is a zero-communication clip-shift-max on the boundary
// vectors, compatible with the single-GPU kernel.  The sequence is cut into
// chunks of equal length L starting at multiples of L.  For a (query chunk,
// key chunk) pair, localize_kernel writes the vectors of the local problem of
// size L; the pair then runs through the ordinary forward / backward, and the
// partial results of a query chunk's pairs are combined:
// - merge_kernel, merge_lse_kernel: log-sum-exp merge of a partial (O, LSE)
//   into fp32 running values; finish_kernel: the merged O as bf16 and its LSE;
// - accumulate_kernel / to_bf16_kernel: fp32 sums of partial gradients.
// All of them are elementwise and bound by HBM bandwidth.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fm_device.cuh"
#include "fm_internal.h"

namespace fm {
namespace {

// Local vectors of one pair: x' = max(min(clamp(x, 0, N), q0 + L) - q0, 0).
// An absent interval is written empty (LT = [L, L), UT = [0, 0)).
__global__ void __launch_bounds__(256) localize_kernel(
    int N, int rows, int q0, int k0, int L, const int32_t *__restrict__ lts,
    const int32_t *__restrict__ lte, const int32_t *__restrict__ uts,
    const int32_t *__restrict__ ute, int32_t *__restrict__ olts, int32_t *__restrict__ olte,
    int32_t *__restrict__ outs, int32_t *__restrict__ oute) {
    const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<long long>(rows) * L) return;
    const int r = static_cast<int>(idx / L), jl = static_cast<int>(idx % L);
    const size_t src = static_cast<size_t>(r) * N + k0 + jl;
    auto loc = [&](const int32_t *v, int absent) {
        int x = v ? v[src] : absent;
        x = min(max(x, 0), N);
        return max(min(x, q0 + L) - q0, 0);
    };
    olts[idx] = loc(lts, N);
    olte[idx] = loc(lte, N);
    outs[idx] = loc(uts, 0);
    oute[idx] = loc(ute, 0);
}

// O [L, H, dv] with 8 values per thread; LSE [H, L] (row (i, h) -> h * L + i).
__global__ void __launch_bounds__(256) merge_init_kernel(long long n8, int L, int H, int dv,
                                                         float *__restrict__ o_acc,
                                                         float *__restrict__ lse_acc) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t < n8) {
        reinterpret_cast<float4 *>(o_acc)[2 * t] = make_float4(0.f, 0.f, 0.f, 0.f);
        reinterpret_cast<float4 *>(o_acc)[2 * t + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (t < static_cast<long long>(L) * H) lse_acc[t] = -INFINITY;
}

// Weights of the log-sum-exp merge of a (running) and b (new part).
__device__ __forceinline__ void merge_weights(float a, float b, float &wa, float &wb,
                                              float &lse) {
    const float m = fmaxf(a, b);
    if (m == -INFINITY) {  // neither has a visible key yet
        wa = 0.f;
        wb = 0.f;
        lse = -INFINITY;
        return;
    }
    const float ea = expf(a - m), eb = expf(b - m);
    const float s = ea + eb;
    wa = ea / s;
    wb = eb / s;
    lse = m + logf(s);
}

// One thread per 8 consecutive values of one (row, head): its weights come
// from the two LSEs of that (row, head).
__global__ void __launch_bounds__(256) merge_kernel(long long n8, int L, int H, int dv,
                                                    const uint4 *__restrict__ o_part,
                                                    const float *__restrict__ lse_part,
                                                    float *__restrict__ o_acc,
                                                    float *__restrict__ lse_acc) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= n8) return;
    const long long row = (t * 8) / dv;  // (i, h) in [L, H] order
    const int i = static_cast<int>(row / H), h = static_cast<int>(row % H);
    const size_t li = static_cast<size_t>(h) * L + i;
    float wa, wb, lse;
    merge_weights(lse_acc[li], lse_part[li], wa, wb, lse);
    (void)lse;
    const uint4 p = o_part[t];
    const uint32_t pw[4] = {p.x, p.y, p.z, p.w};
    float4 *acc = reinterpret_cast<float4 *>(o_acc) + 2 * t;
    float4 a0 = acc[0], a1 = acc[1];
    float pv[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pw[k]));
        pv[2 * k] = f.x;
        pv[2 * k + 1] = f.y;
    }
    a0 = make_float4(a0.x * wa + pv[0] * wb, a0.y * wa + pv[1] * wb, a0.z * wa + pv[2] * wb,
                     a0.w * wa + pv[3] * wb);
    a1 = make_float4(a1.x * wa + pv[4] * wb, a1.y * wa + pv[5] * wb, a1.z * wa + pv[6] * wb,
                     a1.w * wa + pv[7] * wb);
    acc[0] = a0;
    acc[1] = a1;
}

// The merged LSE, after merge_kernel has read the old one (next in the stream).
__global__ void __launch_bounds__(256) merge_lse_kernel(long long rows,
                                                        const float *__restrict__ lse_part,
                                                        float *__restrict__ lse_acc) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= rows) return;
    float wa, wb, lse;
    merge_weights(lse_acc[t], lse_part[t], wa, wb, lse);
    lse_acc[t] = lse;
}

// Merged O (already normalised: the parts are) to bf16; LSE to the caller's
// layout, head h of the chunk at lse_out + h * lse_stride.
__global__ void __launch_bounds__(256) finish_kernel(long long n8, int L, int H, int dv,
                                                     const float *__restrict__ o_acc,
                                                     const float *__restrict__ lse_acc,
                                                     uint4 *__restrict__ o_out,
                                                     float *__restrict__ lse_out,
                                                     long long lse_stride) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t < n8) {
        const float4 a0 = reinterpret_cast<const float4 *>(o_acc)[2 * t];
        const float4 a1 = reinterpret_cast<const float4 *>(o_acc)[2 * t + 1];
        o_out[t] = make_uint4(pack_bf16(a0.x, a0.y), pack_bf16(a0.z, a0.w),
                              pack_bf16(a1.x, a1.y), pack_bf16(a1.z, a1.w));
    }
    if (t < static_cast<long long>(L) * H) {
        const int h = static_cast<int>(t / L), i = static_cast<int>(t % L);
        lse_out[h * lse_stride + i] = lse_acc[t];
    }
}

__global__ void __launch_bounds__(256) accumulate_kernel(long long n8,
                                                         const uint4 *__restrict__ part,
                                                         float *__restrict__ acc) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= n8) return;
    const uint4 p = part[t];
    const uint32_t pw[4] = {p.x, p.y, p.z, p.w};
    float4 *a = reinterpret_cast<float4 *>(acc) + 2 * t;
    float4 a0 = a[0], a1 = a[1];
    float2 f[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
        f[k] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&pw[k]));
    a[0] = make_float4(a0.x + f[0].x, a0.y + f[0].y, a0.z + f[1].x, a0.w + f[1].y);
    a[1] = make_float4(a1.x + f[2].x, a1.y + f[2].y, a1.z + f[3].x, a1.w + f[3].y);
}

__global__ void __launch_bounds__(256) to_bf16_kernel(long long n8, const float *__restrict__ src,
                                                      uint4 *__restrict__ dst) {
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= n8) return;
    const float4 a0 = reinterpret_cast<const float4 *>(src)[2 * t];
    const float4 a1 = reinterpret_cast<const float4 *>(src)[2 * t + 1];
    dst[t] = make_uint4(pack_bf16(a0.x, a0.y), pack_bf16(a0.z, a0.w), pack_bf16(a1.x, a1.y),
                        pack_bf16(a1.z, a1.w));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

unsigned blocks_for(long long n) { return static_cast<unsigned>((n + 255) / 256); }

fm_status launched(const char *what) {
    const cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) return FM_OK;
    set_error_detail(what);
    return FM_ERR_CUDA;
}

// Shape checks of the merge entry points: O chunk [L, H, dv] bf16 / fp32.
bool merge_shape_ok(int L, int H, int dv) {
    return L >= 1 && H >= 1 && dv >= 8 && dv % 8 == 0 &&
           static_cast<long long>(L) * H * dv / 8 < (1LL << 40) &&
           static_cast<long long>(L) * H < 2147483647LL / 2;
}

}  // namespace
}  // namespace fm

using namespace fm;

extern "C" {

fm_status flashmask_localize(const fm_problem *p, const int32_t *lts, const int32_t *lte,
                             const int32_t *uts, const int32_t *ute, int q0, int k0, int len,
                             int32_t *out_lts, int32_t *out_lte, int32_t *out_uts,
                             int32_t *out_ute, int *local_causal, void *stream) {
    CallerContext keep;
    if (!p || !local_causal || !out_lts || !out_lte || !out_uts || !out_ute)
        return FM_ERR_INVALID_ARG;
    if (p->B < 1 || p->N < 1 || !(p->Hm == 1 || p->Hm == p->H) || p->H < 1)
        return FM_ERR_INVALID_ARG;
    if (p->causal != 0 && p->causal != 1) return FM_ERR_INVALID_ARG;
    if ((lts == nullptr) != (lte == nullptr) || (uts == nullptr) != (ute == nullptr))
        return FM_ERR_INVALID_ARG;
    if (len < 1 || q0 < 0 || k0 < 0 || q0 > p->N - len || k0 > p->N - len ||
        (q0 - k0) % len != 0)
        return FM_ERR_INVALID_ARG;
    if (p->causal && k0 > q0) {  // the key chunk lies after the query chunk: all masked
        *local_causal = -1;
        return FM_OK;
    }
    *local_causal = (p->causal && k0 == q0) ? 1 : 0;
    if (!bind_device(out_lts)) return FM_ERR_UNSUPPORTED;
    const int rows = p->B * p->Hm;
    localize_kernel<<<blocks_for(static_cast<long long>(rows) * len), 256, 0,
                      static_cast<cudaStream_t>(stream)>>>(p->N, rows, q0, k0, len, lts, lte,
                                                           uts, ute, out_lts, out_lte, out_uts,
                                                           out_ute);
    return launched("flashmask_localize: launch");
}

fm_status flashmask_merge_init(int L, int H, int dv, float *o_acc, float *lse_acc,
                               void *stream) {
    CallerContext keep;
    if (!merge_shape_ok(L, H, dv) || !o_acc || !lse_acc || !aligned16(o_acc))
        return FM_ERR_INVALID_ARG;
    if (!bind_device(o_acc)) return FM_ERR_UNSUPPORTED;
    const long long n8 = static_cast<long long>(L) * H * dv / 8;
    const long long n = n8 > static_cast<long long>(L) * H ? n8 : static_cast<long long>(L) * H;
    merge_init_kernel<<<blocks_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        n8, L, H, dv, o_acc, lse_acc);
    return launched("flashmask_merge_init: launch");
}

fm_status flashmask_merge(int L, int H, int dv, const void *o_part, const float *lse_part,
                          float *o_acc, float *lse_acc, void *stream) {
    CallerContext keep;
    if (!merge_shape_ok(L, H, dv) || !o_part || !lse_part || !o_acc || !lse_acc ||
        !aligned16(o_part) || !aligned16(o_acc))
        return FM_ERR_INVALID_ARG;
    if (!bind_device(o_acc)) return FM_ERR_UNSUPPORTED;
    const long long n8 = static_cast<long long>(L) * H * dv / 8;
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    merge_kernel<<<blocks_for(n8), 256, 0, st>>>(n8, L, H, dv,
                                                 static_cast<const uint4 *>(o_part), lse_part,
                                                 o_acc, lse_acc);
    const fm_status s = launched("flashmask_merge: launch");
    if (s != FM_OK) return s;
    const long long rows = static_cast<long long>(L) * H;
    merge_lse_kernel<<<blocks_for(rows), 256, 0, st>>>(rows, lse_part, lse_acc);
    return launched("flashmask_merge: launch");
}

fm_status flashmask_merge_finish(int L, int H, int dv, const float *o_acc, const float *lse_acc,
                                 void *o_out, float *lse_out, long long lse_stride,
                                 void *stream) {
    CallerContext keep;
    if (!merge_shape_ok(L, H, dv) || !o_acc || !lse_acc || !o_out || !lse_out ||
        !aligned16(o_acc) || !aligned16(o_out) || lse_stride < L)
        return FM_ERR_INVALID_ARG;
    if (!bind_device(o_acc)) return FM_ERR_UNSUPPORTED;
    const long long n8 = static_cast<long long>(L) * H * dv / 8;
    const long long n = n8 > static_cast<long long>(L) * H ? n8 : static_cast<long long>(L) * H;
    finish_kernel<<<blocks_for(n), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        n8, L, H, dv, o_acc, lse_acc, static_cast<uint4 *>(o_out), lse_out, lse_stride);
    return launched("flashmask_merge_finish: launch");
}

fm_status flashmask_accumulate(long long n, const void *part, float *acc, void *stream) {
    CallerContext keep;
    if (n < 0 || n % 8 != 0 || !part || !acc || !aligned16(part) || !aligned16(acc))
        return FM_ERR_INVALID_ARG;
    if (n == 0) return FM_OK;
    if (!bind_device(acc)) return FM_ERR_UNSUPPORTED;
    accumulate_kernel<<<blocks_for(n / 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        n / 8, static_cast<const uint4 *>(part), acc);
    return launched("flashmask_accumulate: launch");
}

fm_status flashmask_to_bf16(long long n, const float *src, void *dst, void *stream) {
    CallerContext keep;
    if (n < 0 || n % 8 != 0 || !src || !dst || !aligned16(src) || !aligned16(dst))
        return FM_ERR_INVALID_ARG;
    if (n == 0) return FM_OK;
    if (!bind_device(src)) return FM_ERR_UNSUPPORTED;
    to_bf16_kernel<<<blocks_for(n / 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        n / 8, src, static_cast<uint4 *>(dst));
    return launched("flashmask_to_bf16: launch");
}

}  // extern "C"
