// bwd.cu -- backward of FlashMask masked attention on tcgen05 tensor cores.
//
// The derivative of O = softmax(Q K^T * scale + M) V (FlashMask README,
// "Formulation").  P is rebuilt from the forward's LSE:
//   P = exp(S * scale - LSE),  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
//   dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// The backward walks the same tile map as the forward: fully masked tiles are
// skipped, and the mask is applied elementwise only on partial tiles.
//
// The dP and dV products run in fp16 (10 mantissa bits against bf16's 7), on
// copies of dO and V scaled by powers of two, one per (batch, head) and
// tensor, that put the tensor's largest magnitude in [2^14, 2^15): inside
// fp16's range, with its precision, over the whole bf16 input range.  D is
// stored times s_o s_v, so the kernels form dS * s_o s_v (exact: a power of
// two changes no rounding, and bf16 keeps fp32's exponent range), and the
// epilogues undo the scales in fp32: dQ and dK times scale / (s_o s_v), dV
// times 1 / s_o.  |dO s_o|, |V s_v| < 2^15 bound every scaled product by
// dv * 2^30 and |D s_o s_v| by dv * 2^30 too (|O| <= max |V|).
//
// Kernels:
//   range        largest |dO| and |V| per 128-row tile of each (batch, head)
//   scale        the per-(batch, head) scales from those maxima
//   preprocess   D * s_o s_v (fp32) and the log2-domain LSE per row, padded
//                to whole tiles; padding rows and fully masked rows get
//                LSE = +inf, so their P is 0; the scaled fp16 copies of dO, V.
//   dq kernel    one CTA per 128-row query tile walks its key tiles:
//                S = Q K^T (bf16) and dP = dO V^T (fp16 copies) as SS MMAs
//                (at d = 192 and 256, dO sits in TMEM and dP is a TS MMA);
//                dS -> TMEM (bf16);
//                dQ += dS K (TS MMA, dS read from TMEM).  Writes dQ once.
//   dkdv kernel  one CTA per 128-key tile walks its query tiles:
//                S^T = K Q^T (bf16) and dP^T = V dO^T (fp16 copies) as SS MMAs
//                (at d = 192 and 256, V sits in TMEM and dP^T is a TS MMA);
//                P^T -> TMEM as fp16, dS^T as bf16; dV += P^T dO (fp16) and
//                dK += dS^T Q (bf16) as TS MMAs.
// No atomics are used.  In deterministic mode the accumulations run in tile
// order, so every gradient is bit-reproducible; otherwise whichever compute
// group is ready goes first.  For d = dv = 256 the accumulators dK and dV do
// not fit in TMEM together, so the dkdv kernel runs twice: once for dV, once
// for dK.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <type_traits>

#include "fm_device.cuh"
#include "fm_internal.h"

namespace fm {

static __device__ unsigned g_err_bwd;

namespace {

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t tmo,
                                          volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, tmo, abort, &g_err_bwd);
    return __all_sync(0xffffffffu, ok);
}

// 32 values of a 128-row output tile (columns 32c .. 32c + 31 of row `row`),
// times `mul`, as bf16 into the 128B-swizzled shared-memory layout of a
// 64-column x 128-row TMA box: box c / 2, 16-byte units 4 (c % 2) .. + 3.
__device__ __forceinline__ void stage_row_bf16(uint8_t *stage, int c, int row,
                                               const float (&v)[32], float mul) {
    uint8_t *box_row = stage + (c / 2) * (128 * 128) + row * 128;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16(v[q * 8 + 0] * mul, v[q * 8 + 1] * mul);
        w.y = pack_bf16(v[q * 8 + 2] * mul, v[q * 8 + 3] * mul);
        w.z = pack_bf16(v[q * 8 + 4] * mul, v[q * 8 + 5] * mul);
        w.w = pack_bf16(v[q * 8 + 6] * mul, v[q * 8 + 7] * mul);
        const int unit = (c % 2) * 4 + q;
        *reinterpret_cast<uint4 *>(box_row + ((unit ^ (row & 7)) * 16)) = w;
    }
}

// --------------------------------------------------------- range and scale
// Magnitudes of bf16 values compare as the unsigned integers of their low 15
// bits (sign cleared); NaN patterns sort above infinity, and both above every
// finite value.
constexpr uint32_t BF16X2_ABS = 0x7fff7fffu;
constexpr uint32_t BF16_INF_BITS = 0x7f80u;

__device__ __forceinline__ uint32_t max_abs_bf16x8(uint32_t m, uint4 a) {
    const uint32_t x = __vmaxu2(a.x & BF16X2_ABS, a.y & BF16X2_ABS);
    const uint32_t y = __vmaxu2(a.z & BF16X2_ABS, a.w & BF16X2_ABS);
    return __vmaxu2(m, __vmaxu2(x, y));
}

// One CTA per (128-row tile, head, batch): the tile's largest |dO| and |V|
// as bf16 bit patterns (8 values per load).
__global__ void __launch_bounds__(256) range_kernel(int N, int H, int dv, int T,
                                                    const uint4 *__restrict__ dout,
                                                    const uint4 *__restrict__ v,
                                                    uint2 *__restrict__ range_part) {
    __shared__ uint32_t red[2][8];
    pdl_wait();  // dO and V may come from the kernels before
    pdl_trigger();
    const int t = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int bh = b * H + h;
    const int r0 = t * TILE, rows = min(TILE, N - r0);
    const int vpr = dv / 8;  // 16-byte vectors per row
    uint32_t mo = 0, mv = 0;
    for (int idx = threadIdx.x; idx < rows * vpr; idx += 256) {
        const int r = idx / vpr, c = idx - r * vpr;
        const size_t off = ((static_cast<size_t>(b) * N + r0 + r) * H + h) * vpr + c;
        mo = max_abs_bf16x8(mo, dout[off]);
        mv = max_abs_bf16x8(mv, v[off]);
    }
    mo = max(mo & 0xffffu, mo >> 16);
    mv = max(mv & 0xffffu, mv >> 16);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        mo = max(mo, __shfl_xor_sync(0xffffffffu, mo, off));
        mv = max(mv, __shfl_xor_sync(0xffffffffu, mv, off));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[0][warp] = mo;
        red[1][warp] = mv;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
        for (int w = 1; w < 8; ++w) {
            mo = max(mo, red[0][w]);
            mv = max(mv, red[1][w]);
        }
        range_part[static_cast<size_t>(bh) * T + t] = make_uint2(mo, mv);
    }
}

// 2^k as a float, for integer k in [-126, 127].
__device__ __forceinline__ float pow2i(int k) {
    return __uint_as_float(static_cast<uint32_t>(k + 127) << 23);
}

// Exponent k of the power of two that puts a largest magnitude (bf16 bits)
// in [2^14, 2^15), kept in [-63, 63] so that 2^-(k_o + k_v) is a normal fp32;
// 0 (no scaling) for an all-zero tensor and when infinity or NaN is present,
// which then propagate as they would unscaled.
__device__ __forceinline__ int range_exponent(uint32_t amax_bits) {
    if (amax_bits == 0 || amax_bits >= BF16_INF_BITS) return 0;
    const int e = static_cast<int>((amax_bits >> 7) & 0xffu);  // biased exponent
    const int k = 14 - (e - 127);  // a subnormal (e = 0) lands far above 63
    return max(-63, min(63, k));
}

// One CTA per (batch, head): the maxima of its row tiles, then the scales.
__global__ void __launch_bounds__(256) scale_kernel(int T, const uint2 *__restrict__ range_part,
                                                    float4 *__restrict__ scales) {
    __shared__ uint32_t red[2][8];
    pdl_wait();  // the range kernel's maxima
    pdl_trigger();
    const int bh = blockIdx.x;
    uint32_t mo = 0, mv = 0;
    for (int t = threadIdx.x; t < T; t += 256) {
        const uint2 m = range_part[static_cast<size_t>(bh) * T + t];
        mo = max(mo, m.x);
        mv = max(mv, m.y);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        mo = max(mo, __shfl_xor_sync(0xffffffffu, mo, off));
        mv = max(mv, __shfl_xor_sync(0xffffffffu, mv, off));
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        red[0][warp] = mo;
        red[1][warp] = mv;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
        for (int w = 1; w < 8; ++w) {
            mo = max(mo, red[0][w]);
            mv = max(mv, red[1][w]);
        }
        const int ko = range_exponent(mo), kv = range_exponent(mv);
        scales[bh] = make_float4(pow2i(ko), pow2i(kv), pow2i(-ko), pow2i(-(ko + kv)));
    }
}

// fp32 accumulation (fm_options.accumulate_f32, the ACC32 instantiations of
// the gradient kernels): 32 values of one output row
// (columns 32c .. 32c + 31), times `mul`, added to that row of an fp32 array.
// Each element has one writer per call, so a plain load and store suffice.
__device__ __forceinline__ void add_row_f32(float *row_ptr, int c, const uint32_t (&r)[32],
                                            float mul) {
    float4 *dst = reinterpret_cast<float4 *>(row_ptr + c * 32);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float4 a = dst[q];
        a.x = fmaf(__uint_as_float(r[4 * q + 0]), mul, a.x);
        a.y = fmaf(__uint_as_float(r[4 * q + 1]), mul, a.y);
        a.z = fmaf(__uint_as_float(r[4 * q + 2]), mul, a.z);
        a.w = fmaf(__uint_as_float(r[4 * q + 3]), mul, a.w);
        dst[q] = a;
    }
}

// ---------------------------------------------------------------- preprocess
// 16 threads per row; each takes 8 consecutive bf16 of dO, O and V at a time.
// Besides D and LSE2 it writes the fp16 copies of dO and V, times their
// (batch, head)'s powers of two s_o and s_v (V only for the split backward:
// the one-pass kernel converts its resident V tile itself).
__device__ __forceinline__ uint4 bf16x8_to_fp16x8(uint4 a, float mul) {
    const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a);
    uint4 r;
    uint32_t *r32 = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(a2[e]);
        r32[e] = pack_fp16(f.x * mul, f.y * mul);
    }
    return r;
}

__global__ void __launch_bounds__(256) preprocess_kernel(
    int N, int H, int dv, int Npad, int rows_total, const __nv_bfloat16 *__restrict__ o,
    const __nv_bfloat16 *__restrict__ dout, const __nv_bfloat16 *__restrict__ v,
    const float *__restrict__ lse, float *__restrict__ lse2, float *__restrict__ delta,
    uint4 *__restrict__ v16, uint4 *__restrict__ do16, const float4 *__restrict__ scales,
    const float *__restrict__ sink, float *__restrict__ sink_part, float4 *__restrict__ dqacc,
    int dq4) {
    __shared__ float sink_rows[16];
    pdl_wait();  // the scales, and the inputs of the kernels before
    pdl_trigger();
    const int r0 = blockIdx.x * 16 + (threadIdx.x >> 4);  // over B*H*Npad
    const int t = threadIdx.x & 15;
    const bool valid = r0 < rows_total;
    const int r = valid ? r0 : 0;
    const int bh = r / Npad, i = r % Npad;
    const int b = bh / H, h = bh % H;
    // fused dQ: the fp32 buffer [B*H][d/4][Npad] starts at 0.  Each block zeroes
    // one contiguous piece of 16 d/4 float4 (the grid, rows_total / 16 blocks,
    // covers it exactly): full lines in address order, issued before the loads.
    if (dqacc) {
        float4 *z = dqacc + static_cast<size_t>(blockIdx.x) * 16 * dq4;
        for (int k = threadIdx.x; k < 16 * dq4; k += 256) z[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    // the row's LSE, loaded with the rest rather than after the row sum
    const float l_row = (valid && t == 0 && i < N) ? lse[static_cast<size_t>(bh) * N + i] : 0.f;
    float acc = 0.f;
    const float4 sc = scales[bh];
    const float sc_o = sc.x, sc_v = sc.y;
    if (valid && i < N) {
        const size_t base = ((static_cast<size_t>(b) * N + i) * H + h) * dv;
        for (int c = t * 8; c < dv; c += 128) {
            const uint4 a = *reinterpret_cast<const uint4 *>(o + base + c);
            const uint4 g = *reinterpret_cast<const uint4 *>(dout + base + c);
            do16[(base + c) / 8] = bf16x8_to_fp16x8(g, sc.x);
            if (v16) {  // the one-pass backward converts V in its own kernel
                const uint4 vv = *reinterpret_cast<const uint4 *>(v + base + c);
                v16[(base + c) / 8] = bf16x8_to_fp16x8(vv, sc.y);
            }
            const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a);
            const __nv_bfloat162 *g2 = reinterpret_cast<const __nv_bfloat162 *>(&g);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 fa = __bfloat1622float2(a2[e]);
                const float2 fg = __bfloat1622float2(g2[e]);
                acc = fmaf(fa.x, fg.x, acc);
                acc = fmaf(fa.y, fg.y, acc);
            }
        }
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off, 16);
    float sink_term = 0.f;  // the row's term of the sink-logit gradient
    if (valid && t == 0) {
        float l2 = INFINITY;
        if (i < N) {
            const float l = l_row;
            l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
            if (sink && l != -INFINITY) sink_term = -expf(sink[h] - l) * acc;
        }
        lse2[r] = l2;
        delta[r] = i < N ? acc * (sc_o * sc_v) : 0.f;
    }
    // The block's 16 rows belong to one (batch, head) (Npad is a multiple of
    // 16): their terms are summed in row order into the block's slot.
    if (sink_part) {
        if (t == 0) sink_rows[threadIdx.x >> 4] = sink_term;
        __syncthreads();
        if (threadIdx.x == 0) {
            float s = 0.f;
#pragma unroll
            for (int k = 0; k < 16; ++k) s += sink_rows[k];
            sink_part[blockIdx.x] = s;
        }
    }
}

// Gradient of head h's sink logit: the per-block sums of every (batch, head h)
// row block, added in a fixed order (threads stride the blocks, then a fixed
// tree), so the result is the same from run to run.
__global__ void __launch_bounds__(256) sink_grad_kernel(int B, int H, int blocks_per_head,
                                                        const float *__restrict__ sink_part,
                                                        float *__restrict__ dsink) {
    __shared__ float red[256];
    pdl_wait();  // the preprocess kernel's block sums
    pdl_trigger();
    const int h = blockIdx.x;
    float s = 0.f;
    for (int b = 0; b < B; ++b) {
        const float *part = sink_part + (static_cast<size_t>(b) * H + h) * blocks_per_head;
        for (int j = threadIdx.x; j < blocks_per_head; j += 256) s += part[j];
    }
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (static_cast<int>(threadIdx.x) < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) dsink[h] = red[0];
}

// Fused dQ: the fp32 buffer [B*H][d/4][Npad] (float4) to dQ [B, N, H, d] bf16,
// times scale / (s_o s_v); or (ACC32) added to an fp32 dQ of that layout.
// A CTA takes CONV_ROWS rows of one (batch, head): coalesced float4 reads down the
// buffer's columns into a padded shared tile, then coalesced 16-byte writes
// along the output rows.
constexpr int CONV_ROWS = 16;

template <bool ACC32, int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(int N, int H, int Npad,
                                                         const float4 *__restrict__ dqacc,
                                                         const float4 *__restrict__ scales,
                                                         float scale, void *__restrict__ dq) {
    constexpr int LD = D + 4;  // row stride in floats: consecutive rows 16 bytes apart in banks
    __shared__ __align__(16) float tile[CONV_ROWS * LD];
    pdl_wait();  // the fused kernel's sums
    pdl_trigger();
    const int i0 = blockIdx.x * CONV_ROWS;
    const int h = blockIdx.y, b = blockIdx.z;
    const size_t bh = static_cast<size_t>(b) * H + h;
    const float mul = scale * scales[bh].w;
    const float4 *src = dqacc + bh * (D / 4) * static_cast<size_t>(Npad) + i0;
#pragma unroll
    for (int k = 0; k < (D / 4) * CONV_ROWS / 256; ++k) {
        const int idx = threadIdx.x + 256 * k;
        const int c4 = idx / CONV_ROWS, r = idx % CONV_ROWS;  // i0 + r < Npad always
        *reinterpret_cast<float4 *>(&tile[r * LD + c4 * 4]) = src[static_cast<size_t>(c4) * Npad + r];
    }
    __syncthreads();
    if constexpr (ACC32) {
        constexpr int CH = D / 4;  // float4 chunks per row
#pragma unroll
        for (int k = 0; k < CH * CONV_ROWS / 256; ++k) {
            const int idx = threadIdx.x + 256 * k;
            const int r = idx / CH, ch = idx % CH;
            if (i0 + r >= N) continue;
            const float4 x = *reinterpret_cast<const float4 *>(&tile[r * LD + ch * 4]);
            float4 *o = reinterpret_cast<float4 *>(static_cast<float *>(dq) +
                                                   ((static_cast<size_t>(b) * N + i0 + r) * H + h) * D) + ch;
            float4 a = *o;
            a.x = fmaf(x.x, mul, a.x);
            a.y = fmaf(x.y, mul, a.y);
            a.z = fmaf(x.z, mul, a.z);
            a.w = fmaf(x.w, mul, a.w);
            *o = a;
        }
    } else {
        constexpr int CH = D / 8;  // 16-byte chunks (8 bf16) per row
#pragma unroll
        for (int k = 0; k < (CH * CONV_ROWS + 255) / 256; ++k) {
            const int idx = threadIdx.x + 256 * k;
            const int r = idx / CH, ch = idx % CH;
            if (idx >= CH * CONV_ROWS || i0 + r >= N) continue;
            const float4 x = *reinterpret_cast<const float4 *>(&tile[r * LD + ch * 8]);
            const float4 y = *reinterpret_cast<const float4 *>(&tile[r * LD + ch * 8 + 4]);
            uint4 w;
            w.x = pack_bf16(x.x * mul, x.y * mul);
            w.y = pack_bf16(x.z * mul, x.w * mul);
            w.z = pack_bf16(y.x * mul, y.y * mul);
            w.w = pack_bf16(y.z * mul, y.w * mul);
            reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(dq) +
                                      ((static_cast<size_t>(b) * N + i0 + r) * H + h) * D)[ch] = w;
        }
    }
}

struct BwdParams {
    const int4 *vec;
    const int *list;  // fwd list (dq kernel) or bwd list (dkdv kernel)
    const int *cnt;
    const float *lse2;
    const float *delta;
    const void *do16;  // [B, N, H, dv] fp16 copy of dO * s_o
    const void *v16;   // [B, N, H, dv] fp16 copy of V * s_v
    const float4 *scales;  // [B*H] (s_o, s_v, 1/s_o, 1/(s_o s_v))
    float4 *dqacc;         // fused dQ: fp32 [B*H][d/4][Npad] (float4), zeroed by preprocess
    void *dq, *dk, *dv;  // bf16 outputs, or fp32 accumulators (ACC32 instantiations)
    int N, H, Hm, T, Npad, causal;
    float sl2;    // scale * log2(e)
    float scale;
    uint64_t timeout_ns;
    int ordered;  // deterministic mode: accumulate the tiles in tile order
};

// ------------------------------------------------------------------ dq kernel
// One CTA per 128-row query tile; NWG compute warpgroups take alternate key
// sub-tiles of BN keys.  Each group owns one BN-column TMEM region that holds,
// in turn, S (fp32), then dP (fp32), then dS (bf16, packed); all groups feed
// one dQ accumulator, and dQ += dS K reads dS straight from TMEM.
// Rings: K in KS stages shared in tile order (S and dQ read it), V in one
// stage per group (dP reads it).  The MMA thread serves whichever group is
// ready, so one group's late operand never stalls the other group's work;
// only the dQ accumulation keeps tile order (bit-reproducible sums).
// DO_TM: the query tile's dO, the same for every key sub-tile, is put into
// TMEM once by compute group 0 (from the fp16 copy), and dP = dO V^T reads it
// from there (TS MMA).  Shared memory then holds only Q, the K ring and the V
// stages, which lets d = 192 run 128-key sub-tiles (N = 128 MMAs for S and
// dP instead of N = 64 ones, which take the pipe as long); at d <= 128, where
// the sub-tiles are 128 keys anyway, the extra TMEM reads made the kernel
// slower, so there dO stays in shared memory.
template <int D_, int DV_, int BN_, int KS_, int NWG_, bool DO_TM_ = false>
struct DqCfg {
    static constexpr int D = D_, DV = DV_, BN = BN_, KS = KS_, NWG = NWG_;
    static constexpr bool DO_TM = DO_TM_;
    static constexpr int BM = 128;
    static constexpr int SUB = TILE / BN;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int DO_BYTES = DO_TM ? 0 : BM * DV * 2;  // dO in shared memory
    static constexpr int K_BYTES = BN * D * 2;
    static constexpr int V_BYTES = BN * DV * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = OFF_Q + Q_BYTES;
    static constexpr int OFF_K = OFF_DO + DO_BYTES;
    static constexpr int OFF_V = OFF_K + KS * K_BYTES;
    static constexpr int OFF_BAR = OFF_V + NWG * V_BYTES;
    // q_full, k_full[KS], k_empty[KS], v_full[NWG], v_empty[NWG],
    // s_full[NWG], p_full[NWG], dp_full[NWG], ds_full[NWG], dq_done, do_ready
    static constexpr int NBAR = 1 + 2 * KS + 6 * NWG + 2;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int TM_DQ = NWG * BN;  // group w's region: columns [w*BN, (w+1)*BN)
    static constexpr int TM_DO = TM_DQ + D;  // dO as fp16 pairs (DO_TM)
    static constexpr int TM_COLS = 512;
    static constexpr int THREADS = 64 + NWG * 128;
    static_assert(TM_DQ + D + (DO_TM ? DV / 2 : 0) <= TM_COLS, "TMEM budget");
    static_assert(!DO_TM || DV % 64 == 0, "dO columns in 32-column stores");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(BN == 64 || BN == 128, "key sub-tile");
    static_assert(KS >= NWG, "ring depth");
    static_assert(KS * K_BYTES >= BM * D * 2, "dQ staging aliases the K ring");
    // The compute frees a K stage when it sees the group's next S; that S must
    // not need the stage itself.
    static constexpr bool RELAY_K = KS > NWG;
    static_assert((D / 32) % NWG == 0, "epilogue column split");
};

// The query-side work for query tile qt_ of (batch b_, head h_); runs in the
// split backward's single launch (split_bwd_kernel).
template <class C, bool ACC32>
__device__ __forceinline__ void dq_body(uint8_t *smem, const CUtensorMap &tm_q,
                                        const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                        const CUtensorMap &tm_do, const CUtensorMap &tm_dq,
                                        const BwdParams &p, int qt_, int h_, int b_) {
    pdl_wait();  // lists, LSE2, D and the fp16 copies of the kernels before
    pdl_trigger();
    if (smem_u32(smem) & 1023u) {  // swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(&g_err_bwd, ERR_SMEM_ALIGN);
        return;
    }
    uint8_t *sQ = smem + C::OFF_Q, *sDO = smem + C::OFF_DO;
    uint8_t *sK = smem + C::OFF_K, *sV = smem + C::OFF_V;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *q_full = bars, *k_full = bars + 1, *k_empty = k_full + C::KS;
    uint64_t *v_full = k_empty + C::KS, *v_empty = v_full + C::NWG;
    uint64_t *s_full = v_empty + C::NWG, *p_full = s_full + C::NWG, *dp_full = p_full + C::NWG;
    uint64_t *ds_full = dp_full + C::NWG, *dq_done = ds_full + C::NWG;
    uint64_t *do_ready = dq_done + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    int *issued = reinterpret_cast<int *>(smem + C::OFF_MISC + 8);  // loads per ring

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = qt_;
    const int h = h_, b = b_;
    const int bm = b * p.Hm + (p.Hm == 1 ? 0 : h);
    const int n_entries = p.cnt[static_cast<size_t>(bm) * p.T + qt];
    const int *entries = p.list + (static_cast<size_t>(bm) * p.T + qt) * p.T;
    // After a bounded wait gave up anywhere, later CTAs do no work.
    const int n = (*reinterpret_cast<volatile unsigned *>(&g_err_bwd) != 0) ? 0
                                                                            : n_entries * C::SUB;
    const uint64_t tmo = p.timeout_ns;
    auto n_of = [&](int w) { return n > w ? (n - w + C::NWG - 1) / C::NWG : 0; };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < C::KS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < C::NWG; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&dp_full[i], 1);
            mbar_init(&ds_full[i], 128);
        }
        mbar_init(dq_done, 1);
        mbar_init(do_ready, 128);
        *abort = 0;
        issued[0] = issued[1] = 0;
        fence_barrier_init();
        if (n > 0) {  // Q and dO before the CTA-wide barrier: latency overlaps the setup
            mbar_arrive_expect_tx(q_full, C::Q_BYTES + C::DO_BYTES);
#pragma unroll
            for (int c = 0; c < C::D / 64; ++c)
                tma_load_4d(sQ + c * C::BM * 128, &tm_q, q_full, c * 64, h, qt * TILE, b);
            if constexpr (!C::DO_TM) {
#pragma unroll
                for (int c = 0; c < C::DV / 64; ++c)
                    tma_load_4d(sDO + c * C::BM * 128, &tm_do, q_full, c * 64, h, qt * TILE, b);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto key0_of = [&](int u) {
        return (entries[u / C::SUB] >> 1) * TILE + (u % C::SUB) * C::BN;
    };

    if (warp == 0) {
        if (lane == 0 && n > 0) {
            prefetch_tmap(&tm_k);
            int u = 0;
            for (; u < n; ++u) {
                const int s = u % C::KS;
                if (u >= C::KS &&
                    !mbar_wait(&k_empty[s], ((u / C::KS) - 1) & 1, tmo, abort, &g_err_bwd))
                    break;
                mbar_arrive_expect_tx(&k_full[s], C::K_BYTES);
                const int key0 = key0_of(u);
#pragma unroll
                for (int c = 0; c < C::D / 64; ++c)
                    tma_load_4d(sK + s * C::K_BYTES + c * C::BN * 128, &tm_k, &k_full[s], c * 64,
                                h, key0, b);
            }
            issued[0] = u;
        } else if (lane == 1 && n > 0) {
            prefetch_tmap(&tm_v);
            int u = 0;
            for (; u < n; ++u) {
                const int w = u % C::NWG, lw = u / C::NWG;
                if (lw >= 1 && !mbar_wait(&v_empty[w], (lw - 1) & 1, tmo, abort, &g_err_bwd))
                    break;
                mbar_arrive_expect_tx(&v_full[w], C::V_BYTES);
                const int key0 = key0_of(u);
#pragma unroll
                for (int c = 0; c < C::DV / 64; ++c)
                    tma_load_4d(sV + w * C::V_BYTES + c * C::BN * 128, &tm_v, &v_full[w], c * 64,
                                h, key0, b);
            }
            issued[1] = u;
        }
    } else if (warp == 1) {
        if (lane == 0 && n > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(128, C::BN, false, false);
            constexpr uint32_t IDESC_DP = idesc_fp16(128, C::BN, false, false);
            constexpr uint32_t IDESC_DQ = idesc_bf16(128, C::D, false, true);
            // Descriptors are built once; an MMA step only adds its byte offset
            // (in 16-byte units) to the start-address field.
            const uint64_t q_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t do_desc = sdesc_sw128(smem_u32(sDO), 16, 1024);
            const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t k_desc_mn = sdesc_sw128(smem_u32(sK), C::BN * 128, 1024);
            const uint64_t v_desc = sdesc_sw128(smem_u32(sV), 16, 1024);
            int lu_[C::NWG], st_[C::NWG];
            int remaining = 0;
#pragma unroll
            for (int w = 0; w < C::NWG; ++w) {
                lu_[w] = 0;
                st_[w] = 0;
                remaining += n_of(w) > 0;
            }
            // Deterministic mode issues the S tiles and the dQ accumulations in
            // tile order, so the fp32 sums are the same on every run.  Otherwise
            // whichever group is ready goes first: the sums' order, and their
            // last bits, vary, but neither group waits for the other.  The K
            // ring is filled in tile order; a group gets at most one ring length
            // ahead, since a stage is refilled only after its older tile's dQ.
            int next_s = 0, next_q = 0;
            // A tcgen05.commit costs this thread about as long as an MMA, time in
            // which the tensor pipe runs dry, so commits are kept to the two the
            // compute waits for (S, dP).  The compute frees the V stage when it
            // sees dP, and the K stage of its tile lu - 1 when it sees S of tile
            // lu (the pipe ran that dQ first); the MMA thread commits the K
            // stage only after a group's last dQ.  A dQ and the group's next S
            // go out as one run.
            auto issue_s = [&](int w, int u) {  // S = Q K^T into group w's region
                const uint64_t ks =
                    k_desc + static_cast<uint64_t>(((u % C::KS) * C::K_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < C::D / 16; ++k) {
                    const uint32_t a_off = ((k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4;
                    const uint32_t b_off = ((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4;
                    mma_ss(tmem + w * C::BN, q_desc + a_off, ks + b_off, IDESC_S,
                           k > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[w]);
                ++next_s;
            };
            auto s_ready = [&](int u) {
                return (!p.ordered || u == next_s) &&
                       mbar_test(&k_full[u % C::KS], (u / C::KS) & 1) != 0;
            };
            bool ok = mbar_wait(q_full, 0, tmo, abort, &g_err_bwd);
            bool idle = false;
            uint64_t idle_t0 = 0;
            while (ok && remaining > 0) {
                bool prog = false;
#pragma unroll
                for (int w = 0; w < C::NWG; ++w) {
                    const int lu = lu_[w];
                    if (lu >= n_of(w)) continue;
                    const int u = lu * C::NWG + w;
                    const int s = u % C::KS;
                    const uint32_t t_r = tmem + w * C::BN;
                    if (st_[w] == 0) {  // S = Q K^T
                        if (!s_ready(u)) continue;
                        tc_fence_after();
                        issue_s(w, u);
                        st_[w] = 1;
                        prog = true;
                    } else if (st_[w] == 1) {  // dP = dO V^T, once the group has read S
                        if (!mbar_test(&p_full[w], lu & 1) || !mbar_test(&v_full[w], lu & 1))
                            continue;
                        if (C::DO_TM && !mbar_test(do_ready, 0)) continue;
                        tc_fence_after();
                        const uint64_t vsd = v_desc + static_cast<uint64_t>((w * C::V_BYTES) >> 4);
#pragma unroll
                        for (int k = 0; k < C::DV / 16; ++k) {
                            const uint32_t a_off = ((k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4;
                            const uint32_t b_off = ((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4;
                            if constexpr (C::DO_TM)  // A = dO from TMEM, 16 fp16 = 8 columns
                                mma_ts(t_r, tmem + C::TM_DO + k * 8, vsd + b_off, IDESC_DP,
                                       k > 0 ? 1u : 0u);
                            else
                                mma_ss(t_r, do_desc + a_off, vsd + b_off, IDESC_DP,
                                       k > 0 ? 1u : 0u);
                        }
                        mma_commit(&dp_full[w]);
                        st_[w] = 2;
                        prog = true;
                    } else {  // dQ += dS K (dS from TMEM, K MN-major over d), then next S
                        if ((p.ordered && u != next_q) || !mbar_test(&ds_full[w], lu & 1)) continue;
                        tc_fence_after();
                        const uint64_t kmn =
                            k_desc_mn + static_cast<uint64_t>((s * C::K_BYTES) >> 4);
#pragma unroll
                        for (int k = 0; k < C::BN / 16; ++k)
                            mma_ts(tmem + C::TM_DQ, t_r + k * 8, kmn + ((k * 2048) >> 4), IDESC_DQ,
                                   (next_q > 0 || k > 0) ? 1u : 0u);
                        ++next_q;
                        lu_[w] = lu + 1;
                        st_[w] = 0;
                        // no later S of this group frees the stage (or, with no
                        // more stages than groups, that S would need it first)
                        if (!C::RELAY_K || lu + 1 >= n_of(w)) mma_commit(&k_empty[s]);
                        if (lu + 1 >= n_of(w)) {
                            --remaining;
                        } else if (s_ready(u + C::NWG)) {
                            issue_s(w, u + C::NWG);
                            st_[w] = 1;
                        }
                        prog = true;
                    }
                }
                if (prog) {
                    idle = false;
                } else if (*abort) {
                    ok = false;
                } else {
                    const uint64_t now = globaltimer();
                    if (!idle) {
                        idle = true;
                        idle_t0 = now;
                    } else if (now - idle_t0 > tmo) {
                        *abort = 1;
                        atomicExch(&g_err_bwd, ERR_TIMEOUT);
                        ok = false;
                    }
                }
            }
            mma_commit(dq_done);
        }
    } else {
        // compute warpgroups: thread = query row
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int grow = qt * TILE + row;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const uint32_t t_r = lane_base + wg * C::BN;
        const size_t bh = static_cast<size_t>(b) * p.H + h;
        const float lse2 = p.lse2[bh * p.Npad + grow];
        const float Drow = p.delta[bh * p.Npad + grow];  // D * s_o s_v
        const float sl2 = p.sl2;
        const int n_my = n_of(wg);
        const int4 *vec = p.vec + static_cast<size_t>(bm) * p.Npad;
        if constexpr (C::DO_TM) {
            // Group 0 puts the query tile's dO rows (fp16 pairs; zeros past N)
            // into TMEM, where every dP of the CTA reads them.
            if (wg == 0 && n > 0) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    static_cast<const __half *>(p.do16) +
                    ((static_cast<size_t>(b) * p.N + (grow < p.N ? grow : 0)) * p.H + h) *
                        C::DV);
#pragma unroll 1
                for (int c = 0; c < C::DV / 64; ++c) {
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 w4 = grow < p.N ? src[c * 8 + i] : make_uint4(0u, 0u, 0u, 0u);
                        r[4 * i] = w4.x;
                        r[4 * i + 1] = w4.y;
                        r[4 * i + 2] = w4.z;
                        r[4 * i + 3] = w4.w;
                    }
                    tmem_st32(lane_base + C::TM_DO + c * 32, r);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(do_ready);
            }
        }
        // The next tile's list entry and mask boundaries are read one tile ahead.
        int4 cv_next[C::BN / 64][2];
        auto load_bounds = [&](int u, int entry) {
            if (!(entry & 1)) return;
            const int key0 = (entry >> 1) * TILE + (u % C::SUB) * C::BN;
#pragma unroll
            for (int c = 0; c < C::BN / 64; ++c) {
                cv_next[c][0] = __ldg(vec + key0 + c * 64 + lane);
                cv_next[c][1] = __ldg(vec + key0 + c * 64 + 32 + lane);
            }
        };
        int entry_next = n_my > 0 ? entries[wg / C::SUB] : 0;
        if (n_my > 0) load_bounds(wg, entry_next);
        for (int lu = 0; lu < n_my; ++lu) {
            const int u = lu * C::NWG + wg;
            const int entry = entry_next;
            const bool masked_tile = entry & 1;
            const int key0 = (entry >> 1) * TILE + (u % C::SUB) * C::BN;
            // Partial tiles: the mask bits of this lane's row, built before the
            // wait for S.  Lane l holds the boundaries of key columns l and
            // l + 32 of each 64-column chunk; their row bits over this warp's
            // rows are transposed so that each lane gets its row's column bits.
            uint32_t mbits[C::BN / 64][2];
            if (masked_tile) {
                const int R = grow - lane;
#pragma unroll
                for (int c = 0; c < C::BN / 64; ++c)
#pragma unroll
                    for (int e = 0; e < 2; ++e)
                        mbits[c][e] = warp_transpose32(
                            column_row_bits(R, key0 + c * 64 + e * 32 + lane, cv_next[c][e],
                                            p.causal),
                            lane);
#pragma unroll
                for (int c = 0; c < C::BN / 64; ++c)
                    asm volatile("" ::"r"(mbits[c][0]), "r"(mbits[c][1]));
            }
            if (u + C::NWG < n) entry_next = entries[(u + C::NWG) / C::SUB];
            if (!warp_wait(&s_full[wg], lu & 1, tmo, abort)) break;
            tc_fence_after();
            // S of this tile ran after the group's previous dQ: that K stage is free.
            if (C::RELAY_K && ((warp - 2) & 3) == 0 && lane == 0 && lu > 0)
                mbar_arrive(&k_empty[(u - C::NWG) % C::KS]);
            // phase 1: P = exp2(S * scale * log2e - LSE2), masked, kept as fp16 pairs
            uint32_t pk[C::BN / 2];
#pragma unroll
            for (int c = 0; c < C::BN / 64; ++c) {
                float x[64];
                tmem_ld64f(t_r + c * 64, x);
#pragma unroll
                for (int i = 0; i < 32; ++i) {  // paired fp32 FMA for the exponents
                    const float2 t = __ffma2_rn(make_float2(x[2 * i], x[2 * i + 1]),
                                                make_float2(sl2, sl2), make_float2(-lse2, -lse2));
                    x[2 * i] = ex2(t.x);
                    x[2 * i + 1] = ex2(t.y);
                }
                if (masked_tile) {
                    const uint32_t wa = mbits[c][0], wb = mbits[c][1];
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        if ((wa >> jj) & 1u) x[jj] = 0.f;
                        if ((wb >> jj) & 1u) x[32 + jj] = 0.f;
                    }
                }
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[c * 32 + i] = pack_fp16(x[2 * i], x[2 * i + 1]);
            }
            tc_fence_before();
            mbar_arrive(&p_full[wg]);  // S read: the region may take dP
            if (u + C::NWG < n) load_bounds(u + C::NWG, entry_next);
            // phase 2: dS = P * (dP - D) -> the region, bf16
            if (!warp_wait(&dp_full[wg], lu & 1, tmo, abort)) break;
            tc_fence_after();
            if (((warp - 2) & 3) == 0 && lane == 0) mbar_arrive(&v_empty[wg]);  // dP read V
#pragma unroll
            for (int c = 0; c < C::BN / 64; ++c) {
                float dp[64];
                tmem_ld64f(t_r + c * 64, dp);
                uint32_t r[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {  // paired fp32 add and multiply
                    __half2 h2 = *reinterpret_cast<__half2 *>(&pk[c * 32 + i]);
                    const float2 ds = __fmul2_rn(
                        __half22float2(h2),
                        __fadd2_rn(make_float2(dp[2 * i], dp[2 * i + 1]), make_float2(-Drow, -Drow)));
                    r[i] = pack_bf16(ds.x, ds.y);
                }
                tmem_st32(t_r + c * 32, r);  // columns already read
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&ds_full[wg]);
        }
        if (n > 0) warp_wait(dq_done, 0, tmo, abort);
        tc_fence_after();
        // dQ (times scale / (s_o s_v)): added to the fp32 output (acc32), or as
        // bf16 to the 128B-swizzled layout of the output map in the idle K ring,
        // then TMA stores of its 64-column boxes (rows past N clipped).
        const float dq_mul = p.scale * p.scales[bh].w;
        constexpr int CPW = (C::D / 32) / C::NWG;  // 32-column chunks per group
        if constexpr (ACC32) {
            // fp32 accumulation: each row adds its own values (rows past N and
            // CTAs without work add nothing).
            float *dst = static_cast<float *>(p.dq) +
                         ((static_cast<size_t>(b) * p.N + grow) * p.H + h) * C::D;
#pragma unroll 1
            for (int c = wg * CPW; c < (wg + 1) * CPW && n > 0; ++c) {
                uint32_t r[32];
                tmem_ld32(lane_base + C::TM_DQ + c * 32, r);
                if (grow < p.N) add_row_f32(dst, c, r, dq_mul);
            }
        } else {
#pragma unroll 1
            for (int c = wg * CPW; c < (wg + 1) * CPW; ++c) {
                uint32_t r[32];
                tmem_ld32(lane_base + C::TM_DQ + c * 32, r);
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = n > 0 ? __uint_as_float(r[i]) : 0.f;
                stage_row_bf16(sK, c, row, v, dq_mul);
            }
            fence_proxy_async_smem();
            named_bar_sync(1, C::NWG * 128);
            if (threadIdx.x == 64) {
                for (int box = 0; box < C::D / 64; ++box)
                    tma_store_4d(&tm_dq, sK + box * (128 * 128), box * 64, h, qt * TILE, b);
                bulk_commit_wait_read();
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // After a wait gave up, what this CTA still has in flight lands before it
    // frees TMEM and exits: both rings' loads, the tiles loaded at the start and
    // the MMAs.  Past the barrier *abort is final and the same for every
    // thread; on the normal path every load was consumed and every MMA waited
    // for, and nothing is left to drain.
    if (*abort) {
        if (threadIdx.x == 0 && n > 0) {
            drain_ring(k_full, C::KS, issued[0], -1, tmo, &g_err_bwd);
            drain_ring(v_full, C::NWG, issued[1], -1, tmo, &g_err_bwd);
            mbar_wait_drain(q_full, 0, tmo, &g_err_bwd);
            mbar_wait_drain(dq_done, 0, tmo, &g_err_bwd);
        }
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

// ---------------------------------------------------------------- dkdv kernel
// One CTA per 128-key tile; NWG compute warpgroups take alternate query
// sub-tiles of BM rows.  Each group owns one BM-column TMEM region that holds,
// in turn, S^T (fp32) then P^T (fp16, packed), then dP^T (fp32) then dS^T
// (bf16, packed); all groups feed the one dK and the one dV accumulator.
// Rings: Q in QS stages shared in tile order (S^T and dK read it); dO with
// the tile's LSE2 and D in one stage per group (dV, dP^T and the compute read
// them).  The MMA thread serves whichever group is ready; the dV and dK
// accumulations keep tile order (bit-reproducible sums).
// V_TM: the CTA's V tile, the same for every query sub-tile, is put into TMEM
// once by compute group 0 (from the fp16 copy) and dP^T = V dO^T reads it from
// there (TS MMA).  Its shared memory goes to a second compute group and a
// deeper Q ring at d = dv = 256 (where only the dK pass needs V), and to a
// deeper Q ring at d = 192.
// FDQ (fused dQ, the default backward at d <= 128): each sub-tile also gives
// dQ_tile = dS K.  The compute writes dS^T, besides TMEM, to shared memory as
// the MN-major A operand of that product (over the group's dO stage, spent
// once dP^T ran, when it is large enough); the product lands in the group's
// TMEM region after dK has read dS^T from it (the pipe runs them in order);
// the group then adds the tile to the fp32 dQ buffer (coalesced red.add, the
// buffer laid out [B*H][d/4][Npad] in float4) before the region takes the
// group's next S^T.  S and dP are computed once per pair.
template <int D_, int DV_, int BM_, int QS_, bool DK_, bool DV_ON_, int NWG_,
          bool V_TM_ = false, bool FDQ_ = false>
struct DkdvCfg {
    static constexpr int D = D_, DV = DV_, BM = BM_, QS = QS_, NWG = NWG_;
    static constexpr bool DO_DK = DK_, DO_DV = DV_ON_, V_TM = V_TM_, FDQ = FDQ_;
    static constexpr int BN = 128;            // keys per CTA (TMEM lanes)
    static constexpr int SUB = TILE / BM;     // query sub-tiles per list entry
    static constexpr bool NEED_V = DO_DK;     // V only feeds dP^T
    static constexpr int K_BYTES = BN * D * 2;
    static constexpr int V_BYTES = (NEED_V && !V_TM) ? BN * DV * 2 : 0;  // V in shared memory
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int DO_BYTES = BM * DV * 2;
    static constexpr int LD_BYTES = 2 * BM * 4;  // LSE2 then D of the sub-tile's rows
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + K_BYTES;
    static constexpr int OFF_Q = OFF_V + V_BYTES;
    static constexpr int OFF_DO = OFF_Q + QS * Q_BYTES;
    static constexpr int OFF_LD = OFF_DO + NWG * DO_BYTES;
    // FDQ: dS tile per group, bf16 [BN keys][BM queries], 64-query blocks
    static constexpr int DS_BYTES = FDQ ? BN * BM * 2 : 0;
    static constexpr bool DS_IN_DO = FDQ && DO_BYTES >= DS_BYTES;
    static constexpr int OFF_DS = OFF_LD + NWG * LD_BYTES;
    static constexpr int DS_STRIDE = DS_IN_DO ? DO_BYTES : DS_BYTES;  // between groups' tiles
    static constexpr int OFF_BAR = OFF_DS + ((FDQ && !DS_IN_DO) ? NWG * DS_BYTES : 0);
    // FDQ: the first DQ_TMA_COLS columns of a dQ tile leave through a TMA bulk
    // reduction, staged as fp32 [column / 4][128 rows] float4 in the sub-tile's
    // Q stage (spent once dK ran: dQ does not read Q); the rest through red.add
    // from registers.  The bulk path moves its bytes without the compute warps.
    static constexpr int DQ_TMA_COLS = FDQ ? Q_BYTES / (BM * 4) : 0;
    static constexpr bool Q_BY_REDUCER = DQ_TMA_COLS > 0;  // Q stages freed by the reducer
    // kv_full, q_full[QS], q_empty[QS], o_full[NWG], o_empty[NWG],
    // s_full[NWG], p_full[NWG], dp_full[NWG], ds_full[NWG], done, v_ready,
    // FDQ: dq_full[NWG], dq_free[NWG], staged[NWG]
    static constexpr int NBAR = 1 + 2 * QS + 6 * NWG + 2 + (FDQ ? 3 * NWG : 0);
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int TM_DK = 0;
    static constexpr int TM_DV = DO_DK ? D : 0;
    static constexpr int TM_W0 = TM_DV + (DO_DV ? DV : 0);  // group w: [TM_W0 + w*BM, +BM)
    static constexpr int TM_END = TM_W0 + NWG * BM;
    static constexpr int TM_V = TM_END;      // V as fp16 pairs (V_TM)
    static constexpr int TM_COLS = 512;
    static constexpr int THREADS = 64 + NWG * 128;
    static_assert(TM_END + (V_TM ? DV / 2 : 0) <= TM_COLS, "TMEM budget");
    static_assert(!V_TM || (NEED_V && DV % 64 == 0), "V in TMEM only feeds dP^T");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(D <= 256 && DV <= 256 && (BM == 64 || BM == 128), "MMA shape");
    static_assert(QS >= NWG, "ring depth");
    static_assert(QS * Q_BYTES + NWG * DO_BYTES >=
                      (DO_DK ? BN * D * 2 : 0) + (DO_DV ? BN * DV * 2 : 0),
                  "dK / dV staging aliases the Q ring and the dO stages");
    // The compute frees a Q stage when it sees the group's next S^T; that S^T
    // must not need the stage itself.
    static constexpr bool RELAY_Q = QS > NWG;
    static_assert((D / 32) % NWG == 0 && (DV / 32) % NWG == 0, "epilogue column split");
    static_assert(!FDQ || (DO_DK && DO_DV && !V_TM && BM == 128 && D <= BM),
                  "fused dQ: one pass, 128-query sub-tiles, dQ tile within a group region");
    static_assert(OFF_DS % 1024 == 0, "swizzled dS tiles need 1024-byte alignment");
    static_assert(DQ_TMA_COLS % 32 == 0 && DQ_TMA_COLS <= D, "dQ columns staged in 32s");
    static_assert(!FDQ || NWG * DO_BYTES >= (D / 64 + DV / 64) * 128 * 128,
                  "fused dQ: dK and dV staging fits the dO stages");
    static_assert(OFF_DO % 1024 == 0, "swizzled staging needs 1024-byte alignment");
};

// The key-side work for key tile kt_ of (batch b_, head h_): the body of
// dkdv_kernel and of the key-side part of split_bwd_kernel.
template <class C, bool ACC32>
__device__ __forceinline__ void dkdv_body(uint8_t *smem, const CUtensorMap &tm_q,
                                          const CUtensorMap &tm_k, const CUtensorMap &tm_v,
                                          const CUtensorMap &tm_do, const CUtensorMap &tm_dk,
                                          const CUtensorMap &tm_dv, const BwdParams &p, int kt_,
                                          int h_, int b_) {
    pdl_wait();  // lists, LSE2, D and the fp16 copies of the kernels before
    pdl_trigger();
    if (smem_u32(smem) & 1023u) {  // swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(&g_err_bwd, ERR_SMEM_ALIGN);
        return;
    }
    uint8_t *sK = smem + C::OFF_K, *sV = smem + C::OFF_V, *sQ = smem + C::OFF_Q;
    uint8_t *sDO = smem + C::OFF_DO, *sLD = smem + C::OFF_LD;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *kv_full = bars, *q_full = bars + 1, *q_empty = q_full + C::QS;
    uint64_t *o_full = q_empty + C::QS, *o_empty = o_full + C::NWG;
    uint64_t *s_full = o_empty + C::NWG, *p_full = s_full + C::NWG, *dp_full = p_full + C::NWG,
             *ds_full = dp_full + C::NWG, *done = ds_full + C::NWG;
    uint64_t *v_ready = done + 1;
    uint64_t *dq_full = v_ready + 1, *dq_free = dq_full + C::NWG;  // FDQ only
    uint64_t *staged = dq_free + C::NWG;  // FDQ only
    uint8_t *sDS = C::DS_IN_DO ? sDO : smem + C::OFF_DS;             // FDQ only
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    int *issued = reinterpret_cast<int *>(smem + C::OFF_MISC + 8);  // loads per ring

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kt = kt_;
    const int h = h_, b = b_;
    const int bm = b * p.Hm + (p.Hm == 1 ? 0 : h);
    const int n_entries = p.cnt[static_cast<size_t>(bm) * p.T + kt];
    const int *entries = p.list + (static_cast<size_t>(bm) * p.T + kt) * p.T;
    // After a bounded wait gave up anywhere, later CTAs do no work.
    const int n = (*reinterpret_cast<volatile unsigned *>(&g_err_bwd) != 0) ? 0
                                                                            : n_entries * C::SUB;
    const uint64_t tmo = p.timeout_ns;
    const size_t bh = static_cast<size_t>(b) * p.H + h;
    auto n_of = [&](int w) { return n > w ? (n - w + C::NWG - 1) / C::NWG : 0; };

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int i = 0; i < C::QS; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
        }
        for (int i = 0; i < C::NWG; ++i) {
            mbar_init(&o_full[i], 1);
            mbar_init(&o_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&dp_full[i], 1);
            mbar_init(&ds_full[i], 128);
        }
        mbar_init(done, 1);
        mbar_init(v_ready, 128);
        issued[0] = issued[1] = 0;
        if constexpr (C::FDQ) {
            for (int i = 0; i < C::NWG; ++i) {
                mbar_init(&dq_full[i], 1);
                mbar_init(&dq_free[i], 128);
                mbar_init(&staged[i], 128);
            }
        }
        *abort = 0;
        fence_barrier_init();
        if (n > 0) {  // K and V before the CTA-wide barrier: latency overlaps the setup
            mbar_arrive_expect_tx(kv_full, C::K_BYTES + C::V_BYTES);
#pragma unroll
            for (int c = 0; c < C::D / 64; ++c)
                tma_load_4d(sK + c * C::BN * 128, &tm_k, kv_full, c * 64, h, kt * TILE, b);
            if constexpr (C::NEED_V && !C::V_TM) {
#pragma unroll
                for (int c = 0; c < C::DV / 64; ++c)
                    tma_load_4d(sV + c * C::BN * 128, &tm_v, kv_full, c * 64, h, kt * TILE, b);
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto q0_of = [&](int u) { return (entries[u / C::SUB] >> 1) * TILE + (u % C::SUB) * C::BM; };

    if (warp == 0) {
        if (lane == 0 && n > 0) {
            prefetch_tmap(&tm_q);
            int u = 0;
            for (; u < n; ++u) {
                const int s = u % C::QS;
                if (u >= C::QS &&
                    !mbar_wait(&q_empty[s], ((u / C::QS) - 1) & 1, tmo, abort, &g_err_bwd))
                    break;
                mbar_arrive_expect_tx(&q_full[s], C::Q_BYTES);
                const int q0 = q0_of(u);
#pragma unroll
                for (int c = 0; c < C::D / 64; ++c)
                    tma_load_4d(sQ + s * C::Q_BYTES + c * C::BM * 128, &tm_q, &q_full[s], c * 64,
                                h, q0, b);
            }
            issued[0] = u;
        } else if (lane == 1 && n > 0) {
            prefetch_tmap(&tm_do);
            int u = 0;
            for (; u < n; ++u) {
                const int w = u % C::NWG, lw = u / C::NWG;
                // The stage is free once the group's previous tile no longer
                // needs it: with dK, when its compute has written dS^T (the dV
                // and dP^T MMAs, the last readers of dO, completed before dP^T
                // was handed over); without dK, when the dV MMA has completed;
                // with fused dQ, when the dQ MMA has read the dS tile (written
                // over the spent dO, or beside it).
                uint64_t *free_bar =
                    C::FDQ ? &dq_full[w] : (C::DO_DK ? &ds_full[w] : &o_empty[w]);
                if (lw >= 1 && !mbar_wait(free_bar, (lw - 1) & 1, tmo, abort, &g_err_bwd))
                    break;
                mbar_arrive_expect_tx(&o_full[w], C::DO_BYTES + C::LD_BYTES);
                const int q0 = q0_of(u);
#pragma unroll
                for (int c = 0; c < C::DV / 64; ++c)
                    tma_load_4d(sDO + w * C::DO_BYTES + c * C::BM * 128, &tm_do, &o_full[w],
                                c * 64, h, q0, b);
                uint8_t *ld = sLD + w * C::LD_BYTES;
                bulk_load(ld, p.lse2 + bh * p.Npad + q0, C::BM * 4, &o_full[w]);
                bulk_load(ld + C::BM * 4, p.delta + bh * p.Npad + q0, C::BM * 4, &o_full[w]);
            }
            issued[1] = u;
        } else if (lane == 2 && n > 0 && C::Q_BY_REDUCER) {
            // dQ reducer: once a group has staged a tile's first DQ_TMA_COLS
            // columns in the tile's Q stage, add them to the fp32 buffer with
            // bulk reductions (2 KB: 128 rows of one float4 column), wait until
            // the engine has read the stage, and hand the stage back to the Q
            // producer.
            for (int u = 0; u < n; ++u) {
                const int w = u % C::NWG, lw = u / C::NWG;
                if (!mbar_wait(&staged[w], lw & 1, tmo, abort, &g_err_bwd)) break;
                float4 *g = p.dqacc + bh * (C::D / 4) * static_cast<size_t>(p.Npad) + q0_of(u);
                const uint8_t *src = sQ + (u % C::QS) * C::Q_BYTES;
#pragma unroll 1
                for (int c4 = 0; c4 < C::DQ_TMA_COLS / 4; ++c4)
                    bulk_reduce_add_f32(g + static_cast<size_t>(c4) * p.Npad, src + c4 * 2048, 2048);
                bulk_commit();
                bulk_wait_read_all();
                mbar_arrive(&q_empty[u % C::QS]);
            }
            bulk_wait_all();  // the reductions' global writes, before the CTA exits
        }
    } else if (warp == 1) {
        if (lane == 0 && n > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(128, C::BM, false, false);
            constexpr uint32_t IDESC_DP = idesc_fp16(128, C::BM, false, false);
            constexpr uint32_t IDESC_DV = idesc_fp16(128, C::DV, false, true);
            constexpr uint32_t IDESC_DK = idesc_bf16(128, C::D, false, true);
            // fused dQ = dS K: A = dS, MN-major over the 128 queries of the
            // sub-tile; B = K, MN-major over d
            constexpr uint32_t IDESC_DQ = idesc_bf16(128, C::D, true, true);
            // Descriptors are built once; an MMA step only adds its byte offset
            // (in 16-byte units) to the start-address field.
            const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t k_desc_mn = sdesc_sw128(smem_u32(sK), C::BN * 128, 1024);
            const uint64_t ds_desc = sdesc_sw128(smem_u32(sDS), C::BN * 128, 1024);
            const uint64_t v_desc = sdesc_sw128(smem_u32(sV), 16, 1024);
            const uint64_t q_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t q_desc_mn = sdesc_sw128(smem_u32(sQ), C::BM * 128, 1024);
            const uint64_t do_desc = sdesc_sw128(smem_u32(sDO), 16, 1024);
            const uint64_t do_desc_mn = sdesc_sw128(smem_u32(sDO), C::BM * 128, 1024);
            int lu_[C::NWG], st_[C::NWG];
            int remaining = 0;
#pragma unroll
            for (int w = 0; w < C::NWG; ++w) {
                lu_[w] = 0;
                st_[w] = 0;
                remaining += n_of(w) > 0;
            }
            // Deterministic mode issues the S^T tiles and the dV and dK
            // accumulations in tile order, so the fp32 sums are the same on
            // every run.  Otherwise whichever group is ready goes first: the
            // sums' order, and their last bits, vary, but neither group waits
            // for the other.  The Q ring is filled in tile order; a stage is
            // refilled only after its older tile's dK.
            int next_s = 0, next_v = 0, next_k = 0;
            // A tcgen05.commit costs this thread about as long as an MMA, time in
            // which the tensor pipe runs dry, so commits are kept to the two the
            // compute waits for (S^T, dP^T).  The compute frees the Q stage of
            // its tile lu - 1 when it sees S^T of tile lu (the pipe ran that dK
            // first); the MMA thread commits the Q stage only after a group's
            // last dK.  A dK and the group's next S^T go out as one run.
            auto issue_s = [&](int w, int u) {  // S^T = K Q^T into group w's region
                const uint64_t qs =
                    q_desc + static_cast<uint64_t>(((u % C::QS) * C::Q_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < C::D / 16; ++k) {
                    const uint32_t a_off = ((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4;
                    const uint32_t b_off = ((k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4;
                    mma_ss(tmem + C::TM_W0 + w * C::BM, k_desc + a_off, qs + b_off, IDESC_S,
                           k > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[w]);
                ++next_s;
            };
            auto s_ready = [&](int u) {
                return (!p.ordered || u == next_s) &&
                       mbar_test(&q_full[u % C::QS], (u / C::QS) & 1) != 0;
            };
            bool ok = mbar_wait(kv_full, 0, tmo, abort, &g_err_bwd);
            bool idle = false;
            uint64_t idle_t0 = 0;
            while (ok && remaining > 0) {
                bool prog = false;
#pragma unroll
                for (int w = 0; w < C::NWG; ++w) {
                    const int lu = lu_[w];
                    if (lu >= n_of(w)) continue;
                    const int u = lu * C::NWG + w;
                    const int s = u % C::QS;
                    const uint32_t t_r = tmem + C::TM_W0 + w * C::BM;
                    if (st_[w] == 0) {  // S^T = K Q^T
                        if (!s_ready(u)) continue;
                        // fused dQ: the region holds the group's previous dQ tile
                        // until the group has added it to the buffer
                        if (C::FDQ && lu > 0 && !mbar_test(&dq_free[w], (lu - 1) & 1)) continue;
                        tc_fence_after();
                        issue_s(w, u);
                        st_[w] = 1;
                        prog = true;
                    } else if (st_[w] == 1) {
                        // The group has read S^T (and written P^T): dV += P^T dO,
                        // then dP^T = V dO^T into the same region.
                        if ((p.ordered && u != next_v) || !mbar_test(&p_full[w], lu & 1) ||
                            !mbar_test(&o_full[w], lu & 1))
                            continue;
                        if ((C::V_TM || C::FDQ) && !mbar_test(v_ready, 0)) continue;
                        tc_fence_after();
                        const bool acc_v = next_v > 0;  // the first dV product initialises
                        ++next_v;
                        if constexpr (C::DO_DV) {
                            const uint64_t dmn =
                                do_desc_mn + static_cast<uint64_t>((w * C::DO_BYTES) >> 4);
#pragma unroll
                            for (int k = 0; k < C::BM / 16; ++k)
                                mma_ts(tmem + C::TM_DV, t_r + k * 8, dmn + ((k * 2048) >> 4),
                                       IDESC_DV, (acc_v || k > 0) ? 1u : 0u);
                        }
                        if constexpr (C::DO_DK) {
                            const uint64_t dd =
                                do_desc + static_cast<uint64_t>((w * C::DO_BYTES) >> 4);
#pragma unroll
                            for (int k = 0; k < C::DV / 16; ++k) {
                                const uint32_t a_off =
                                    ((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4;
                                const uint32_t b_off =
                                    ((k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4;
                                if constexpr (C::V_TM)  // A = V from TMEM, 16 fp16 = 8 columns
                                    mma_ts(t_r, tmem + C::TM_V + k * 8, dd + b_off, IDESC_DP,
                                           k > 0 ? 1u : 0u);
                                else
                                    mma_ss(t_r, v_desc + a_off, dd + b_off, IDESC_DP,
                                           k > 0 ? 1u : 0u);
                            }
                            mma_commit(&dp_full[w]);
                        } else {
                            mma_commit(&o_empty[w]);  // dO and LSE2 read
                        }
                        st_[w] = 2;
                        prog = true;
                    } else {
                        // The group has written dS^T: dK += dS^T Q, then the
                        // group's next S^T.
                        if ((p.ordered && u != next_k) || !mbar_test(&ds_full[w], lu & 1)) continue;
                        tc_fence_after();
                        const bool acc_k = next_k > 0;  // the first dK product initialises
                        ++next_k;
                        if constexpr (C::DO_DK) {
                            const uint64_t qmn =
                                q_desc_mn + static_cast<uint64_t>((s * C::Q_BYTES) >> 4);
#pragma unroll
                            for (int k = 0; k < C::BM / 16; ++k)
                                mma_ts(tmem + C::TM_DK, t_r + k * 8, qmn + ((k * 2048) >> 4),
                                       IDESC_DK, (acc_k || k > 0) ? 1u : 0u);
                        }
                        if constexpr (C::FDQ) {
                            // dQ_tile = dS K into the region dK has just read
                            const uint64_t dsd =
                                ds_desc + static_cast<uint64_t>((w * C::DS_STRIDE) >> 4);
#pragma unroll
                            for (int k = 0; k < C::BN / 16; ++k)
                                mma_ss(t_r, dsd + ((k * 2048) >> 4), k_desc_mn + ((k * 2048) >> 4),
                                       IDESC_DQ, k > 0 ? 1u : 0u);
                            mma_commit(&dq_full[w]);
                        }
                        lu_[w] = lu + 1;
                        st_[w] = 0;
                        // no later S^T of this group frees the stage (or, with no
                        // more stages than groups, that S^T would need it first)
                        if (!C::Q_BY_REDUCER && (!C::RELAY_Q || lu + 1 >= n_of(w)))
                            mma_commit(&q_empty[s]);
                        if (lu + 1 >= n_of(w)) {
                            --remaining;
                        } else if (!C::FDQ && s_ready(u + C::NWG)) {
                            issue_s(w, u + C::NWG);
                            st_[w] = 1;
                        }
                        prog = true;
                    }
                }
                if (prog) {
                    idle = false;
                } else if (*abort) {
                    ok = false;
                } else {
                    const uint64_t now = globaltimer();
                    if (!idle) {
                        idle = true;
                        idle_t0 = now;
                    } else if (now - idle_t0 > tmo) {
                        *abort = 1;
                        atomicExch(&g_err_bwd, ERR_TIMEOUT);
                        ok = false;
                    }
                }
            }
            mma_commit(done);
        }
    } else {
        // compute warpgroups: thread = key column (TMEM lane)
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int gkey = kt * TILE + row;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const uint32_t t_r = lane_base + C::TM_W0 + wg * C::BM;
        const int4 cv = p.vec[static_cast<size_t>(bm) * p.Npad + gkey];
        const float sl2 = p.sl2;

        const int n_my = n_of(wg);
        const float *slse = reinterpret_cast<const float *>(sLD + wg * C::LD_BYTES);
        const float *sd = slse + C::BM;
        if constexpr (C::FDQ) {
            // Group 0 turns the key tile's V (bf16, loaded once) into the scaled
            // fp16 operand of dP^T in place: 8 values per 16-byte unit, so the
            // swizzled layout is unchanged.
            if (wg == 0 && n > 0) {
                if (warp_wait(kv_full, 0, tmo, abort)) {
                    const float sv = p.scales[bh].y;
                    uint4 *vb = reinterpret_cast<uint4 *>(sV);
#pragma unroll 4
                    for (int k = row; k < C::V_BYTES / 16; k += 128) vb[k] = bf16x8_to_fp16x8(vb[k], sv);
                    fence_proxy_async_smem();
                }
                mbar_arrive(v_ready);
            }
        }
        if constexpr (C::V_TM) {
            // Group 0 puts the key tile's V rows (fp16 pairs; zeros past N) into
            // TMEM, where every dP^T of the CTA reads them.
            if (wg == 0 && n > 0) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    static_cast<const __half *>(p.v16) +
                    ((static_cast<size_t>(b) * p.N + (gkey < p.N ? gkey : 0)) * p.H + h) *
                        C::DV);
#pragma unroll 1
                for (int c = 0; c < C::DV / 64; ++c) {
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint4 w4 = gkey < p.N ? src[c * 8 + i] : make_uint4(0u, 0u, 0u, 0u);
                        r[4 * i] = w4.x;
                        r[4 * i + 1] = w4.y;
                        r[4 * i + 2] = w4.z;
                        r[4 * i + 3] = w4.w;
                    }
                    tmem_st32(lane_base + C::TM_V + c * 32, r);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(v_ready);
            }
        }
        int entry_next = n_my > 0 ? entries[wg / C::SUB] : 0;
        for (int lu = 0; lu < n_my; ++lu) {
            const int u = lu * C::NWG + wg;
            const int entry = entry_next;
            if (u + C::NWG < n) entry_next = entries[(u + C::NWG) / C::SUB];
            const bool need_mask = entry & 1;
            const int q0 = (entry >> 1) * TILE + (u % C::SUB) * C::BM;
            if (!warp_wait(&s_full[wg], lu & 1, tmo, abort)) break;
            if (!warp_wait(&o_full[wg], lu & 1, tmo, abort)) break;
            tc_fence_after();
            // S^T of this tile ran after the group's previous dK: that Q stage is free.
            if (C::RELAY_Q && !C::Q_BY_REDUCER && ((warp - 2) & 3) == 0 && lane == 0 && lu > 0)
                mbar_arrive(&q_empty[(u - C::NWG) % C::QS]);
            // phase 1: P^T = exp2(S^T * scale * log2e - LSE2), masked; fp16 pairs
            uint32_t pk[C::BM / 2];
#pragma unroll
            for (int c = 0; c < C::BM / 64; ++c) {
                float x[64];
                tmem_ld64f(t_r + c * 64, x);
                // Partial tiles: this thread's key column's masked query rows of
                // the chunk as bits, applied after the exponent (two loop copies,
                // so that full tiles carry no selects).
                auto exp_pack = [&](auto masked, uint32_t mw0, uint32_t mw1) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float4 l4 =
                            *reinterpret_cast<const float4 *>(slse + c * 64 + 4 * (i / 2));
                        const float2 l2 =
                            (i & 1) ? make_float2(l4.z, l4.w) : make_float2(l4.x, l4.y);
                        const float2 t =
                            __ffma2_rn(make_float2(x[2 * i], x[2 * i + 1]), make_float2(sl2, sl2),
                                       make_float2(-l2.x, -l2.y));
                        float p0 = ex2(t.x);
                        float p1 = ex2(t.y);
                        if constexpr (decltype(masked)::value) {
                            const uint32_t w = (2 * i < 32) ? mw0 : mw1;
                            if ((w >> ((2 * i) & 31)) & 1u) p0 = 0.f;
                            if ((w >> ((2 * i + 1) & 31)) & 1u) p1 = 0.f;
                        }
                        pk[c * 32 + i] = pack_fp16(p0, p1);
                    }
                };
                if (need_mask)
                    exp_pack(std::true_type{}, column_row_bits(q0 + c * 64, gkey, cv, p.causal),
                             column_row_bits(q0 + c * 64 + 32, gkey, cv, p.causal));
                else
                    exp_pack(std::false_type{}, 0u, 0u);
                if constexpr (C::DO_DV) {
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = pk[c * 32 + i];
                    tmem_st32(t_r + c * 32, r);  // columns already read
                }
            }
            if constexpr (C::DO_DV) tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[wg]);  // S^T read (and P^T written)
            if constexpr (C::DO_DK) {
                // phase 2: dS^T = P^T * (dP^T - D) -> the region, bf16
                if (!warp_wait(&dp_full[wg], lu & 1, tmo, abort)) break;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < C::BM / 64; ++c) {
                    float dp[64];
                    tmem_ld64f(t_r + c * 64, dp);
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {  // paired fp32 add and multiply
                        const float4 d4 = *reinterpret_cast<const float4 *>(sd + c * 64 + 4 * (i / 2));
                        const float2 dd = (i & 1) ? make_float2(d4.z, d4.w) : make_float2(d4.x, d4.y);
                        __half2 h2 = *reinterpret_cast<__half2 *>(&pk[c * 32 + i]);
                        const float2 ds = __fmul2_rn(
                            __half22float2(h2),
                            __fadd2_rn(make_float2(dp[2 * i], dp[2 * i + 1]),
                                       make_float2(-dd.x, -dd.y)));
                        r[i] = pack_bf16(ds.x, ds.y);
                    }
                    tmem_st32(t_r + c * 32, r);  // columns already read
                    if constexpr (C::FDQ) {
                        // this key's row of the dS tile: queries 64c .. 64c + 63 in
                        // block c, 16-byte units swizzled by the row (128B pattern)
                        uint8_t *ds_row = sDS + wg * C::DS_STRIDE + c * (C::BN * 128) + row * 128;
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            *reinterpret_cast<uint4 *>(ds_row + ((q ^ (row & 7)) * 16)) =
                                make_uint4(r[4 * q], r[4 * q + 1], r[4 * q + 2], r[4 * q + 3]);
                    }
                }
                if constexpr (C::FDQ) fence_proxy_async_smem();  // dS tile -> the MMA
                tmem_st_wait();
                tc_fence_before();
            }
            mbar_arrive(&ds_full[wg]);
            if constexpr (C::FDQ) {
                // phase 3: the tile's dQ rows (TMEM lane = query row q0 + row)
                // added to the fp32 buffer; then the region is free
                if (!warp_wait(&dq_full[wg], lu & 1, tmo, abort)) break;
                tc_fence_after();
                if constexpr (C::DQ_TMA_COLS > 0) {
                    // the first columns to the tile's spent Q stage, for the reducer
                    float4 *stg = reinterpret_cast<float4 *>(sQ + (u % C::QS) * C::Q_BYTES) + row;
#pragma unroll 1
                    for (int c = 0; c < C::DQ_TMA_COLS / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld32(t_r + c * 32, r);
#pragma unroll
                        for (int q = 0; q < 8; ++q)
                            stg[(c * 8 + q) * 128] =
                                make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                            __uint_as_float(r[4 * q + 2]),
                                            __uint_as_float(r[4 * q + 3]));
                    }
                    fence_proxy_async_smem();
                    mbar_arrive(&staged[wg]);  // release: the engine reads these writes
                }
                float4 *dst = p.dqacc + bh * (C::D / 4) * static_cast<size_t>(p.Npad) + q0 + row;
#pragma unroll 1
                for (int c = C::DQ_TMA_COLS / 32; c < C::D / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld32(t_r + c * 32, r);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        red_add_v4(dst + static_cast<size_t>(c * 8 + q) * p.Npad,
                                   __uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                   __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3]));
                }
                // Only the TMEM reads (complete at tcgen05.wait::ld) must precede
                // the next S^T; the reductions need no ordering inside the CTA.
                tc_fence_before();
                mbar_arrive_relaxed(&dq_free[wg]);
            }
        }
        if (n > 0) warp_wait(done, 0, tmo, abort);
        tc_fence_after();
        // dK (times scale / (s_o s_v)) and dV (times 1 / s_o): added to the fp32
        // outputs (acc32), or as bf16 to the 128B-swizzled layouts of the output
        // maps in idle shared memory (the Q ring, or with fused dQ the dO
        // stages), then TMA stores of their 64-column boxes (rows past N
        // clipped).
        const float4 sc = p.scales[bh];
        if constexpr (ACC32) {
            // fp32 accumulation: each key row adds its own values (rows past N
            // and CTAs without work add nothing).
            const size_t grow_off = (static_cast<size_t>(b) * p.N + gkey) * p.H + h;
            if constexpr (C::DO_DK) {
                constexpr int CPW = (C::D / 32) / C::NWG;
                float *dst = static_cast<float *>(p.dk) + grow_off * C::D;
#pragma unroll 1
                for (int c = wg * CPW; c < (wg + 1) * CPW && n > 0; ++c) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + C::TM_DK + c * 32, r);
                    if (gkey < p.N) add_row_f32(dst, c, r, p.scale * sc.w);
                }
            }
            if constexpr (C::DO_DV) {
                constexpr int CPW = (C::DV / 32) / C::NWG;
                float *dst = static_cast<float *>(p.dv) + grow_off * C::DV;
#pragma unroll 1
                for (int c = wg * CPW; c < (wg + 1) * CPW && n > 0; ++c) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + C::TM_DV + c * 32, r);
                    if (gkey < p.N) add_row_f32(dst, c, r, sc.z);
                }
            }
        } else {
            // Staging: the Q ring, or (fused dQ) the dO stages, spent once every
            // MMA ran (their dS tiles included), while the dQ reducer may still
            // be reading its last tile from the Q ring.
            uint8_t *stage_dk = C::FDQ ? sDO : sQ;
            uint8_t *stage_dv = stage_dk + (C::DO_DK ? C::D / 64 : 0) * (128 * 128);
            if constexpr (C::DO_DK) {
                constexpr int CPW = (C::D / 32) / C::NWG;
#pragma unroll 1
                for (int c = wg * CPW; c < (wg + 1) * CPW; ++c) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + C::TM_DK + c * 32, r);
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = n > 0 ? __uint_as_float(r[i]) : 0.f;
                    stage_row_bf16(stage_dk, c, row, v, p.scale * sc.w);
                }
            }
            // dK's boxes go out while dV is staged; the wait for the reads at
            // the end covers both stores.  In the split backward a group that
            // owns whole 64-column boxes of dK and dV stores them itself, after
            // its own barrier; otherwise one thread stores every box after
            // CTA-wide barriers.  (Measured: dK first 0.6 % faster for the
            // one-pass kernel, per-group stores another 0.4 % for the split
            // one and 0.3 % slower for the one-pass one.)
            constexpr bool OWN_BOXES = !C::FDQ && C::DO_DK && C::DO_DV &&
                                       ((C::D / 32) / C::NWG) % 2 == 0 &&
                                       ((C::DV / 32) / C::NWG) % 2 == 0;
            const bool g_leader = ((threadIdx.x - 64) & 127) == 0;
            if constexpr (C::DO_DK && C::DO_DV) {
                fence_proxy_async_smem();
                if constexpr (OWN_BOXES) {
                    named_bar_sync(2 + wg, 128);
                    if (g_leader) {
                        constexpr int BPW = (C::D / 64) / C::NWG;
                        for (int box = wg * BPW; box < (wg + 1) * BPW; ++box)
                            tma_store_4d(&tm_dk, stage_dk + box * (128 * 128), box * 64, h,
                                         kt * TILE, b);
                        bulk_commit();
                    }
                } else {
                    named_bar_sync(1, C::NWG * 128);
                    if (threadIdx.x == 64) {
                        for (int box = 0; box < C::D / 64; ++box)
                            tma_store_4d(&tm_dk, stage_dk + box * (128 * 128), box * 64, h,
                                         kt * TILE, b);
                        bulk_commit();
                    }
                }
            }
            if constexpr (C::DO_DV) {
                constexpr int CPW = (C::DV / 32) / C::NWG;
#pragma unroll 1
                for (int c = wg * CPW; c < (wg + 1) * CPW; ++c) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + C::TM_DV + c * 32, r);
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = n > 0 ? __uint_as_float(r[i]) : 0.f;
                    stage_row_bf16(stage_dv, c, row, v, sc.z);  // dV = (P^T dO s_o) / s_o
                }
            }
            fence_proxy_async_smem();
            if constexpr (OWN_BOXES) {
                named_bar_sync(2 + wg, 128);
                if (g_leader) {
                    constexpr int BPW = (C::DV / 64) / C::NWG;
                    for (int box = wg * BPW; box < (wg + 1) * BPW; ++box)
                        tma_store_4d(&tm_dv, stage_dv + box * (128 * 128), box * 64, h,
                                     kt * TILE, b);
                    bulk_commit_wait_read();
                }
            } else {
                named_bar_sync(1, C::NWG * 128);
                if (threadIdx.x == 64) {
                    if constexpr (C::DO_DK && !C::DO_DV)
                        for (int box = 0; box < C::D / 64; ++box)
                            tma_store_4d(&tm_dk, stage_dk + box * (128 * 128), box * 64, h,
                                         kt * TILE, b);
                    if constexpr (C::DO_DV)
                        for (int box = 0; box < C::DV / 64; ++box)
                            tma_store_4d(&tm_dv, stage_dv + box * (128 * 128), box * 64, h,
                                         kt * TILE, b);
                    bulk_commit_wait_read();
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    // After a wait gave up, what this CTA still has in flight lands before it
    // frees TMEM and exits: both rings' loads, the tiles loaded at the start and
    // the MMAs.  Past the barrier *abort is final and the same for every
    // thread; on the normal path every load was consumed and every MMA waited
    // for, and nothing is left to drain.
    if (*abort) {
        if (threadIdx.x == 0 && n > 0) {
            drain_ring(q_full, C::QS, issued[0], -1, tmo, &g_err_bwd);
            drain_ring(o_full, C::NWG, issued[1], -1, tmo, &g_err_bwd);
            mbar_wait_drain(kv_full, 0, tmo, &g_err_bwd);
            mbar_wait_drain(done, 0, tmo, &g_err_bwd);
        }
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

// One key tile per CTA: grid (T, H, B).
template <class C, bool ACC32>
__global__ void __launch_bounds__(C::THREADS, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                const BwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    dkdv_body<C, ACC32>(smem, tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv, p, blockIdx.x, blockIdx.y,
                        blockIdx.z);
}

// The split backward (deterministic mode, d >= 192) as one launch: CTAs
// [0, T H B) take the key side (key tile fastest, then head, then batch), the
// rest the query side (heaviest query tiles first).  One griddepcontrol.wait
// orders both after the kernels before, and the query-side CTAs, last in block
// order, start on the SMs the key side's tail frees.
template <class KV, class DQ, bool ACC32>
__global__ void __launch_bounds__(KV::THREADS, 1)
    split_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                     const __grid_constant__ CUtensorMap tm_dk,
                     const __grid_constant__ CUtensorMap tm_dv,
                     const __grid_constant__ CUtensorMap tm_q_dq,
                     const __grid_constant__ CUtensorMap tm_k_dq,
                     const __grid_constant__ CUtensorMap tm_v_dq,
                     const __grid_constant__ CUtensorMap tm_do_dq,
                     const __grid_constant__ CUtensorMap tm_dq, const BwdParams pkv,
                     const BwdParams pdq) {
    static_assert(KV::THREADS == DQ::THREADS, "one block shape for both roles");
    extern __shared__ __align__(1024) uint8_t smem[];
    const int half = static_cast<int>(gridDim.x) / 2;  // T H B CTAs per role
    const int c = static_cast<int>(blockIdx.x);
    const int TH = pkv.T * pkv.H;
    if (c < half)
        dkdv_body<KV, ACC32>(smem, tm_q, tm_k, tm_v, tm_do, tm_dk, tm_dv, pkv, c % pkv.T,
                             (c / pkv.T) % pkv.H, c / TH);
    else
        dq_body<DQ, ACC32>(smem, tm_q_dq, tm_k_dq, tm_v_dq, tm_do_dq, tm_dq, pdq,
                           pdq.T - 1 - (c - half) % pdq.T, ((c - half) / pdq.T) % pdq.H,
                           (c - half) / TH);
}

BwdParams make_params(const Geometry &g, const Workspace &ws, const BwdArgs &a, bool dq_side) {
    BwdParams p;
    p.vec = ws.vec;
    p.list = dq_side ? ws.fwd_list : ws.bwd_list;
    p.cnt = dq_side ? ws.fwd_cnt : ws.bwd_cnt;
    p.lse2 = ws.lse2;
    p.delta = ws.delta;
    p.do16 = ws.do16;
    p.v16 = ws.v16;
    p.scales = ws.scales;
    p.dqacc = ws.dqacc;
    p.dq = a.dq;
    p.dk = a.dk;
    p.dv = a.dv;
    p.N = g.N;
    p.H = g.H;
    p.Hm = g.Hm;
    p.T = g.T;
    p.Npad = g.Npad;
    p.causal = g.causal;
    p.sl2 = g.scale * 1.4426950408889634f;
    p.scale = g.scale;
    p.timeout_ns = g.timeout_ns;
    p.ordered = g.deterministic != 0;
    return p;
}

template <class C>
cudaError_t launch_dkdv(const Geometry &g, const Workspace &ws, const BwdArgs &a,
                        cudaStream_t st) {
    if (a.kv_q_rows != C::BM) return cudaErrorInvalidValue;  // map boxes must match the tile
    auto kern = g.acc32 ? dkdv_kernel<C, true> : dkdv_kernel<C, false>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(g.T, g.H, g.B), dim3(C::THREADS), C::SMEM_BYTES, st, *a.tm_q,
                      *a.tm_k, *a.tm_v, *a.tm_do, *a.tm_dk_out, *a.tm_dv_out,
                      make_params(g, ws, a, false));
}

template <class KV, class DQ>
cudaError_t launch_pair(const Geometry &g, const Workspace &ws, const BwdArgs &a, cudaStream_t st,
                        Recorder &rec) {
    if (a.kv_q_rows != KV::BM || a.dq_k_rows != DQ::BN)
        return cudaErrorInvalidValue;  // map boxes must match the tiles
    auto kern = g.acc32 ? split_bwd_kernel<KV, DQ, true> : split_bwd_kernel<KV, DQ, false>;
    constexpr int SMEM = KV::SMEM_BYTES > DQ::SMEM_BYTES ? KV::SMEM_BYTES : DQ::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    rec.before(st);
    e = launch_pdl(kern, dim3(2 * g.T * g.H * g.B), dim3(KV::THREADS), SMEM, st, *a.tm_q, *a.tm_k,
                   *a.tm_v, *a.tm_do, *a.tm_dk_out, *a.tm_dv_out, *a.tm_q_dq, *a.tm_k_dq,
                   *a.tm_v_dq, *a.tm_do_dq, *a.tm_dq_out, make_params(g, ws, a, false),
                   make_params(g, ws, a, true));
    rec.after(st);
    return e;
}

}  // namespace

// Key sub-tile of the query-side kernel (128 up to d = 192, with dO in TMEM at
// d = 192) and query sub-tile of the key-side kernel (128 up to d = 128): 128
// gives full-rate N = 128 MMAs, 64 is what shared memory holds above.
int dq_key_rows(int d, int) { return d <= 192 ? 128 : 64; }
int dkdv_query_rows(int d, int) { return d <= 128 ? 128 : 64; }

cudaError_t launch_bwd(const Geometry &g, const Workspace &ws, const BwdArgs &a,
                       cudaStream_t st, Recorder &rec) {
    const int rows_total = g.B * g.H * g.Npad;
    // The preprocess step: input ranges, their scales, then D, LSE2 and the
    // scaled fp16 copies (one event pair around the three launches).
    rec.before(st);
    cudaError_t e = launch_pdl(range_kernel, dim3(g.T, g.H, g.B), dim3(256), 0, st, g.N, g.H,
                               g.dv, g.T, static_cast<const uint4 *>(a.dout),
                               static_cast<const uint4 *>(a.v), ws.range_part);
    if (e == cudaSuccess)
        e = launch_pdl(scale_kernel, dim3(g.B * g.H), dim3(256), 0, st, g.T,
                       static_cast<const uint2 *>(ws.range_part), ws.scales);
    if (e == cudaSuccess)
        e = launch_pdl(preprocess_kernel, dim3((rows_total + 15) / 16), dim3(256), 0, st, g.N,
                       g.H, g.dv, g.Npad, rows_total, static_cast<const __nv_bfloat16 *>(a.o),
                       static_cast<const __nv_bfloat16 *>(a.dout),
                       static_cast<const __nv_bfloat16 *>(a.v), static_cast<const float *>(a.lse),
                       ws.lse2, ws.delta, static_cast<uint4 *>(ws.v16),
                       static_cast<uint4 *>(ws.do16), static_cast<const float4 *>(ws.scales),
                       g.sink, g.dsink ? ws.sink_part : nullptr, ws.dqacc, g.d / 4);
    rec.after(st);
    if (e == cudaSuccess && g.dsink)
        e = launch_pdl(sink_grad_kernel, dim3(g.H), dim3(256), 0, st, g.B, g.H, g.Npad / 16,
                       static_cast<const float *>(ws.sink_part), g.dsink);
    if (e != cudaSuccess) return e;
    if (fused_dq(g)) {
        // One key-side pass with dQ reduced into the fp32 buffer, then dQ out.
        rec.before(st);
        e = g.d == 64 ? launch_dkdv<DkdvCfg<64, 64, 128, 5, true, true, 2, false, true>>(g, ws, a, st)
                      : launch_dkdv<DkdvCfg<128, 128, 128, 3, true, true, 2, false, true>>(g, ws,
                                                                                            a, st);
        rec.after(st);
        if (e != cudaSuccess) return e;
        rec.before(st);
        const dim3 cgrid((g.N + CONV_ROWS - 1) / CONV_ROWS, g.H, g.B);
        auto conv = g.d == 64 ? (g.acc32 ? dq_convert_kernel<true, 64> : dq_convert_kernel<false, 64>)
                              : (g.acc32 ? dq_convert_kernel<true, 128>
                                         : dq_convert_kernel<false, 128>);
        e = launch_pdl(conv, cgrid, dim3(256), 0, st, g.N, g.H, g.Npad,
                       static_cast<const float4 *>(ws.dqacc), static_cast<const float4 *>(ws.scales),
                       g.scale, a.dq);
        rec.after(st);
        return e;
    }
    // DkdvCfg<d, dv, query sub-tile, Q stages, dK, dV, groups>;
    // DqCfg<d, dv, key sub-tile, K stages, groups>
    if (g.d == 64 && g.dv == 64)
        return launch_pair<DkdvCfg<64, 64, 128, 3, true, true, 2>, DqCfg<64, 64, 128, 3, 2>>(
            g, ws, a, st, rec);
    if (g.d == 128 && g.dv == 128)
        return launch_pair<DkdvCfg<128, 128, 128, 3, true, true, 2>, DqCfg<128, 128, 128, 3, 2>>(
            g, ws, a, st, rec);
    if (g.d == 192 && g.dv == 128)
        return launch_pair<DkdvCfg<192, 128, 64, 4, true, true, 2, true>,
                           DqCfg<192, 128, 128, 2, 2, true>>(
            g, ws, a, st, rec);
    if (g.d == 256 && g.dv == 256) {
        rec.before(st);
        e = launch_dkdv<DkdvCfg<256, 256, 64, 2, false, true, 2>>(g, ws, a, st);
        rec.after(st);
        if (e != cudaSuccess) return e;
        return launch_pair<DkdvCfg<256, 256, 64, 3, true, false, 2, true>,
                           DqCfg<256, 256, 64, 3, 2, true>>(
            g, ws, a, st, rec);
    }
    return cudaErrorInvalidValue;
}

unsigned read_clear_error_bwd() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_bwd, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_err_bwd, &zero, sizeof(zero));
    return v;
}

}  // namespace fm
