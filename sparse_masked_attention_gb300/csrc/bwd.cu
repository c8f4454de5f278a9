// bwd.cu -- backward of FlashMask masked attention on tcgen05 tensor cores.
//
// The derivative of O = softmax(Q K^T * scale + M) V (FlashMask README,
// "Formulation").  P is rebuilt from the forward's LSE:
//   P = exp(S * scale - LSE),  dP = dO V^T,  D_i = sum_c dO_ic O_ic,
//   dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// The backward walks the same tile map as the forward: fully masked tiles are
// skipped, and the mask is applied elementwise only on partial tiles.
//
// Three kernels:
//   preprocess   D (fp32) and the log2-domain LSE per row, padded to whole
//                tiles; padding rows and fully masked rows get LSE = +inf, so
//                their P is 0.
//   dq kernel    one CTA per 128-row query tile walks its key tiles:
//                S = Q K^T (bf16), dP = dO V^T (fp16 copies) as SS MMAs;
//                dS -> shared memory (bf16);
//                dQ += dS K (SS MMA).  Writes dQ once, in a fixed order.
//   dkdv kernel  one CTA per 128-key tile walks its query tiles:
//                S^T = K Q^T (bf16), dP^T = V dO^T (fp16 copies) as SS MMAs;
//                P^T -> TMEM as fp16, dS^T as bf16; dV += P^T dO (fp16) and
//                dK += dS^T Q (bf16) as TS MMAs.
// No atomics are used, so every gradient is bit-reproducible.  For
// d = dv = 256 the accumulators dK and dV do not fit in TMEM together, so
// the dkdv kernel runs twice: once for dV, once for dK.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

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

__device__ __forceinline__ void store_row_bf16(__nv_bfloat16 *dst, const float (&v)[32],
                                               float mul) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16(v[q * 8 + 0] * mul, v[q * 8 + 1] * mul);
        w.y = pack_bf16(v[q * 8 + 2] * mul, v[q * 8 + 3] * mul);
        w.z = pack_bf16(v[q * 8 + 4] * mul, v[q * 8 + 5] * mul);
        w.w = pack_bf16(v[q * 8 + 6] * mul, v[q * 8 + 7] * mul);
        d4[q] = w;
    }
}

// ---------------------------------------------------------------- preprocess
// 16 threads per row; each takes 8 consecutive bf16 of dO, O and V at a time.
// Besides D and LSE2 it writes fp16 copies of V and dO: the backward's dP and
// dV products run in fp16 (10 mantissa bits against bf16's 7), which keeps the
// probabilities' rounding well below the bf16 rounding of the outputs.
__device__ __forceinline__ uint4 bf16x8_to_fp16x8(uint4 a) {
    const __nv_bfloat162 *a2 = reinterpret_cast<const __nv_bfloat162 *>(&a);
    uint4 r;
    uint32_t *r32 = reinterpret_cast<uint32_t *>(&r);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(a2[e]);
        r32[e] = pack_fp16(f.x, f.y);
    }
    return r;
}

__global__ void __launch_bounds__(256) preprocess_kernel(
    int N, int H, int dv, int Npad, int rows_total, const __nv_bfloat16 *__restrict__ o,
    const __nv_bfloat16 *__restrict__ dout, const __nv_bfloat16 *__restrict__ v,
    const float *__restrict__ lse, float *__restrict__ lse2, float *__restrict__ delta,
    uint4 *__restrict__ v16, uint4 *__restrict__ do16) {
    const int r0 = blockIdx.x * 16 + (threadIdx.x >> 4);  // over B*H*Npad
    const int t = threadIdx.x & 15;
    const bool valid = r0 < rows_total;
    const int r = valid ? r0 : 0;
    const int bh = r / Npad, i = r % Npad;
    const int b = bh / H, h = bh % H;
    float acc = 0.f;
    if (valid && i < N) {
        const size_t base = ((static_cast<size_t>(b) * N + i) * H + h) * dv;
        for (int c = t * 8; c < dv; c += 128) {
            const uint4 a = *reinterpret_cast<const uint4 *>(o + base + c);
            const uint4 g = *reinterpret_cast<const uint4 *>(dout + base + c);
            const uint4 vv = *reinterpret_cast<const uint4 *>(v + base + c);
            do16[(base + c) / 8] = bf16x8_to_fp16x8(g);
            v16[(base + c) / 8] = bf16x8_to_fp16x8(vv);
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
    if (valid && t == 0) {
        float l2 = INFINITY;
        if (i < N) {
            const float l = lse[static_cast<size_t>(bh) * N + i];
            l2 = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
        }
        lse2[r] = l2;
        delta[r] = i < N ? acc : 0.f;
    }
}

struct BwdParams {
    const int4 *vec;
    const int *list;  // fwd list (dq kernel) or bwd list (dkdv kernel)
    const int *cnt;
    const float *lse2;
    const float *delta;
    __nv_bfloat16 *dq, *dk, *dv;
    int N, H, Hm, T, Npad, causal;
    float sl2;    // scale * log2(e)
    float scale;
    uint64_t timeout_ns;
};

// ------------------------------------------------------------------ dq kernel
// One CTA per 128-row query tile.  NWG compute warpgroups take alternate key
// sub-tiles of BN keys; each has its own S/dP region in TMEM and its own dS
// buffer in shared memory, and all of them feed one dQ accumulator.
template <int D_, int DV_, int BN_, int ST_, int NWG_, int ES_>
struct DqCfg {
    static constexpr int D = D_, DV = DV_, BN = BN_, ST = ST_, NWG = NWG_, ES = ES_;
    static constexpr int BM = 128;
    static constexpr int SUB = TILE / BN;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int DO_BYTES = BM * DV * 2;
    static constexpr int K_BYTES = BN * D * 2;
    static constexpr int V_BYTES = BN * DV * 2;
    static constexpr int DS_BYTES = BM * BN * 2;
    static constexpr int E_BYTES = BN * 16;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_DO = OFF_Q + Q_BYTES;
    static constexpr int OFF_DS = OFF_DO + DO_BYTES;
    static constexpr int OFF_K = OFF_DS + NWG * DS_BYTES;
    static constexpr int OFF_V = OFF_K + ST * K_BYTES;
    static constexpr int OFF_E = OFF_V + ST * V_BYTES;
    static constexpr int OFF_BAR = OFF_E + ES * E_BYTES;
    // q_full, kv_full[ST], kv_empty[ST], e_full[ES], e_empty[ES], s_full[NWG],
    // ds_full[NWG], dq_done
    static constexpr int NBAR = 1 + 2 * ST + 2 * ES + 2 * NWG + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int TM_SDP = 2 * BN;  // per group: S then dP
    static constexpr int TM_DQ = NWG * TM_SDP;
    static constexpr int TM_COLS = 512;
    static constexpr int THREADS = 64 + NWG * 128;
    static_assert(TM_DQ + D <= TM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(BN == 64 || BN == 128, "key sub-tile");
    static_assert(ST >= NWG && ES % NWG == 0, "ring depths");
    static_assert((D / 32) % NWG == 0, "epilogue column split");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
              const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sQ = smem + C::OFF_Q, *sDO = smem + C::OFF_DO, *sDS = smem + C::OFF_DS;
    uint8_t *sK = smem + C::OFF_K, *sV = smem + C::OFF_V, *sE = smem + C::OFF_E;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *q_full = bars, *kv_full = bars + 1, *kv_empty = kv_full + C::ST;
    uint64_t *e_full = kv_empty + C::ST, *e_empty = e_full + C::ES;
    uint64_t *s_full = e_empty + C::ES, *ds_full = s_full + C::NWG, *dq_done = ds_full + C::NWG;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = p.T - 1 - static_cast<int>(blockIdx.x);
    const int h = blockIdx.y, b = blockIdx.z;
    const int bm = b * p.Hm + (p.Hm == 1 ? 0 : h);
    const int n_entries = p.cnt[static_cast<size_t>(bm) * p.T + qt];
    const int *entries = p.list + (static_cast<size_t>(bm) * p.T + qt) * p.T;
    // After a bounded wait gave up anywhere, later CTAs do no work.
    const int n = (*reinterpret_cast<volatile unsigned *>(&g_err_bwd) != 0) ? 0
                                                                            : n_entries * C::SUB;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < C::ST; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
        for (int i = 0; i < C::ES; ++i) {
            mbar_init(&e_full[i], 1);
            mbar_init(&e_empty[i], 128);
        }
        for (int i = 0; i < C::NWG; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&ds_full[i], 128);
        }
        mbar_init(dq_done, 1);
        *abort = 0;
        fence_barrier_init();
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
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            prefetch_tmap(&tm_do);
            mbar_arrive_expect_tx(q_full, C::Q_BYTES + C::DO_BYTES);
#pragma unroll
            for (int c = 0; c < C::D / 64; ++c)
                tma_load_4d(sQ + c * C::BM * 128, &tm_q, q_full, c * 64, h, qt * TILE, b);
#pragma unroll
            for (int c = 0; c < C::DV / 64; ++c)
                tma_load_4d(sDO + c * C::BM * 128, &tm_do, q_full, c * 64, h, qt * TILE, b);
            for (int u = 0; u < n; ++u) {
                const int s = u % C::ST;
                if (u >= C::ST &&
                    !mbar_wait(&kv_empty[s], ((u / C::ST) - 1) & 1, tmo, abort, &g_err_bwd))
                    break;
                mbar_arrive_expect_tx(&kv_full[s], C::K_BYTES + C::V_BYTES);
                const int key0 = key0_of(u);
#pragma unroll
                for (int c = 0; c < C::D / 64; ++c)
                    tma_load_4d(sK + s * C::K_BYTES + c * C::BN * 128, &tm_k, &kv_full[s],
                                c * 64, h, key0, b);
#pragma unroll
                for (int c = 0; c < C::DV / 64; ++c)
                    tma_load_4d(sV + s * C::V_BYTES + c * C::BN * 128, &tm_v, &kv_full[s],
                                c * 64, h, key0, b);
            }
        } else if (lane == 1 && n > 0) {
            const int4 *vec = p.vec + static_cast<size_t>(bm) * p.Npad;
            for (int u = 0; u < n; ++u) {
                const int s = u % C::ES;
                if (u >= C::ES &&
                    !mbar_wait(&e_empty[s], ((u / C::ES) - 1) & 1, tmo, abort, &g_err_bwd))
                    break;
                mbar_arrive_expect_tx(&e_full[s], C::E_BYTES);
                bulk_load(sE + s * C::E_BYTES, vec + key0_of(u), C::E_BYTES, &e_full[s]);
            }
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
            const uint64_t ds_desc = sdesc_sw128(smem_u32(sDS), 16, 1024);
            const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t k_desc_mn = sdesc_sw128(smem_u32(sK), C::BN * 128, 1024);
            const uint64_t v_desc = sdesc_sw128(smem_u32(sV), 16, 1024);
            auto issue_s_dp = [&](int u) -> bool {
                const int s = u % C::ST, w = u % C::NWG;
                if (!mbar_wait(&kv_full[s], (u / C::ST) & 1, tmo, abort, &g_err_bwd)) return false;
                tc_fence_after();
                const uint32_t t_s = tmem + w * C::TM_SDP, t_dp = t_s + C::BN;
                const uint64_t ks = k_desc + static_cast<uint64_t>((s * C::K_BYTES) >> 4);
                const uint64_t vsd = v_desc + static_cast<uint64_t>((s * C::V_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < C::D / 16; ++k) {
                    const uint32_t a_off = ((k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4;
                    const uint32_t b_off = ((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4;
                    mma_ss(t_s, q_desc + a_off, ks + b_off, IDESC_S, k > 0 ? 1u : 0u);
                }
#pragma unroll
                for (int k = 0; k < C::DV / 16; ++k) {
                    const uint32_t a_off = ((k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4;
                    const uint32_t b_off = ((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4;
                    mma_ss(t_dp, do_desc + a_off, vsd + b_off, IDESC_DP, k > 0 ? 1u : 0u);
                }
                mma_commit(&s_full[w]);
                return true;
            };
            bool ok = mbar_wait(q_full, 0, tmo, abort, &g_err_bwd);
            for (int u = 0; u < C::NWG && u < n && ok; ++u) ok = issue_s_dp(u);
            for (int u = 0; u < n && ok; ++u) {
                const int w = u % C::NWG, lu = u / C::NWG, s = u % C::ST;
                if (!mbar_wait(&ds_full[w], lu & 1, tmo, abort, &g_err_bwd)) break;
                tc_fence_after();
                // dQ += dS K_u: A = dS (K-major over BN keys), B = K_u (MN-major over d).
                const uint64_t dsw = ds_desc + static_cast<uint64_t>((w * C::DS_BYTES) >> 4);
                const uint64_t kmn = k_desc_mn + static_cast<uint64_t>((s * C::K_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < C::BN / 16; ++k) {
                    const uint32_t a_off = ((k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4;
                    mma_ss(tmem + C::TM_DQ, dsw + a_off, kmn + ((k * 2048) >> 4), IDESC_DQ,
                           (u > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&kv_empty[s]);
                if (u + C::NWG < n) ok = issue_s_dp(u + C::NWG);
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
        const size_t bh = static_cast<size_t>(b) * p.H + h;
        const float lse2 = p.lse2[bh * p.Npad + grow];
        const float Drow = p.delta[bh * p.Npad + grow];
        const float sl2 = p.sl2;
        const int n_my = n > wg ? (n - wg + C::NWG - 1) / C::NWG : 0;
        // dS row of the K-major swizzled tile: 16-byte chunk c of 64-column box
        // kb lives at kb*BM*128 + r*128 + ((c ^ (r & 7)) * 16).
        uint8_t *ds_row = sDS + wg * C::DS_BYTES + row * 128;
        int entry_next = n_my > 0 ? entries[wg / C::SUB] : 0;
        for (int lu = 0; lu < n_my; ++lu) {
            const int u = lu * C::NWG + wg;
            const int entry = entry_next;
            if (u + C::NWG < n) entry_next = entries[(u + C::NWG) / C::SUB];
            const bool masked_tile = entry & 1;
            const int key0 = (entry >> 1) * TILE + (u % C::SUB) * C::BN;
            const int es = u % C::ES;
            if (!warp_wait(&s_full[wg], lu & 1, tmo, abort)) break;
            if (!warp_wait(&e_full[es], (u / C::ES) & 1, tmo, abort)) break;
            tc_fence_after();
            const uint32_t t_s = lane_base + wg * C::TM_SDP, t_dp = t_s + C::BN;
            const int4 *cv = reinterpret_cast<const int4 *>(sE + es * C::E_BYTES);
#pragma unroll
            for (int c = 0; c < C::BN / 64; ++c) {
                float pr[64], dp[64];
                tmem_ld64f_x2(t_s + c * 64, pr, t_dp + c * 64, dp);
#pragma unroll
                for (int jj = 0; jj < 64; ++jj) pr[jj] = ex2(fmaf(pr[jj], sl2, -lse2));
                if (masked_tile) {
                    // Row bits of key columns lane, lane + 32 over the warp's rows,
                    // transposed so each lane holds its row's column bits.
                    const int R = grow - lane;
                    const int ja = key0 + c * 64 + lane;
                    const uint32_t wa = warp_transpose32(
                        column_row_bits(R, ja, cv[c * 64 + lane], p.causal), lane);
                    const uint32_t wb = warp_transpose32(
                        column_row_bits(R, ja + 32, cv[c * 64 + 32 + lane], p.causal), lane);
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        if ((wa >> jj) & 1u) pr[jj] = 0.f;
                        if ((wb >> jj) & 1u) pr[32 + jj] = 0.f;
                    }
                }
                uint8_t *box = ds_row + c * C::BM * 128;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    uint4 w4;
                    w4.x = pack_bf16(pr[q * 8 + 0] * (dp[q * 8 + 0] - Drow),
                                     pr[q * 8 + 1] * (dp[q * 8 + 1] - Drow));
                    w4.y = pack_bf16(pr[q * 8 + 2] * (dp[q * 8 + 2] - Drow),
                                     pr[q * 8 + 3] * (dp[q * 8 + 3] - Drow));
                    w4.z = pack_bf16(pr[q * 8 + 4] * (dp[q * 8 + 4] - Drow),
                                     pr[q * 8 + 5] * (dp[q * 8 + 5] - Drow));
                    w4.w = pack_bf16(pr[q * 8 + 6] * (dp[q * 8 + 6] - Drow),
                                     pr[q * 8 + 7] * (dp[q * 8 + 7] - Drow));
                    *reinterpret_cast<uint4 *>(box + ((q ^ (row & 7)) * 16)) = w4;
                }
            }
            mbar_arrive(&e_empty[es]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&ds_full[wg]);
        }
        if (n > 0) warp_wait(dq_done, 0, tmo, abort);
        tc_fence_after();
        __nv_bfloat16 *dst =
            p.dq + ((static_cast<size_t>(b) * p.N + grow) * p.H + h) * static_cast<size_t>(C::D);
        constexpr int CPW = (C::D / 32) / C::NWG;  // 32-column chunks per group
#pragma unroll 1
        for (int c = wg * CPW; c < (wg + 1) * CPW; ++c) {
            uint32_t r[32];
            tmem_ld32(lane_base + C::TM_DQ + c * 32, r);
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = n > 0 ? __uint_as_float(r[i]) : 0.f;
            if (grow < p.N) store_row_bf16(dst + c * 32, v, p.scale);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

// ---------------------------------------------------------------- dkdv kernel
// One CTA per 128-key tile.  NWG compute warpgroups take alternate query
// sub-tiles of BM rows; each has its own S^T/dP^T region in TMEM, and all of
// them feed the one dK and the one dV accumulator.
template <int D_, int DV_, int BM_, int ST_, bool DK_, bool DV_ON_, int NWG_>
struct DkdvCfg {
    static constexpr int D = D_, DV = DV_, BM = BM_, ST = ST_, NWG = NWG_;
    static constexpr bool DO_DK = DK_, DO_DV = DV_ON_;
    static constexpr int BN = 128;            // keys per CTA (TMEM lanes)
    static constexpr int SUB = TILE / BM;     // query sub-tiles per list entry
    static constexpr bool NEED_V = DO_DK;     // V only feeds dP^T
    static constexpr int K_BYTES = BN * D * 2;
    static constexpr int V_BYTES = NEED_V ? BN * DV * 2 : 0;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int DO_BYTES = BM * DV * 2;
    static constexpr int STAGE_BYTES = Q_BYTES + DO_BYTES + 2 * BM * 4;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = OFF_K + K_BYTES;
    static constexpr int OFF_ST = OFF_V + V_BYTES;
    static constexpr int ST_Q = 0, ST_DO = Q_BYTES, ST_LSE = Q_BYTES + DO_BYTES,
                         ST_D = ST_LSE + BM * 4;
    static constexpr int STAGE_STRIDE = (STAGE_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_ST + ST * STAGE_STRIDE;
    // kv_full, q_full[ST], q_empty[ST], s_full[NWG], p_full[NWG], ds_full[NWG], done
    static constexpr int NBAR = 1 + 2 * ST + 3 * NWG + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
    static constexpr int TM_DK = 0;
    static constexpr int TM_DV = DO_DK ? D : 0;
    static constexpr int TM_W0 = TM_DV + (DO_DV ? DV : 0);
    static constexpr int TM_SDP = BM + (DO_DK ? BM : 0);  // per group: S^T then dP^T
    static constexpr int TM_END = TM_W0 + NWG * TM_SDP;
    static constexpr int TM_COLS = 512;
    static constexpr int THREADS = 64 + NWG * 128;
    static_assert(TM_END <= TM_COLS, "TMEM budget");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(D <= 256 && DV <= 256 && BM % 64 == 0, "MMA shape");
    static_assert(ST >= NWG, "ring depth");
    static_assert((D / 32) % NWG == 0 && (DV / 32) % NWG == 0, "epilogue column split");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v,
                const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t *sK = smem + C::OFF_K, *sV = smem + C::OFF_V, *sST = smem + C::OFF_ST;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *kv_full = bars, *q_full = bars + 1, *q_empty = q_full + C::ST;
    uint64_t *s_full = q_empty + C::ST, *p_full = s_full + C::NWG, *ds_full = p_full + C::NWG,
             *done = ds_full + C::NWG;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kt = blockIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    const int bm = b * p.Hm + (p.Hm == 1 ? 0 : h);
    const int n_entries = p.cnt[static_cast<size_t>(bm) * p.T + kt];
    const int *entries = p.list + (static_cast<size_t>(bm) * p.T + kt) * p.T;
    // After a bounded wait gave up anywhere, later CTAs do no work.
    const int n = (*reinterpret_cast<volatile unsigned *>(&g_err_bwd) != 0) ? 0
                                                                            : n_entries * C::SUB;
    const uint64_t tmo = p.timeout_ns;
    const size_t bh = static_cast<size_t>(b) * p.H + h;

    if (threadIdx.x == 0) {
        mbar_init(kv_full, 1);
        for (int i = 0; i < C::ST; ++i) {
            mbar_init(&q_full[i], 1);
            mbar_init(&q_empty[i], 1);
        }
        for (int i = 0; i < C::NWG; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&ds_full[i], 128);
        }
        mbar_init(done, 1);
        *abort = 0;
        fence_barrier_init();
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
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_do);
            mbar_arrive_expect_tx(kv_full, C::K_BYTES + C::V_BYTES);
#pragma unroll
            for (int c = 0; c < C::D / 64; ++c)
                tma_load_4d(sK + c * C::BN * 128, &tm_k, kv_full, c * 64, h, kt * TILE, b);
            if constexpr (C::NEED_V) {
                prefetch_tmap(&tm_v);
#pragma unroll
                for (int c = 0; c < C::DV / 64; ++c)
                    tma_load_4d(sV + c * C::BN * 128, &tm_v, kv_full, c * 64, h, kt * TILE, b);
            }
            for (int u = 0; u < n; ++u) {
                const int s = u % C::ST;
                if (u >= C::ST &&
                    !mbar_wait(&q_empty[s], ((u / C::ST) - 1) & 1, tmo, abort, &g_err_bwd))
                    break;
                uint8_t *stg = sST + s * C::STAGE_STRIDE;
                mbar_arrive_expect_tx(&q_full[s], C::STAGE_BYTES);
                const int q0 = q0_of(u);
#pragma unroll
                for (int c = 0; c < C::D / 64; ++c)
                    tma_load_4d(stg + C::ST_Q + c * C::BM * 128, &tm_q, &q_full[s], c * 64, h, q0,
                                b);
#pragma unroll
                for (int c = 0; c < C::DV / 64; ++c)
                    tma_load_4d(stg + C::ST_DO + c * C::BM * 128, &tm_do, &q_full[s], c * 64, h,
                                q0, b);
                bulk_load(stg + C::ST_LSE, p.lse2 + bh * p.Npad + q0, C::BM * 4, &q_full[s]);
                bulk_load(stg + C::ST_D, p.delta + bh * p.Npad + q0, C::BM * 4, &q_full[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && n > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(128, C::BM, false, false);
            constexpr uint32_t IDESC_DP = idesc_fp16(128, C::BM, false, false);
            constexpr uint32_t IDESC_DV = idesc_fp16(128, C::DV, false, true);
            constexpr uint32_t IDESC_DK = idesc_bf16(128, C::D, false, true);
            // Descriptors are built once; an MMA step only adds its byte offset
            // (in 16-byte units) to the start-address field.
            const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t v_desc = sdesc_sw128(smem_u32(sV), 16, 1024);
            const uint64_t st_desc = sdesc_sw128(smem_u32(sST), 16, 1024);
            const uint64_t st_desc_mn = sdesc_sw128(smem_u32(sST), C::BM * 128, 1024);
            auto issue_s = [&](int u) -> bool {
                const int s = u % C::ST, w = u % C::NWG;
                const uint64_t stg = st_desc + static_cast<uint64_t>((s * C::STAGE_STRIDE) >> 4);
                if (!mbar_wait(&q_full[s], (u / C::ST) & 1, tmo, abort, &g_err_bwd)) return false;
                tc_fence_after();
                const uint32_t t_s = tmem + C::TM_W0 + w * C::TM_SDP, t_dp = t_s + C::BM;
                // S^T = K Q^T
#pragma unroll
                for (int k = 0; k < C::D / 16; ++k) {
                    const uint32_t a_off = ((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4;
                    const uint32_t b_off = (C::ST_Q + (k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4;
                    mma_ss(t_s, k_desc + a_off, stg + b_off, IDESC_S, k > 0 ? 1u : 0u);
                }
                if constexpr (C::DO_DK) {
                    // dP^T = V dO^T
#pragma unroll
                    for (int k = 0; k < C::DV / 16; ++k) {
                        const uint32_t a_off = ((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4;
                        const uint32_t b_off =
                            (C::ST_DO + (k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4;
                        mma_ss(t_dp, v_desc + a_off, stg + b_off, IDESC_DP, k > 0 ? 1u : 0u);
                    }
                }
                mma_commit(&s_full[w]);
                return true;
            };
            bool ok = mbar_wait(kv_full, 0, tmo, abort, &g_err_bwd);
            for (int u = 0; u < C::NWG && u < n && ok; ++u) ok = issue_s(u);
            for (int u = 0; u < n && ok; ++u) {
                const int s = u % C::ST, w = u % C::NWG, lu = u / C::NWG;
                const uint64_t stg_mn =
                    st_desc_mn + static_cast<uint64_t>((s * C::STAGE_STRIDE) >> 4);
                const uint32_t t_s = tmem + C::TM_W0 + w * C::TM_SDP, t_dp = t_s + C::BM;
                if constexpr (C::DO_DV) {
                    if (!mbar_wait(&p_full[w], lu & 1, tmo, abort, &g_err_bwd)) break;
                    tc_fence_after();
                    // dV += P^T dO: A = P^T (TMEM, fp16), B = dO (MN-major over dv)
#pragma unroll
                    for (int k = 0; k < C::BM / 16; ++k)
                        mma_ts(tmem + C::TM_DV, t_s + k * 8, stg_mn + ((C::ST_DO + k * 2048) >> 4),
                               IDESC_DV, (u > 0 || k > 0) ? 1u : 0u);
                }
                // The group is done with this sub-tile's S^T / dP^T reads.
                if (!mbar_wait(&ds_full[w], lu & 1, tmo, abort, &g_err_bwd)) break;
                tc_fence_after();
                if constexpr (C::DO_DK) {
                    // dK += dS^T Q: A = dS^T (TMEM, bf16), B = Q (MN-major over d)
#pragma unroll
                    for (int k = 0; k < C::BM / 16; ++k)
                        mma_ts(tmem + C::TM_DK, t_dp + k * 8, stg_mn + ((C::ST_Q + k * 2048) >> 4),
                               IDESC_DK, (u > 0 || k > 0) ? 1u : 0u);
                }
                mma_commit(&q_empty[s]);
                if (u + C::NWG < n) ok = issue_s(u + C::NWG);
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
        const int4 cv = p.vec[static_cast<size_t>(bm) * p.Npad + gkey];
        const float sl2 = p.sl2;
        const int n_my = n > wg ? (n - wg + C::NWG - 1) / C::NWG : 0;
        int entry_next = n_my > 0 ? entries[wg / C::SUB] : 0;
        for (int lu = 0; lu < n_my; ++lu) {
            const int u = lu * C::NWG + wg;
            const int s = u % C::ST;
            const int entry = entry_next;
            if (u + C::NWG < n) entry_next = entries[(u + C::NWG) / C::SUB];
            const bool need_mask = entry & 1;
            const int q0 = (entry >> 1) * TILE + (u % C::SUB) * C::BM;
            const uint8_t *stg = sST + s * C::STAGE_STRIDE;
            const float *slse = reinterpret_cast<const float *>(stg + C::ST_LSE);
            const float *sd = reinterpret_cast<const float *>(stg + C::ST_D);
            if (!warp_wait(&s_full[wg], lu & 1, tmo, abort)) break;
            tc_fence_after();
            const uint32_t t_s = lane_base + C::TM_W0 + wg * C::TM_SDP, t_dp = t_s + C::BM;
#pragma unroll
            for (int c = 0; c < C::BM / 64; ++c) {
                float pr[64];
                tmem_ld64f(t_s + c * 64, pr);
                // This thread's key column: masked query rows of the sub-tile as bits.
                const uint32_t mw0 = need_mask ? column_row_bits(q0 + c * 64, gkey, cv, p.causal) : 0u;
                const uint32_t mw1 =
                    need_mask ? column_row_bits(q0 + c * 64 + 32, gkey, cv, p.causal) : 0u;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const int qi = c * 64 + i;
                    float v = ex2(fmaf(pr[i], sl2, -slse[qi]));
                    if ((((i < 32) ? mw0 : mw1) >> (i & 31)) & 1u) v = 0.f;
                    pr[i] = v;
                }
                if constexpr (C::DO_DV) {
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = pack_fp16(pr[2 * i], pr[2 * i + 1]);
                    tmem_st32(t_s + c * 32, r);
                }
                if constexpr (C::DO_DK) {
                    float dp[64];
                    tmem_ld64f(t_dp + c * 64, dp);
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int qi = c * 64 + 2 * i;
                        r[i] = pack_bf16(pr[2 * i] * (dp[2 * i] - sd[qi]),
                                         pr[2 * i + 1] * (dp[2 * i + 1] - sd[qi + 1]));
                    }
                    tmem_st32(t_dp + c * 32, r);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            if constexpr (C::DO_DV) mbar_arrive(&p_full[wg]);
            mbar_arrive(&ds_full[wg]);
        }
        if (n > 0) warp_wait(done, 0, tmo, abort);
        tc_fence_after();
        const bool store = gkey < p.N;
        const size_t rowoff = (static_cast<size_t>(b) * p.N + gkey) * p.H + h;
        if constexpr (C::DO_DK) {
            constexpr int CPW = (C::D / 32) / C::NWG;
#pragma unroll 1
            for (int c = wg * CPW; c < (wg + 1) * CPW; ++c) {
                uint32_t r[32];
                tmem_ld32(lane_base + C::TM_DK + c * 32, r);
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = n > 0 ? __uint_as_float(r[i]) : 0.f;
                if (store) store_row_bf16(p.dk + rowoff * C::D + c * 32, v, p.scale);
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
                if (store) store_row_bf16(p.dv + rowoff * C::DV + c * 32, v, 1.0f);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

BwdParams make_params(const Geometry &g, const Workspace &ws, const BwdArgs &a, bool dq_side) {
    BwdParams p;
    p.vec = ws.vec;
    p.list = dq_side ? ws.fwd_list : ws.bwd_list;
    p.cnt = dq_side ? ws.fwd_cnt : ws.bwd_cnt;
    p.lse2 = ws.lse2;
    p.delta = ws.delta;
    p.dq = static_cast<__nv_bfloat16 *>(a.dq);
    p.dk = static_cast<__nv_bfloat16 *>(a.dk);
    p.dv = static_cast<__nv_bfloat16 *>(a.dv);
    p.N = g.N;
    p.H = g.H;
    p.Hm = g.Hm;
    p.T = g.T;
    p.Npad = g.Npad;
    p.causal = g.causal;
    p.sl2 = g.scale * 1.4426950408889634f;
    p.scale = g.scale;
    p.timeout_ns = g.timeout_ns;
    return p;
}

template <class C>
cudaError_t launch_dq(const Geometry &g, const Workspace &ws, const BwdArgs &a, cudaStream_t st) {
    if (a.dq_k_rows != C::BN) return cudaErrorInvalidValue;  // map boxes must match the tile
    auto kern = dq_kernel<C>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(g.T, g.H, g.B);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(*a.tm_q_dq, *a.tm_k_dq, *a.tm_v_dq,
                                                  *a.tm_do_dq, make_params(g, ws, a, true));
    return cudaGetLastError();
}

template <class C>
cudaError_t launch_dkdv(const Geometry &g, const Workspace &ws, const BwdArgs &a,
                        cudaStream_t st) {
    if (a.kv_q_rows != C::BM) return cudaErrorInvalidValue;  // map boxes must match the tile
    auto kern = dkdv_kernel<C>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    dim3 grid(g.T, g.H, g.B);
    kern<<<grid, C::THREADS, C::SMEM_BYTES, st>>>(*a.tm_q, *a.tm_k, *a.tm_v, *a.tm_do,
                                                  make_params(g, ws, a, false));
    return cudaGetLastError();
}

template <class KV, class DQ>
cudaError_t launch_pair(const Geometry &g, const Workspace &ws, const BwdArgs &a, cudaStream_t st,
                        Recorder &rec) {
    rec.before(st);
    cudaError_t e = launch_dkdv<KV>(g, ws, a, st);
    rec.after(st);
    if (e != cudaSuccess) return e;
    rec.before(st);
    e = launch_dq<DQ>(g, ws, a, st);
    rec.after(st);
    return e;
}

}  // namespace

// Every DqCfg below uses 64-key sub-tiles and every DkdvCfg 64-query sub-tiles.
int dq_key_rows(int, int) { return 64; }
int dkdv_query_rows(int, int) { return 64; }

cudaError_t launch_bwd(const Geometry &g, const Workspace &ws, const BwdArgs &a,
                       cudaStream_t st, Recorder &rec) {
    const int rows_total = g.B * g.H * g.Npad;
    rec.before(st);
    preprocess_kernel<<<(rows_total + 15) / 16, 256, 0, st>>>(
        g.N, g.H, g.dv, g.Npad, rows_total, static_cast<const __nv_bfloat16 *>(a.o),
        static_cast<const __nv_bfloat16 *>(a.dout), static_cast<const __nv_bfloat16 *>(a.v),
        a.lse, ws.lse2, ws.delta, static_cast<uint4 *>(ws.v16), static_cast<uint4 *>(ws.do16));
    rec.after(st);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // DkdvCfg<d, dv, query sub-tile, stages, dK, dV, groups>;
    // DqCfg<d, dv, key sub-tile, stages, groups, boundary stages>
    if (g.d == 64 && g.dv == 64)
        return launch_pair<DkdvCfg<64, 64, 64, 4, true, true, 2>, DqCfg<64, 64, 64, 4, 2, 4>>(
            g, ws, a, st, rec);
    if (g.d == 128 && g.dv == 128)
        return launch_pair<DkdvCfg<128, 128, 64, 4, true, true, 2>, DqCfg<128, 128, 64, 3, 2, 4>>(
            g, ws, a, st, rec);
    if (g.d == 192 && g.dv == 128)
        return launch_pair<DkdvCfg<192, 128, 64, 2, true, true, 1>, DqCfg<192, 128, 64, 2, 2, 4>>(
            g, ws, a, st, rec);
    if (g.d == 256 && g.dv == 256) {
        rec.before(st);
        e = launch_dkdv<DkdvCfg<256, 256, 64, 2, false, true, 2>>(g, ws, a, st);
        rec.after(st);
        if (e != cudaSuccess) return e;
        return launch_pair<DkdvCfg<256, 256, 64, 1, true, false, 1>, DqCfg<256, 256, 64, 1, 1, 2>>(
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
