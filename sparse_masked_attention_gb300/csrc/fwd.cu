// fwd.cu -- forward of FlashMask masked attention on tcgen05 tensor cores.
//
//   O = softmax(Q K^T * scale + M) V        (FlashMask README, "Formulation")
//
// Only the key tiles the tile map kept are walked ("skip unnecessary
// computation", FlashMask abstract).  Two kernels:
// - fwd_pair_kernel (d <= 128): one CTA per pair of 128-row query tiles of
//   one (batch, head); softmax group g owns query tile 2p + g, and both groups
//   walk the union of the two tiles' key-tile lists, so K / V are loaded once.
// - fwd_kernel (larger heads): one CTA per query tile; with two groups they
//   take alternate key tiles of that tile and merge their halves at the end.
// Roles, by warp:
//   warp 0      TMA producers: lane 0 Q (and, in the pair kernel, the first K
//               and V tiles) and the K ring, lane 1 the V ring
//   warp 1      allocates TMEM; lane 0 issues every tcgen05.mma
//   warps 2..   softmax warpgroups.  Thread t of a group owns query row t,
//               which is TMEM lane t.
// While one group runs its softmax, the tensor core works on the other's tiles.
//
// Per key tile, group g:
//   S_g  = Q K^T                  (SS MMA, fp32 in TMEM)
//   softmax thread: S -> registers; apply the mask elementwise on partial
//   tiles only; online max/sum in the log2 domain with exp2; P -> TMEM as
//   bf16, in place of S (softmax_tile)
//   O_g += P V                    (TS MMA: P read from TMEM, V from smem)
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "fm_device.cuh"
#include "fm_internal.h"

namespace fm {

static __device__ unsigned g_err_fwd;

namespace {

struct FwdParams {
    const int4 *vec;
    const int *list;  // per query tile, or per query-tile pair (pair kernel)
    const int *cnt;
    const int *order;  // pair kernel: pairs by decreasing key-tile count
    float *lse;
    const float *sink;  // [H] attention-sink logits, or nullptr
    int N, H, Hm, T, B, Npad, causal;
    float sl2;  // scale * log2(e)
    uint64_t timeout_ns;
    int drop_load;  // failure-detection test: k > 0 skips the k-th K load (pair kernel)
    int next_stride;  // pair kernel: the CTA this many blocks later gets its first tiles
                      // prefetched into L2 (0: off)
};

template <int D_, int DV_, int BN_, int NWG_, int NSB_, int KS_, int VS_>
struct FwdCfg {
    static constexpr int D = D_, DV = DV_, BN = BN_, NWG = NWG_, NSB = NSB_, KS = KS_, VS = VS_;
    static constexpr int BM = 128;
    static constexpr int SUB = TILE / BN;  // key sub-tiles per list entry
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int K_BYTES = BN * D * 2;
    static constexpr int V_BYTES = BN * DV * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + Q_BYTES;
    static constexpr int OFF_V = OFF_K + KS * K_BYTES;
    static constexpr int OFF_BAR = OFF_V + VS * V_BYTES;
    // q_full, k_full[KS], k_empty[KS], v_full[VS], v_empty[VS],
    // s_full[NWG*NSB], p_full[NWG*NSB], pv_done[NWG*2], mma_done
    static constexpr int NBAR = 1 + 2 * KS + 2 * VS + 2 * NWG * NSB + 2 * NWG + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int TM_O = 0;
    static constexpr int TM_S = NWG * DV;
    static constexpr int TM_COLS = 512;
    static constexpr int THREADS = 64 + NWG * 128;
    static_assert(TM_S + NWG * NSB * BN <= TM_COLS, "TMEM budget");
    static_assert(D % 64 == 0 && DV % 64 == 0 && (BN == 64 || BN == 128), "tile shape");
    static_assert(DV <= 256 && BN % 64 == 0, "MMA shape");
    static_assert(NWG * 128 * 2 * 4 <= K_BYTES, "merge statistics alias K stage 0");
    static_assert((KS - 1) * K_BYTES >= BM * DV * 2, "output tile staging aliases K stages 1..");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(KS % NWG == 0 && VS % NWG == 0, "per-group ring stages");
    // A V stage is freed only once the group has seen a later tile's S, so a
    // single stage would wait on itself.
    static_assert(VS >= 2, "ring depth");
};

// Row normalisation.  O_acc and the row sum l are relative to the row's
// reference max m (log2 units); O = O_acc * factor.  An attention-sink logit
// sink2 (log2 units, -inf for none) adds exp2(sink2 - m) to the denominator,
// a term with no value.  Returns the factor (0 when the row saw no key) and
// writes the row's LSE in log2 units (-inf when it saw neither a key nor a
// sink).
__device__ __forceinline__ float row_finish(float m, float l, float sink2, float &lse2) {
    if (!(l > 0.f)) {  // every key of the row masked
        lse2 = sink2;
        return 0.f;
    }
    if (sink2 == -INFINITY) {
        lse2 = m + lg2(l);
        return 1.0f / l;
    }
    if (sink2 <= m) {
        const float lt = l + ex2(sink2 - m);
        lse2 = m + lg2(lt);
        return 1.0f / lt;
    }
    const float r = ex2(m - sink2);  // the sink dominates: rescale to it
    const float lt = fmaf(l, r, 1.0f);
    lse2 = sink2 + lg2(lt);
    return r / lt;
}

// Warp-uniform bounded wait: every lane polls, the warp agrees on the result.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t tmo,
                                          volatile int *abort) {
    const bool ok = mbar_wait(bar, parity, tmo, abort, &g_err_fwd);
    return __all_sync(0xffffffffu, ok);
}

// Softmax of one S tile (C::BN columns of this thread's row, at TMEM address
// s_addr), in place: P = exp2(S * sl2 - m) as bf16 over S, with the running
// reference max m_ref and row sum l_sum of the row.  Partial tiles set the
// columns whose bit is set in mbits (per 64-column chunk, two 32-bit words) to
// -inf first.  One pass in 64-column chunks:
// - fast path: exponents against the current reference without a row max,
//   valid when every row of the warp has a reference and no row's chunk sum
//   exceeds 2^32 (then no P, row sum or product with V can overflow);
// - otherwise the chunk is reloaded from TMEM (P not stored yet) and takes the
//   reference path: its row max, and when the max grew by more than 2^8 a new
//   reference, with O (at o_addr; has_prev: earlier tiles accumulated into it),
//   the row sum and the P chunks of this tile already written rescaled.
//   wait_prev_pv() is called once before O is first touched; false = give up.
// Returns false when a wait gave up.
template <class C, class WaitPrev>
__device__ __forceinline__ bool softmax_tile(uint32_t s_addr, uint32_t o_addr, bool masked_tile,
                                             const uint32_t (&mbits)[C::BN / 64][2],
                                             bool has_prev, float sl2, float &m_ref,
                                             float &l_sum, WaitPrev wait_prev_pv) {
    const float NEG_INF = -INFINITY;
    bool o_synced = false;  // wait_prev_pv done
    const float2 sl2x2 = make_float2(sl2, sl2);
#pragma unroll
    for (int c = 0; c < C::BN / 64; ++c) {
        // Partial tiles: a chunk every column of which is masked for every row
        // of the warp has P = 0 (nothing to load, exponentiate or add); one in
        // which no row of the warp masks anything needs no masking.
        bool chunk_masked = masked_tile;
        if (masked_tile) {
            const uint32_t wa = mbits[c][0], wb = mbits[c][1];
            if (__all_sync(0xffffffffu, (wa & wb) == 0xffffffffu)) {
                uint32_t z[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) z[i] = 0u;
                tmem_st32(s_addr + c * 32, z);
                continue;
            }
            chunk_masked = __any_sync(0xffffffffu, (wa | wb) != 0u);
        }
        auto load_masked = [&](float (&x)[64]) {
            tmem_ld64f(s_addr + c * 64, x);
            if (chunk_masked) {
                const uint32_t wa = mbits[c][0], wb = mbits[c][1];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    if ((wa >> jj) & 1u) x[jj] = NEG_INF;
                    if ((wb >> jj) & 1u) x[32 + jj] = NEG_INF;
                }
            }
        };
        // P = exp2(x * sl2 - m) as bf16 pairs, and the row sum of P
        auto exp_pack = [&](const float (&x)[64], float m, uint32_t (&r)[32]) {
            const float2 negm = make_float2(-m, -m);
            float2 l4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) l4[i] = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float2 t = __ffma2_rn(make_float2(x[2 * i], x[2 * i + 1]), sl2x2, negm);
                const float2 pp = make_float2(ex2(t.x), ex2(t.y));
                l4[i & 3] = __fadd2_rn(l4[i & 3], pp);
                r[i] = pack_bf16(pp.x, pp.y);
            }
            const float2 la = __fadd2_rn(__fadd2_rn(l4[0], l4[1]), __fadd2_rn(l4[2], l4[3]));
            return la.x + la.y;
        };
        uint32_t r[32];
        float lc = 0.f;
        // A row with no reference yet takes the fast path too when every
        // column of this chunk is masked for it: its P is 0 whatever the
        // reference (as for the rows of a document that starts inside the
        // query tile, over the key tiles of the document before).
        const bool row_empty = masked_tile && (mbits[c][0] & mbits[c][1]) == 0xffffffffu;
        bool fast = __all_sync(0xffffffffu, m_ref != NEG_INF || row_empty);
        if (fast) {
            float x[64];
            load_masked(x);
            lc = exp_pack(x, m_ref == NEG_INF ? 0.0f : m_ref, r);
            fast = __all_sync(0xffffffffu, lc <= 4294967296.0f);  // false for NaN
        }
        if (!fast) {
            float x[64];
            load_masked(x);  // S is still in TMEM: P not stored yet
            // max(m, max(a, b)) steps: one three-input max instruction each
            float mx8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(x[i], x[8 + i]);
#pragma unroll
            for (int jj = 16; jj < 64; jj += 16)
#pragma unroll
                for (int i = 0; i < 8; ++i) mx8[i] = fmaxf(mx8[i], fmaxf(x[jj + i], x[jj + 8 + i]));
            const float mc = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                                   fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]))) *
                             sl2;  // log2 domain (sl2 > 0)
            const bool need = (m_ref == NEG_INF) ? (mc != NEG_INF) : (mc > m_ref + 8.0f);
            if (__any_sync(0xffffffffu, need)) {
                const float m_new = need ? mc : m_ref;
                // alpha = 0 when the row had no visible key yet (O, l, P all 0)
                const float alpha = need ? (m_ref == NEG_INF ? 0.f : ex2(m_ref - m_new)) : 1.0f;
                const bool fix = need && m_ref != NEG_INF;
                m_ref = m_new;
                l_sum *= alpha;
                if (__any_sync(0xffffffffu, fix)) {
                    if (has_prev) {
                        if (!o_synced) {
                            if (!wait_prev_pv()) return false;
                            o_synced = true;
                        }
#pragma unroll 1
                        for (int oc = 0; oc < C::DV / 32; ++oc) {
                            uint32_t ro[32];
                            tmem_ld32(o_addr + oc * 32, ro);
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                ro[i] = __float_as_uint(__uint_as_float(ro[i]) * alpha);
                            tmem_st32(o_addr + oc * 32, ro);
                        }
                    }
                    if (c > 0) tmem_st_wait();  // earlier chunks' P stores landed
#pragma unroll 1
                    for (int pc = 0; pc < c; ++pc) {  // this tile's P already written
                        uint32_t rp[32];
                        tmem_ld32(s_addr + pc * 32, rp);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            __nv_bfloat162 h2 = *reinterpret_cast<__nv_bfloat162 *>(&rp[i]);
                            const float2 f2 = __bfloat1622float2(h2);
                            rp[i] = pack_bf16(f2.x * alpha, f2.y * alpha);
                        }
                        tmem_st32(s_addr + pc * 32, rp);
                    }
                }
            }
            lc = exp_pack(x, (m_ref == NEG_INF) ? 0.0f : m_ref, r);
        }
        tmem_st32(s_addr + c * 32, r);
        l_sum += lc;
    }
    return true;
}

// Mask bits of this lane's row over a partial tile's key columns: lane l loads
// the boundaries of key columns l and l + 32 of each 64-column chunk, builds
// their row bits over this warp's 32 rows (first row R0), and a bit transpose
// hands every lane the column bits of its own row.
template <class C>
__device__ __forceinline__ void tile_mask_bits(const int4 *vec, int key0, int R0, int causal,
                                               int lane, uint32_t (&mbits)[C::BN / 64][2]) {
    int4 cv[C::BN / 64][2];
#pragma unroll
    for (int c = 0; c < C::BN / 64; ++c) {
        cv[c][0] = __ldg(vec + key0 + c * 64 + lane);
        cv[c][1] = __ldg(vec + key0 + c * 64 + 32 + lane);
    }
#pragma unroll
    for (int c = 0; c < C::BN / 64; ++c)
#pragma unroll
        for (int e = 0; e < 2; ++e)
            mbits[c][e] = column_row_bits(R0, key0 + c * 64 + e * 32 + lane, cv[c][e], causal);
#pragma unroll
    for (int c = 0; c < C::BN / 64; ++c)
#pragma unroll
        for (int e = 0; e < 2; ++e) mbits[c][e] = warp_transpose32(mbits[c][e], lane);
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
               const FwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    pdl_wait();  // tile lists of the kernel before
    pdl_trigger();
    if (smem_u32(smem) & 1023u) {  // swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(&g_err_fwd, ERR_SMEM_ALIGN);
        return;
    }
    uint8_t *sQ = smem + C::OFF_Q;
    uint8_t *sK = smem + C::OFF_K;
    uint8_t *sV = smem + C::OFF_V;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *q_full = bars;
    uint64_t *k_full = q_full + 1;
    uint64_t *k_empty = k_full + C::KS;
    uint64_t *v_full = k_empty + C::KS;
    uint64_t *v_empty = v_full + C::VS;
    uint64_t *s_full = v_empty + C::VS;
    uint64_t *p_full = s_full + C::NWG * C::NSB;
    uint64_t *pv_done = p_full + C::NWG * C::NSB;
    uint64_t *mma_done = pv_done + C::NWG * 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    int *issued = reinterpret_cast<int *>(smem + C::OFF_MISC + 8);  // loads per ring

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qt = p.T - 1 - static_cast<int>(blockIdx.x);  // heaviest query tiles first
    const int h = blockIdx.y, b = blockIdx.z;
    const int bm = b * p.Hm + (p.Hm == 1 ? 0 : h);
    const int n_entries = p.cnt[static_cast<size_t>(bm) * p.T + qt];
    const int *entries = p.list + (static_cast<size_t>(bm) * p.T + qt) * p.T;
    // key tiles of BN columns; none after a bounded wait gave up anywhere
    const int n = (*reinterpret_cast<volatile unsigned *>(&g_err_fwd) != 0) ? 0
                                                                            : n_entries * C::SUB;
    const uint64_t tmo = p.timeout_ns;
    auto n_of = [&](int w) { return n > w ? (n - w + C::NWG - 1) / C::NWG : 0; };

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int i = 0; i < C::KS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
        }
        for (int i = 0; i < C::VS; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
        for (int i = 0; i < C::NWG * C::NSB; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
        }
        for (int i = 0; i < C::NWG * 2; ++i) mbar_init(&pv_done[i], 1);
        mbar_init(mma_done, 1);
        *abort = 0;
        issued[0] = issued[1] = 0;
        fence_barrier_init();
        if (n > 0) {  // Q before the CTA-wide barrier: its latency overlaps the setup
            mbar_arrive_expect_tx(q_full, C::Q_BYTES);
#pragma unroll
            for (int c = 0; c < C::D / 64; ++c)
                tma_load_4d(sQ + c * C::BM * 128, &tm_q, q_full, c * 64, h, qt * TILE, b);
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
        // ------------------------------------------------------ TMA producers
        // Two lanes, two independent rings, each filled in the order its
        // consumer drains it: lane 0 Q and K, lane 1 V.
        if (lane == 0 && n > 0) {
            prefetch_tmap(&tm_k);
            int u = 0;
            for (; u < n; ++u) {
                const int s = u % C::KS;
                if (u >= C::KS &&
                    !mbar_wait(&k_empty[s], ((u / C::KS) - 1) & 1, tmo, abort, &g_err_fwd))
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
                const int s = u % C::VS;
                if (u >= C::VS &&
                    !mbar_wait(&v_empty[s], ((u / C::VS) - 1) & 1, tmo, abort, &g_err_fwd))
                    break;
                mbar_arrive_expect_tx(&v_full[s], C::V_BYTES);
                const int key0 = key0_of(u);
#pragma unroll
                for (int c = 0; c < C::DV / 64; ++c)
                    tma_load_4d(sV + s * C::V_BYTES + c * C::BN * 128, &tm_v, &v_full[s], c * 64,
                                h, key0, b);
            }
            issued[1] = u;
        }
    } else if (warp == 1) {
        // --------------------------------------------------- tcgen05 issuer
        if (lane == 0 && n > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(128, C::BN, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, C::DV, false, true);
            // Descriptors are built once; an MMA step only adds its byte offset
            // (in 16-byte units) to the start-address field.
            const uint64_t q_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t v_desc = sdesc_sw128(smem_u32(sV), C::BN * 128, 1024);
            // S = Q K^T of group w's tile ls (K stage landed, S buffer free)
            auto issue_s = [&](int w, int ls) {
                const int u = ls * C::NWG + w, s = u % C::KS;
                const uint32_t d_tmem = tmem + C::TM_S + (w * C::NSB + ls % C::NSB) * C::BN;
                const uint64_t ks = k_desc + static_cast<uint64_t>((s * C::K_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < C::D / 16; ++k) {
                    const uint64_t ad = q_desc + (((k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4);
                    const uint64_t bd = ks + (((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4);
                    mma_ss(d_tmem, ad, bd, IDESC_S, k > 0 ? 1u : 0u);
                }
            };
            // Each commit costs the issuing thread about as long as an MMA, time
            // in which the tensor pipe runs dry, so a step commits once: S done.
            // The softmax group frees the K stage when it sees S, and the V
            // stage of its tile lp - NSB, since the pipe ran that P V before S.
            auto commit_s = [&](int w, int ls) { mma_commit(&s_full[w * C::NSB + ls % C::NSB]); };
            auto k_ready = [&](int w, int ls) {
                const int u = ls * C::NWG + w;
                return mbar_test(&k_full[u % C::KS], (u / C::KS) & 1) != 0;
            };
            // O_w += P V of group w's tile lp (P written, V stage landed)
            auto issue_pv = [&](int w, int lp) {
                const int u = lp * C::NWG + w, vs = u % C::VS;
                const uint32_t o_tmem = tmem + C::TM_O + w * C::DV;
                const uint32_t p_tmem = tmem + C::TM_S + (w * C::NSB + lp % C::NSB) * C::BN;
                const uint64_t vsd = v_desc + static_cast<uint64_t>((vs * C::V_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < C::BN / 16; ++k)
                    mma_ts(o_tmem, p_tmem + k * 8, vsd + ((k * 2048) >> 4), IDESC_PV,
                           (lp > 0 || k > 0) ? 1u : 0u);
            };
            // With one S buffer per group the group's next S implies its P V is
            // done; with two, the rescale of O waits for this commit.
            auto commit_pv = [&](int w, int lp) {
                if constexpr (C::NSB > 1) mma_commit(&pv_done[w * 2 + (lp & 1)]);
            };
            auto pv_ready = [&](int w, int lp) {
                const int u = lp * C::NWG + w;
                return mbar_test(&p_full[w * C::NSB + lp % C::NSB], (lp / C::NSB) & 1) &&
                       mbar_test(&v_full[u % C::VS], (u / C::VS) & 1);
            };
            bool ok = mbar_wait(q_full, 0, tmo, abort, &g_err_fwd);
            // Prologue: S of every group's first NSB tiles, in tile order.
            for (int ls = 0; ok && ls < C::NSB; ++ls)
                for (int w = 0; ok && w < C::NWG; ++w) {
                    if (ls >= n_of(w)) continue;
                    const int u = ls * C::NWG + w;
                    ok = mbar_wait(&k_full[u % C::KS], (u / C::KS) & 1, tmo, abort, &g_err_fwd);
                    if (!ok) break;
                    tc_fence_after();
                    issue_s(w, ls);
                    commit_s(w, ls);
                }
            // Steady state: a step of group w is its P V for tile lp and the S of
            // tile lp + NSB (the buffer P V frees; the tensor pipe runs them in
            // order), issued as one run once P, V and K are all ready, with the
            // commits after the run.  The thread serves the groups in turn and
            // reads the clock only while idle, so consecutive runs follow each
            // other without a gap that would drain the MMA queue.  Both rings
            // hold a multiple of NWG stages: a group waits only on its own
            // older tiles.
            int pv_cnt[C::NWG];
            int remaining = 0;
#pragma unroll
            for (int w = 0; w < C::NWG; ++w) {
                pv_cnt[w] = 0;
                remaining += n_of(w) > 0;
            }
            int w = 0;
            bool idle = false;
            uint64_t idle_t0 = 0;
            while (ok && remaining > 0) {
                bool prog = false;
#pragma unroll
                for (int i = 0; i < C::NWG; ++i) {
                    const int nm = n_of(w), lp = pv_cnt[w];
                    const int ls = lp + C::NSB;
                    if (lp < nm && pv_ready(w, lp) && (ls >= nm || k_ready(w, ls))) {
                        tc_fence_after();
                        issue_pv(w, lp);
                        if (ls < nm) issue_s(w, ls);
                        commit_pv(w, lp);
                        if (ls < nm) commit_s(w, ls);
                        pv_cnt[w] = lp + 1;
                        if (lp + 1 >= nm) --remaining;
                        prog = true;
                    }
                    w = (w + 1 == C::NWG) ? 0 : w + 1;
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
                        atomicExch(&g_err_fwd, ERR_TIMEOUT);
                        ok = false;
                    }
                }
            }
            mma_commit(mma_done);  // every MMA of the CTA has completed
        }
    } else {
        // ------------------------------------------------ softmax warpgroups
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int grow = qt * TILE + row;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const int n_my = n > wg ? (n - wg + C::NWG - 1) / C::NWG : 0;
        const float NEG_INF = -INFINITY;
        const float sl2 = p.sl2;
        const int4 *vec = p.vec + static_cast<size_t>(bm) * p.Npad;
        float m_ref = NEG_INF, l_sum = 0.f;
        // The list entry of the group's next tile is read one tile ahead.
        int entry_next = n_my > 0 ? entries[wg / C::SUB] : 0;

        for (int lu = 0; lu < n_my; ++lu) {
            const int u = lu * C::NWG + wg;
            const int sb = wg * C::NSB + lu % C::NSB;
            const int entry = entry_next;
            if (u + C::NWG < n) entry_next = entries[(u + C::NWG) / C::SUB];
            const bool masked_tile = entry & 1;
            const int key0 = (entry >> 1) * TILE + (u % C::SUB) * C::BN;

            // Partial tiles: the mask bits of this lane's row over the tile's key
            // columns, built before the wait for S (they do not depend on S), so
            // that the wait hides the boundary loads and the bit transposes.
            // Lane l loads the boundaries of key columns l and l + 32 of each
            // 64-column chunk and builds their row bits over this warp's 32
            // rows; a bit transpose hands every lane the column bits of its row.
            uint32_t mbits[C::BN / 64][2];
            if (masked_tile) {
                tile_mask_bits<C>(vec, key0, grow - lane, p.causal, lane, mbits);
                // Keep the bits ahead of the wait: left to itself the compiler
                // sinks this work past the wait, to its first use.
#pragma unroll
                for (int c = 0; c < C::BN / 64; ++c)
                    asm volatile("" ::"r"(mbits[c][0]), "r"(mbits[c][1]));
            }
            if (!warp_wait(&s_full[sb], (lu / C::NSB) & 1, tmo, abort)) break;
            tc_fence_after();
            if (((warp - 2) & 3) == 0 && lane == 0) {
                // S of this tile is done, and so is the group's P V of tile
                // lu - NSB (issued before it): their K and V stages are free.
                mbar_arrive(&k_empty[u % C::KS]);
                if (lu >= C::NSB) mbar_arrive(&v_empty[((lu - C::NSB) * C::NWG + wg) % C::VS]);
            }
            const uint32_t s_addr = lane_base + C::TM_S + sb * C::BN;

            bool failed = !softmax_tile<C>(s_addr, lane_base + C::TM_O + wg * C::DV, masked_tile,
                                           mbits, lu > 0, sl2, m_ref, l_sum, [&]() {
                                               if constexpr (C::NSB > 1) {
                                                   const int pl = lu - 1;
                                                   if (!warp_wait(&pv_done[wg * 2 + (pl & 1)],
                                                                  (pl >> 1) & 1, tmo, abort))
                                                       return false;
                                                   tc_fence_after();
                                               }
                                               return true;
                                           });
            if (failed) break;
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&p_full[sb]);
        }

        // ------------------------------------------------------- epilogue
        // Wait until every MMA of the CTA has completed: O is then final and
        // the K ring is free for the merge statistics.  A group with no tiles
        // waits too.
        if (n > 0) warp_wait(mma_done, 0, tmo, abort);
        tc_fence_after();
        const bool store = grow < p.N;
        float m_all = m_ref, l_all = l_sum, a0 = 1.f, a1 = 0.f;
        float l0 = l_sum, l1 = 0.f;
        int c_begin = 0, c_end = C::DV / 32;
        if constexpr (C::NWG == 2) {
            float *stats = reinterpret_cast<float *>(sK);  // K stage 0 is idle by now
            stats[(wg * 128 + row) * 2 + 0] = m_ref;
            stats[(wg * 128 + row) * 2 + 1] = l_sum;
            tc_fence_before();
            named_bar_sync(1, 256);
            tc_fence_after();
            const float mA = stats[row * 2 + 0], lA = stats[row * 2 + 1];
            const float mB = stats[(128 + row) * 2 + 0], lB = stats[(128 + row) * 2 + 1];
            m_all = fmaxf(mA, mB);
            a0 = lA > 0.f ? ex2(mA - m_all) : 0.f;
            a1 = lB > 0.f ? ex2(mB - m_all) : 0.f;
            l0 = lA;
            l1 = lB;
            l_all = a0 * lA + a1 * lB;
            c_begin = wg * (C::DV / 64);
            c_end = c_begin + C::DV / 64;
        }
        float lse2_row;
        const float sink2 = p.sink ? p.sink[h] * 1.4426950408889634f : NEG_INF;
        const float inv = row_finish(m_all, l_all, sink2, lse2_row);
        // The normalised bf16 row goes to shared memory in the 128B-swizzled
        // layout of the output tensor map (64-column boxes of 128 rows; K
        // stages 1.. are idle by now); TMA then stores whole boxes, clipping
        // rows past N.
        uint8_t *stage = sK + C::K_BYTES;
        for (int c = c_begin; c < c_end; ++c) {
            uint32_t r0[32];
            tmem_ld32(lane_base + C::TM_O + c * 32, r0);
            float o[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = l0 > 0.f ? a0 * __uint_as_float(r0[i]) : 0.f;
            if constexpr (C::NWG == 2) {
                uint32_t r1[32];
                tmem_ld32(lane_base + C::TM_O + C::DV + c * 32, r1);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    o[i] += l1 > 0.f ? a1 * __uint_as_float(r1[i]) : 0.f;
            }
            uint8_t *box_row = stage + (c / 2) * (C::BM * 128) + row * 128;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                uint4 w;
                w.x = pack_bf16(o[v * 8 + 0] * inv, o[v * 8 + 1] * inv);
                w.y = pack_bf16(o[v * 8 + 2] * inv, o[v * 8 + 3] * inv);
                w.z = pack_bf16(o[v * 8 + 4] * inv, o[v * 8 + 5] * inv);
                w.w = pack_bf16(o[v * 8 + 6] * inv, o[v * 8 + 7] * inv);
                const int unit = (c % 2) * 4 + v;  // 16-byte unit of the 128-byte row
                *reinterpret_cast<uint4 *>(box_row + ((unit ^ (row & 7)) * 16)) = w;
            }
        }
        fence_proxy_async_smem();              // generic stores -> visible to TMA
        named_bar_sync(2, C::NWG * 128);       // every row of every box is staged
        if (threadIdx.x == 64) {
            for (int box = 0; box < C::DV / 64; ++box)
                tma_store_4d(&tm_o, stage + box * (C::BM * 128), box * 64, h, qt * TILE, b);
            bulk_commit_wait_read();           // shared memory read before the CTA exits
        }
        if (wg == 0 && store) {
            const float ln2 = 0.69314718055994530942f;
            p.lse[(static_cast<size_t>(b) * p.H + h) * p.N + grow] = lse2_row * ln2;
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
            drain_ring(k_full, C::KS, issued[0], -1, tmo, &g_err_fwd);
            drain_ring(v_full, C::VS, issued[1], -1, tmo, &g_err_fwd);
            mbar_wait_drain(q_full, 0, tmo, &g_err_fwd);
            mbar_wait_drain(mma_done, 0, tmo, &g_err_fwd);
        }
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

template <class C>
cudaError_t launch_cfg(const Geometry &g, const Workspace &ws, const FwdArgs &a,
                       cudaStream_t st) {
    FwdParams p;
    p.vec = ws.vec;
    p.list = ws.fwd_list;
    p.cnt = ws.fwd_cnt;
    p.order = nullptr;
    p.sink = g.sink;
    p.B = g.B;
    p.lse = a.lse;
    p.N = g.N;
    p.H = g.H;
    p.Hm = g.Hm;
    p.T = g.T;
    p.Npad = g.Npad;
    p.causal = g.causal;
    p.sl2 = g.scale * 1.4426950408889634f;
    p.timeout_ns = g.timeout_ns;
    p.drop_load = g.drop_load;
    p.next_stride = 0;
    if (a.k_rows != C::BN) return cudaErrorInvalidValue;  // map boxes must match the tile
    auto kern = fwd_kernel<C>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(g.T, g.H, g.B), dim3(C::THREADS), C::SMEM_BYTES, st, *a.tm_q,
                      *a.tm_k, *a.tm_v, *a.tm_o, p);
}


// ------------------------------------------------------------- pair kernel
// One CTA per pair of 128-row query tiles (2p, 2p+1) of one (batch, head):
// softmax group g owns query tile 2p + g (its Q, its O accumulator, its row
// statistics), and both groups walk the union of the two tiles' key-tile lists,
// so each K / V tile is loaded once for both.  A key tile that one query tile
// skips is processed as a partial tile for it (all its columns masked).
// Per key tile j, group g: S_g = Q_g K_j^T; softmax; O_g += P_g V_j.  The MMA
// steps alternate the groups as in fwd_kernel; each K / V stage is freed by
// both groups (arrival count 2).  Each group finishes on its own: it
// normalises its O, stages it in its Q buffer (idle once its last S ran) and
// stores it with TMA; no statistics cross groups.
template <int D_, int DV_, int KS_, int VS_>
struct PairCfg {
    static constexpr int D = D_, DV = DV_, KS = KS_, VS = VS_;
    static constexpr int BM = 128, BN = 128;
    static constexpr int Q_BYTES = BM * D * 2;  // one per group
    static constexpr int K_BYTES = BN * D * 2;
    static constexpr int V_BYTES = BN * DV * 2;
    static constexpr int OFF_Q = 0;
    static constexpr int OFF_K = OFF_Q + 2 * Q_BYTES;
    static constexpr int OFF_V = OFF_K + KS * K_BYTES;
    static constexpr int OFF_BAR = OFF_V + VS * V_BYTES;
    // q_full[2], k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], s_full[2],
    // p_full[2], o_done[2], mma_idle
    static constexpr int NBAR = 2 + 2 * KS + 2 * VS + 7;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16;
    static constexpr int TM_O = 0;
    static constexpr int TM_S = 2 * DV;
    static constexpr int TM_COLS = 512;
    static constexpr int THREADS = 64 + 2 * 128;
    static_assert(TM_S + 2 * BN <= TM_COLS, "TMEM budget");
    static_assert(D % 64 == 0 && DV % 64 == 0 && DV <= 256, "tile shape");
    static_assert(Q_BYTES >= BM * DV * 2, "output staging aliases the group's Q buffer");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(KS >= 2 && VS >= 2, "ring depth");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    pdl_wait();  // tile lists of the kernel before
    pdl_trigger();
    if (smem_u32(smem) & 1023u) {  // swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(&g_err_fwd, ERR_SMEM_ALIGN);
        return;
    }
    uint8_t *sQ = smem + C::OFF_Q;
    uint8_t *sK = smem + C::OFF_K;
    uint8_t *sV = smem + C::OFF_V;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *q_full = bars;  // per group
    uint64_t *k_full = q_full + 2;
    uint64_t *k_empty = k_full + C::KS;
    uint64_t *v_full = k_empty + C::KS;
    uint64_t *v_empty = v_full + C::VS;
    uint64_t *s_full = v_empty + C::VS;
    uint64_t *p_full = s_full + 2;
    uint64_t *o_done = p_full + 2;
    uint64_t *mma_idle = o_done + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
    int *issued = reinterpret_cast<int *>(smem + C::OFF_MISC + 8);  // loads per ring

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int TP = (p.T + 1) / 2;
    // CTA c takes the pair of rank c / (H B) (heaviest first) of head-batch
    // c % (H B): every head's heaviest pairs start in the first waves.
    const int hb = static_cast<int>(blockIdx.x) % (p.H * p.B);
    const int h = hb % p.H, b = hb / p.H;
    const int bm = b * p.Hm + (p.Hm == 1 ? 0 : h);
    const int pp = p.order[static_cast<size_t>(bm) * TP + static_cast<int>(blockIdx.x) / (p.H * p.B)];
    const int *entries = p.list + (static_cast<size_t>(bm) * TP + pp) * p.T;
    // The pair's key-tile count and first entry are read together, both right
    // after its index (the row holds T entries, so entry 0 is in bounds even
    // for an empty list).
    const int cnt = p.cnt[static_cast<size_t>(bm) * TP + pp];
    const int entry0 = entries[0];
    // key tiles; none after a bounded wait gave up anywhere
    const int n = (*reinterpret_cast<volatile unsigned *>(&g_err_fwd) != 0) ? 0 : cnt;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        mbar_init(&q_full[0], 1);
        mbar_init(&q_full[1], 1);
        for (int i = 0; i < C::KS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 2);
        }
        for (int i = 0; i < C::VS; ++i) {
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 2);
        }
        for (int g = 0; g < 2; ++g) {
            mbar_init(&s_full[g], 1);
            mbar_init(&p_full[g], 4);  // one arrival per softmax warp
            mbar_init(&o_done[g], 1);
        }
        mbar_init(mma_idle, 1);
        *abort = 0;
        issued[0] = issued[1] = 0;
        fence_barrier_init();
        if (n > 0) {  // both Q tiles before the CTA-wide barrier: latency overlaps the setup
            // a barrier per group: group 0's first S need not wait for Q_1;
            // issued Q_0, K_0, Q_1, V_0, in the order the first MMAs need them
            const int key0 = (entry0 >> 2) * TILE;
#pragma unroll
            for (int g = 0; g < 2; ++g) {
                mbar_arrive_expect_tx(&q_full[g], C::Q_BYTES);
#pragma unroll
                for (int c = 0; c < C::D / 64; ++c)
                    tma_load_4d(sQ + g * C::Q_BYTES + c * C::BM * 128, &tm_q, &q_full[g], c * 64,
                                h, (2 * pp + g) * TILE, b);
                // the first K tile (unless the test drops that load)
                if (g == 0 && p.drop_load != 1) {
                    mbar_arrive_expect_tx(&k_full[0], C::K_BYTES);
#pragma unroll
                    for (int c = 0; c < C::D / 64; ++c)
                        tma_load_4d(sK + c * C::BN * 128, &tm_k, &k_full[0], c * 64, h, key0, b);
                }
            }
            mbar_arrive_expect_tx(&v_full[0], C::V_BYTES);
#pragma unroll
            for (int c = 0; c < C::DV / 64; ++c)
                tma_load_4d(sV + c * C::BN * 128, &tm_v, &v_full[0], c * 64, h, key0, b);
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

    if (warp == 0) {
        // ------------------------------------------------------ TMA producers
        // lane 0 the K ring, lane 1 the V ring, both in tile order
        if (lane < 2 && n > 0) {
            const bool is_k = lane == 0;
            const int S = is_k ? C::KS : C::VS;
            // failure-detection test only: this K load is never issued
            const int skip = is_k ? p.drop_load - 1 : -1;
            if (is_k) prefetch_tmap(&tm_k); else prefetch_tmap(&tm_v);
            int j = 1;  // tile 0 was loaded before the CTA-wide barrier
            for (; j < n; ++j) {
                const int s = j % S;
                uint64_t *full = is_k ? &k_full[s] : &v_full[s];
                uint64_t *empty = is_k ? &k_empty[s] : &v_empty[s];
                if (j >= S && !mbar_wait(empty, ((j / S) - 1) & 1, tmo, abort, &g_err_fwd)) break;
                if (j == skip) continue;
                const int key0 = (entries[j] >> 2) * TILE;
                if (is_k) {
                    mbar_arrive_expect_tx(full, C::K_BYTES);
#pragma unroll
                    for (int c = 0; c < C::D / 64; ++c)
                        tma_load_4d(sK + s * C::K_BYTES + c * C::BN * 128, &tm_k, full, c * 64, h,
                                    key0, b);
                } else {
                    mbar_arrive_expect_tx(full, C::V_BYTES);
#pragma unroll
                    for (int c = 0; c < C::DV / 64; ++c)
                        tma_load_4d(sV + s * C::V_BYTES + c * C::BN * 128, &tm_v, full, c * 64, h,
                                    key0, b);
                }
            }
            issued[is_k ? 0 : 1] = j;
            // Its last K load issued, this CTA has a few key tiles left: the
            // CTA about one wave later (about when this one ends) gets its two
            // Q tiles and its first K and V tiles prefetched into L2, so that
            // it starts on L2 latency (8K causal-document forward 0.8 % faster,
            // 32K block-sparse 0.5 % slower).
            const int nx = static_cast<int>(blockIdx.x) + p.next_stride;
            if (is_k && p.next_stride > 0 && nx < static_cast<int>(gridDim.x)) {
                const int hb2 = nx % (p.H * p.B);
                const int h2 = hb2 % p.H, b2 = hb2 / p.H;
                const int bm2 = b2 * p.Hm + (p.Hm == 1 ? 0 : h2);
                const int pp2 = p.order[static_cast<size_t>(bm2) * TP + nx / (p.H * p.B)];
#pragma unroll
                for (int g = 0; g < 2; ++g)
                    if (2 * pp2 + g < p.T)
#pragma unroll
                        for (int c = 0; c < C::D / 64; ++c)
                            tma_prefetch_l2_4d(&tm_q, c * 64, h2, (2 * pp2 + g) * TILE, b2);
                const size_t r2 = static_cast<size_t>(bm2) * TP + pp2;
                if (p.cnt[r2] > 0) {
                    const int k2 = (p.list[r2 * p.T] >> 2) * TILE;
#pragma unroll
                    for (int c = 0; c < C::D / 64; ++c) tma_prefetch_l2_4d(&tm_k, c * 64, h2, k2, b2);
#pragma unroll
                    for (int c = 0; c < C::DV / 64; ++c) tma_prefetch_l2_4d(&tm_v, c * 64, h2, k2, b2);
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------- tcgen05 issuer
        if (lane == 0 && n > 0) {
            constexpr uint32_t IDESC_S = idesc_bf16(128, C::BN, false, false);
            constexpr uint32_t IDESC_PV = idesc_bf16(128, C::DV, false, true);
            const uint64_t q_desc = sdesc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t k_desc = sdesc_sw128(smem_u32(sK), 16, 1024);
            const uint64_t v_desc = sdesc_sw128(smem_u32(sV), C::BN * 128, 1024);
            // S_g = Q_g K_j^T into group g's S buffer
            auto issue_s = [&](int g, int j) {
                const uint32_t d_tmem = tmem + C::TM_S + g * C::BN;
                const uint64_t qs = q_desc + static_cast<uint64_t>((g * C::Q_BYTES) >> 4);
                const uint64_t ks = k_desc + static_cast<uint64_t>(((j % C::KS) * C::K_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < C::D / 16; ++k) {
                    const uint64_t ad = qs + (((k / 4) * (C::BM * 128) + (k % 4) * 32) >> 4);
                    const uint64_t bd = ks + (((k / 4) * (C::BN * 128) + (k % 4) * 32) >> 4);
                    mma_ss(d_tmem, ad, bd, IDESC_S, k > 0 ? 1u : 0u);
                }
            };
            // O_g += P_g V_j (P from the group's S buffer)
            auto issue_pv = [&](int g, int j) {
                const uint32_t o_tmem = tmem + C::TM_O + g * C::DV;
                const uint32_t p_tmem = tmem + C::TM_S + g * C::BN;
                const uint64_t vsd =
                    v_desc + static_cast<uint64_t>(((j % C::VS) * C::V_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < C::BN / 16; ++k)
                    mma_ts(o_tmem, p_tmem + k * 8, vsd + ((k * 2048) >> 4), IDESC_PV,
                           (j > 0 || k > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(&k_full[0], 0, tmo, abort, &g_err_fwd);
            for (int g = 0; g < 2 && ok; ++g) {
                ok = mbar_wait(&q_full[g], 0, tmo, abort, &g_err_fwd);
                if (ok) {
                    tc_fence_after();
                    issue_s(g, 0);
                    mma_commit(&s_full[g]);
                }
            }
            // A step of group g: its P V for tile j and its S of tile j + 1 (the
            // buffer P V frees), one run with one commit.  The softmax group that
            // sees S of tile j + 1 frees (with the other group) the K stage of
            // j + 1 and the V stage of j.
            int pv_cnt[2] = {0, 0};
            int remaining = 2;
            int g = 0;
            bool idle = false;
            uint64_t idle_t0 = 0;
            while (ok && remaining > 0) {
                bool prog = false;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int j = pv_cnt[g];
                    if (j < n && mbar_test(&p_full[g], j & 1) &&
                        mbar_test(&v_full[j % C::VS], (j / C::VS) & 1) &&
                        (j + 1 >= n || mbar_test(&k_full[(j + 1) % C::KS], ((j + 1) / C::KS) & 1))) {
                        tc_fence_after();
                        issue_pv(g, j);
                        if (j + 1 < n) {
                            issue_s(g, j + 1);
                            mma_commit(&s_full[g]);
                        } else {
                            mma_commit(&o_done[g]);  // the group's O is final
                            --remaining;
                        }
                        pv_cnt[g] = j + 1;
                        prog = true;
                    }
                    g ^= 1;
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
                        atomicExch(&g_err_fwd, ERR_TIMEOUT);
                        ok = false;
                    }
                }
            }
            mma_commit(mma_idle);  // waited for only after a wait gave up
        }
    } else {
        // ------------------------------------------------ softmax warpgroups
        const int wg = (warp - 2) >> 2;
        const int quad = warp & 3;
        const int row = quad * 32 + lane;
        const int qt = 2 * pp + wg;
        const int grow = qt * TILE + row;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quad * 32) << 16);
        const uint32_t s_addr = lane_base + C::TM_S + wg * C::BN;
        const float NEG_INF = -INFINITY;
        const float sl2 = p.sl2;
        const int4 *vec = p.vec + static_cast<size_t>(bm) * p.Npad;
        const bool leader = ((warp - 2) & 3) == 0 && lane == 0;
        float m_ref = NEG_INF, l_sum = 0.f;
        bool failed = false;
        // The list entry of the next tile is read one tile ahead.
        int entry_next = entry0;
        for (int j = 0; j < n; ++j) {
            const int entry = entry_next;
            if (j + 1 < n) entry_next = entries[j + 1];
            const bool masked_tile = (entry >> (1 - wg)) & 1;
            const int key0 = (entry >> 2) * TILE;
            uint32_t mbits[C::BN / 64][2];
            if (masked_tile) {
                tile_mask_bits<C>(vec, key0, grow - lane, p.causal, lane, mbits);
                // Keep the bits ahead of the wait: left to itself the compiler
                // sinks this work past the wait, to its first use.
#pragma unroll
                for (int c = 0; c < C::BN / 64; ++c)
                    asm volatile("" ::"r"(mbits[c][0]), "r"(mbits[c][1]));
            }
            if (!warp_wait(&s_full[wg], j & 1, tmo, abort)) {
                failed = true;
                break;
            }
            tc_fence_after();
            if (leader) {
                // S of tile j is done, and so is this group's P V of tile j - 1
                // (issued before it): this group's part of their stages is free.
                mbar_arrive(&k_empty[j % C::KS]);
                if (j > 0) mbar_arrive(&v_empty[(j - 1) % C::VS]);
            }
            if (!softmax_tile<C>(s_addr, lane_base + C::TM_O + wg * C::DV, masked_tile, mbits,
                                 j > 0, sl2, m_ref, l_sum, []() { return true; })) {
                failed = true;
                break;
            }
            // Every lane's P stores have landed (wait::st) and are fenced; one
            // lane per warp arrives for the warp, after the warp converges.
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full[wg]);
        }

        // ------------------------------------------------------- epilogue
        // O_g final once the group's last P V completed; the group's Q buffer
        // (its last S has run) stages the normalised bf16 rows for TMA.
        if (n > 0 && !failed) failed = !warp_wait(&o_done[wg], 0, tmo, abort);
        tc_fence_after();
        float lse2_row;
        const float sink2 = p.sink ? p.sink[h] * 1.4426950408889634f : NEG_INF;
        const float inv = row_finish(m_ref, l_sum, sink2, lse2_row);
        uint8_t *stage = sQ + wg * C::Q_BYTES;
        for (int c = 0; c < C::DV / 32; ++c) {
            float o[32];
            if (n > 0 && !failed) {
                uint32_t r0[32];
                tmem_ld32(lane_base + C::TM_O + wg * C::DV + c * 32, r0);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = l_sum > 0.f ? __uint_as_float(r0[i]) : 0.f;
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = 0.f;
            }
            uint8_t *box_row = stage + (c / 2) * (C::BM * 128) + row * 128;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                uint4 w;
                w.x = pack_bf16(o[v * 8 + 0] * inv, o[v * 8 + 1] * inv);
                w.y = pack_bf16(o[v * 8 + 2] * inv, o[v * 8 + 3] * inv);
                w.z = pack_bf16(o[v * 8 + 4] * inv, o[v * 8 + 5] * inv);
                w.w = pack_bf16(o[v * 8 + 6] * inv, o[v * 8 + 7] * inv);
                const int unit = (c % 2) * 4 + v;  // 16-byte unit of the 128-byte row
                *reinterpret_cast<uint4 *>(box_row + ((unit ^ (row & 7)) * 16)) = w;
            }
        }
        fence_proxy_async_smem();        // generic stores -> visible to TMA
        named_bar_sync(1 + wg, 128);     // the group's rows are all staged
        if (leader) {
            if (!failed && qt < p.T)
                for (int box = 0; box < C::DV / 64; ++box)
                    tma_store_4d(&tm_o, stage + box * (C::BM * 128), box * 64, h, qt * TILE, b);
            bulk_commit_wait_read();     // shared memory read before the CTA exits
        }
        if (grow < p.N && !failed) {
            const float ln2 = 0.69314718055994530942f;
            p.lse[(static_cast<size_t>(b) * p.H + h) * p.N + grow] = lse2_row * ln2;
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
            drain_ring(k_full, C::KS, issued[0], p.drop_load - 1, tmo, &g_err_fwd);
            drain_ring(v_full, C::VS, issued[1], -1, tmo, &g_err_fwd);
            mbar_wait_drain(&q_full[0], 0, tmo, &g_err_fwd);
            mbar_wait_drain(&q_full[1], 0, tmo, &g_err_fwd);
            mbar_wait_drain(mma_idle, 0, tmo, &g_err_fwd);
        }
        __syncthreads();
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::TM_COLS);
    }
}

template <class C>
cudaError_t launch_pair(const Geometry &g, const Workspace &ws, const FwdArgs &a,
                        cudaStream_t st) {
    FwdParams p;
    p.vec = ws.vec;
    p.list = ws.pair_list;
    p.cnt = ws.pair_cnt;
    p.order = ws.pair_order;
    p.sink = g.sink;
    p.B = g.B;
    p.lse = a.lse;
    p.N = g.N;
    p.H = g.H;
    p.Hm = g.Hm;
    p.T = g.T;
    p.Npad = g.Npad;
    p.causal = g.causal;
    p.sl2 = g.scale * 1.4426950408889634f;
    p.timeout_ns = g.timeout_ns;
    p.drop_load = g.drop_load;
    p.next_stride = current_sm_count();
    if (a.k_rows != C::BN) return cudaErrorInvalidValue;  // map boxes must match the tile
    auto kern = fwd_pair_kernel<C>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const long long ctas = static_cast<long long>((g.T + 1) / 2) * g.H * g.B;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3(static_cast<unsigned>(ctas)), dim3(C::THREADS), C::SMEM_BYTES,
                      st, *a.tm_q, *a.tm_k, *a.tm_v, *a.tm_o, p);
}

}  // namespace

int fwd_key_rows(int d, int dv) { return (d == 256 && dv == 256) ? 64 : 128; }

cudaError_t launch_fwd(const Geometry &g, const Workspace &ws, const FwdArgs &a,
                       cudaStream_t st) {
    // <d, dv, key tile, softmax groups, S buffers per group, K / V ring stages>
    // d <= 128: a pair of query tiles per CTA, <d, dv, K / V ring stages>
    if (g.d == 64 && g.dv == 64) return launch_pair<PairCfg<64, 64, 2, 2>>(g, ws, a, st);
    if (g.d == 128 && g.dv == 128) return launch_pair<PairCfg<128, 128, 2, 2>>(g, ws, a, st);
    if (g.d == 192 && g.dv == 128)
        return launch_cfg<FwdCfg<192, 128, 128, 2, 1, 2, 2>>(g, ws, a, st);
    if (g.d == 256 && g.dv == 256)
        return launch_cfg<FwdCfg<256, 256, 64, 1, 2, 3, 2>>(g, ws, a, st);
    return cudaErrorInvalidValue;
}

unsigned read_clear_error_fwd() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_fwd, sizeof(v)) != cudaSuccess) return 0;
    if (v) cudaMemcpyToSymbol(g_err_fwd, &zero, sizeof(zero));
    return v;
}

}  // namespace fm
